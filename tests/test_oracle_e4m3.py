"""Pins for the oracle's E4M3 table, encoder, store and gather-cast.

The oracle is checked against things other than itself: the format
definition's landmark values (tests/golden), PyTorch's float8_e4m3fn and
bfloat16 conversions (library routines), and an exact brute-force nearest
search written here in numpy.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def _torch_e4m3_to_f32(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.float().numpy()


def test_table_landmarks():
    tab = oracle.e4m3_table()
    for hexbyte, val in _lines("e4m3_landmarks.txt"):
        b = int(hexbyte, 16)
        if val == "nan":
            assert np.isnan(tab[b]), hexbyte
        else:
            v = float(val)
            assert tab[b] == v, hexbyte
            assert np.signbit(tab[b]) == np.signbit(v), hexbyte


def test_table_matches_torch_float8():
    tab = oracle.e4m3_table()
    ref = _torch_e4m3_to_f32(np.arange(256, dtype=np.uint8)).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(tab))
    assert np.array_equal(ref[~nan], tab[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(tab[~nan]))


def test_table_strictly_increasing_and_symmetric():
    tab = oracle.e4m3_table()
    pos = tab[:0x7F]
    assert np.all(np.diff(pos) > 0)
    assert pos[-1] == 448.0
    assert np.array_equal(tab[0x80:0xFF], -pos)
    assert np.isnan(tab[0x7F]) and np.isnan(tab[0xFF])


def test_encode_golden_cases():
    for val, hexbyte, *_ in _lines("e4m3_encode_cases.txt"):
        x = np.float32(float(val))
        got = int(oracle.e4m3_encode([x])[0])
        assert got == int(hexbyte, 16), (val, hex(got), hexbyte)


def _bruteforce_encode(x: np.ndarray) -> np.ndarray:
    """Nearest of the 127 finite magnitudes, ties to the even code, |x|>448
    saturates, NaN -> 0x7F, sign kept.  Distances are exact in float64 for
    every x whose two candidates are close to it."""
    tab = oracle.e4m3_table()[:0x7F]
    a = np.abs(x.astype(np.float64))
    out = np.empty(x.shape, np.uint8)
    chunk = 8192
    for i in range(0, x.size, chunk):
        aa = a[i:i + chunk]
        d = np.abs(aa[:, None] - tab[None, :])
        dmin = d.min(axis=1, keepdims=True)
        ties = d == dmin
        first = ties.argmax(axis=1)
        two = ties.sum(axis=1) > 1
        code = np.where(two & (first % 2 == 1), first + 1, first)
        code = np.where(aa > 448.0, 0x7E, code)
        out[i:i + chunk] = code
    out |= np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    out[np.isnan(x)] = 0x7F
    return out


@pytest.mark.parametrize("k_scale", [1.0, 0.5, 3.0 / 448.0, 0.0123, 7.0, 2.0 ** -12,
                                     0.00634765625])
def test_encode_bruteforce_all_bf16_inputs(k_scale):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = W.bf16_bits_to_float(bits)
    x = x[~np.isnan(x)]
    with np.errstate(over="ignore"):                   # overflow to inf saturates
        y = (x / np.float32(k_scale)).astype(np.float32)   # one IEEE fp32 division
    got = oracle.e4m3_encode(y)
    ref = _bruteforce_encode(y)
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, (y[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_encode_matches_torch_in_range():
    g = np.random.default_rng(7)
    x = np.concatenate([
        g.standard_normal(200000).astype(np.float32) * np.float32(50),
        g.standard_normal(100000).astype(np.float32) * np.float32(0.01),
        (oracle.e4m3_table()[:0x7E] + oracle.e4m3_table()[1:0x7F]).astype(np.float32) / 2,
    ])
    x = x[np.abs(x) < 464]
    x = np.concatenate([x, -x])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x)
    assert np.array_equal(got, ref)


def test_encode_decode_roundtrip():
    tab = oracle.e4m3_table()
    codes = np.array([b for b in range(256) if (b & 0x7F) != 0x7F], np.uint8)
    enc = oracle.e4m3_encode(tab[codes].astype(np.float32))
    assert np.array_equal(enc, codes)


def test_store_writes_encoded_rows_only():
    g = np.random.default_rng(3)
    n, P = 9, 40
    lat = torch.from_numpy(g.standard_normal((n, 576)).astype(np.float32) * 0.5)
    bits = lat.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    slots = g.choice(P, size=n, replace=False).astype(np.int64)
    slots[4] = P + 3                                  # out of range: skipped
    k = 0.0071
    pool = np.full((P, 576), 0x11, np.uint8)
    bad = oracle.kv_store_fp8(bits[:, :512], bits[:, 512:], slots, k, pool[:, :512],
                              pool[:, 512:])
    assert bad == 1
    x = (W.bf16_bits_to_float(bits) / np.float32(k)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for i, s in enumerate(slots):
        if i == 4:
            continue
        assert np.array_equal(pool[s], ref[i])
    untouched = np.setdiff1d(np.arange(P), slots)
    assert np.all(pool[untouched] == 0x11)


def test_store_separate_pools_with_padding_strides():
    g = np.random.default_rng(4)
    n = 5
    bits = torch.from_numpy(g.standard_normal((n, 576)).astype(np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    slots = np.array([0, 7, 3, 9, 1], np.int64)
    ckv = np.zeros((10, 528), np.uint8)[:, :512]          # row stride 528
    kpe = np.zeros((10, 80), np.uint8)[:, :64]            # row stride 80
    oracle.kv_store_fp8(bits[:, :512], bits[:, 512:], slots, 1.0, ckv, kpe)
    joined = np.zeros((10, 576), np.uint8)
    oracle.kv_store_fp8(bits[:, :512], bits[:, 512:], slots, 1.0, joined[:, :512],
                        joined[:, 512:])
    assert np.array_equal(ckv, joined[:, :512]) and np.array_equal(kpe, joined[:, 512:])


@pytest.mark.parametrize("k_scale,page_size", [(1.0, 1), (1.0, 4), (0.0063, 1), (3.5, 2)])
def test_gather_cast_matches_torch(k_scale, page_size):
    g = np.random.default_rng(5)
    pages = 12
    pool = W.random_fill_bytes(g, (pages * page_size, 576))
    idx = g.permutation(pages)[:7].astype(np.int32)
    ckv, kpe = oracle.kv_gather_cast(pool[:, :512], pool[:, 512:], idx, page_size, k_scale)
    rows = (idx[:, None].astype(np.int64) * page_size + np.arange(page_size)).ravel()
    f8 = torch.from_numpy(pool[rows]).view(torch.float8_e4m3fn)
    if k_scale == 1.0:
        ref = f8.to(torch.bfloat16)                      # the pages' .to(bfloat16)
    else:
        ref = (f8.float() * torch.tensor(k_scale, dtype=torch.float32)).to(torch.bfloat16)
    ref = ref.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ckv, ref[:, :512]) and np.array_equal(kpe, ref[:, 512:])


def test_gather_cast_rejects_out_of_range_page():
    pool = np.zeros((8, 576), np.uint8)
    with pytest.raises(IndexError):
        oracle.kv_gather_cast(pool[:, :512], pool[:, 512:], np.array([1, 8], np.int32), 1, 1.0)


def test_float_to_bf16_matches_torch():
    g = np.random.default_rng(6)
    x = g.standard_normal(3000).astype(np.float32) * np.float32(1e3)
    # exact ties: a BF16 value plus half of its ulp (ulp = 2^(exponent - 7))
    base = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    half_ulp = np.ldexp(np.float32(1.0), np.frexp(base)[1] - 9).astype(np.float32)
    ties = (base + np.sign(base) * half_ulp).astype(np.float32)
    x = np.concatenate([x, ties, np.float32([0.0, -0.0, 1e-40, -3e-39, 3.3e38, -3.38e38])])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.float_to_bf16(x)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("k_scale", [1.0, 0.37, 2.0 ** -7])
def test_gather_cast_all_256_bytes_including_nan(k_scale):
    """Every byte value, the two NaN codes included.  At k_scale = 1 the
    oracle is PyTorch's float8_e4m3fn -> bfloat16 cast bit for bit (the
    pages' .to(bfloat16); it gives the quiet NaN 0x7FC0 for 0x7F and 0xFF).
    At any other scale the finite bytes follow one fp32 multiply and a BF16
    rounding, and the NaN codes still give 0x7FC0."""
    rows = np.arange(256 * 9, dtype=np.int64).reshape(-1, 576) % 256
    pool = rows.astype(np.uint8)                    # 4 rows, each byte value 9 times
    idx = np.arange(pool.shape[0], dtype=np.int32)
    ckv, kpe = oracle.kv_gather_cast(pool[:, :512], pool[:, 512:], idx, 1, k_scale)
    got = np.concatenate([ckv, kpe], axis=1)
    f8 = torch.from_numpy(pool).view(torch.float8_e4m3fn)
    nan = (pool & 0x7F) == 0x7F
    assert nan.sum() == 2 * 9
    assert np.all(got[nan] == 0x7FC0)
    if k_scale == 1.0:
        ref = f8.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, ref)
    else:
        ref = (f8.float() * torch.tensor(k_scale, dtype=torch.float32)).to(torch.bfloat16)
        ref = ref.view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got[~nan], ref[~nan])
