"""Pins for the oracle's paged MLA decode attention.

Checked against: a brute force written here in a different formulation
(PyTorch's float8_e4m3fn dequant, exact-rounded math.fsum sums, no max
subtraction), scipy's softmax / logsumexp on explicit rows, and invariants
that hold for any correct implementation (weights sum to one, a one-token
context returns that row, slot order does not matter, a zero query averages
the values, heads are independent, the BF16 cast-then-attend path equals the
FP8 path).
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads as W

SCALE = 1.0 / math.sqrt(192.0)


def _f8(pool_rows: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(pool_rows)).view(
        torch.float8_e4m3fn).float().numpy().astype(np.float64)


def _tiny_case(seed, B=2, H=3, lens=(5, 8), ps=1, pool_pages=20, k_scale=0.37, std=1.0):
    g = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int32)
    pages = (lens + ps - 1) // ps
    indptr = np.zeros(B + 1, np.int32)
    indptr[1:] = np.cumsum(pages)
    indices = g.permutation(pool_pages)[: indptr[-1]].astype(np.int32)
    pool = W.random_fill_bytes(g, (pool_pages * ps, 576))
    # keep magnitudes moderate so the brute force needs no max subtraction
    pool[(pool & 0x78) > 0x50] &= 0x87
    q = torch.from_numpy(g.standard_normal((B, H, 576)).astype(np.float32) * std).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return q, pool, indptr, indices, lens, ps, k_scale


def _brute(q, pool, indptr, indices, lens, ps, k_scale, scale=SCALE):
    B, H, _ = q.shape
    qf = W.bf16_bits_to_float(q).astype(np.float64)
    o = np.zeros((B, H, 512))
    lse = np.zeros((B, H))
    for b in range(B):
        rows = []
        for t in range(int(lens[b])):
            slot = int(indices[indptr[b] + t // ps]) * ps + t % ps
            rows.append(_f8(pool[slot]) * k_scale)
        for h in range(H):
            if not rows:
                lse[b, h] = -math.inf
                continue
            e = [math.exp(scale * math.fsum(qf[b, h] * r)) for r in rows]
            z = math.fsum(e)
            for d in range(512):
                o[b, h, d] = math.fsum(e[t] / z * rows[t][d] for t in range(len(rows)))
            lse[b, h] = math.log(z)
    return o, lse


@pytest.mark.parametrize("seed,ps,lens", [(0, 1, (5, 8)), (1, 3, (7, 2)), (2, 1, (1, 6)),
                                          (3, 4, (8, 5))])
def test_matches_bruteforce(seed, ps, lens):
    q, pool, indptr, indices, lens, ps, k = _tiny_case(seed, lens=lens, ps=ps)
    o, lse = oracle.decode_fp8(q, pool[:, :512], pool[:, 512:], indptr, indices, lens, ps, k,
                               SCALE)
    bo, blse = _brute(q, pool, indptr, indices, lens, ps, k)
    np.testing.assert_allclose(o, bo, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, blse, rtol=1e-12, atol=1e-13)


def test_core_matches_scipy_softmax():
    g = np.random.default_rng(11)
    q = g.standard_normal((5, 576))
    k = g.standard_normal((700, 576)) * 0.5
    o, lse, p = oracle.attention_f64(q, k, SCALE, want_p=True)
    s = SCALE * q @ k.T
    np.testing.assert_allclose(lse, scipy.special.logsumexp(s, axis=1), rtol=1e-13)
    ps = scipy.special.softmax(s, axis=1)
    np.testing.assert_allclose(p, ps, rtol=1e-11, atol=1e-16)
    np.testing.assert_allclose(o, ps @ k[:, :512], rtol=1e-10, atol=1e-13)


def test_weights_sum_to_one_and_vanish_past_the_context():
    q, pool, indptr, indices, lens, ps, k = _tiny_case(4, lens=(5, 8))
    o, lse, p = oracle.decode_fp8(q, pool[:, :512], pool[:, 512:], indptr, indices, lens, ps,
                                  k, SCALE, want_p=True)
    for b in range(2):
        np.testing.assert_allclose(p[b, :, : lens[b]].sum(axis=1), 1.0, atol=1e-12)
        assert np.all(p[b, :, lens[b]:] == 0)


def test_single_token_returns_that_row():
    q, pool, indptr, indices, lens, ps, k = _tiny_case(5, lens=(1, 1))
    o, lse = oracle.decode_fp8(q, pool[:, :512], pool[:, 512:], indptr, indices, lens, ps, k,
                               SCALE)
    qf = W.bf16_bits_to_float(q).astype(np.float64)
    for b in range(2):
        row = _f8(pool[indices[b]]) * k
        for h in range(3):
            assert np.array_equal(o[b, h], row[:512])
            assert lse[b, h] == pytest.approx(SCALE * math.fsum(qf[b, h] * row), rel=1e-13)


@pytest.mark.parametrize("ps", [1, 4])
def test_slot_order_does_not_matter(ps):
    q, pool, indptr, indices, lens, ps, k = _tiny_case(6, lens=(16, 12), ps=ps, pool_pages=32)
    o, lse = oracle.decode_fp8(q, pool[:, :512], pool[:, 512:], indptr, indices, lens, ps, k,
                               SCALE)
    # move every token to a new slot (and the page table with it)
    g = np.random.default_rng(60)
    lens2 = lens.copy()
    rows = []
    for b in range(2):
        for t in range(lens[b]):
            rows.append((b, pool[int(indices[indptr[b] + t // ps]) * ps + t % ps].copy()))
    pool2 = W.random_fill_bytes(g, (64 * ps, 576))
    new_slots = g.permutation(64 * ps)
    indptr2 = np.zeros(3, np.int32)
    indptr2[1:] = np.cumsum(lens2)
    per_b = [[r for (bb, r) in rows if bb == b] for b in range(2)]
    idx2 = []
    n = 0
    for b in range(2):
        order = g.permutation(len(per_b[b]))
        for j in order:
            pool2[new_slots[n]] = per_b[b][j]
            idx2.append(new_slots[n])
            n += 1
    o2, lse2 = oracle.decode_fp8(q, pool2[:, :512], pool2[:, 512:], indptr2,
                                 np.array(idx2, np.int32), lens2, 1, k, SCALE)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13)


def test_zero_query_averages_values():
    q, pool, indptr, indices, lens, ps, k = _tiny_case(7, lens=(6, 3))
    q[:] = 0
    o, lse = oracle.decode_fp8(q, pool[:, :512], pool[:, 512:], indptr, indices, lens, ps, k,
                               SCALE)
    for b in range(2):
        v = np.stack([_f8(pool[indices[indptr[b] + t]])[:512] * k for t in range(lens[b])])
        for h in range(3):
            np.testing.assert_allclose(o[b, h], v.mean(axis=0), rtol=1e-13, atol=1e-16)
            assert lse[b, h] == pytest.approx(math.log(lens[b]), abs=1e-14)


def test_zero_rope_keys_reduce_to_512_dim_attention():
    q, pool, indptr, indices, lens, ps, k = _tiny_case(8, lens=(7, 4))
    pool[:, 512:] = 0
    o, lse = oracle.decode_fp8(q, pool[:, :512], pool[:, 512:], indptr, indices, lens, ps, k,
                               SCALE)
    qf = W.bf16_bits_to_float(q).astype(np.float64)
    for b in range(2):
        kk = np.stack([_f8(pool[indices[indptr[b] + t]]) * k for t in range(lens[b])])
        q512 = qf[b].copy()
        q512[:, 512:] = 0                      # the rope query no longer matters
        o2, lse2 = oracle.attention_f64(q512, kk, SCALE)
        np.testing.assert_allclose(o[b], o2, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(lse[b], lse2, rtol=1e-13)


def test_heads_are_independent():
    q, pool, indptr, indices, lens, ps, k = _tiny_case(9, H=4, lens=(9, 5))
    o, lse = oracle.decode_fp8(q, pool[:, :512], pool[:, 512:], indptr, indices, lens, ps, k,
                               SCALE)
    for h in range(4):
        oh, lh = oracle.decode_fp8(np.ascontiguousarray(q[:, h:h + 1]), pool[:, :512],
                                   pool[:, 512:], indptr, indices, lens, ps, k, SCALE)
        assert np.array_equal(oh[:, 0], o[:, h]) and np.array_equal(lh[:, 0], lse[:, h])


def test_empty_context():
    q, pool, indptr, indices, lens, ps, k = _tiny_case(10, lens=(0, 3))
    o, lse = oracle.decode_fp8(q, pool[:, :512], pool[:, 512:], indptr, indices, lens, ps, k,
                               SCALE)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


@pytest.mark.parametrize("ps", [1, 2])
def test_gather_cast_then_sequential_replan_equals_fp8_path(ps):
    """The gather-then-cast fix: cast only the active pages, then attend over
    the compact BF16 copy with indices 0..n-1; the result must equal the
    direct FP8 read."""
    q, pool, indptr, indices, lens, ps, k = _tiny_case(12, lens=(9, 6), ps=ps)
    o, lse = oracle.decode_fp8(q, pool[:, :512], pool[:, 512:], indptr, indices, lens, ps, k,
                               SCALE)
    ckv, kpe = oracle.kv_gather_cast(pool[:, :512], pool[:, 512:], indices, ps, 1.0)
    seq_idx = np.arange(indices.shape[0], dtype=np.int32)
    o2, lse2 = oracle.decode_bf16(q, ckv, kpe, indptr, seq_idx, lens, ps, k, SCALE)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_rejects_short_page_table_and_bad_slot():
    q, pool, indptr, indices, lens, ps, k = _tiny_case(13, lens=(4, 4))
    with pytest.raises(IndexError):
        oracle.decode_fp8(q, pool[:, :512], pool[:, 512:], indptr, indices,
                          np.array([5, 4], np.int32), 1, k, SCALE)
    bad = indices.copy()
    bad[2] = 10_000
    with pytest.raises(IndexError):
        oracle.decode_fp8(q, pool[:, :512], pool[:, 512:], indptr, bad, lens, 1, k, SCALE)
