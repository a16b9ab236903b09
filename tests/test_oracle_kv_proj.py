"""Pins for the oracle's fused KV projection + quantize-on-store.

Checked against: exact rational arithmetic (Python fractions: the dot
product of BF16 values summed exactly, then rounded to BF16 by a rounding
written here from the format: 8 significant bits, ties to even, subnormal
spacing 2^-133); printed tie cases; the identity projection, which must
store exactly what kv_store_fp8 stores; linearity in the weights.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads as W


def _bf16(x) -> np.ndarray:
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _exact_bf16_bits(v: Fraction) -> int:
    """Round an exact rational to BF16 (nearest, ties to even)."""
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator)) + 1
    while Fraction(2) ** (e - 1) > a:        # make 2^(e-1) <= a < 2^e exactly
        e -= 1
    while Fraction(2) ** e <= a:
        e += 1
    q = max(e - 8, -133)
    scaled = a / Fraction(2) ** q
    r = math.floor(scaled)
    rem = scaled - r
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and r % 2 == 1):
        r += 1
    val = Fraction(r) * Fraction(2) ** q
    if val >= Fraction(2) ** 128:
        return sign | 0x7F80
    bits = int(np.array([float(val)], np.float32).view(np.uint32)[0] >> 16)
    return sign | bits


@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3F80), (1 + 2 ** -8, 0x3F80), (1 + 3 * 2 ** -8, 0x3F82), (-(1 + 2 ** -8), 0xBF80),
    (1.5 * 2 ** -133, 0x0002), (0.5 * 2 ** -133, 0x0000), (2.0 ** 128, 0x7F80),
    (255.5, 0x4380), (2 ** -126, 0x0080),
])
def test_double_to_bf16_cases(x, bits):
    assert int(oracle.double_to_bf16([x])[0]) == bits
    assert _exact_bf16_bits(Fraction(x)) == bits


def _case(seed, n, d, scale=1.0):
    g = np.random.default_rng(seed)
    x = _bf16(g.standard_normal((n, d)) * scale)
    w = _bf16(g.standard_normal((576, d)) / math.sqrt(d))
    return x, w


@pytest.mark.parametrize("seed,n,d", [(0, 3, 64), (1, 2, 128), (2, 1, 200)])
def test_latent_is_the_exact_dot_rounded_once(seed, n, d):
    x, w = _case(seed, n, d)
    g = np.random.default_rng(seed + 10)
    P = 16
    slots = g.permutation(P)[:n].astype(np.int64)
    pool = W.random_fill_bytes(g, (P, 576))
    lat, bad = oracle.kv_proj_fp8(x, w, slots, 0.0123, pool[:, :512], pool[:, 512:])
    assert bad == 0
    xf = W.bf16_bits_to_float(x)
    wf = W.bf16_bits_to_float(w)
    for i in range(n):
        xi = [Fraction(float(v)) for v in xf[i]]
        for j in range(0, 576, 7):               # a spread of channels, both parts
            exact = sum(a * Fraction(float(b)) for a, b in zip(xi, wf[j]))
            assert int(lat[i, j]) == _exact_bf16_bits(exact), (i, j)
    # the pool rows are the store of those latents
    again = pool.copy()
    oracle.kv_store_fp8(lat[:, :512], lat[:, 512:], slots, 0.0123, again[:, :512], again[:, 512:])
    assert np.array_equal(again, pool)


def test_identity_projection_stores_the_input():
    g = np.random.default_rng(5)
    n, d = 4, 640
    x = _bf16(g.standard_normal((n, d)) * 3)
    w = np.zeros((576, d), np.uint16)
    w[np.arange(576), np.arange(576)] = 0x3F80       # 1.0
    slots = np.array([7, 2, 9, 0], np.int64)
    pool_a = W.random_fill_bytes(g, (12, 576))
    pool_b = pool_a.copy()
    lat, _ = oracle.kv_proj_fp8(x, w, slots, 0.02, pool_a[:, :512], pool_a[:, 512:])
    assert np.array_equal(lat, x[:, :576])
    oracle.kv_store_fp8(x[:, :512], x[:, 512:576], slots, 0.02, pool_b[:, :512], pool_b[:, 512:])
    assert np.array_equal(pool_a, pool_b)


def test_doubling_the_weights_doubles_the_latent():
    x, w = _case(6, 3, 96)
    w2 = _bf16(W.bf16_bits_to_float(w) * 2)          # exact: a power of two
    slots = np.arange(3, dtype=np.int64)
    p1 = np.zeros((3, 576), np.uint8)
    p2 = np.zeros((3, 576), np.uint8)
    l1, _ = oracle.kv_proj_fp8(x, w, slots, 0.01, p1[:, :512], p1[:, 512:])
    l2, _ = oracle.kv_proj_fp8(x, w2, slots, 0.02, p2[:, :512], p2[:, 512:])
    assert np.array_equal(W.bf16_bits_to_float(l2), 2 * W.bf16_bits_to_float(l1))
    assert np.array_equal(p1, p2)                    # k_scale doubled with the weights


def test_out_of_range_slot_is_counted_and_skipped():
    x, w = _case(7, 2, 64)
    pool = np.full((4, 576), 0x11, np.uint8)
    _, bad = oracle.kv_proj_fp8(x, w, np.array([1, 4], np.int64), 0.01, pool[:, :512],
                                pool[:, 512:])
    assert bad == 1
    assert np.all(pool[[0, 2, 3]] == 0x11) and not np.all(pool[1] == 0x11)
