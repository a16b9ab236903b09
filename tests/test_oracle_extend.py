"""Pins for the oracle's causal extend attention (new tokens of a request
attending to its cached prefix and to the new tokens before them).

Checked against: a dense formulation written here with library routines
(PyTorch's float8_e4m3fn dequant, an explicit lower-triangular mask,
torch.softmax and torch.logsumexp in float64); the pinned decode oracle, to
which a one-token extend and the last new token of any extend reduce; and a
closed form (the first token of a request without a prefix sees only itself,
so its output is its own value row and its lse its own score).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W

SCALE = 1.0 / math.sqrt(192.0)


def _f8(rows: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(rows)).view(torch.float8_e4m3fn).to(torch.float64)


def _case(seed, lens, q_lens, H=3, ps=1, k_scale=0.37, std=1.0):
    g = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int32)
    q_lens = np.asarray(q_lens, np.int32)
    B = lens.shape[0]
    pages = (lens + ps - 1) // ps
    indptr = np.zeros(B + 1, np.int32)
    indptr[1:] = np.cumsum(pages)
    pool_pages = int(indptr[-1]) + 7
    indices = g.permutation(pool_pages)[: indptr[-1]].astype(np.int32)
    pool = W.random_fill_bytes(g, (pool_pages * ps, 576))
    pool[(pool & 0x78) > 0x50] &= 0x87          # moderate magnitudes (exponent field <= 10)
    qo = np.zeros(B + 1, np.int32)
    qo[1:] = np.cumsum(q_lens)
    q = torch.from_numpy(g.standard_normal((int(qo[-1]), H, 576)).astype(np.float32) * std).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return q, pool, qo, indptr, indices, lens, ps, k_scale


def _run(case):
    q, pool, qo, indptr, indices, lens, ps, k = case
    return oracle.extend_fp8(q, pool[:, :512], pool[:, 512:], qo, indptr, indices, lens, ps, k,
                             SCALE)


def _dense(case):
    """Per request: all its keys, all its new queries, a causal mask."""
    q, pool, qo, indptr, indices, lens, ps, k = case
    H = q.shape[1]
    qf = torch.from_numpy(W.bf16_bits_to_float(q).astype(np.float64))
    o = torch.zeros(q.shape[0], H, 512, dtype=torch.float64)
    lse = torch.zeros(q.shape[0], H, dtype=torch.float64)
    for b in range(lens.shape[0]):
        L, n = int(lens[b]), int(qo[b + 1] - qo[b])
        if n == 0:
            continue
        t = np.arange(L)
        slots = indices[indptr[b] + t // ps].astype(np.int64) * ps + t % ps
        kk = _f8(pool[slots]) * k                                   # [L, 576]
        qq = qf[qo[b]:qo[b + 1]]                                    # [n, H, 576]
        s = SCALE * torch.einsum("nhd,ld->nhl", qq, kk)
        pos = torch.arange(L - n, L).view(n, 1, 1)                  # each new token's position
        s = s.masked_fill(torch.arange(L).view(1, 1, L) > pos, -math.inf)
        o[qo[b]:qo[b + 1]] = torch.einsum("nhl,ld->nhd", torch.softmax(s, dim=-1), kk[:, :512])
        lse[qo[b]:qo[b + 1]] = torch.logsumexp(s, dim=-1)
    return o.numpy(), lse.numpy()


@pytest.mark.parametrize("seed,ps,lens,q_lens", [
    (0, 1, (6, 9, 12), (2, 0, 5)),
    (1, 3, (7, 10), (7, 3)),          # a pure prefill (no prefix) and an extend
    (2, 4, (13, 1, 8), (1, 1, 8)),
    (3, 1, (16,), (11,)),
])
def test_matches_dense_causal_formulation(seed, ps, lens, q_lens):
    case = _case(seed, lens, q_lens, ps=ps)
    o, lse = _run(case)
    do, dlse = _dense(case)
    np.testing.assert_allclose(o, do, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, dlse, rtol=1e-12, atol=1e-13)


def test_one_new_token_is_decode():
    case = _case(4, (9, 5, 14), (1, 1, 1), H=4, ps=2)
    q, pool, qo, indptr, indices, lens, ps, k = case
    o, lse = _run(case)
    do, dlse = oracle.decode_fp8(q, pool[:, :512], pool[:, 512:], indptr, indices, lens, ps, k,
                                 SCALE)
    assert np.array_equal(o, do) and np.array_equal(lse, dlse)


def test_each_new_token_is_decode_over_its_visible_prefix():
    case = _case(5, (11, 8), (4, 8), H=2, ps=1)
    q, pool, qo, indptr, indices, lens, ps, k = case
    o, lse = _run(case)
    for b in range(2):
        n = int(qo[b + 1] - qo[b])
        for i in range(n):
            visible = int(lens[b]) - n + i + 1
            row = int(qo[b]) + i
            do, dlse = oracle.decode_fp8(q[row:row + 1], pool[:, :512], pool[:, 512:],
                                         np.array([0, visible], np.int32),
                                         indices[indptr[b]:indptr[b] + visible],
                                         np.array([visible], np.int32), 1, k, SCALE)
            assert np.array_equal(o[row], do[0]) and np.array_equal(lse[row], dlse[0])


def test_first_token_of_a_prefill_sees_only_itself():
    case = _case(6, (5, 9), (5, 9), H=3)
    q, pool, qo, indptr, indices, lens, ps, k = case
    o, lse = _run(case)
    qf = W.bf16_bits_to_float(q).astype(np.float64)
    for b in range(2):
        row = _f8(pool[indices[indptr[b]]]).numpy() * k
        for h in range(3):
            assert np.array_equal(o[qo[b], h], row[:512])
            assert lse[qo[b], h] == pytest.approx(SCALE * math.fsum(qf[qo[b], h] * row), rel=1e-13)


def test_rejects_more_new_tokens_than_context():
    case = _case(7, (4, 6), (2, 3))
    q, pool, qo, indptr, indices, lens, ps, k = case
    with pytest.raises(IndexError):
        oracle.extend_fp8(q, pool[:, :512], pool[:, 512:], qo, indptr, indices,
                          np.array([4, 2], np.int32), ps, k, SCALE)
