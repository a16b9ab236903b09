"""GPU parity on inputs that drive the FP8 tensor-core kernel's less common
branches, against the CPU oracle:

  * scores that rise across a context, so that the online softmax's running
    maximum moves on most 64-token tiles and the output accumulator is
    rescaled in tensor memory (decode at full batch-40 size, the 128-head
    paged call on sampled requests, and speculative extend);
  * raw random cache bytes at k_scale = 1 (scores in the tens, peaky and
    jumping), the same branch reached another way;
  * query rows whose entries span a wide range (one entry in the hundreds
    next to entries near 1e-3, or entries 2^-10 .. 2^-16 of the row's
    largest), which the first two E4M3 terms of the split query cannot hold;
  * all-zero query rows (out = mean of the values, lse = ln L);
  * an "attention sink": one token per request far above thousands of
    others, whose small weights must still reach the output;
  * query rows holding an infinity or a NaN (that head's output and lse are
    NaN, every other head is unaffected).

Tolerance: the contract's |err| <= 1e-2 + 1e-2 |ref| on the BF16 output and
1e-3 on the LSE, and for the wide-range queries also the four times tighter
bound of the kernel's own precision test.
"""
import numpy as np
import pytest
import torch

import mla_decode_attention_run_gb300 as M
import oracle
import workloads as W
from gpu_util import check_attention, dev_bf16, dev_i32, gpu_decode, oracle_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    M.mla_get_last_error()


def _bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def _token_index(w: W.Workload, requests) -> np.ndarray:
    """Token position of each drawn latent row (rows are per request, in
    token order, for the requests whose latents were drawn)."""
    return np.concatenate([np.arange(int(w.seq_lens[b])) for b in requests])


def _set_latents(w: W.Workload, lat: np.ndarray):
    """Replace the workload's latents (float32 [n, 576], rounded to BF16)
    and take k_scale = absmax / 448 again."""
    w.latent_bf16 = _bf16(lat)
    amax = float(np.abs(W.bf16_bits_to_float(w.latent_bf16)).max())
    w.k_scale = float(np.float32(amax / 448.0))


RAMP_CHANNELS = 64


def _ramp(w: W.Workload, requests, per_token: float):
    """c_kv channels 0-63 of token t of a request of L tokens move by
    per_token / 64 * (t - L) (on top of the drawn noise, which dithers their
    E4M3 rounding) and q channels 0-63 are 2 (2.5 for odd heads): each head's
    score rises by about softmax_scale * 2 * per_token per token, several
    log2 units per tile, up to ordinary values at the context's end (so the
    largest scores, and the lse, stay where fp32 resolves 1e-3)."""
    lat = W.bf16_bits_to_float(w.latent_bf16).copy()
    lens = np.concatenate([np.full(int(w.seq_lens[b]), int(w.seq_lens[b])) for b in requests])
    lat[:, :RAMP_CHANNELS] += (per_token / RAMP_CHANNELS) * (_token_index(w, requests) - lens)[:, None]
    _set_latents(w, lat)
    q = W.bf16_bits_to_float(w.q_bf16).copy()
    q[:, :, :RAMP_CHANNELS] = np.where(np.arange(w.heads) % 2 == 0, 2.0, 2.5)[None, :, None]
    w.q_bf16 = _bf16(q)


def _oracle_decode(w, pool, sel=None):
    if sel is None:
        return oracle.decode_fp8(w.q_bf16, pool[:, :512], pool[:, 512:], w.kv_indptr,
                                 w.kv_indices, w.seq_lens, w.page_size, w.k_scale,
                                 w.softmax_scale)
    indptr = np.zeros(len(sel) + 1, np.int32)
    idx = []
    for i, b in enumerate(sel):
        idx.append(w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]])
        indptr[i + 1] = indptr[i] + idx[-1].size
    return oracle.decode_fp8(np.ascontiguousarray(w.q_bf16[sel]), pool[:, :512], pool[:, 512:],
                             indptr, np.concatenate(idx), w.seq_lens[sel], w.page_size,
                             w.k_scale, w.softmax_scale)


def _gpu(w, pool_np):
    pool = torch.from_numpy(pool_np).cuda()
    out, lse, _ = gpu_decode(w, pool[:, :512], pool[:, 512:])
    assert M.mla_get_last_error() == 0
    return out, lse


def _rescales_per_tile(w, pool, request, head, tau=4.0):
    """The fraction of one request's 64-token tiles after the first on which
    the kernel's running maximum moves (a score more than tau log2 units
    above it), from the oracle's exact scores: it shows that a case really
    exercises the rescale."""
    _, _, p = oracle.decode_fp8(w.q_bf16[request:request + 1, head:head + 1].copy(),
                                pool[:, :512], pool[:, 512:],
                                np.array([0, w.kv_indptr[request + 1] - w.kv_indptr[request]],
                                         np.int32),
                                w.kv_indices[w.kv_indptr[request]:w.kv_indptr[request + 1]],
                                w.seq_lens[request:request + 1], w.page_size, w.k_scale,
                                w.softmax_scale, want_p=True)
    s = np.log2(np.maximum(p[0, 0, :w.seq_lens[request]], 1e-300))   # scores up to a constant
    moves, m = 0, s[:64].max()
    for t0 in range(64, s.size, 64):
        tile = s[t0:t0 + 64]
        if tile.max() > m + tau:
            moves += 1
            m = tile.max()
    return moves / max(1, (s.size - 1) // 64)


# ------------------------------------------------------------ rescale path

def test_rescale_rising_scores_concurrency_full_size():
    """Batch 40, contexts U[1024, 8192], the full 495,552-slot pool: scores
    rise by about 5 log2 units per tile, so the running maximum moves on
    most tiles of every request and the output is rescaled in place before
    each PV."""
    w = W.make_workload("concurrency")
    _ramp(w, range(w.batch), per_token=0.4)
    pool = oracle_pool(w)
    assert _rescales_per_tile(w, pool, request=3, head=0) > 0.75
    out, lse = _gpu(w, pool)
    o_ref, lse_ref = _oracle_decode(w, pool)
    check_attention(out, lse, o_ref, lse_ref, "rising scores, batch 40")


def test_rescale_rising_scores_gentle_slope():
    """A slope of about 2.5 log2 units per tile: the maximum moves on every
    second tile or so, and the tiles between add to an accumulator that was
    rescaled earlier."""
    w = W.make_workload("concurrency", batch=8, num_slots=100_000, seed=61)
    _ramp(w, range(w.batch), per_token=0.2)
    pool = oracle_pool(w)
    frac = _rescales_per_tile(w, pool, request=0, head=0)
    assert 0.2 < frac < 0.9
    out, lse = _gpu(w, pool)
    o_ref, lse_ref = _oracle_decode(w, pool)
    check_attention(out, lse, o_ref, lse_ref, "gentle slope")


def test_rescale_random_cache_bytes_unit_scale():
    """Raw random E4M3 bytes (exponent capped at 2^3, so |value| <= 15) at
    k_scale = 1 in every active slot of the batch-40 page table: scores with
    a spread in the tens, peaky softmax, maxima that jump."""
    w = W.make_workload("concurrency", latent_requests=[])
    g = np.random.default_rng(62)
    pool = W.random_fill_bytes(g, (w.num_slots, 576))
    pool[(pool & 0x78) > 0x50] &= 0x87
    w.k_scale = 1.0
    assert _rescales_per_tile(w, pool, request=5, head=2) > 0
    out, lse = _gpu(w, pool)
    o_ref, lse_ref = _oracle_decode(w, pool)
    check_attention(out, lse, o_ref, lse_ref, "random bytes, k_scale 1")


def test_rescale_large_head_paged_sampled():
    """H = 128 (32-head CTAs, four head groups), page size 64, 32,768-token
    contexts: the full 2.4 GB launch, with rising scores on 4 sampled
    requests compared in full."""
    sample = [0, 40, 99, 127]
    w = W.make_workload("large_head", latent_requests=sample)
    _ramp(w, sample, per_token=0.4)
    pool = oracle_pool(w)
    out, lse = _gpu(w, pool)
    o_ref, lse_ref = _oracle_decode(w, pool, sel=np.array(sample))
    sel = torch.tensor(sample, device="cuda")
    check_attention(out[sel], lse[sel], o_ref, lse_ref, "rising scores, H = 128")


def test_rescale_rising_scores_extend():
    """Speculative extend (40 requests x 4 new tokens, the decode workload's
    contexts) on rising scores, every row's causal limit inside the ramp."""
    w = W.make_extend_workload("spec_decode")
    _ramp(w, range(w.batch), per_token=0.4)
    pool = oracle_pool(w)
    o_ref, lse_ref = oracle.extend_fp8(w.q_bf16, pool[:, :512], pool[:, 512:],
                                       w.extra["qo_indptr"], w.kv_indptr, w.kv_indices,
                                       w.seq_lens, w.page_size, w.k_scale, w.softmax_scale)
    dpool = torch.from_numpy(pool).cuda()
    qo = w.extra["qo_indptr"]
    plan = M.mla_extend_plan(qo, w.kv_indptr, w.seq_lens, w.batch, w.heads, w.page_size)
    n_q = int(qo[-1])
    out = torch.full((n_q, w.heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((n_q, w.heads), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    M.mla_extend_run(plan, dev_bf16(w.q_bf16), dpool[:, :512], dpool[:, 512:], w.num_slots,
                     dev_i32(w.kv_indptr), dev_i32(w.kv_indices), dev_i32(w.seq_lens),
                     w.k_scale, w.softmax_scale, out, lse, ws)
    assert M.mla_get_last_error() == 0
    check_attention(out, lse, o_ref, lse_ref, "rising scores, extend")


# ------------------------------------------------------ wide-range queries

def _tight(out, lse, o_ref, lse_ref, where):
    o = out.float().cpu().numpy()
    err = np.abs(o - o_ref) - (2.5e-3 + 2.5e-3 * np.abs(o_ref))
    assert err.max() <= 0, f"{where}: output off by {np.abs(o - o_ref).max():.3e}"
    dl = np.abs(lse.cpu().numpy().astype(np.float64) - lse_ref)
    assert dl.max() <= 2.5e-4, f"{where}: lse off by {dl.max():.3e}"


def _wide_range_q(w: W.Workload, seed: int) -> np.ndarray:
    """Per (request, head) one of four query rows: (0) one entry of +-300 at
    a random channel, every other entry N(0, 1e-3); (1) largest entry 1,
    the others +-2^-u with u uniform in [10, 16]; (2) all zero; (3) N(0, 1)."""
    g = np.random.default_rng(seed)
    B, H = w.batch, w.heads
    q = np.zeros((B, H, 576), np.float32)
    kind = np.arange(B * H).reshape(B, H) % 4
    for b in range(B):
        for h in range(H):
            if kind[b, h] == 0:
                q[b, h] = g.normal(0, 1e-3, 576)
                q[b, h, g.integers(576)] = 300.0 * g.choice([-1, 1])
            elif kind[b, h] == 1:
                q[b, h] = g.choice([-1, 1], 576) * np.exp2(-g.uniform(10, 16, 576))
                q[b, h, g.integers(576)] = 1.0
            elif kind[b, h] == 3:
                q[b, h] = g.standard_normal(576)
    return q


def test_wide_range_and_zero_queries_concurrency_full_size():
    w = W.make_workload("concurrency")
    q = _wide_range_q(w, 63)
    w.q_bf16 = _bf16(q)
    pool = oracle_pool(w)
    out, lse = _gpu(w, pool)
    o_ref, lse_ref = _oracle_decode(w, pool)
    check_attention(out, lse, o_ref, lse_ref, "wide-range q")
    _tight(out, lse, o_ref, lse_ref, "wide-range q")
    # zero rows: every score is 0, so lse = ln L exactly (the closed form)
    zero = np.all(q == 0, axis=2)
    assert zero.sum() == w.batch * w.heads // 4
    ln_l = np.log(w.seq_lens.astype(np.float64))[:, None].repeat(w.heads, 1)
    assert np.abs(lse.cpu().numpy()[zero] - ln_l[zero]).max() <= 1e-3


def test_wide_range_queries_large_head_sampled():
    sample = [5, 77, 126]
    w = W.make_workload("large_head", latent_requests=sample)
    w.q_bf16 = _bf16(_wide_range_q(w, 64))
    pool = oracle_pool(w)
    out, lse = _gpu(w, pool)
    o_ref, lse_ref = _oracle_decode(w, pool, sel=np.array(sample))
    sel = torch.tensor(sample, device="cuda")
    check_attention(out[sel], lse[sel], o_ref, lse_ref, "wide-range q, H = 128")
    _tight(out[sel], lse[sel], o_ref, lse_ref, "wide-range q, H = 128")


def test_wide_range_queries_extend():
    w = W.make_extend_workload("concurrency", q_lens=[3, 1, 4, 2], batch=4, num_slots=60_000,
                               seed=65)
    n_q = int(w.extra["qo_indptr"][-1])
    g = np.random.default_rng(66)
    q = g.normal(0, 1e-3, (n_q, w.heads, 576)).astype(np.float32)
    q[np.arange(n_q)[:, None], np.arange(w.heads)[None, :], g.integers(576, size=(n_q, w.heads))] = 300.0
    w.q_bf16 = _bf16(q)
    pool = oracle_pool(w)
    o_ref, lse_ref = oracle.extend_fp8(w.q_bf16, pool[:, :512], pool[:, 512:],
                                       w.extra["qo_indptr"], w.kv_indptr, w.kv_indices,
                                       w.seq_lens, w.page_size, w.k_scale, w.softmax_scale)
    dpool = torch.from_numpy(pool).cuda()
    qo = w.extra["qo_indptr"]
    plan = M.mla_extend_plan(qo, w.kv_indptr, w.seq_lens, w.batch, w.heads, w.page_size)
    out = torch.full((n_q, w.heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((n_q, w.heads), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    M.mla_extend_run(plan, dev_bf16(w.q_bf16), dpool[:, :512], dpool[:, 512:], w.num_slots,
                     dev_i32(w.kv_indptr), dev_i32(w.kv_indices), dev_i32(w.seq_lens),
                     w.k_scale, w.softmax_scale, out, lse, ws)
    assert M.mla_get_last_error() == 0
    check_attention(out, lse, o_ref, lse_ref, "wide-range q, extend")
    _tight(out, lse, o_ref, lse_ref, "wide-range q, extend")


# ------------------------------------------------------------ small weights

@pytest.mark.parametrize("gap_log2", [12.0, 14.0, 15.5, 17.0])
def test_attention_sink_small_weights_reach_the_output(gap_log2):
    """Token 0 of each request scores gap_log2 log2 units above the other
    ~4,000 tokens, whose weights (2^-gap each) add up to 3-25 % of the
    sink's, and whose c_kv channels 1-64 sit 1.0 above the sink's: output
    channels 1-64 are then about the tail's share of the weight, which a
    kernel that dropped weights below 2^-14 of the maximum would lose."""
    w = W.make_workload("concurrency", batch=6, lens=[4096, 3000, 5000, 4500, 3500, 4096],
                        num_slots=60_000, seed=67)
    lat = W.bf16_bits_to_float(w.latent_bf16).copy()
    tok = _token_index(w, range(w.batch))
    lat[tok == 0, 0] = 200.0
    lat[tok != 0, 1:65] += 1.0
    _set_latents(w, lat)
    g = np.random.default_rng(68)
    q = g.normal(0, 0.05, (w.batch, w.heads, 576)).astype(np.float32)
    # sink score - typical score = softmax_scale * q0 * 200 (natural log)
    q[:, :, 0] = gap_log2 * np.log(2.0) / (w.softmax_scale * 200.0)
    w.q_bf16 = _bf16(q)
    pool = oracle_pool(w)
    out, lse = _gpu(w, pool)
    o_ref, lse_ref = _oracle_decode(w, pool)
    check_attention(out, lse, o_ref, lse_ref, f"sink, gap {gap_log2}")


# ------------------------------------------------------ non-finite queries

def test_nonfinite_query_rows_give_nan_rows_only():
    w = W.make_workload("concurrency", batch=3, lens=[300, 2000, 77], num_slots=10_000, seed=69)
    q = W.bf16_bits_to_float(w.q_bf16).copy()
    q[0, 3, 5] = np.inf
    q[1, 7, 100] = np.nan
    q[2, 0, 575] = -np.inf
    w.q_bf16 = _bf16(q)
    pool = oracle_pool(w)
    out, lse = _gpu(w, pool)
    o_ref, lse_ref = _oracle_decode(w, pool)
    bad = np.zeros((w.batch, w.heads), bool)
    bad[0, 3] = bad[1, 7] = bad[2, 0] = True
    assert np.all(np.isnan(o_ref[bad])) and np.all(np.isnan(lse_ref[bad]))
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    assert np.all(np.isnan(o[bad])) and np.all(np.isnan(l[bad]))
    assert not np.isnan(o[~bad]).any() and not np.isnan(l[~bad]).any()
    keep = torch.from_numpy(~bad).cuda()
    check_attention(out[keep], lse[keep], o_ref[~bad], lse_ref[~bad], "finite heads")
