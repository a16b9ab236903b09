"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Store and gather-cast must be bit-exact; decode must be within
|err| <= 1e-2 + 1e-2 |ref| on the BF16 output and 1e-3 on the LSE (the
precision the method states for a BF16 output over an FP8 cache)."""
import numpy as np
import pytest
import torch

import mla_decode_attention_run_gb300 as M
import oracle
import workloads as W
from gpu_util import bf16_bits, check_attention, dev_bf16, dev_i32, gpu_decode, oracle_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    M.mla_get_last_error()       # clear flags left by anything earlier


# ------------------------------------------------------------ quantize-on-store

@pytest.mark.parametrize("k_scale", [1.0, 0.00634765625, 3.0 / 448.0, 7.0, 2.0 ** -12])
def test_store_bitexact_on_every_bf16_pattern(k_scale):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    rows = (bits.size + 575) // 576
    lat = np.zeros(rows * 576, np.uint16)
    lat[:bits.size] = bits
    lat = lat.reshape(rows, 576)
    g = np.random.default_rng(1)
    P = 400
    slots = g.permutation(P)[:rows].astype(np.int64)
    pool0 = W.random_fill_bytes(g, (P, 576))
    ref = pool0.copy()
    oracle.kv_store_fp8(lat[:, :512], lat[:, 512:], slots, k_scale, ref[:, :512], ref[:, 512:])
    pool = torch.from_numpy(pool0).cuda()
    lat_d = dev_bf16(lat)
    M.kv_store_fp8(lat_d[:, :512].contiguous(), lat_d[:, 512:].contiguous(),
                   torch.from_numpy(slots).cuda(), k_scale, pool[:, :512], pool[:, 512:])
    assert M.mla_get_last_error() == 0
    got = pool.cpu().numpy()
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{bad.shape[0]} bytes differ, first at {bad[:3]}"


def test_store_separate_padded_pools_and_oob_slot():
    g = np.random.default_rng(2)
    n, P = 37, 90
    lat = bf16_bits((torch.randn(n, 576) * 0.3).to(torch.bfloat16))
    slots = g.permutation(P)[:n].astype(np.int64)
    slots[5] = P                                    # out of range: skipped and flagged
    ckv0 = W.random_fill_bytes(g, (P, 544))         # row stride 544
    kpe0 = W.random_fill_bytes(g, (P, 80))          # row stride 80
    ref_ckv, ref_kpe = ckv0.copy(), kpe0.copy()
    bad = oracle.kv_store_fp8(lat[:, :512], lat[:, 512:], slots, 0.0041, ref_ckv[:, :512],
                              ref_kpe[:, :64])
    assert bad == 1
    ckv, kpe = torch.from_numpy(ckv0).cuda(), torch.from_numpy(kpe0).cuda()
    lat_d = dev_bf16(lat)
    M.kv_store_fp8(lat_d[:, :512].contiguous(), lat_d[:, 512:].contiguous(),
                   torch.from_numpy(slots).cuda(), 0.0041, ckv[:, :512], kpe[:, :64],
                   num_pool_slots=P)
    assert M.mla_get_last_error() == M.FLAG_INDEX_OOB
    assert np.array_equal(ckv.cpu().numpy(), ref_ckv)
    assert np.array_equal(kpe.cpu().numpy(), ref_kpe)


# ------------------------------------------------------------------ gather-cast

@pytest.mark.parametrize("page_size,k_scale", [(1, 1.0), (1, 0.00634765625), (64, 1.0),
                                               (3, 0.37)])
def test_gather_cast_bitexact(page_size, k_scale):
    g = np.random.default_rng(3)
    pages = 300
    pool0 = W.random_fill_bytes(g, (pages * page_size, 576))
    idx = g.permutation(pages)[:211].astype(np.int32)
    ref_ckv, ref_kpe = oracle.kv_gather_cast(pool0[:, :512], pool0[:, 512:], idx, page_size,
                                             k_scale)
    pool = torch.from_numpy(pool0).cuda()
    n = idx.size * page_size
    ck = torch.empty(n, 512, dtype=torch.bfloat16, device="cuda")
    kp = torch.empty(n, 64, dtype=torch.bfloat16, device="cuda")
    M.kv_gather_cast(pool[:, :512], pool[:, 512:], dev_i32(idx), page_size, k_scale, ck, kp)
    assert M.mla_get_last_error() == 0
    assert np.array_equal(bf16_bits(ck), ref_ckv)
    assert np.array_equal(bf16_bits(kp), ref_kpe)


@pytest.mark.parametrize("page_size,k_scale", [(1, 1.0), (3, 0.37), (1, 2.0 ** -7)])
def test_gather_cast_bitexact_on_every_byte_including_nan(page_size, k_scale):
    """Pools holding all 256 byte values, the NaN codes 0x7F and 0xFF
    included, in every channel position: bit-exact with the oracle (NaN ->
    0x7FC0)."""
    g = np.random.default_rng(41)
    pages = 120
    rows = pages * page_size
    pool0 = ((np.arange(rows * 576, dtype=np.int64) * 7 + 3) % 256).astype(np.uint8).reshape(rows, 576)
    pool0 = pool0[g.permutation(rows)]
    assert np.count_nonzero((pool0 & 0x7F) == 0x7F) > 100
    idx = g.permutation(pages)[:97].astype(np.int32)
    ref_ckv, ref_kpe = oracle.kv_gather_cast(pool0[:, :512], pool0[:, 512:], idx, page_size,
                                             k_scale)
    pool = torch.from_numpy(pool0).cuda()
    n = idx.size * page_size
    ck = torch.empty(n, 512, dtype=torch.bfloat16, device="cuda")
    kp = torch.empty(n, 64, dtype=torch.bfloat16, device="cuda")
    M.kv_gather_cast(pool[:, :512], pool[:, 512:], dev_i32(idx), page_size, k_scale, ck, kp)
    assert M.mla_get_last_error() == 0
    assert np.array_equal(bf16_bits(ck), ref_ckv)
    assert np.array_equal(bf16_bits(kp), ref_kpe)


def test_gather_cast_equals_torch_cast_at_unit_scale():
    """With k_scale = 1 the gather-cast of every page equals the pages'
    full-pool .to(bfloat16) restricted to those rows."""
    g = np.random.default_rng(4)
    pool = torch.from_numpy(W.random_fill_bytes(g, (5000, 576))).cuda()
    idx = torch.from_numpy(g.permutation(5000)[:1234].astype(np.int32)).cuda()
    ck = torch.empty(1234, 512, dtype=torch.bfloat16, device="cuda")
    kp = torch.empty(1234, 64, dtype=torch.bfloat16, device="cuda")
    M.kv_gather_cast(pool[:, :512], pool[:, 512:], idx, 1, 1.0, ck, kp)
    full = pool.view(torch.float8_e4m3fn).to(torch.bfloat16)
    assert torch.equal(ck, full[idx.long(), :512]) and torch.equal(kp, full[idx.long(), 512:])


def test_gather_cast_oob_page_flagged():
    pool = torch.zeros(64, 576, dtype=torch.uint8, device="cuda")
    idx = dev_i32([3, 64, 5])
    ck = torch.full((3, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    kp = torch.full((3, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    M.kv_gather_cast(pool[:, :512], pool[:, 512:], idx, 1, 1.0, ck, kp)
    assert M.mla_get_last_error() == M.FLAG_INDEX_OOB
    assert torch.all(ck[1] == 7.0) and torch.all(ck[0] == 0) and torch.all(ck[2] == 0)


# ----------------------------------------------------------------------- decode

def _decode_case(w, pool_np, **kw):
    pool = torch.from_numpy(pool_np).cuda()
    out, lse, plan = gpu_decode(w, pool[:, :512], pool[:, 512:], **kw)
    flags = M.mla_get_last_error()
    return out, lse, flags


def test_decode_tiny_config():
    w = W.make_workload("tiny")
    pool = oracle_pool(w)
    out, lse, flags = _decode_case(w, pool)
    assert flags == 0
    o_ref, lse_ref = oracle.decode_fp8(w.q_bf16, pool[:, :512], pool[:, 512:], w.kv_indptr,
                                       w.kv_indices, w.seq_lens, 1, w.k_scale, w.softmax_scale)
    check_attention(out, lse, o_ref, lse_ref, "tiny")


def test_decode_single_stream_full_size():
    w = W.make_workload("single")
    pool = oracle_pool(w)
    out, lse, flags = _decode_case(w, pool)
    assert flags == 0
    o_ref, lse_ref = oracle.decode_fp8(w.q_bf16, pool[:, :512], pool[:, 512:], w.kv_indptr,
                                       w.kv_indices, w.seq_lens, 1, w.k_scale, w.softmax_scale)
    check_attention(out, lse, o_ref, lse_ref, "single")


def test_decode_concurrency_full_size():
    """Batch 40, contexts U[1024, 8192], full 495,552-slot pool, every output
    element against the oracle."""
    w = W.make_workload("concurrency")
    pool = oracle_pool(w)
    out, lse, flags = _decode_case(w, pool)
    assert flags == 0
    o_ref, lse_ref = oracle.decode_fp8(w.q_bf16, pool[:, :512], pool[:, 512:], w.kv_indptr,
                                       w.kv_indices, w.seq_lens, 1, w.k_scale, w.softmax_scale)
    check_attention(out, lse, o_ref, lse_ref, "concurrency")


def test_decode_large_head_full_size_sampled():
    """Batch 128 x 32,768 tokens, H = 128, page size 64 (2.4 GB pool): the
    launch is full size; 6 requests carry oracle-encoded latents and are
    compared in full (all heads)."""
    sample = [0, 17, 63, 64, 101, 127]
    w = W.make_workload("large_head", latent_requests=sample)
    pool = oracle_pool(w)
    out, lse, flags = _decode_case(w, pool)
    assert flags == 0
    sel = np.array(sample)
    indptr = np.zeros(len(sel) + 1, np.int32)
    idx = []
    for i, b in enumerate(sel):
        idx.append(w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]])
        indptr[i + 1] = indptr[i] + idx[-1].size
    o_ref, lse_ref = oracle.decode_fp8(np.ascontiguousarray(w.q_bf16[sel]), pool[:, :512],
                                       pool[:, 512:], indptr, np.concatenate(idx),
                                       w.seq_lens[sel], 64, w.k_scale, w.softmax_scale)
    check_attention(out[torch.from_numpy(sel).cuda()], lse[torch.from_numpy(sel).cuda()],
                    o_ref, lse_ref, "large_head")


@pytest.mark.parametrize("heads,ps,lens", [
    (1, 1, [1, 2, 3]),
    (4, 3, [0, 65, 64, 63, 1]),
    (16, 1, [129, 0, 7]),
    (16, 64, [1, 4096, 130]),
    (32, 2, [300, 77]),
    (48, 1, [513]),
    (64, 1, [2000, 5, 700, 64]),                   # 32-head CTAs in two head groups
    (96, 8, [777, 64, 1, 130]),                    # three 32-head groups, paged
    (128, 64, [1000, 64, 3]),
])
def test_decode_edge_shapes(heads, ps, lens):
    w = W.make_workload("concurrency", batch=len(lens), heads=heads, lens=lens, page_size=ps,
                        num_slots=6000 * ps // ps * 1 if ps == 1 else 200 * ps, seed=77 + heads)
    pool = oracle_pool(w, fill_seed=heads)
    out, lse, flags = _decode_case(w, pool)
    assert flags == 0
    o_ref, lse_ref = oracle.decode_fp8(w.q_bf16, pool[:, :512], pool[:, 512:], w.kv_indptr,
                                       w.kv_indices, w.seq_lens, ps, w.k_scale, w.softmax_scale)
    check_attention(out, lse, o_ref, lse_ref, f"H={heads} ps={ps} lens={lens}")


@pytest.mark.parametrize("heads", [16, 64, 128])
def test_decode_strided_q_and_separate_pools(heads):
    """Padded c_kv and k_pe pools of their own, at 16 heads and at 64 and
    128 (32-head CTAs, two and four head groups per token range)."""
    w = W.make_workload("concurrency", batch=3, heads=heads, lens=[200, 1, 777], num_slots=3000,
                        seed=5)
    pool = oracle_pool(w)
    ckv0 = np.zeros((w.num_slots, 528), np.uint8)
    kpe0 = np.zeros((w.num_slots, 96), np.uint8)
    ckv0[:, :512] = pool[:, :512]
    kpe0[:, :64] = pool[:, 512:]
    ckv, kpe = torch.from_numpy(ckv0).cuda(), torch.from_numpy(kpe0).cuda()
    big = torch.zeros(3, 2 * w.heads, 600, dtype=torch.bfloat16, device="cuda")
    big[:, ::2, :576] = dev_bf16(w.q_bf16)
    q = big[:, ::2, :576]                       # strides (2*H*600, 1200, 1)
    out, lse, _ = gpu_decode(w, ckv[:, :512], kpe[:, :64], q=q)
    assert M.mla_get_last_error() == 0
    o_ref, lse_ref = oracle.decode_fp8(w.q_bf16, pool[:, :512], pool[:, 512:], w.kv_indptr,
                                       w.kv_indices, w.seq_lens, 1, w.k_scale, w.softmax_scale)
    check_attention(out, lse, o_ref, lse_ref, f"strided H={heads}")


def test_decode_many_short_requests_past_the_segment_table():
    """12,000 requests of 1-99 tokens: every 16-head CTA serves 73-82
    segments, more than the 64 it keeps in shared memory, so it reads the
    rest from the plan as it reaches them."""
    B = 12000
    lens = np.random.default_rng(5).integers(1, 100, B)
    w = W.make_workload("concurrency", batch=B, heads=16, lens=list(lens), num_slots=650000, seed=91)
    sched, info = M.mla_decode_schedule(w.kv_indptr, w.seq_lens, B, 16, 1, M.MLA_KV_FP8_E4M3)
    per_cta = np.bincount(np.asarray(sched)[:, 0])
    assert info["kernel"] == 1 and per_cta.min() > 64
    pool = oracle_pool(w)
    out, lse, flags = _decode_case(w, pool)
    assert flags == 0
    o_ref, lse_ref = oracle.decode_fp8(w.q_bf16, pool[:, :512], pool[:, 512:], w.kv_indptr,
                                       w.kv_indices, w.seq_lens, 1, w.k_scale, w.softmax_scale)
    check_attention(out, lse, o_ref, lse_ref, "12,000 short requests")


def test_decode_is_deterministic():
    w = W.make_workload("concurrency", batch=6, num_slots=60000, seed=9)
    pool = torch.from_numpy(oracle_pool(w)).cuda()
    o1, l1, _ = gpu_decode(w, pool[:, :512], pool[:, 512:])
    o2, l2, _ = gpu_decode(w, pool[:, :512], pool[:, 512:])
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_out_of_range_index_is_excluded_and_flagged():
    w = W.make_workload("concurrency", batch=2, lens=[100, 50], num_slots=1000, seed=11)
    pool = oracle_pool(w)
    bad = w.kv_indices.copy()
    bad[10] = 5000                                  # request 0, token 10
    out, lse, flags = _decode_case(w, pool, kv_indices=bad)
    assert flags & M.FLAG_INDEX_OOB
    keep = np.delete(w.kv_indices, 10)
    lens = w.seq_lens.copy()
    lens[0] -= 1
    indptr = np.array([0, lens[0], lens[0] + lens[1]], np.int32)
    o_ref, lse_ref = oracle.decode_fp8(w.q_bf16, pool[:, :512], pool[:, 512:], indptr, keep, lens,
                                       1, w.k_scale, w.softmax_scale)
    check_attention(out, lse, o_ref, lse_ref, "oob excluded")


def test_decode_plan_mismatch_flagged():
    w = W.make_workload("concurrency", batch=2, lens=[100, 50], num_slots=1000, seed=12)
    pool = torch.from_numpy(oracle_pool(w)).cuda()
    plan = M.mla_decode_plan(w.kv_indptr, w.seq_lens, 2, 16, 1)
    out = torch.empty(2, 16, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(2, 16, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    short = w.seq_lens.copy()
    short[0] = 20                                  # device lengths shorter than planned
    M.mla_decode_run(plan, dev_bf16(w.q_bf16), pool[:, :512], pool[:, 512:], 1000,
                     dev_i32(w.kv_indptr), dev_i32(w.kv_indices), dev_i32(short), w.k_scale,
                     w.softmax_scale, out, lse, ws)
    assert M.mla_get_last_error() & M.FLAG_PLAN_MISMATCH


def test_decode_rejects_small_workspace():
    w = W.make_workload("concurrency", batch=1, lens=[8192], num_slots=9000, seed=13)
    pool = torch.zeros(9000, 576, dtype=torch.uint8, device="cuda")
    plan = M.mla_decode_plan(w.kv_indptr, w.seq_lens, 1, 16, 1)
    assert plan.workspace_bytes > 0
    out = torch.empty(1, 16, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 16, dtype=torch.float32, device="cuda")
    ws = torch.empty(plan.workspace_bytes - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.MLAError) as e:
        M.mla_decode_run(plan, dev_bf16(w.q_bf16), pool[:, :512], pool[:, 512:], 9000,
                         dev_i32(w.kv_indptr), dev_i32(w.kv_indices), dev_i32(w.seq_lens),
                         w.k_scale, w.softmax_scale, out, lse, ws)
    assert e.value.status == 3


def test_plan_rebuilt_in_place_across_steps():
    """One plan handle reused over growing contexts (a decode step appends a
    token per request)."""
    w = W.make_workload("concurrency", batch=4, lens=[100, 300, 64, 5], num_slots=4000, seed=14)
    pool_np = oracle_pool(w)
    pool = torch.from_numpy(pool_np).cuda()
    plan = None
    for step in range(3):
        lens = w.seq_lens - 2 + step
        indptr = np.zeros(5, np.int32)
        indptr[1:] = np.cumsum(lens)
        idx = np.concatenate([w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b] + lens[b]]
                              for b in range(4)])
        out, lse, plan = gpu_decode(w, pool[:, :512], pool[:, 512:], kv_indptr=indptr,
                                    kv_indices=idx, seq_lens=lens, plan=plan)
        o_ref, lse_ref = oracle.decode_fp8(w.q_bf16, pool_np[:, :512], pool_np[:, 512:], indptr,
                                           idx, lens, 1, w.k_scale, w.softmax_scale)
        check_attention(out, lse, o_ref, lse_ref, f"step {step}")
    assert M.mla_get_last_error() == 0


# ----------------------------------------------------- the two baselines' paths

def test_gather_then_cast_then_bf16_decode():
    """Baseline 2: gather-cast the active pages (k_scale 1), replan with
    sequential indices, BF16 decode with k_scale applied in attention."""
    w = W.make_workload("concurrency", batch=8, num_slots=W.POOL_SLOTS, seed=15)
    pool_np = oracle_pool(w)
    pool = torch.from_numpy(pool_np).cuda()
    n = w.kv_indices.size
    ck = torch.empty(n, 512, dtype=torch.bfloat16, device="cuda")
    kp = torch.empty(n, 64, dtype=torch.bfloat16, device="cuda")
    M.kv_gather_cast(pool[:, :512], pool[:, 512:], dev_i32(w.kv_indices), 1, 1.0, ck, kp)
    seq_idx = np.arange(n, dtype=np.int32)
    out, lse, _ = gpu_decode(w, ck, kp, kv_dtype=M.MLA_KV_BF16, kv_indices=seq_idx)
    assert M.mla_get_last_error() == 0
    o_ref, lse_ref = oracle.decode_fp8(w.q_bf16, pool_np[:, :512], pool_np[:, 512:], w.kv_indptr,
                                       w.kv_indices, w.seq_lens, 1, w.k_scale, w.softmax_scale)
    check_attention(out, lse, o_ref, lse_ref, "gather-then-cast")


def test_full_pool_cast_then_bf16_decode():
    """Baseline 1: the pages' full-pool .to(bfloat16), then BF16 decode on
    the original indices."""
    w = W.make_workload("concurrency", batch=4, num_slots=W.POOL_SLOTS, seed=16)
    pool_np = oracle_pool(w)
    pool = torch.from_numpy(pool_np).cuda()
    full = pool.view(torch.float8_e4m3fn).to(torch.bfloat16)
    out, lse, _ = gpu_decode(w, full[:, :512], full[:, 512:], kv_dtype=M.MLA_KV_BF16)
    assert M.mla_get_last_error() == 0
    o_ref, lse_ref = oracle.decode_fp8(w.q_bf16, pool_np[:, :512], pool_np[:, 512:], w.kv_indptr,
                                       w.kv_indices, w.seq_lens, 1, w.k_scale, w.softmax_scale)
    check_attention(out, lse, o_ref, lse_ref, "full-pool cast")


def test_fp8_tensor_core_path_precision():
    """The FP8 tensor-core kernel (E4M3 cache bytes as MMA operands, q and P
    each split exactly into two E4M3 terms) is checked against the oracle at
    a bound four times tighter than the contract: a lost second term (about
    2^-5 relative in P, 2^-4 in q) would fail it."""
    w = W.make_workload("concurrency", batch=12, num_slots=W.POOL_SLOTS, seed=31)
    segs, info = M.mla_decode_schedule(w.kv_indptr, w.seq_lens, w.batch, w.heads, 1)
    assert info["kernel"] == 1                       # the tcgen05 kernel serves this plan
    pool = oracle_pool(w)
    out, lse, flags = _decode_case(w, pool)
    assert flags == 0
    o_ref, lse_ref = oracle.decode_fp8(w.q_bf16, pool[:, :512], pool[:, 512:], w.kv_indptr,
                                       w.kv_indices, w.seq_lens, 1, w.k_scale, w.softmax_scale)
    o = out.float().cpu().numpy()
    assert np.all(np.abs(o - o_ref) <= 2.5e-3 + 2.5e-3 * np.abs(o_ref))
    assert np.all(np.abs(lse.cpu().numpy() - lse_ref) <= 2.5e-4)
