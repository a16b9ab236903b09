"""GPU parity of causal extend attention (several new tokens per request)
through the C ABI against the CPU oracle, within the decode tolerance
(|err| <= 1e-2 + 1e-2 |ref| on the BF16 output, 1e-3 on the LSE)."""
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


def gpu_extend(w: W.Workload, ckv, kpe, qo=None, plan=None):
    dev = ckv.device
    qo = w.extra["qo_indptr"] if qo is None else qo
    plan = M.mla_extend_plan(qo, w.kv_indptr, w.seq_lens, w.batch, w.heads, w.page_size,
                             plan=plan)
    n_q = int(qo[-1])
    q = dev_bf16(w.q_bf16, dev)
    out = torch.full((n_q, w.heads, 512), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((n_q, w.heads), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    M.mla_extend_run(plan, q, ckv, kpe, ckv.shape[0], dev_i32(w.kv_indptr, dev),
                     dev_i32(w.kv_indices, dev), dev_i32(w.seq_lens, dev), w.k_scale,
                     w.softmax_scale, out, lse, ws)
    return out, lse, plan


def _run_case(w: W.Workload, where: str):
    pool = oracle_pool(w)
    o_ref, lse_ref = oracle.extend_fp8(w.q_bf16, pool[:, :512], pool[:, 512:],
                                       w.extra["qo_indptr"], w.kv_indptr, w.kv_indices,
                                       w.seq_lens, w.page_size, w.k_scale, w.softmax_scale)
    dpool = torch.from_numpy(pool).cuda()
    out, lse, plan = gpu_extend(w, dpool[:, :512], dpool[:, 512:])
    assert M.mla_get_last_error() == 0
    check_attention(out, lse, o_ref, lse_ref, where)
    return out, lse, plan


@pytest.mark.parametrize("heads,lens,q_lens,ps", [
    (16, [100, 300, 65, 1000], [4, 64, 65, 1], 1),     # ragged, a pure prefill (65 of 65)
    (16, [3000, 2500], [2, 3], 1),                     # speculative-style, split contexts
    (4, [40, 17, 33], [0, 17, 5], 1),                  # padded blocks, a request with no new token
    (128, [700, 300], [3, 1], 64),                     # 32-row blocks over 4 head groups, paged
    (16, [130, 200], [130, 77], 16),                   # the causal edge inside and across tiles
    (32, [513, 64], [40, 64], 1),
])
def test_extend_matches_oracle(heads, lens, q_lens, ps):
    w = W.make_extend_workload("tiny", q_lens, batch=len(lens), heads=heads, lens=lens,
                               page_size=ps, num_slots=max(sum(lens) * 2, 128) // ps * ps + ps,
                               std=0.5, k_scale=None)
    _run_case(w, f"H={heads} lens={lens} q={q_lens}")


def test_extend_splits_long_blocks_across_ctas():
    """Few blocks, long contexts: every block is split, and rows whose causal
    limit lies before a later segment get an empty partial (lse -inf) that the
    merge must weigh 0."""
    w = W.make_extend_workload("single", 7, batch=1, lens=[4096])
    _, _, plan = _run_case(w, "split")
    assert M.mla_decode_plan_info(plan)["num_partials"] > 1


def test_one_new_token_is_bitwise_the_decode_call():
    w = W.make_extend_workload("tiny", 1, batch=5, heads=16, lens=[1000, 77, 4096, 1, 300],
                               num_slots=8192, std=0.5)
    pool = torch.from_numpy(oracle_pool(w)).cuda()
    out_e, lse_e, _ = gpu_extend(w, pool[:, :512], pool[:, 512:])
    out_d, lse_d, _ = gpu_decode(w, pool[:, :512], pool[:, 512:], q=dev_bf16(w.q_bf16))
    assert torch.equal(out_e.view(torch.int16), out_d.view(torch.int16))
    assert torch.equal(lse_e, lse_d)


def test_plans_are_not_interchangeable():
    w = W.make_extend_workload("tiny", 2, batch=2, heads=4, lens=[17, 33])
    pool = torch.from_numpy(oracle_pool(w)).cuda()
    _, _, eplan = gpu_extend(w, pool[:, :512], pool[:, 512:])
    q = dev_bf16(w.q_bf16)
    out = torch.empty((4, 4, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((4, 4), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(eplan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    with pytest.raises(M.MLAError) as e:
        M.mla_decode_run(eplan, q, pool[:, :512], pool[:, 512:], pool.shape[0],
                         dev_i32(w.kv_indptr), dev_i32(w.kv_indices), dev_i32(w.seq_lens),
                         w.k_scale, w.softmax_scale, out, lse, ws)
    assert e.value.status == 1
    dplan = M.mla_decode_plan(w.kv_indptr, w.seq_lens, 2, 4, 1)
    with pytest.raises(M.MLAError) as e:
        M.mla_extend_run(dplan, q, pool[:, :512], pool[:, 512:], pool.shape[0],
                         dev_i32(w.kv_indptr), dev_i32(w.kv_indices), dev_i32(w.seq_lens),
                         w.k_scale, w.softmax_scale, out, lse, ws)
    assert e.value.status == 1


@pytest.mark.parametrize("name,requests", [("spec_decode", [0, 17, 39]), ("extend_chunk", [2])])
def test_extend_full_size_sampled(name, requests):
    """The bench's extend workloads at full size, in the bench's launch
    configuration; the oracle checks every row of the sampled requests."""
    w = W.make_extend_workload(name, latent_requests=requests)
    pool = oracle_pool(w)
    dpool = torch.from_numpy(pool).cuda()
    out, lse, _ = gpu_extend(w, dpool[:, :512], dpool[:, 512:])
    assert M.mla_get_last_error() == 0
    qo = w.extra["qo_indptr"]
    for b in requests:
        sub_indptr = np.array([0, w.kv_indptr[b + 1] - w.kv_indptr[b]], np.int32)
        sub_idx = w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]]
        sub_qo = np.array([0, qo[b + 1] - qo[b]], np.int32)
        o_ref, lse_ref = oracle.extend_fp8(w.q_bf16[qo[b]:qo[b + 1]], pool[:, :512],
                                           pool[:, 512:], sub_qo, sub_indptr, sub_idx,
                                           w.seq_lens[b:b + 1], w.page_size, w.k_scale,
                                           w.softmax_scale)
        check_attention(out[qo[b]:qo[b + 1]], lse[qo[b]:qo[b + 1]], o_ref, lse_ref,
                        f"{name} request {b}")


def test_long_prefill_sampled_rows():
    """A 1,024-token prefill (no cached prefix): 512 blocks of 32 rows, split
    over the CTAs; sampled new tokens (first, tile edges, last) against the
    oracle's decode over each token's visible prefix."""
    L = 1024
    w = W.make_extend_workload("single", L, batch=1, lens=[L], num_slots=4096, std=0.5)
    pool = oracle_pool(w)
    dpool = torch.from_numpy(pool).cuda()
    out, lse, plan = gpu_extend(w, dpool[:, :512], dpool[:, 512:])
    assert M.mla_get_last_error() == 0
    assert M.mla_decode_plan_info(plan)["num_ctas"] > 100
    for i in (0, 1, 63, 64, 65, 127, 500, 1022, 1023):
        visible = i + 1
        o_ref, lse_ref = oracle.decode_fp8(w.q_bf16[i:i + 1], pool[:, :512], pool[:, 512:],
                                           np.array([0, visible], np.int32),
                                           w.kv_indices[:visible], np.array([visible], np.int32),
                                           1, w.k_scale, w.softmax_scale)
        check_attention(out[i:i + 1], lse[i:i + 1], o_ref, lse_ref, f"prefill token {i}")
