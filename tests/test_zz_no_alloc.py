"""mla_decode_run_static_scratch: the decode call for callers that cannot
allocate device memory (a plugin inside a framework that owns all GPU
memory, a loop that must not pay cudaMalloc's implicit synchronisation).
It keeps the split-KV partials in a fixed array inside the library instead
of a caller workspace.  These tests check that it gives the same answer as
mla_decode_run with a workspace, twice in a row (the array is reused and
keeps the previous call's contents), and that plans needing more scratch
than the array holds are refused.

This file is named to be collected last, so that a run stopping at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import mla_decode_attention_run_gb300 as M
import workloads as W
from gpu_util import ATOL, LSE_TOL, RTOL, dev_bf16, dev_i32, oracle_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    M.mla_get_last_error()


def _identical(out, lse, ref_out, ref_lse):
    """Both calls run the same deterministic kernels on the same plan and
    inputs, only with the scratch elsewhere: the results agree bit for bit
    (which is also within the attention tolerance the other tests use)."""
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
    o, r = out.float().cpu().numpy(), ref_out.float().cpu().numpy()
    assert np.all(np.abs(o - r) <= ATOL + RTOL * np.abs(r))
    assert np.all(np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy()) <= LSE_TOL)


def test_static_scratch_matches_workspace_call_twice_in_a_row():
    w = W.make_workload("concurrency", batch=8, num_slots=100_000, seed=21)
    pool = torch.from_numpy(oracle_pool(w)).cuda()
    ckv, kpe = pool[:, :512], pool[:, 512:]
    q = dev_bf16(w.q_bf16)
    indptr, idx, lens = dev_i32(w.kv_indptr), dev_i32(w.kv_indices), dev_i32(w.seq_lens)
    plan = M.mla_decode_plan(w.kv_indptr, w.seq_lens, w.batch, w.heads, 1)
    # the split-KV partials really go through scratch in this case
    assert 0 < plan.workspace_bytes <= M.STATIC_SCRATCH_BYTES

    ref_out = torch.empty(w.batch, w.heads, 512, dtype=torch.bfloat16, device="cuda")
    ref_lse = torch.empty(w.batch, w.heads, dtype=torch.float32, device="cuda")
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    M.mla_decode_run(plan, q, ckv, kpe, w.num_slots, indptr, idx, lens, w.k_scale,
                     w.softmax_scale, ref_out, ref_lse, ws)
    for _ in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        M.mla_decode_run_static_scratch(plan, q, ckv, kpe, w.num_slots, indptr, idx, lens,
                                        w.k_scale, w.softmax_scale, out, lse)
        assert M.mla_get_last_error() == 0
        _identical(out, lse, ref_out, ref_lse)
    M.mla_decode_plan_destroy(plan)


def test_static_scratch_refuses_plans_that_need_more():
    """A plan whose scratch exceeds the array is refused with status 3 before
    any launch, and one that fits is accepted.  The plan's scratch depends on
    the GPU's SM count, so which of the two shapes needs more is read from
    the plans (on a 152-SM GPU the 128-head, 128 x 32,768-token one does)."""
    tiny = torch.zeros(64, 576, dtype=torch.uint8, device="cuda")
    q = torch.zeros(128, 128, 576, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(128, 128, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(128, 128, dtype=torch.float32, device="cuda")
    refused = expected = 0
    for lens, heads, ps in (([32768] * 128, 128, 64), ([5000, 3000], 16, 1)):
        lens = np.asarray(lens, np.int32)
        indptr = np.zeros(len(lens) + 1, np.int32)
        indptr[1:] = np.cumsum((lens + ps - 1) // ps)
        plan = M.mla_decode_plan(indptr, lens, len(lens), heads, ps)
        expected += plan.workspace_bytes > M.STATIC_SCRATCH_BYTES
        if plan.workspace_bytes > M.STATIC_SCRATCH_BYTES:
            with pytest.raises(M.MLAError) as e:
                M.mla_decode_run_static_scratch(plan, q[:len(lens), :heads], tiny[:, :512],
                                                tiny[:, 512:], 64, dev_i32(indptr),
                                                dev_i32(np.zeros(indptr[-1], np.int32)),
                                                dev_i32(lens), 1.0, 0.07,
                                                out[:len(lens), :heads], lse[:len(lens), :heads])
            assert e.value.status == 3
            refused += 1
        M.mla_decode_plan_destroy(plan)
    assert refused == expected >= 1
