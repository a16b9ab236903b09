"""Failure handling of the FP8 decode kernels, tested without faulting the
GPU: every wait of a CTA on an in-kernel barrier is bounded, and a wait that
runs out sets MLA_FLAG_WAIT_TIMEOUT, makes the CTA abandon its work, let its
copies and MMAs finish, free its tensor memory and exit.  The test shortens
the limit through the library's test hook to 1 ns, so that the first wait
of a CTA that finds its phase incomplete runs out, checks the flag,
restores the limit and checks that the next call on the same context is
correct again.  Covered: 16-head CTAs (two
query buffers) and 32-head CTAs that each serve one segment.
"""
import pytest
import torch

import mla_decode_attention_run_gb300 as M
import oracle
import workloads as W
from gpu_util import check_attention, gpu_decode, oracle_pool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    M.mla_get_last_error()
    yield
    M.mla_debug_set_wait_limit(0)


def _timed_out_then_correct(run, check):
    torch.cuda.synchronize()
    M.mla_debug_set_wait_limit(1)                  # 1 ns: the first wait that has to wait gives up
    try:
        run()
        flags = M.mla_get_last_error()
    finally:
        M.mla_debug_set_wait_limit(0)
    assert flags & M.FLAG_WAIT_TIMEOUT, f"flags {flags:#x}"
    out, lse = run()
    assert M.mla_get_last_error() == 0
    check(out, lse)


@pytest.mark.parametrize("heads,lens", [(4, None), (64, [700, 90])])
def test_decode_wait_timeout_flags_and_recovers(heads, lens):
    """16-head CTAs (the tiny configuration) and 32-head CTAs (H = 64)."""
    if lens is None:
        w = W.make_workload("tiny")
    else:
        w = W.make_workload("concurrency", batch=len(lens), heads=heads, lens=lens,
                            num_slots=5000, seed=71)
    pool = oracle_pool(w)
    dpool = torch.from_numpy(pool).cuda()
    o_ref, lse_ref = oracle.decode_fp8(w.q_bf16, pool[:, :512], pool[:, 512:], w.kv_indptr,
                                       w.kv_indices, w.seq_lens, w.page_size, w.k_scale,
                                       w.softmax_scale)

    def run():
        out, lse, _ = gpu_decode(w, dpool[:, :512], dpool[:, 512:])
        return out, lse

    _timed_out_then_correct(run, lambda o, l: check_attention(o, l, o_ref, lse_ref, "after timeout"))
