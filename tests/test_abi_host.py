"""Host-side tests of libmla_decode.so: it loads without a GPU, exports every
entry point include/mla_decode.h declares, validates arguments before any
CUDA call, and builds a balanced split-KV schedule."""
import ctypes
import os
import re

import numpy as np
import pytest

import mla_decode_attention_run_gb300 as M
import workloads as W

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mla_decode.h")
# [q1;q2] as 2 x 16 rows of 576 E4M3 bytes, then 16 fp32 score multipliers and
# 16 int32 causal limits
QIMAGE_BYTES = 3 * 16 * 576 + 16 * 12      # [q1;q2;q3] rows + two multipliers and a limit per row
SEGMENT_COST = 2          # tiles' worth of CTA time the tcgen05 schedule charges per segment


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mla_decode_attention_run_gb300 import build
    build.build()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:mla_status_t|const char\*)\s+(\w+)\s*\(", src, re.M)))


def test_every_declared_symbol_is_exported():
    decl = _declared_functions()
    assert len(decl) >= 9
    lib = M.library()
    for name in decl:
        assert hasattr(lib, name), name
    assert set(decl) <= set(M.exported_symbols())


def test_status_strings():
    lib = M.library()
    for st in range(6):
        assert lib.mla_status_string(st)
    assert lib.mla_status_string(99) == b"unknown status"


def _indptr(lens, ps):
    pages = (np.asarray(lens, np.int64) + ps - 1) // ps
    out = np.zeros(len(lens) + 1, np.int32)
    out[1:] = np.cumsum(pages)
    return out


def _check_schedule(segs, info, lens, heads, num_sms=152):
    lens = np.asarray(lens)
    tile = info["tile_tokens"]
    assert tile == 64
    tc = info["kernel"] == 1
    # every request's tokens are covered exactly once, in order
    for b in range(len(lens)):
        mine = segs[segs[:, 1] == b]
        if lens[b] == 0:
            assert mine.shape[0] == 0
            continue
        assert mine[0, 2] == 0 and mine[-1, 3] == lens[b]
        assert np.all(mine[1:, 2] == mine[:-1, 3])
        assert np.all(mine[:, 3] > mine[:, 2])
        assert np.all(mine[:, 2] % tile == 0)
        if mine.shape[0] == 1:
            assert mine[0, 4] == -1
        else:
            parts = mine[:, 4]
            assert np.all(parts >= 0) and np.all(np.diff(parts) == 1)
    # partial indices are a permutation of 0..n-1
    parts = segs[segs[:, 4] >= 0, 4]
    assert np.array_equal(np.sort(parts), np.arange(info["num_partials"]))
    ctas = info["num_ctas"]
    # CTAs per token range: 32 heads each on the tcgen05 path when they divide H, else 16
    hg = heads // 32 if (tc and heads % 32 == 0) else (heads + 15) // 16
    assert ctas <= max(1, num_sms // hg)
    tiles = np.zeros(ctas, np.int64)
    cost = np.zeros(ctas, np.int64)
    for c, b, t0, t1, _ in segs:
        tiles[c] += (t1 - t0 + tile - 1) // tile
        cost[c] += (t1 - t0 + tile - 1) // tile + SEGMENT_COST
    assert np.all(np.diff(segs[:, 0]) >= 0)
    if tc:
        # tcgen05 schedule: the largest CTA cost (tiles + a fixed cost per
        # segment) is within one segment of the even share
        n_req = int(np.sum(lens > 0))
        total = int(np.sum((lens + tile - 1) // tile)) + SEGMENT_COST * n_req
        assert cost.max() <= -(-total // max(ctas, 1)) + SEGMENT_COST + 1
        assert np.all(cost > 0)
    else:
        # mma.sync schedule: contiguous ranges balanced to within one tile
        assert tiles.max() - tiles.min() <= 1
    ws = info["workspace_bytes"]
    need = info["num_partials"] * heads * (512 + 1) * 4
    if tc and ctas > 0:                    # tcgen05 path: one q image per request and head group
        need += len(lens) * ((heads + 15) // 16) * QIMAGE_BYTES
    assert ws >= need
    if need == 0:
        assert ws == 0


@pytest.mark.parametrize("name", ["tiny", "single", "concurrency"])
def test_schedule_of_named_workloads(name):
    cfg = W.CONFIGS[name]
    g = np.random.default_rng(cfg["number"])
    if cfg["lens"] == "uniform":
        lens = g.integers(1024, 8193, cfg["batch"])
    else:
        lens = np.asarray(cfg["lens"])
    segs, info = M.mla_decode_schedule(_indptr(lens, 1), lens, len(lens), cfg["heads"], 1)
    _check_schedule(segs, info, lens, cfg["heads"])


def test_schedule_large_head_paged():
    lens = np.full(128, 32768)
    segs, info = M.mla_decode_schedule(_indptr(lens, 64), lens, 128, 128, 64)
    _check_schedule(segs, info, lens, 128)
    assert info["num_ctas"] == 152 // 4          # 32-head CTAs: four per token range


def test_schedule_ragged_and_empty_requests():
    lens = np.array([0, 1, 63, 64, 65, 0, 1000, 3])
    segs, info = M.mla_decode_schedule(_indptr(lens, 3), lens, len(lens), 4, 3, num_sms=5)
    _check_schedule(segs, info, lens, 4, num_sms=5)


def test_schedule_many_short_requests_over_sm_counts():
    """Several one-tile requests and few CTAs: every request costs a segment,
    so the search for the cost cap must start from a cap that one CTA can
    always meet (every request whole, one segment each)."""
    g = np.random.default_rng(5)
    cases = [np.array([1, 2, 3]), np.array([64, 1, 1, 1, 65]), np.full(9, 5),
             g.integers(0, 200, 17), g.integers(1, 70, 40)]
    for lens in cases:
        for heads in (16, 64):
            for num_sms in (1, 2, 3, 4, 7, 19, 152):
                segs, info = M.mla_decode_schedule(_indptr(lens, 1), lens, len(lens), heads, 1,
                                                   num_sms=num_sms)
                assert info["num_ctas"] >= 1
                _check_schedule(segs, info, lens, heads, num_sms=num_sms)


def test_schedule_picks_the_tensor_core_kernel_for_fp8_pools():
    lens = np.array([1000, 3000])
    _, fp8_16 = M.mla_decode_schedule(_indptr(lens, 1), lens, 2, 16, 1, M.MLA_KV_FP8_E4M3)
    _, bf16_16 = M.mla_decode_schedule(_indptr(lens, 1), lens, 2, 16, 1, M.MLA_KV_BF16)
    _, fp8_32 = M.mla_decode_schedule(_indptr(lens, 1), lens, 2, 32, 1, M.MLA_KV_FP8_E4M3)
    assert fp8_16["kernel"] == 1 and fp8_32["kernel"] == 1
    assert bf16_16["kernel"] == 0


def test_schedule_all_empty():
    lens = np.zeros(3, np.int64)
    segs, info = M.mla_decode_schedule(_indptr(lens, 1), lens, 3, 16, 1)
    assert segs.shape[0] == 0 and info["num_ctas"] == 0 and info["workspace_bytes"] == 0


@pytest.mark.parametrize("mutate,status", [
    (lambda ip, sl: (ip, np.array([5, -1], np.int32)), 1),          # negative length
    (lambda ip, sl: (np.array([0, 4, 9], np.int32), sl), 1),        # wrong page count
    (lambda ip, sl: (np.array([0, 5, 4], np.int32), sl), 1),        # non-monotone
    (lambda ip, sl: (np.array([-1, 4, 8], np.int32), sl), 1),       # negative start
])
def test_schedule_rejects_bad_page_tables(mutate, status):
    indptr, lens = mutate(np.array([0, 5, 9], np.int32), np.array([5, 4], np.int32))
    with pytest.raises(M.MLAError) as e:
        M.mla_decode_schedule(indptr, lens, 2, 16, 1)
    assert e.value.status == status


@pytest.mark.parametrize("heads,ps,status", [(0, 1, 2), (17, 1, 2), (144, 1, 2), (24, 1, 2),
                                             (16, 0, 1)])
def test_schedule_rejects_bad_shapes(heads, ps, status):
    lens = np.array([5, 4], np.int32)
    indptr = _indptr(lens, max(ps, 1))
    with pytest.raises(M.MLAError) as e:
        M.mla_decode_schedule(indptr, lens, 2, heads, ps)
    assert e.value.status == status


def test_plan_validates_before_touching_cuda():
    lib = M.library()
    plan = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    lens = np.array([5, 4], np.int32)
    bad = np.array([0, 5, 8], np.int32)
    st = lib.mla_decode_plan(ctypes.byref(plan), bad.ctypes.data, lens.ctypes.data, 2, 16, 1, 0,
                             ctypes.byref(ws), None)
    assert st == 1 and not plan.value
    st = lib.mla_decode_plan(ctypes.byref(plan), bad.ctypes.data, lens.ctypes.data, 2, 20, 1, 0,
                             ctypes.byref(ws), None)
    assert st == 2
    assert lib.mla_decode_plan(None, bad.ctypes.data, lens.ctypes.data, 2, 16, 1, 0,
                               ctypes.byref(ws), None) == 1


def test_entry_points_reject_null_and_accept_empty_without_cuda():
    lib = M.library()
    # n = 0 / n_pages = 0 are no-ops
    assert lib.kv_store_fp8(None, None, None, 0, 1.0, None, 576, None, 576, 10, None) == 0
    assert lib.kv_gather_cast(None, 576, None, 576, 10, None, 0, 1, 1.0, None, None, None) == 0
    # NULL pointers / bad sizes
    assert lib.kv_store_fp8(None, None, None, 3, 1.0, None, 576, None, 576, 10, None) == 1
    assert lib.kv_store_fp8(16, 16, 16, -1, 1.0, 16, 576, 16, 576, 10, None) == 1
    assert lib.kv_gather_cast(16, 576, 16, 576, 10, 16, 2, 0, 1.0, 16, 16, None) == 1
    # bad scale
    assert lib.kv_store_fp8(16, 16, 16, 3, 0.0, 16, 576, 16, 576, 10, None) == 1
    assert lib.kv_store_fp8(16, 16, 16, 3, float("inf"), 16, 576, 16, 576, 10, None) == 1
    # misaligned pool / stride
    assert lib.kv_store_fp8(16, 16, 16, 3, 1.0, 17, 576, 16, 576, 10, None) == 2
    assert lib.kv_store_fp8(16, 16, 16, 3, 1.0, 16, 570, 16, 576, 10, None) == 2
    assert lib.kv_gather_cast(16, 576, 16, 577, 10, 16, 2, 1, 1.0, 16, 16, None) == 2
    # decode run without a plan
    assert lib.mla_decode_run(None, 16, 0, 576, 16, 576, 16, 576, 10, 16, 16, 16, 1.0, 0.07, 16,
                              16, None, 0, None) == 1
    assert M.library().mla_decode_plan_destroy(None) == 0
    # fused projection store: n = 0 is a no-op; bad sizes, scale and alignment
    assert lib.kv_proj_store_fp8(None, 64, None, 64, 0, 64, None, 1.0, None, 576, None, 576, 10,
                                 None, None) == 0
    assert lib.kv_proj_store_fp8(16, 64, 16, 64, -1, 64, 16, 1.0, 16, 576, 16, 576, 10, None,
                                 None) == 1
    assert lib.kv_proj_store_fp8(16, 96, 16, 96, 3, 96, 16, 1.0, 16, 576, 16, 576, 10, None,
                                 None) == 1                       # d_model not a multiple of 64
    assert lib.kv_proj_store_fp8(16, 64, 16, 64, 3, 64, 16, 0.0, 16, 576, 16, 576, 10, None,
                                 None) == 1
    assert lib.kv_proj_store_fp8(17, 64, 16, 64, 3, 64, 16, 1.0, 16, 576, 16, 576, 10, None,
                                 None) == 2                       # misaligned x
    assert lib.kv_proj_store_fp8(16, 64, 16, 64, 3, 64, 16, 1.0, 16, 576, 16, 576, 10, 24,
                                 None) == 2                       # misaligned latent_out
