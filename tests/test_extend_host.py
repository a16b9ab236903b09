"""Host-side tests of the extend (causal, several new tokens per request)
plan: query rows are cut into blocks that cover every request's rows once,
each block's context ends at its last row's causal limit, the segments
cover each block's context once, and bad inputs are rejected before any
CUDA call."""
import ctypes

import numpy as np
import pytest

import mla_decode_attention_run_gb300 as M

QIMAGE_BYTES = 3 * 16 * 576 + 16 * 12      # [q1;q2;q3] rows + two multipliers and a limit per row
TILE = 64
EXTEND_SEGMENT_COST = 4   # tiles' worth of CTA time the extend schedule charges per segment


@pytest.fixture(scope="module", autouse=True)
def _built():
    from mla_decode_attention_run_gb300 import build
    build.build()


def _tables(lens, q_lens, ps=1):
    lens = np.asarray(lens, np.int32)
    pages = (lens.astype(np.int64) + ps - 1) // ps
    indptr = np.zeros(len(lens) + 1, np.int32)
    indptr[1:] = np.cumsum(pages)
    qo = np.zeros(len(lens) + 1, np.int32)
    qo[1:] = np.cumsum(q_lens)
    return qo, indptr, lens


def _check(lens, q_lens, heads, ps=1, num_sms=152):
    qo, indptr, lens = _tables(lens, q_lens, ps)
    B = len(lens)
    segs, blocks, info = M.mla_extend_schedule(qo, indptr, lens, B, heads, ps, num_sms=num_sms)
    G = info["block_rows"]
    assert G in (16, 32)
    # blocks tile each request's rows (token * H + head) in order
    for b in range(B):
        mine = blocks[blocks[:, 0] == b]
        lo, hi = int(qo[b]) * heads, int(qo[b + 1]) * heads
        if hi == lo:
            assert mine.shape[0] == 0
            continue
        assert mine[0, 1] == lo and mine[-1, 1] + mine[-1, 2] == hi
        assert np.all(mine[1:, 1] == mine[:-1, 1] + mine[:-1, 2])
        assert np.all(mine[:-1, 2] == G) and 1 <= mine[-1, 2] <= G
        # causal base: the last new token (row hi - 1) sees the whole context
        assert np.all(mine[:, 3] == lens[b] + 1 - qo[b + 1])
        assert mine[-1, 3] + (hi - 1) // heads == lens[b]
    # each block's context (its last row's limit) is covered once, tile-aligned
    for v, (b, r0, rows, base) in enumerate(blocks):
        length = base + (r0 + rows - 1) // heads
        assert 1 <= length <= lens[b]
        mine = segs[segs[:, 1] == v]
        assert mine[0, 2] == 0 and mine[-1, 3] == length
        assert np.all(mine[1:, 2] == mine[:-1, 3]) and np.all(mine[:, 2] % TILE == 0)
        if mine.shape[0] == 1:
            assert mine[0, 4] == -1
        else:
            assert np.all(np.diff(mine[:, 4]) == 1) and mine[0, 4] >= 0
    parts = segs[segs[:, 4] >= 0, 4]
    assert np.array_equal(np.sort(parts), np.arange(info["num_partials"]))
    assert info["num_ctas"] <= num_sms
    need = info["num_partials"] * G * (512 + 1) * 4
    if info["num_ctas"] > 0:
        need += info["num_blocks"] * (G // 16) * QIMAGE_BYTES
    assert info["workspace_bytes"] >= need
    return segs, blocks, info


@pytest.mark.parametrize("lens,q_lens,heads,ps", [
    ([100, 300, 65], [4, 64, 65], 16, 1),          # extend, and a pure prefill (q_len = L)
    ([5000, 1200], [2, 3], 16, 1),                 # speculative-style
    ([40, 17, 33], [0, 17, 5], 4, 1),              # a request without new tokens
    ([700, 900], [8, 1], 128, 64),                 # many heads, paged
    ([64, 128], [64, 128], 16, 16),
    ([0, 50, 0], [0, 7, 0], 16, 1),                # empty contexts beside an extend
])
def test_extend_schedule_covers_rows_and_contexts(lens, q_lens, heads, ps):
    _check(lens, q_lens, heads, ps)


@pytest.mark.parametrize("lens,q_lens", [
    ([5000, 1200, 3000, 800], [4, 4, 4, 4]),
    (list(np.random.default_rng(3).integers(1024, 8193, 40)), [4] * 40),   # speculative, batch 40
    ([4000] * 8, [256] * 8),                                              # prefill chunks
])
def test_extend_schedule_balances_cost(lens, q_lens):
    """The largest CTA cost (tiles + a fixed cost per segment) is within one
    segment of the even share, and with tiles enough every CTA has work (the
    plan splits the costliest range until none is idle)."""
    segs, blocks, info = _check(lens, q_lens, 16)
    ctas = info["num_ctas"]
    tiles = np.zeros(ctas, np.int64)
    nseg = np.zeros(ctas, np.int64)
    for c, _, t0, t1, _ in segs:
        tiles[c] += (t1 - t0 + TILE - 1) // TILE
        nseg[c] += 1
    total = int(tiles.sum()) + EXTEND_SEGMENT_COST * blocks.shape[0]
    cost = tiles + EXTEND_SEGMENT_COST * nseg
    assert cost.max() <= -(-total // ctas) + EXTEND_SEGMENT_COST + 1
    if tiles.sum() >= 152:
        assert ctas == 152 and tiles.min() >= 1


def test_one_new_token_per_request_reads_each_whole_context():
    lens = [1000, 77, 4096]
    segs, blocks, info = _check(lens, [1, 1, 1], 16)
    assert info["block_rows"] == 16 and info["num_blocks"] == 3
    assert np.array_equal(blocks[:, 0], [0, 1, 2])
    for v in range(3):
        assert segs[segs[:, 1] == v][-1, 3] == lens[v]


@pytest.mark.parametrize("q_lens,heads,rows", [([1, 1], 16, 16), ([4, 4], 16, 32),
                                               ([3, 3], 4, 16), ([2, 1], 128, 32)])
def test_block_rows(q_lens, heads, rows):
    _, _, info = _check([500, 600], q_lens, heads)
    assert info["block_rows"] == rows


def test_all_requests_without_new_tokens():
    segs, blocks, info = _check([10, 20], [0, 0], 16)
    assert info["num_ctas"] == 0 and info["num_blocks"] == 0 and info["workspace_bytes"] == 0


@pytest.mark.parametrize("mutate,status", [
    (lambda qo, ip, l: qo.__setitem__(2, 9), 1),          # more new tokens than context
    (lambda qo, ip, l: qo.__setitem__(0, 1), 1),          # qo_indptr must start at 0
    (lambda qo, ip, l: qo.__setitem__(1, 5), 1),          # decreasing qo_indptr
    (lambda qo, ip, l: ip.__setitem__(1, 3), 1),          # page table of the wrong length
])
def test_extend_rejects_bad_tables(mutate, status):
    qo, indptr, lens = _tables([6, 4], [2, 2])
    mutate(qo, indptr, lens)
    with pytest.raises(M.MLAError) as e:
        M.mla_extend_schedule(qo, indptr, lens, 2, 16, 1)
    assert e.value.status == status


def test_extend_rejects_bf16_pools_and_bad_heads():
    qo, indptr, lens = _tables([6, 4], [2, 2])
    with pytest.raises(M.MLAError) as e:
        M.mla_extend_schedule(qo, indptr, lens, 2, 16, 1, kv_dtype=M.MLA_KV_BF16)
    assert e.value.status == 2
    with pytest.raises(M.MLAError) as e:
        M.mla_extend_schedule(qo, indptr, lens, 2, 20, 1)
    assert e.value.status == 2


def test_extend_entry_points_validate_before_cuda():
    lib = M.library()
    plan = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    qo, indptr, lens = _tables([6, 4], [2, 7])          # 7 > 4
    st = lib.mla_extend_plan(ctypes.byref(plan), qo.ctypes.data, indptr.ctypes.data,
                             lens.ctypes.data, 2, 16, 1, 0, ctypes.byref(ws), None)
    assert st == 1 and not plan.value
    assert lib.mla_extend_plan(ctypes.byref(plan), None, indptr.ctypes.data, lens.ctypes.data,
                               2, 16, 1, 0, ctypes.byref(ws), None) == 1
    assert lib.mla_extend_run(None, 16, 576 * 16, 576, 16, 576, 16, 576, 10, 16, 16, 16, 1.0,
                              0.07, 16, 16, None, 0, None) == 1
