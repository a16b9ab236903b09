"""Paged MLA decode over an FP8 E4M3 KV cache on GB300 (sm_103a).

Thin Python binding of libmla_decode.so (C ABI in include/mla_decode.h).  The
functions below carry the C entry points' names and only marshal arguments:
torch tensors provide device memory and streams, every step of the path runs
in the library's CUDA kernels.  There is no CPU fallback: if the library is
missing or cannot load, importing a function raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "MLA_KV_FP8_E4M3", "MLA_KV_BF16", "MLAError", "library", "library_path",
    "mla_decode_plan", "mla_decode_run", "mla_decode_plan_destroy", "mla_decode_plan_info",
    "mla_decode_schedule", "kv_store_fp8", "kv_gather_cast", "mla_get_last_error",
    "exported_symbols", "D_CKV", "D_KPE", "D_QK", "mla_decode_run_static_scratch",
    "STATIC_SCRATCH_BYTES", "mla_extend_plan", "mla_extend_run", "mla_extend_schedule",
    "kv_proj_store_fp8", "mla_debug_set_wait_limit",
]

D_CKV, D_KPE, D_QK = 512, 64, 576
MLA_KV_FP8_E4M3, MLA_KV_BF16 = 0, 1
FLAG_INDEX_OOB, FLAG_PLAN_MISMATCH, FLAG_WAIT_TIMEOUT = 0x1, 0x2, 0x4
STATIC_SCRATCH_BYTES = 8 << 20       # MLA_STATIC_SCRATCH_BYTES

library_path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmla_decode.so")
_lib = None

_P = ctypes.c_void_p
_i32, _i64, _f32, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_PI32 = ctypes.POINTER(ctypes.c_int32)


class MLAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = library().mla_status_string(status).decode() if _lib else str(status)
        super().__init__(f"{where}: status {status} ({msg})")


def library():
    """Load libmla_decode.so (built by build.py); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise RuntimeError(
            f"{library_path} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` "
            "(or python mla_decode_attention_run_gb300/build.py)")
    lib = ctypes.CDLL(library_path)
    lib.mla_decode_plan.argtypes = [ctypes.POINTER(_P), _P, _P, _i32, _i32, _i32, ctypes.c_int,
                                    ctypes.POINTER(_sz), _P]
    lib.mla_decode_run.argtypes = [_P, _P, _i64, _i64, _P, _i64, _P, _i64, _i64, _P, _P, _P, _f32,
                                   _f32, _P, _P, _P, _sz, _P]
    lib.mla_decode_run_static_scratch.argtypes = [_P, _P, _i64, _i64, _P, _i64, _P, _i64, _i64,
                                                  _P, _P, _P, _f32, _f32, _P, _P, _P]
    lib.mla_decode_plan_destroy.argtypes = [_P]
    lib.mla_decode_plan_info.argtypes = [_P, _PI32, _PI32, _PI32, ctypes.POINTER(_sz)]
    lib.mla_decode_schedule.argtypes = [_P, _P, _i32, _i32, _i32, ctypes.c_int, _i32, _P, _i32,
                                        _PI32, _PI32, _PI32, _PI32, _PI32, ctypes.POINTER(_sz)]
    lib.mla_extend_plan.argtypes = [ctypes.POINTER(_P), _P, _P, _P, _i32, _i32, _i32, ctypes.c_int,
                                    ctypes.POINTER(_sz), _P]
    lib.mla_extend_run.argtypes = lib.mla_decode_run.argtypes
    lib.mla_extend_schedule.argtypes = [_P, _P, _P, _i32, _i32, _i32, ctypes.c_int, _i32, _P, _i32,
                                        _P, _i32, _P, ctypes.POINTER(_sz)]
    lib.kv_store_fp8.argtypes = [_P, _P, _P, _i64, _f32, _P, _i64, _P, _i64, _i64, _P]
    lib.kv_proj_store_fp8.argtypes = [_P, _i64, _P, _i64, _i64, _i32, _P, _f32, _P, _i64, _P, _i64,
                                      _i64, _P, _P]
    lib.kv_gather_cast.argtypes = [_P, _i64, _P, _i64, _i64, _P, _i64, _i32, _f32, _P, _P, _P]
    lib.mla_get_last_error.argtypes = [_P, ctypes.POINTER(ctypes.c_uint32)]
    lib.mla_debug_set_wait_limit.argtypes = [ctypes.c_uint64]
    lib.mla_status_string.argtypes = [ctypes.c_int]
    lib.mla_status_string.restype = ctypes.c_char_p
    for name in ("mla_decode_plan", "mla_decode_run", "mla_decode_plan_destroy",
                 "mla_decode_plan_info", "mla_decode_schedule", "kv_store_fp8", "kv_gather_cast",
                 "mla_get_last_error", "mla_decode_run_static_scratch", "mla_extend_plan",
                 "mla_extend_run", "mla_extend_schedule", "kv_proj_store_fp8",
                 "mla_debug_set_wait_limit"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def exported_symbols() -> list[str]:
    """Names of the C entry points declared in include/mla_decode.h that the
    loaded library resolves."""
    lib = library()
    names = []
    for n in ("mla_decode_plan", "mla_decode_run", "mla_decode_plan_destroy",
              "mla_decode_plan_info", "mla_decode_schedule", "kv_store_fp8", "kv_gather_cast",
              "mla_get_last_error", "mla_status_string", "mla_decode_run_static_scratch",
              "mla_extend_plan", "mla_extend_run", "mla_extend_schedule", "kv_proj_store_fp8",
              "mla_debug_set_wait_limit"):
        getattr(lib, n)
        names.append(n)
    return names


def _check(status: int, where: str):
    if status != 0:
        raise MLAError(status, where)


def _stream(stream):
    if stream is None:
        import torch
        return _P(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return _P(stream)
    return _P(stream.cuda_stream)


def _host_i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _dptr(t) -> int:
    return t.data_ptr() if t is not None else 0


def _row_stride_bytes(t) -> int:
    return t.stride(0) * t.element_size()


class Plan:
    """Owns a plan handle; destroyed explicitly or when garbage collected."""

    def __init__(self):
        self.handle = _P(None)
        self.workspace_bytes = 0

    def __del__(self):
        try:
            if self.handle and self.handle.value and _lib is not None:
                _lib.mla_decode_plan_destroy(self.handle)
                self.handle = _P(None)
        except Exception:
            pass


def mla_decode_plan(kv_indptr_host, seq_lens_host, batch: int, num_heads: int, page_size: int,
                    kv_dtype: int = MLA_KV_FP8_E4M3, stream=None, plan: Plan | None = None) -> Plan:
    """Build (or rebuild in place) a plan; returns it with .workspace_bytes."""
    lib = library()
    indptr, lens = _host_i32(kv_indptr_host), _host_i32(seq_lens_host)
    plan = plan if plan is not None else Plan()
    ws = _sz(0)
    _check(lib.mla_decode_plan(ctypes.byref(plan.handle), indptr.ctypes.data, lens.ctypes.data,
                               batch, num_heads, page_size, kv_dtype, ctypes.byref(ws),
                               _stream(stream)), "mla_decode_plan")
    plan.workspace_bytes = ws.value
    plan._keep = (indptr, lens)          # host arrays live until the upload is done
    return plan


def mla_decode_run(plan: Plan, q, ckv_pool, kpe_pool, num_pool_slots: int, kv_indptr_dev,
                   kv_indices_dev, seq_lens_dev, k_scale: float, softmax_scale: float, out, lse,
                   workspace=None, stream=None):
    """q: bf16 [B, H, 576] (any strides with contiguous last dim); pools:
    uint8 / float8 (FP8 plans) or bf16 (BF16 plans) with rows along dim 0;
    out: bf16 [B, H, 512]; lse: fp32 [B, H]; workspace: >= plan.workspace_bytes."""
    lib = library()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.mla_decode_run(plan.handle, q.data_ptr(), q.stride(0), q.stride(1),
                              ckv_pool.data_ptr(), _row_stride_bytes(ckv_pool),
                              kpe_pool.data_ptr(), _row_stride_bytes(kpe_pool), num_pool_slots,
                              kv_indptr_dev.data_ptr(), _dptr(kv_indices_dev),
                              seq_lens_dev.data_ptr(), k_scale, softmax_scale, out.data_ptr(),
                              lse.data_ptr(), _dptr(workspace), ws_bytes, _stream(stream)),
           "mla_decode_run")


def mla_decode_run_static_scratch(plan: Plan, q, ckv_pool, kpe_pool, num_pool_slots: int,
                                  kv_indptr_dev, kv_indices_dev, seq_lens_dev, k_scale: float,
                                  softmax_scale: float, out, lse, stream=None):
    """mla_decode_run without a workspace argument, for callers that cannot
    allocate device memory: the split-KV partials go to a fixed array inside
    the library (STATIC_SCRATCH_BYTES per GPU, kept until exit).  Calls that
    overlap on the GPU share that array and race; calls on one stream are
    ordered.  Raises MLAError (status 3) if the plan needs more scratch."""
    _check(library().mla_decode_run_static_scratch(
        plan.handle, q.data_ptr(), q.stride(0), q.stride(1), ckv_pool.data_ptr(),
        _row_stride_bytes(ckv_pool), kpe_pool.data_ptr(), _row_stride_bytes(kpe_pool),
        num_pool_slots, kv_indptr_dev.data_ptr(), _dptr(kv_indices_dev),
        seq_lens_dev.data_ptr(), k_scale, softmax_scale, out.data_ptr(), lse.data_ptr(),
        _stream(stream)), "mla_decode_run_static_scratch")


def mla_decode_plan_destroy(plan: Plan):
    if plan.handle and plan.handle.value:
        _check(library().mla_decode_plan_destroy(plan.handle), "mla_decode_plan_destroy")
        plan.handle = _P(None)


def mla_decode_plan_info(plan: Plan) -> dict:
    c, s, p, w = _i32(), _i32(), _i32(), _sz()
    _check(library().mla_decode_plan_info(plan.handle, ctypes.byref(c), ctypes.byref(s),
                                          ctypes.byref(p), ctypes.byref(w)), "mla_decode_plan_info")
    return dict(num_ctas=c.value, num_segments=s.value, num_partials=p.value,
                workspace_bytes=w.value)


def mla_decode_schedule(kv_indptr_host, seq_lens_host, batch: int, num_heads: int,
                        page_size: int, kv_dtype: int = MLA_KV_FP8_E4M3, num_sms: int = 152):
    """Host-only schedule: returns (segments int32 [n, 5] = cta, request, t0,
    t1, partial; info dict with kernel 0 = mma.sync, 1 = tcgen05).  Raises
    MLAError on invalid input."""
    lib = library()
    indptr, lens = _host_i32(kv_indptr_host), _host_i32(seq_lens_host)
    n, p, c, t, k, w = _i32(), _i32(), _i32(), _i32(), _i32(), _sz()
    args = (indptr.ctypes.data, lens.ctypes.data, batch, num_heads, page_size, kv_dtype, num_sms)
    outs = (ctypes.byref(n), ctypes.byref(p), ctypes.byref(c), ctypes.byref(t), ctypes.byref(k),
            ctypes.byref(w))
    _check(lib.mla_decode_schedule(*args, None, 0, *outs), "mla_decode_schedule")
    segs = np.zeros((max(n.value, 1), 5), np.int32)
    _check(lib.mla_decode_schedule(*args, segs.ctypes.data, n.value, *outs),
           "mla_decode_schedule")
    return segs[:n.value], dict(num_ctas=c.value, num_partials=p.value, tile_tokens=t.value,
                                kernel=k.value, workspace_bytes=w.value)


def mla_extend_plan(qo_indptr_host, kv_indptr_host, seq_lens_host, batch: int, num_heads: int,
                    page_size: int, kv_dtype: int = MLA_KV_FP8_E4M3, stream=None,
                    plan: Plan | None = None) -> Plan:
    """Plan causal extend attention: request b's new tokens are query rows
    qo_indptr[b] .. qo_indptr[b+1]-1 and already count in seq_lens[b]."""
    lib = library()
    qo, indptr, lens = _host_i32(qo_indptr_host), _host_i32(kv_indptr_host), _host_i32(seq_lens_host)
    plan = plan if plan is not None else Plan()
    ws = _sz(0)
    _check(lib.mla_extend_plan(ctypes.byref(plan.handle), qo.ctypes.data, indptr.ctypes.data,
                               lens.ctypes.data, batch, num_heads, page_size, kv_dtype,
                               ctypes.byref(ws), _stream(stream)), "mla_extend_plan")
    plan.workspace_bytes = ws.value
    plan._keep = (qo, indptr, lens)
    return plan


def mla_extend_run(plan: Plan, q, ckv_pool, kpe_pool, num_pool_slots: int, kv_indptr_dev,
                   kv_indices_dev, seq_lens_dev, k_scale: float, softmax_scale: float, out, lse,
                   workspace=None, stream=None):
    """q: bf16 [n_q, H, 576] (contiguous last dim); out: bf16 [n_q, H, 512];
    lse: fp32 [n_q, H]; the rest as mla_decode_run."""
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(library().mla_extend_run(plan.handle, q.data_ptr(), q.stride(0), q.stride(1),
                                    ckv_pool.data_ptr(), _row_stride_bytes(ckv_pool),
                                    kpe_pool.data_ptr(), _row_stride_bytes(kpe_pool),
                                    num_pool_slots, kv_indptr_dev.data_ptr(),
                                    _dptr(kv_indices_dev), seq_lens_dev.data_ptr(), k_scale,
                                    softmax_scale, out.data_ptr(), lse.data_ptr(),
                                    _dptr(workspace), ws_bytes, _stream(stream)),
           "mla_extend_run")


def mla_extend_schedule(qo_indptr_host, kv_indptr_host, seq_lens_host, batch: int,
                        num_heads: int, page_size: int, kv_dtype: int = MLA_KV_FP8_E4M3,
                        num_sms: int = 152):
    """Host-only extend schedule: (segments int32 [n, 5] = cta, block, t0, t1,
    partial; blocks int32 [m, 4] = request, first row, rows, causal base;
    info dict)."""
    lib = library()
    qo, indptr, lens = _host_i32(qo_indptr_host), _host_i32(kv_indptr_host), _host_i32(seq_lens_host)
    counts = np.zeros(5, np.int32)
    w = _sz()
    args = (qo.ctypes.data, indptr.ctypes.data, lens.ctypes.data, batch, num_heads, page_size,
            kv_dtype, num_sms)
    _check(lib.mla_extend_schedule(*args, None, 0, None, 0, counts.ctypes.data, ctypes.byref(w)),
           "mla_extend_schedule")
    segs = np.zeros((max(int(counts[0]), 1), 5), np.int32)
    blocks = np.zeros((max(int(counts[3]), 1), 4), np.int32)
    _check(lib.mla_extend_schedule(*args, segs.ctypes.data, int(counts[0]), blocks.ctypes.data,
                                   int(counts[3]), counts.ctypes.data, ctypes.byref(w)),
           "mla_extend_schedule")
    return segs[:counts[0]], blocks[:counts[3]], dict(
        num_segments=int(counts[0]), num_partials=int(counts[1]), num_ctas=int(counts[2]),
        num_blocks=int(counts[3]), block_rows=int(counts[4]), workspace_bytes=w.value)


def kv_store_fp8(ckv_new, kpe_new, slots, k_scale: float, ckv_pool, kpe_pool,
                 num_pool_slots: int | None = None, stream=None):
    """ckv_new bf16 [n, 512], kpe_new bf16 [n, 64] (contiguous), slots int64 [n]."""
    n = slots.shape[0]
    nps = ckv_pool.shape[0] if num_pool_slots is None else num_pool_slots
    _check(library().kv_store_fp8(ckv_new.data_ptr(), kpe_new.data_ptr(), slots.data_ptr(), n,
                                  k_scale, ckv_pool.data_ptr(), _row_stride_bytes(ckv_pool),
                                  kpe_pool.data_ptr(), _row_stride_bytes(kpe_pool), nps,
                                  _stream(stream)), "kv_store_fp8")


def kv_proj_store_fp8(x, w, slots, k_scale: float, ckv_pool, kpe_pool,
                      num_pool_slots: int | None = None, latent_out=None, stream=None):
    """x bf16 [n, d_model], w bf16 [576, d_model] (row j = channel j's
    weights), slots int64 [n]: latent = BF16(x @ w.T) quantized into the pool
    rows like kv_store_fp8; latent_out (optional) bf16 [n, 576] receives the
    rounded latents."""
    n, d = x.shape
    nps = ckv_pool.shape[0] if num_pool_slots is None else num_pool_slots
    _check(library().kv_proj_store_fp8(x.data_ptr(), x.stride(0), w.data_ptr(), w.stride(0), n, d,
                                       slots.data_ptr(), k_scale, ckv_pool.data_ptr(),
                                       _row_stride_bytes(ckv_pool), kpe_pool.data_ptr(),
                                       _row_stride_bytes(kpe_pool), nps, _dptr(latent_out),
                                       _stream(stream)), "kv_proj_store_fp8")


def kv_gather_cast(ckv_pool, kpe_pool, kv_indices, page_size: int, k_scale: float, ckv_out,
                   kpe_out, num_pool_slots: int | None = None, stream=None):
    """Gather the listed pages into compact bf16 [n_pages*page_size, 512 / 64]."""
    nps = ckv_pool.shape[0] if num_pool_slots is None else num_pool_slots
    _check(library().kv_gather_cast(ckv_pool.data_ptr(), _row_stride_bytes(ckv_pool),
                                    kpe_pool.data_ptr(), _row_stride_bytes(kpe_pool), nps,
                                    kv_indices.data_ptr(), kv_indices.shape[0], page_size,
                                    k_scale, ckv_out.data_ptr(), kpe_out.data_ptr(),
                                    _stream(stream)), "kv_gather_cast")


def mla_get_last_error(stream=None) -> int:
    """Synchronise the stream; return and clear the device flag word."""
    flags = ctypes.c_uint32(0)
    st = library().mla_get_last_error(_stream(stream), ctypes.byref(flags))
    if st not in (0, 4):
        raise MLAError(st, "mla_get_last_error")
    return flags.value


def mla_debug_set_wait_limit(limit_ns: int):
    """Time limit (ns) of the decode kernels' bounded in-kernel waits on the
    current device; 0 restores the default (2 s).  A test hook: a tiny limit
    makes the next decode calls give up and set FLAG_WAIT_TIMEOUT."""
    _check(library().mla_debug_set_wait_limit(ctypes.c_uint64(int(limit_ns))),
           "mla_debug_set_wait_limit")
