"""CPU oracle for paged MLA decode over an FP8 E4M3 KV cache.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the benchmark's CPU-baseline leg may import this package.  The CUDA
library never calls it, and it shares no code with the CUDA library.

The arithmetic lives in ``mla_oracle.c`` (plain C, fp64 attention); this
module only compiles it and marshals numpy arrays through ctypes.  What each
function computes, and which web page it follows, is stated in the C file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

D_CKV, D_KPE = 512, 64
D_ALL = D_CKV + D_KPE


def build(force: bool = False) -> str:
    """Compile mla_oracle.c into liboracle.so next to it (gcc, no fast math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_double
        lib.oracle_e4m3_table.argtypes = [P]
        lib.oracle_e4m3_encode.argtypes = [f32]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_float_to_bf16.argtypes = [f32]
        lib.oracle_float_to_bf16.restype = ctypes.c_uint16
        lib.oracle_e4m3_encode_array.argtypes = [P, i64, P]
        lib.oracle_kv_store_fp8.argtypes = [P, P, P, i64, f32, P, i64, P, i64, i64]
        lib.oracle_kv_store_fp8.restype = i64
        lib.oracle_kv_proj_fp8.argtypes = [P, P, i64, i32, P, f32, P, i64, P, i64, i64, P]
        lib.oracle_kv_proj_fp8.restype = i64
        lib.oracle_double_to_bf16.argtypes = [f64]
        lib.oracle_double_to_bf16.restype = ctypes.c_uint16
        lib.oracle_kv_gather_cast.argtypes = [P, i64, P, i64, i64, P, i64, i32, f32, P, P]
        lib.oracle_kv_gather_cast.restype = i64
        dec_args = [P, P, i64, P, i64, i64, P, P, P, i32, i32, i32, f64, f64, P, P, P, i64,
                    ctypes.c_int]
        lib.oracle_decode_fp8.argtypes = dec_args
        lib.oracle_decode_fp8.restype = ctypes.c_int
        lib.oracle_decode_bf16.argtypes = dec_args
        lib.oracle_decode_bf16.restype = ctypes.c_int
        lib.oracle_extend_fp8.argtypes = [P, P, i64, P, i64, i64, P, P, P, P, i32, i32, i32,
                                          f64, f64, P, P, ctypes.c_int]
        lib.oracle_extend_fp8.restype = ctypes.c_int
        lib.oracle_attention_f64.argtypes = [P, P, i64, i32, f64, P, P, P]
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def e4m3_table() -> np.ndarray:
    """float64[256]: the value of every E4M3 byte (NaN for 0x7F / 0xFF)."""
    out = np.empty(256, np.float64)
    _load().oracle_e4m3_table(_ptr(out))
    return out


def e4m3_encode(x) -> np.ndarray:
    """Encode float32 values to E4M3 bytes (nearest, ties to even, saturating)."""
    x = np.ascontiguousarray(np.asarray(x, np.float32))
    out = np.empty(x.shape, np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def float_to_bf16(x) -> np.ndarray:
    """Round float32 values to BF16 bit patterns (nearest, ties to even)."""
    lib = _load()
    x = np.asarray(x, np.float32)
    return np.array([lib.oracle_float_to_bf16(float(v)) for v in x.ravel()],
                    np.uint16).reshape(x.shape)


def kv_store_fp8(ckv_new_bf16: np.ndarray, kpe_new_bf16: np.ndarray, slots: np.ndarray,
                 k_scale: float, ckv_pool: np.ndarray, kpe_pool: np.ndarray) -> int:
    """In-place quantize-on-store into uint8 pools [num_slots, stride].

    ckv_new_bf16: uint16 [n, 512]; kpe_new_bf16: uint16 [n, 64]; slots: int64 [n].
    The pools may be views of one [num_slots, 576] array (kpe = columns 512:).
    Returns the number of out-of-range slots skipped.
    """
    ckv = np.ascontiguousarray(ckv_new_bf16, np.uint16)
    kpe = np.ascontiguousarray(kpe_new_bf16, np.uint16)
    slots = np.ascontiguousarray(slots, np.int64)
    n = slots.shape[0]
    assert ckv.shape == (n, D_CKV) and kpe.shape == (n, D_KPE)
    return int(_load().oracle_kv_store_fp8(
        _ptr(ckv), _ptr(kpe), _ptr(slots), n, np.float32(k_scale),
        ckv_pool.ctypes.data, ckv_pool.strides[0], kpe_pool.ctypes.data,
        kpe_pool.strides[0], ckv_pool.shape[0]))


def double_to_bf16(x) -> np.ndarray:
    """BF16 bits of float64 values rounded once to nearest, ties to even."""
    lib = _load()
    x = np.asarray(x, np.float64)
    return np.array([lib.oracle_double_to_bf16(float(v)) for v in x.ravel()],
                    np.uint16).reshape(x.shape)


def kv_proj_fp8(x_bf16: np.ndarray, w_bf16: np.ndarray, slots: np.ndarray, k_scale: float,
                ckv_pool: np.ndarray, kpe_pool: np.ndarray):
    """KV projection + quantize-on-store.  x_bf16: uint16 [n, d]; w_bf16:
    uint16 [576, d] (row j = weights of latent channel j); pools as for
    kv_store_fp8 (written in place).  Returns (latent BF16 bits [n, 576],
    number of out-of-range slots)."""
    x = np.ascontiguousarray(x_bf16, np.uint16)
    w = np.ascontiguousarray(w_bf16, np.uint16)
    n, d = x.shape
    assert w.shape == (D_ALL, d)
    sl = np.ascontiguousarray(slots, np.int64)
    assert sl.shape == (n,)
    lat = np.zeros((n, D_ALL), np.uint16)
    bad = _load().oracle_kv_proj_fp8(_ptr(x), _ptr(w), n, d, _ptr(sl), float(k_scale),
                                     ckv_pool.ctypes.data, ckv_pool.strides[0],
                                     kpe_pool.ctypes.data, kpe_pool.strides[0], ckv_pool.shape[0],
                                     _ptr(lat))
    return lat, int(bad)


def kv_gather_cast(ckv_pool: np.ndarray, kpe_pool: np.ndarray, kv_indices: np.ndarray,
                   page_size: int, k_scale: float):
    """Gather the listed pages into compact BF16 buffers.

    Returns (ckv_out uint16 [n_pages*page_size, 512], kpe_out uint16 [.., 64]).
    """
    idx = np.ascontiguousarray(kv_indices, np.int32)
    n_rows = idx.shape[0] * page_size
    ckv_out = np.zeros((n_rows, D_CKV), np.uint16)
    kpe_out = np.zeros((n_rows, D_KPE), np.uint16)
    num_slots = ckv_pool.shape[0]
    bad = _load().oracle_kv_gather_cast(
        ckv_pool.ctypes.data, ckv_pool.strides[0], kpe_pool.ctypes.data, kpe_pool.strides[0],
        num_slots, _ptr(idx), idx.shape[0], page_size, np.float32(k_scale),
        _ptr(ckv_out), _ptr(kpe_out))
    if bad:
        raise IndexError(f"{bad} page(s) out of range")
    return ckv_out, kpe_out


def _decode(fn, q_bf16, ckv_pool, kpe_pool, kv_indptr, kv_indices, seq_lens, page_size,
            k_scale, softmax_scale, want_p, nthreads):
    q = np.ascontiguousarray(q_bf16, np.uint16)
    B, H, D = q.shape
    assert D == D_ALL
    indptr = np.ascontiguousarray(kv_indptr, np.int32)
    indices = np.ascontiguousarray(kv_indices, np.int32)
    lens = np.ascontiguousarray(seq_lens, np.int32)
    assert indptr.shape == (B + 1,) and lens.shape == (B,)
    o = np.zeros((B, H, D_CKV), np.float64)
    lse = np.zeros((B, H), np.float64)
    max_len = int(lens.max()) if B else 0
    p = np.zeros((B, H, max(max_len, 1)), np.float64) if want_p else None
    rc = fn(_ptr(q), ckv_pool.ctypes.data, ckv_pool.strides[0], kpe_pool.ctypes.data,
            kpe_pool.strides[0], ckv_pool.shape[0], _ptr(indptr), _ptr(indices), _ptr(lens),
            B, H, int(page_size), float(k_scale), float(softmax_scale), _ptr(o), _ptr(lse),
            _ptr(p), max(max_len, 1), int(nthreads))
    if rc != 0:
        raise IndexError("page table out of range or too short for a sequence")
    return (o, lse, p) if want_p else (o, lse)


def decode_fp8(q_bf16, ckv_pool, kpe_pool, kv_indptr, kv_indices, seq_lens, page_size,
               k_scale, softmax_scale, want_p=False, nthreads=0):
    """fp64 paged MLA decode over E4M3 uint8 pools.

    q_bf16: uint16 [B, H, 576]; pools: uint8 [num_slots, stride] (views allowed).
    Returns o float64 [B, H, 512], lse float64 [B, H] (natural log) and, with
    want_p, the softmax weights p [B, H, max_len].  nthreads 0 = OpenMP default.
    """
    return _decode(_load().oracle_decode_fp8, q_bf16, ckv_pool, kpe_pool, kv_indptr,
                   kv_indices, seq_lens, page_size, k_scale, softmax_scale, want_p, nthreads)


def decode_bf16(q_bf16, ckv_pool, kpe_pool, kv_indptr, kv_indices, seq_lens, page_size,
                k_scale, softmax_scale, want_p=False, nthreads=0):
    """fp64 paged MLA decode over BF16 pools (uint16 [num_slots, stride])."""
    return _decode(_load().oracle_decode_bf16, q_bf16, ckv_pool, kpe_pool, kv_indptr,
                   kv_indices, seq_lens, page_size, k_scale, softmax_scale, want_p, nthreads)


def extend_fp8(q_bf16, ckv_pool, kpe_pool, qo_indptr, kv_indptr, kv_indices, seq_lens,
               page_size, k_scale, softmax_scale, nthreads=0):
    """fp64 causal extend attention over E4M3 uint8 pools.

    q_bf16: uint16 [n_q, H, 576], the new tokens of request b in rows
    qo_indptr[b] .. qo_indptr[b+1]-1; seq_lens count the new tokens.  New
    token i of request b sees the first seq_lens[b] - q_len_b + i + 1 tokens.
    Returns o float64 [n_q, H, 512] and lse float64 [n_q, H] (natural log).
    """
    q = np.ascontiguousarray(q_bf16, np.uint16)
    n_q, H, D = q.shape
    assert D == D_ALL
    qo = np.ascontiguousarray(qo_indptr, np.int32)
    indptr = np.ascontiguousarray(kv_indptr, np.int32)
    indices = np.ascontiguousarray(kv_indices, np.int32)
    lens = np.ascontiguousarray(seq_lens, np.int32)
    B = lens.shape[0]
    assert qo.shape == (B + 1,) and indptr.shape == (B + 1,) and int(qo[-1]) == n_q
    o = np.zeros((n_q, H, D_CKV), np.float64)
    lse = np.zeros((n_q, H), np.float64)
    rc = _load().oracle_extend_fp8(
        _ptr(q), ckv_pool.ctypes.data, ckv_pool.strides[0], kpe_pool.ctypes.data,
        kpe_pool.strides[0], ckv_pool.shape[0], _ptr(qo), _ptr(indptr), _ptr(indices),
        _ptr(lens), B, H, int(page_size), float(k_scale), float(softmax_scale), _ptr(o),
        _ptr(lse), int(nthreads))
    if rc != 0:
        raise IndexError("query lengths, page table or slots inconsistent with the contexts")
    return o, lse


def attention_f64(q: np.ndarray, k: np.ndarray, softmax_scale: float, want_p=False):
    """The attention core on explicit rows: q [H, 576], k [L, 576] (float64)."""
    q = np.ascontiguousarray(q, np.float64)
    k = np.ascontiguousarray(k, np.float64)
    H, L = q.shape[0], k.shape[0]
    o = np.zeros((H, D_CKV), np.float64)
    lse = np.zeros(H, np.float64)
    p = np.zeros((H, max(L, 1)), np.float64) if want_p else None
    _load().oracle_attention_f64(_ptr(q), _ptr(k), L, H, float(softmax_scale), _ptr(o),
                                 _ptr(lse), _ptr(p))
    return (o, lse, p) if want_p else (o, lse)
