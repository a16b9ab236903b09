// Shared device helpers for libmla_decode.so (sm_103a only).
//
// Inline PTX wrappers for the few instructions the kernels need: 16-byte
// cp.async with zero fill, ldmatrix, mma.sync, E4M3 <-> f16 / f32
// conversions, and exp2.  Nothing here computes the method by itself.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/mla_decode.h"

#define MLA_DEVINLINE __device__ __forceinline__

namespace mla {

constexpr int kDCkv = MLA_D_CKV;   // 512
constexpr int kDKpe = MLA_D_KPE;   // 64
constexpr int kDQk = MLA_D_QK;     // 576

// ---------------------------------------------------------------- host side

// Device pointer of this library's flag word on the current device.
uint32_t* device_flags_ptr();
// SM count of the current device (cached per device).
int device_sm_count();
// Maps a cudaError_t to a status, recording nothing else.
inline mla_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------- device side

MLA_DEVINLINE uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Split-KV partials are written by the decode and read once by the merge at
// the end of the call, and query images are written by the q split and read
// at each segment start, while the call streams far more than L2 holds: both
// are stored with L2 priority evict_last; the merge reads the partials with
// evict_first (cache-policy operands covering every access they are given to).
MLA_DEVINLINE uint64_t l2_policy(bool keep) {
    uint64_t pol;
    if (keep) asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol));
    else asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}
MLA_DEVINLINE void st_f32_hint(float* ptr, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;\n" :: "l"(ptr), "f"(v), "l"(pol) : "memory");
}
MLA_DEVINLINE void st_v4_hint(void* ptr, const uint4& v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;\n"
                 :: "l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol) : "memory");
}
MLA_DEVINLINE float ld_f32_hint(const float* ptr, uint64_t pol) {
    float v;
    asm volatile("ld.global.L2::cache_hint.f32 %0, [%1], %2;\n" : "=f"(v) : "l"(ptr), "l"(pol));
    return v;
}
MLA_DEVINLINE float4 ld_f32x4_hint(const float4* ptr, uint64_t pol) {
    float4 v;
    asm volatile("ld.global.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(ptr), "l"(pol));
    return v;
}

// 16-byte async copy global -> shared.  src_bytes = 0 writes zeros and reads
// nothing (used for masked rows).
MLA_DEVINLINE void cp_async16(void* smem, const void* gmem, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
                 :: "r"(smem_u32(smem)), "l"(gmem), "r"(src_bytes) : "memory");
}
MLA_DEVINLINE void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
MLA_DEVINLINE void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" :: "n"(N) : "memory"); }

MLA_DEVINLINE void ldmatrix_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                               const void* smem_row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(smem_u32(smem_row)));
}
MLA_DEVINLINE void ldmatrix_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                     const void* smem_row) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(smem_u32(smem_row)));
}

// D += A * B, m16n8k16, fp32 accumulate; A/B both f16 or both bf16.
template <bool kBf16>
MLA_DEVINLINE void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (kBf16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
}

// Two E4M3 bytes (low byte = first element) -> f16x2 (low half = first).
// Exact: every E4M3 value is an f16 value.
MLA_DEVINLINE uint32_t e4m3x2_to_f16x2(uint16_t two) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(two));
    return r;
}

// Two floats -> two E4M3 bytes (round to nearest even, saturating finite).
// Returns first element in the low byte.
MLA_DEVINLINE uint16_t f32x2_to_e4m3x2(float first, float second) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(second), "f"(first));
    return r;
}

// Quantize-on-store of two BF16 values (one 32-bit word, first value in the
// low half): each is widened exactly to fp32, divided by k_scale in one IEEE
// division and rounded to E4M3 (nearest even, saturating; NaN -> 0x7F).
// Returns the first byte in the low byte.
MLA_DEVINLINE uint16_t bf16x2_to_e4m3x2_scaled(uint32_t word, float k_scale) {
    const float a = __fdiv_rn(__uint_as_float(word << 16), k_scale);
    const float b = __fdiv_rn(__uint_as_float(word & 0xFFFF0000u), k_scale);
    uint16_t two = f32x2_to_e4m3x2(a, b);
    // NaN encodes as the canonical 0x7F whatever its sign
    if (a != a) two = static_cast<uint16_t>((two & 0xFF00u) | 0x7Fu);
    if (b != b) two = static_cast<uint16_t>((two & 0x00FFu) | 0x7F00u);
    return two;
}

// Two f16 (low half = first) -> two E4M3 bytes (nearest even, saturating).
MLA_DEVINLINE uint16_t f16x2_to_e4m3x2(uint32_t h) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;\n" : "=h"(r) : "r"(h));
    return r;
}
MLA_DEVINLINE uint32_t sub_f16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
MLA_DEVINLINE uint32_t mul_f16x2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

MLA_DEVINLINE uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
MLA_DEVINLINE uint32_t pack_f16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

MLA_DEVINLINE float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before its predecessor in the stream finishes;
// griddep_wait() blocks the calling thread until the predecessor grid has
// completed and its writes are visible, and griddep_launch_dependents() lets
// the next such kernel start once every block of this grid has called it.
MLA_DEVINLINE void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
MLA_DEVINLINE void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// Out of line: it runs only on an error, and each inlined copy of the atomic
// costs code in the paths that call it.
static __device__ __noinline__ void raise_flag(uint32_t* flags, uint32_t bit) {
    if (flags) atomicOr(flags, bit);
}

}  // namespace mla
