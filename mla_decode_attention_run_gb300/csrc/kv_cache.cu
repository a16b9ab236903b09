// Companion kernels of the FP8 KV cache:
//  * kv_store_fp8   -- quantize-on-store scatter of new BF16 latents into the
//    E4M3 pools ("When a Faster Kernel Doesn't Speed Up Serving", section
//    "Step 3: Source Validation", CastToFP8 in set_kv_buffer: the BF16->FP8
//    cast and the scatter become one pass);
//  * kv_gather_cast -- active-page gather + E4M3->BF16 cast into a compact
//    buffer ("The Gather-Then-Cast Pivot", section "The Reasoning Process").
// Both are HBM-bound streaming kernels: 16-byte loads and stores per thread,
// grid sized in multiples of the SM count.
#include "common.cuh"

namespace mla {
namespace {

constexpr uint32_t kBf16QuietNaN = 0x7FC0u;
constexpr int kStoreUnitsPerRow = (kDCkv + kDKpe) / 8;   // 8 elements per thread
constexpr int kGatherUnitsPerRow = (kDCkv + kDKpe) / 16; // 16 bytes per thread

__global__ void __launch_bounds__(256)
kv_store_fp8_kernel(const uint16_t* __restrict__ ckv_new, const uint16_t* __restrict__ kpe_new,
                    const int64_t* __restrict__ slots, int64_t n, float k_scale,
                    uint8_t* __restrict__ ckv_pool, int64_t ckv_stride,
                    uint8_t* __restrict__ kpe_pool, int64_t kpe_stride, int64_t num_slots,
                    uint32_t* flags) {
    const int64_t total = n * kStoreUnitsPerRow;
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = u / kStoreUnitsPerRow;
        const int k = static_cast<int>(u % kStoreUnitsPerRow);
        const int64_t slot = slots[i];
        if (slot < 0 || slot >= num_slots) {
            if (k == 0) raise_flag(flags, MLA_FLAG_INDEX_OOB);
            continue;
        }
        const uint16_t* src;
        uint8_t* dst;
        if (k < kDCkv / 8) {
            src = ckv_new + i * kDCkv + 8 * k;
            dst = ckv_pool + slot * ckv_stride + 8 * k;
        } else {
            src = kpe_new + i * kDKpe + 8 * (k - kDCkv / 8);
            dst = kpe_pool + slot * kpe_stride + 8 * (k - kDCkv / 8);
        }
        const uint4 in = *reinterpret_cast<const uint4*>(src);
        const uint32_t w[4] = {in.x, in.y, in.z, in.w};
        uint32_t packed[2];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            uint32_t bytes = 0;
#pragma unroll
            for (int q = 0; q < 2; ++q)
                bytes |= static_cast<uint32_t>(bf16x2_to_e4m3x2_scaled(w[2 * p + q], k_scale)) << (16 * q);
            packed[p] = bytes;
        }
        *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
    }
}

__global__ void __launch_bounds__(256)
kv_gather_cast_kernel(const uint8_t* __restrict__ ckv_pool, int64_t ckv_stride,
                      const uint8_t* __restrict__ kpe_pool, int64_t kpe_stride,
                      int64_t num_slots, const int32_t* __restrict__ kv_indices,
                      int64_t n_pages, int32_t page_size, float k_scale,
                      uint16_t* __restrict__ ckv_out, uint16_t* __restrict__ kpe_out,
                      uint32_t* flags) {
    const int64_t rows = n_pages * page_size;
    const int64_t total = rows * kGatherUnitsPerRow;
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < total;
         u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = u / kGatherUnitsPerRow;
        const int c = static_cast<int>(u % kGatherUnitsPerRow);
        const int64_t j = row / page_size;
        const int64_t r = row % page_size;
        const int64_t page = kv_indices[j];
        if (page < 0 || page * page_size + page_size > num_slots) {
            if (c == 0) raise_flag(flags, MLA_FLAG_INDEX_OOB);
            continue;
        }
        const int64_t slot = page * page_size + r;
        const uint8_t* src;
        uint16_t* dst;
        if (c < kDCkv / 16) {
            src = ckv_pool + slot * ckv_stride + 16 * c;
            dst = ckv_out + row * kDCkv + 16 * c;
        } else {
            src = kpe_pool + slot * kpe_stride + 16 * (c - kDCkv / 16);
            dst = kpe_out + row * kDKpe + 16 * (c - kDCkv / 16);
        }
        const uint4 in = *reinterpret_cast<const uint4*>(src);
        const uint32_t w[4] = {in.x, in.y, in.z, in.w};
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t f16x2 = e4m3x2_to_f16x2(static_cast<uint16_t>(w[q] >> (16 * h)));
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&f16x2));
                uint32_t v = pack_bf16x2(__fmul_rn(f.x, k_scale), __fmul_rn(f.y, k_scale));
                // the NaN codes 0x7F / 0xFF give the quiet NaN 0x7FC0 whatever
                // their sign, as PyTorch's float8_e4m3fn -> bfloat16 cast does
                if (f.x != f.x) v = (v & 0xFFFF0000u) | kBf16QuietNaN;
                if (f.y != f.y) v = (v & 0x0000FFFFu) | (kBf16QuietNaN << 16);
                o[2 * q + h] = v;
            }
        }
        uint4* d = reinterpret_cast<uint4*>(dst);
        d[0] = make_uint4(o[0], o[1], o[2], o[3]);
        d[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

int grid_for(int64_t units, int threads) {
    const int64_t want = (units + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(device_sm_count() > 0 ? device_sm_count() : 148) * 16;
    return static_cast<int>(want < cap ? want : cap);
}

bool scale_ok(float k) { return k > 0.0f && k < __builtin_huge_valf(); }

}  // namespace
}  // namespace mla

extern "C" mla_status_t kv_store_fp8(const void* ckv_new, const void* kpe_new,
                                     const int64_t* slots, int64_t n, float k_scale,
                                     void* ckv_pool, int64_t ckv_row_stride_bytes,
                                     void* kpe_pool, int64_t kpe_row_stride_bytes,
                                     int64_t num_pool_slots, void* stream) {
    using namespace mla;
    if (n < 0 || num_pool_slots < 0) return MLA_ERR_INVALID_ARG;
    if (n == 0) return MLA_OK;
    if (!ckv_new || !kpe_new || !slots || !ckv_pool || !kpe_pool) return MLA_ERR_INVALID_ARG;
    if (!scale_ok(k_scale)) return MLA_ERR_INVALID_ARG;
    if (!aligned16(ckv_new) || !aligned16(kpe_new) || !aligned16(ckv_pool) ||
        !aligned16(kpe_pool) || (reinterpret_cast<uintptr_t>(slots) & 7u))
        return MLA_ERR_UNSUPPORTED;
    if (ckv_row_stride_bytes <= 0 || kpe_row_stride_bytes <= 0 || (ckv_row_stride_bytes & 15) ||
        (kpe_row_stride_bytes & 15))
        return MLA_ERR_UNSUPPORTED;
    const int threads = 256;
    const int grid = grid_for(n * kStoreUnitsPerRow, threads);
    kv_store_fp8_kernel<<<grid, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(ckv_new), static_cast<const uint16_t*>(kpe_new), slots, n,
        k_scale, static_cast<uint8_t*>(ckv_pool), ckv_row_stride_bytes,
        static_cast<uint8_t*>(kpe_pool), kpe_row_stride_bytes, num_pool_slots,
        device_flags_ptr());
    return cuda_status(cudaGetLastError());
}

extern "C" mla_status_t kv_gather_cast(const void* ckv_pool, int64_t ckv_row_stride_bytes,
                                       const void* kpe_pool, int64_t kpe_row_stride_bytes,
                                       int64_t num_pool_slots, const int32_t* kv_indices,
                                       int64_t n_pages, int32_t page_size, float k_scale,
                                       void* ckv_out, void* kpe_out, void* stream) {
    using namespace mla;
    if (n_pages < 0 || page_size <= 0 || num_pool_slots < 0) return MLA_ERR_INVALID_ARG;
    if (n_pages == 0) return MLA_OK;
    if (!ckv_pool || !kpe_pool || !kv_indices || !ckv_out || !kpe_out) return MLA_ERR_INVALID_ARG;
    if (!scale_ok(k_scale)) return MLA_ERR_INVALID_ARG;
    if (!aligned16(ckv_pool) || !aligned16(kpe_pool) || !aligned16(ckv_out) ||
        !aligned16(kpe_out))
        return MLA_ERR_UNSUPPORTED;
    if (ckv_row_stride_bytes <= 0 || kpe_row_stride_bytes <= 0 || (ckv_row_stride_bytes & 15) ||
        (kpe_row_stride_bytes & 15))
        return MLA_ERR_UNSUPPORTED;
    const int threads = 256;
    const int grid = grid_for(n_pages * page_size * kGatherUnitsPerRow, threads);
    kv_gather_cast_kernel<<<grid, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(ckv_pool), ckv_row_stride_bytes,
        static_cast<const uint8_t*>(kpe_pool), kpe_row_stride_bytes, num_pool_slots, kv_indices,
        n_pages, page_size, k_scale, static_cast<uint16_t*>(ckv_out),
        static_cast<uint16_t*>(kpe_out), device_flags_ptr());
    return cuda_status(cudaGetLastError());
}
