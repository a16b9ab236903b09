// mla_decode_run_static_scratch: the decode call for callers that cannot
// allocate device memory.
//
// Who needs it: code that has no device allocator of its own to hand out a
// workspace -- for example a plugin running inside another framework that
// owns all GPU memory, a real-time loop where cudaMalloc's implicit device
// synchronisation is not acceptable, or a caller that must not touch the
// allocator between steps.  mla_decode_run wants a caller-provided workspace
// for its split-KV partials; this variant uses a fixed array compiled into
// the library instead, so the call itself allocates nothing (the plan is
// still built beforehand by mla_decode_plan).
//
// The array (MLA_STATIC_SCRATCH_BYTES) exists once per GPU that loads the
// library and stays allocated until the process exits.  Every call shares
// it, so two calls whose GPU work overlaps (different streams, or several
// host threads) race on it; calls on one stream are ordered and safe.  The
// decode kernel writes every partial it later reads in the same call, so
// nothing in the array has to start at zero and old contents are harmless.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[MLA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (the first call on a device does this; make that first call before
// any stream capture begins).  The address is kept for the life of the
// process: a cudaDeviceReset of the device discards the array with the
// context, so a process that resets a device must not use this call on it
// afterwards.
mla_status_t scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return MLA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MLA_OK;
}

}  // namespace

extern "C" mla_status_t mla_decode_run_static_scratch(
    mla_plan_t plan, const void* q, int64_t q_stride_b, int64_t q_stride_h, const void* ckv_pool,
    int64_t ckv_row_stride_bytes, const void* kpe_pool, int64_t kpe_row_stride_bytes,
    int64_t num_pool_slots, const int32_t* kv_indptr_dev, const int32_t* kv_indices_dev,
    const int32_t* seq_lens_dev, float k_scale, float softmax_scale, void* out, float* lse,
    void* stream) {
    if (!plan) return MLA_ERR_INVALID_ARG;
    size_t need = 0;
    const mla_status_t st = mla_decode_plan_info(plan, nullptr, nullptr, nullptr, &need);
    if (st != MLA_OK) return st;
    if (need > MLA_STATIC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;   // plan needs more scratch
    void* scratch = nullptr;
    const mla_status_t sst = scratch_address(&scratch);
    if (sst != MLA_OK) return sst;
    return mla_decode_run(plan, q, q_stride_b, q_stride_h, ckv_pool, ckv_row_stride_bytes,
                          kpe_pool, kpe_row_stride_bytes, num_pool_slots, kv_indptr_dev,
                          kv_indices_dev, seq_lens_dev, k_scale, softmax_scale, out, lse, scratch,
                          MLA_STATIC_SCRATCH_BYTES, stream);
}
