// Library-wide state: the device flag word, per-device caches, status text,
// and mla_get_last_error.
#include <mutex>
#include <vector>

#include "common.cuh"

namespace {
// OR-ed by kernels on device-detected problems; read and cleared by
// mla_get_last_error.  One word per device (a __device__ variable exists
// once per device context).
__device__ uint32_t g_mla_flags;

std::mutex g_mu;
std::vector<uint32_t*> g_flag_ptr;   // per device ordinal
std::vector<int> g_sm_count;
}  // namespace

namespace mla {

uint32_t* device_flags_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if ((int)g_flag_ptr.size() <= dev) g_flag_ptr.resize(dev + 1, nullptr);
    if (!g_flag_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_mla_flags) != cudaSuccess) return nullptr;
        g_flag_ptr[dev] = static_cast<uint32_t*>(p);
    }
    return g_flag_ptr[dev];
}

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if ((int)g_sm_count.size() <= dev) g_sm_count.resize(dev + 1, 0);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

}  // namespace mla

extern "C" mla_status_t mla_get_last_error(void* stream, uint32_t* device_flags_out) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
    uint32_t* dflags = mla::device_flags_ptr();
    if (!dflags) return MLA_ERR_CUDA;
    uint32_t host = 0;
    if (cudaMemcpy(&host, dflags, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (host != 0) {
        const uint32_t zero = 0;
        if (cudaMemcpy(dflags, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return MLA_ERR_CUDA;
    }
    if (device_flags_out) *device_flags_out = host;
    return host ? MLA_ERR_INDEX_OOB : MLA_OK;
}

extern "C" const char* mla_status_string(mla_status_t status) {
    switch (status) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARG: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
        case MLA_ERR_WORKSPACE: return "workspace missing or too small";
        case MLA_ERR_INDEX_OOB: return "device reported an out-of-range index";
        case MLA_ERR_CUDA: return "CUDA runtime error";
    }
    return "unknown status";
}
