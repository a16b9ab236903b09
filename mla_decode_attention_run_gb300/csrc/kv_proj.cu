// kv_proj_store_fp8: the KV projection with the FP8 cache write fused into its
// epilogue.  Each step's new latent (512 c_kv + 64 k_pe channels) leaves the
// attention projection in BF16 and, in the unfused path, is quantized into
// the E4M3 cache by a separate copy ("When a Faster Kernel Doesn't Speed Up
// Serving", section "Step 3: Source Validation", CastToFP8 in
// set_kv_buffer); the same page's "From Attribution to Optimization Targets"
// asks for a projection kernel that emits FP8 itself.  Here one kernel does
// latent = x . W^T on the tensor cores, rounds it to BF16 (the value the
// unfused path would store), quantizes it exactly as kv_store_fp8 does and
// writes the bytes into the tokens' pool rows.
//
// Tiles: 128 tokens (MMA M) x 64 latent channels (MMA N); K in 64-element
// (128-byte) chunks through a 6-stage cp.async ring, 128-byte swizzle.  The
// weights are the bytes that matter when few tokens come in (a decode step:
// 576 x d_model BF16 per layer), so K is split over a thread-block cluster
// of up to 16 CTAs, as wide as still lets every cluster run at once.  Row r
// of the tile belongs to CTA r mod S of the cluster: every CTA writes its
// fp32 partial of row r straight into that CTA's shared memory (distributed
// shared memory), and after one cluster barrier each CTA sums its rows'
// partials in a fixed order (deterministic), rounds, quantizes and stores
// them.  Token rows past the batch are never loaded: warps 3-5 zero them
// once per stage buffer while the first loads are in flight.  No workspace,
// no second launch.
//
// A batch of at most 64 tokens runs M = 64 MMAs: 8 KB token tiles and 4
// stages keep a CTA at 86 KB of shared memory, two per SM.  The kernel is
// launched as a programmatic dependent of the kernel before it: the first
// weight chunks are requested before griddepcontrol.wait, the hidden states
// after it.
//
// Warps: 0-1 load, lane 0 of warp 2 issues the MMAs, warps 2-5 (one per TMEM
// lane quadrant) read the accumulator out.  Waits are bounded; after a
// timeout the CTA still reaches the cluster barrier, so no CTA of its
// cluster waits forever.
#include <array>
#include <cmath>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "tc.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int kPM = 128;                     // token rows per tile beyond 64 tokens (MMA M)
constexpr int kPK = 64;                      // K elements per stage: one 128-byte row
constexpr int kPLoadWarps = 2;
constexpr int kPThreads = 192;
constexpr int kPMaxSplit = 16;               // cluster size (8 is portable; 16 where allowed)

// Shared-memory map for M token rows (MMA M: 128, or 64 for a batch of at
// most 64 tokens, whose smaller tiles let two CTAs share an SM) and N latent
// channels per tile.
template <int N, int M>
struct ProjShape {
    static constexpr int kATile = M * 128;
    static constexpr int kBTile = N * 128;
    static constexpr int kStage = kATile + kBTile;
    static constexpr int kStages = M == 64 ? 4 : 6;
    static constexpr int kRedStride = N + 4;            // floats per partial-tile row (spreads banks)
    static constexpr int kOffRed = kStages * kStage;
    // partial rows received from the cluster: split x ceil(M / split) rows
    static constexpr int kRedRows = M + kPMaxSplit;
    static constexpr int kOffBar = kOffRed + kRedRows * kRedStride * 4;
    static constexpr int kNumBars = 2 * kStages + 2;    // full[], empty[], done, zero
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmem = kOffMisc + 16 + 1024;
    static constexpr uint32_t kTmemCols = N;
    static_assert(kSmem <= 227 * 1024, "shared memory budget");
    static_assert(kDCkv % N == 0 && kDKpe % N == 0, "a channel tile lies in c_kv or in k_pe");
    static_assert(kStage % 1024 == 0 && kATile % 1024 == 0, "swizzle atoms need 1 KB alignment");
};
static_assert(kDQk % 64 == 0 && kDCkv % 64 == 0, "a channel tile lies in c_kv or in k_pe");

struct ProjParams {
    const uint16_t* x;       // BF16 [n][d_model], row stride x_stride (elements)
    int64_t x_stride;
    const uint16_t* w;       // BF16 [576][d_model], row j = weights of latent channel j
    int64_t w_stride;
    int64_t n;
    int32_t kchunks;         // d_model / 64
    const int64_t* slots;
    float k_scale;
    uint8_t* ckv;
    int64_t ckv_stride;
    uint8_t* kpe;
    int64_t kpe_stride;
    int64_t num_slots;
    uint16_t* latent;        // optional BF16 [n][576]
    uint32_t* flags;
};

template <int N, int M>
__global__ void __launch_bounds__(kPThreads, 1) kv_proj_store_kernel(const ProjParams p) {
    using S = ProjShape<N, M>;
    constexpr int kStages = S::kStages;
    constexpr int FULL = 0, EMPTY = kStages, DONE = 2 * kStages, ZERO = 2 * kStages + 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + S::kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + S::kOffMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(base + S::kOffMisc + 4);
    float* red = reinterpret_cast<float*>(base + S::kOffRed);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = gridDim.x;                  // = the cluster size along K
    const int rank = static_cast<int>(cluster_ctarank());
    const int n0 = blockIdx.y * N;
    const int64_t m0 = int64_t(blockIdx.z) * M;
    const int rows = p.n - m0 < M ? static_cast<int>(p.n - m0) : M;   // token rows of this tile
    const int c_lo = p.kchunks * rank / split, c_hi = p.kchunks * (rank + 1) / split;
    const int nch = c_hi - c_lo;                  // >= 1: the host keeps split <= kchunks

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars[FULL + s], 32 * kPLoadWarps);
            mbar_init(&bars[EMPTY + s], 1);
        }
        mbar_init(&bars[DONE], 1);
        mbar_init(&bars[ZERO], 96);
        *abort = 0;
        mbar_fence_init();
    }
    if (warp == 2) tmem_alloc(tmem_slot, S::kTmemCols);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp < kPLoadWarps) {
        // stage = A: M token rows x 128 B (rows past the batch stay zero),
        // B: N weight rows x 128 B; 16-byte chunk c of row r at c ^ (r & 7).
        // The weights do not depend on the kernel before this one (the launch
        // is its programmatic dependent): the first ring's weight chunks go
        // out at once, the hidden states after griddepcontrol.wait.
        const int pre = nch < kStages ? nch : kStages;
        auto load_b = [&](int i) {
            uint8_t* b = base + (i % kStages) * S::kStage + S::kATile;
            const int64_t k0 = int64_t(c_lo + i) * kPK;
#pragma unroll
            for (int j = 0; j < N * 8 / (32 * kPLoadWarps); ++j) {
                const int q = tid + 32 * kPLoadWarps * j, r = q >> 3, c = q & 7;
                cp_async16(b + r * 128 + ((c ^ (r & 7)) << 4), p.w + int64_t(n0 + r) * p.w_stride + k0 + c * 8, 16u);
            }
        };
        auto load_a = [&](int i) {
            uint8_t* a = base + (i % kStages) * S::kStage;
            const int64_t k0 = int64_t(c_lo + i) * kPK;
            for (int q = tid; q < rows * 8; q += 32 * kPLoadWarps) {
                const int r = q >> 3, c = q & 7;
                cp_async16(a + r * 128 + ((c ^ (r & 7)) << 4), p.x + (m0 + r) * p.x_stride + k0 + c * 8, 16u);
            }
        };
        for (int i = 0; i < pre; ++i) load_b(i);        // stages start empty: no wait
        griddep_wait();
        for (int i = 0; i < nch; ++i) {
            const int s = i % kStages;
            const uint32_t u = static_cast<uint32_t>(i / kStages);
            if (!mbar_wait(&bars[EMPTY + s], (u & 1) ^ 1, abort, p.flags)) break;
            if (i >= pre) load_b(i);
            load_a(i);
            // arrives once this thread's copies so far (this stage's among
            // them) have landed
            mbar_arrive_cp_async(&bars[FULL + s]);
        }
        cp_async_wait<0>();
    } else if (warp == 2) {
        if (lane == 0) {
        const uint32_t idesc = idesc_bf16_f32(M, N);
        // the zeroed rows must be in place before the first MMA reads them
        const bool zeroed = mbar_wait(&bars[ZERO], 0, abort, p.flags);
        for (int i = 0; zeroed && i < nch; ++i) {
            const int s = i % kStages;
            const uint32_t u = static_cast<uint32_t>(i / kStages);
            if (!mbar_wait(&bars[FULL + s], u & 1, abort, p.flags)) break;
            fence_after_sync();
            fence_proxy_async_smem();
            const uint32_t sa = smem_u32(base + s * S::kStage);
            const uint64_t ad = smem_desc(sa, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(sa + S::kATile, 16, 1024, kSwizzle128B);
#pragma unroll
            for (int ks = 0; ks < kPK / 16; ++ks)       // K = 16 per MMA: 32 bytes along the row
                mma_bf16(tmem, ad + static_cast<uint64_t>(ks * 2), bd + static_cast<uint64_t>(ks * 2), idesc,
                         i > 0 || ks > 0);
            mma_commit(&bars[EMPTY + s]);                 // the stage may be refilled
        }
        mma_commit(&bars[DONE]);                          // every MMA issued has completed
        }
    } else {
        // warps 3-5: token rows past the batch, zero in every stage, once
        for (int q = rows * 8 + (tid - 96); q < M * 8; q += 96) {
            const int r = q >> 3, c = q & 7;
#pragma unroll 1
            for (int s = 0; s < kStages; ++s)
                *reinterpret_cast<uint4*>(base + s * S::kStage + r * 128 + ((c ^ (r & 7)) << 4)) =
                    make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();                         // visible to the tensor core's reads
        mbar_arrive(&bars[ZERO]);
    }
    __syncwarp();

    // this CTA's partial of tile row r goes to CTA r mod S of the cluster,
    // partial slot [rank][r / S].  M = 128: row r in TMEM lane r; M = 64:
    // rows 16 q .. 16 q + 15 in lanes 0-15 of lane quadrant q
    const int rpo = (M + split - 1) / split;              // rows per owning CTA
    if (warp >= 2) {
        const int q = warp & 3;
        const int row = M == 128 ? q * 32 + lane : (lane < 16 ? q * 16 + lane : M);
        // a drain: the MMA thread commits DONE on every path, and TMEM is read
        // (and later released) only once its MMAs have completed
        volatile int never = 0;
        const bool ok = mbar_wait(&bars[DONE], 0, &never, p.flags, 1000000000ull) && *abort == 0;
        fence_after_sync();
        const int prow = row < rows ? row : 0;            // address only used when row < rows
        const uint32_t dst = cluster_map(smem_u32(red + (rank * rpo + prow / split) * S::kRedStride),
                                         static_cast<uint32_t>(prow % split));
#pragma unroll
        for (int c = 0; c < N; c += 16) {
            uint32_t r[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + c, r);
            tmem_wait_ld();
            if (row < rows) {                             // (a row of M never is)
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                    st_cluster_f4(dst + 4 * (c + e),
                                  ok ? make_float4(__uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                                                   __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]))
                                     : make_float4(0.f, 0.f, 0.f, 0.f));
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    cluster_sync();                                       // every partial row has arrived
    // the next kernel may be launched (a programmatic dependent still waits
    // for this grid to complete before it reads what this grid wrote);
    // signalling here rather than at the start measured faster
    if (tid == 0) griddep_launch_dependents();

    // rows rank, rank + S, ...: sum the S partials (in rank order), round to
    // BF16, quantize, store
    if (warp >= 2) {
        constexpr int kChunks = N / 4;                    // float4 per row
        constexpr int kRowsPerPass = 128 / kChunks;
        const int t = tid - 64;                           // 0..127
        const int c4 = t % kChunks;
        for (int lr = t / kChunks; rank + lr * split < rows; lr += kRowsPerPass) {
            const int r = rank + lr * split;
            float4 acc = *reinterpret_cast<const float4*>(red + lr * S::kRedStride + 4 * c4);
            for (int src = 1; src < split; ++src) {
                const float4 v = *reinterpret_cast<const float4*>(red + (src * rpo + lr) * S::kRedStride + 4 * c4);
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            const uint32_t w01 = pack_bf16x2(acc.x, acc.y), w23 = pack_bf16x2(acc.z, acc.w);
            const int64_t tok = m0 + r;
            if (p.latent)
                *reinterpret_cast<uint2*>(p.latent + tok * kDQk + n0 + 4 * c4) = make_uint2(w01, w23);
            const int64_t slot = p.slots[tok];
            if (slot < 0 || slot >= p.num_slots) {
                if (c4 == 0) raise_flag(p.flags, MLA_FLAG_INDEX_OOB);
                continue;
            }
            const uint32_t bytes = static_cast<uint32_t>(bf16x2_to_e4m3x2_scaled(w01, p.k_scale)) |
                                   (static_cast<uint32_t>(bf16x2_to_e4m3x2_scaled(w23, p.k_scale)) << 16);
            uint8_t* dst = n0 < kDCkv ? p.ckv + slot * p.ckv_stride + n0 : p.kpe + slot * p.kpe_stride + (n0 - kDCkv);
            *reinterpret_cast<uint32_t*>(dst + 4 * c4) = bytes;
        }
    }
    // no CTA touches another's shared memory after the barrier: nobody waits
    if (warp == 2) tmem_dealloc(tmem, S::kTmemCols);
}

std::mutex g_proj_mu;
std::vector<char> g_proj_attr;      // per device: bit (N / 32 - 1): attributes set
std::vector<std::array<int, 2>> g_proj_max_split;  // per device and M: widest cluster accepted
std::vector<std::vector<int>> g_proj_fit;   // per device, per (M, split): clusters that fit at once

template <int N, int M>
mla_status_t launch_proj(const ProjParams& p, int64_t m_tiles, int dev, cudaStream_t stream) {
    using S = ProjShape<N, M>;
    {
        std::lock_guard<std::mutex> lk(g_proj_mu);
        if ((int)g_proj_attr.size() <= dev) g_proj_attr.resize(dev + 1, 0);
        const char bit = static_cast<char>(1 << (M / 64 - 1));
        if (!(g_proj_attr[dev] & bit)) {
            if (cudaFuncSetAttribute(kv_proj_store_kernel<N, M>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     S::kSmem) != cudaSuccess)
                return MLA_ERR_CUDA;
            if ((int)g_proj_max_split.size() <= dev) g_proj_max_split.resize(dev + 1);
            // clusters of 16 are not portable: use them where the device allows
            g_proj_max_split[dev][M / 64 - 1] =
                cudaFuncSetAttribute(kv_proj_store_kernel<N, M>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                        cudaSuccess
                    ? kPMaxSplit
                    : 8;
            cudaGetLastError();
            g_proj_attr[dev] |= bit;
        }
    }
    // split K over the widest cluster (up to 16 CTAs) whose clusters all fit
    // on the GPU at once: a second wave of clusters costs more than a
    // narrower split (measured on GB300 at 40 tokens: 9 tiles split 16
    // 8.3 us, split 8 8.9 us; 32-channel tiles split 8, two waves, 17.3 us)
    const int64_t tiles = m_tiles * (kDQk / N);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = S::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // a programmatic dependent of the kernel before it: CTAs may start (and
    // stream weights) while that kernel finishes; they wait for it on the
    // device before reading the hidden states or writing the pool
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int split = 1;
    int max_split = 8;
    {
        std::lock_guard<std::mutex> lk(g_proj_mu);
        max_split = g_proj_max_split[dev][M / 64 - 1];
    }
    for (int s = max_split < p.kchunks ? max_split : p.kchunks; s > 1; --s) {
        if (tiles * s > device_sm_count()) continue;
        cfg.gridDim = dim3(static_cast<unsigned>(s), kDQk / N, static_cast<unsigned>(m_tiles));
        attr[0].val.clusterDim.x = static_cast<unsigned>(s);
        int fit = -1;
        {
            std::lock_guard<std::mutex> lk(g_proj_mu);
            if ((int)g_proj_fit.size() <= dev) g_proj_fit.resize(dev + 1);
            if (g_proj_fit[dev].empty()) g_proj_fit[dev].assign(2 * (kPMaxSplit + 1), -1);
            int& slot = g_proj_fit[dev][(M / 64 - 1) * (kPMaxSplit + 1) + s];
            if (slot < 0) {
                if (cudaOccupancyMaxActiveClusters(&slot, kv_proj_store_kernel<N, M>, &cfg) != cudaSuccess) {
                    cudaGetLastError();
                    slot = 0;
                }
            }
            fit = slot;
        }
        if (fit >= tiles) {
            split = s;
            break;
        }
    }
    cfg.gridDim = dim3(static_cast<unsigned>(split), kDQk / N, static_cast<unsigned>(m_tiles));
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kv_proj_store_kernel<N, M>, p) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace
}  // namespace mla

extern "C" mla_status_t kv_proj_store_fp8(const void* x, int64_t x_row_stride, const void* w,
                                          int64_t w_row_stride, int64_t n, int32_t d_model,
                                          const int64_t* slots, float k_scale, void* ckv_pool,
                                          int64_t ckv_row_stride_bytes, void* kpe_pool,
                                          int64_t kpe_row_stride_bytes, int64_t num_pool_slots,
                                          void* latent_out, void* stream) {
    using namespace mla;
    if (n < 0) return MLA_ERR_INVALID_ARG;
    if (n == 0) return MLA_OK;
    if (!x || !w || !slots || !ckv_pool || !kpe_pool) return MLA_ERR_INVALID_ARG;
    if (d_model < kPK || d_model > (1 << 16) || d_model % kPK) return MLA_ERR_INVALID_ARG;
    if (x_row_stride < d_model || w_row_stride < d_model || num_pool_slots < 0) return MLA_ERR_INVALID_ARG;
    if (!(k_scale > 0.f) || !std::isfinite(k_scale)) return MLA_ERR_INVALID_ARG;
    if (ckv_row_stride_bytes < kDCkv || kpe_row_stride_bytes < kDKpe) return MLA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || (x_row_stride & 7) || (w_row_stride & 7) || !aligned16(ckv_pool) ||
        !aligned16(kpe_pool) || (ckv_row_stride_bytes & 15) || (kpe_row_stride_bytes & 15) ||
        (latent_out && !aligned16(latent_out)))
        return MLA_ERR_UNSUPPORTED;
    const int64_t m_tiles = (n + kPM - 1) / kPM;
    if (m_tiles > 65535) return MLA_ERR_UNSUPPORTED;
    const bool small = n <= 64;         // one 64-row token tile
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    ProjParams p;
    p.x = static_cast<const uint16_t*>(x);
    p.x_stride = x_row_stride;
    p.w = static_cast<const uint16_t*>(w);
    p.w_stride = w_row_stride;
    p.n = n;
    p.kchunks = d_model / kPK;
    p.slots = slots;
    p.k_scale = k_scale;
    p.ckv = static_cast<uint8_t*>(ckv_pool);
    p.ckv_stride = ckv_row_stride_bytes;
    p.kpe = static_cast<uint8_t*>(kpe_pool);
    p.kpe_stride = kpe_row_stride_bytes;
    p.num_slots = num_pool_slots;
    p.latent = static_cast<uint16_t*>(latent_out);
    p.flags = device_flags_ptr();
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    return small ? launch_proj<64, 64>(p, 1, dev, cs) : launch_proj<64, 128>(p, m_tiles, dev, cs);
}
