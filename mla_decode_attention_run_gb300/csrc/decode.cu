// mla_decode_run: paged MLA decode attention reading the KV pools in place.
//
// What is computed (per request b, head h; k_t = value(row_t) * k_scale over
// 576 channels, v_t = its first 512): s_t = softmax_scale * q.k_t,
// out = softmax(s) . v, lse = ln sum exp(s).  The pages motivate reading the
// FP8 rows directly instead of casting the pool to BF16 first ("The KV Cache
// Cast Bottleneck", sections "The Context" and "The Message"; "The
// Gather-Then-Cast Pivot", section "The Subject Message"), and the 576 =
// 512 + 64 row split comes from "The KV Cache Cast Bottleneck", "The Context".
//
// Kernel design (one CTA = one token range x 16 heads, 4 warps):
//  * the 16 heads share every KV row (MLA: one latent KV head), so a CTA
//    loads each gathered row once for all 16 heads: QK^T is a [16 x 576] x
//    [576 x 64] tile contraction and PV a [16 x 64] x [64 x 512] one, both on
//    tensor cores (mma.sync m16n8k16, fp32 accumulate);
//  * rows are gathered with 16-byte cp.async (zero fill for masked rows) into
//    a two-stage ring, slot indices prefetched one tile ahead;
//  * E4M3 rows are widened to f16 in shared memory (exact: E4M3 is a subset
//    of f16); q is brought to f16 with a per-head power-of-two scale, so the
//    product is exact and the scale folds into the score multiplier;
//  * online softmax in the log2 domain; warps split QK^T by tokens and PV by
//    output channels (128 each), exchanging the tile max and P through smem;
//  * split-KV: segments of a request spread over CTAs write fp32 partials
//    (normalised o and lse) that the warp-shuffle merge kernel combines.
#include <cmath>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "decode_params.h"
#include "plan.h"

namespace mla {
namespace {

constexpr int kT = kTileTokens;      // 64 tokens per tile
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kRow16 = kDQk + 8;     // padded 16-bit row (584 elements = 1168 B)
constexpr int kPRow = kT + 8;        // padded P row (72 elements)

template <bool kFp8>
struct Smem {
    static constexpr int kRawRow = kFp8 ? kDQk : kRow16 * 2;              // bytes
    static constexpr size_t kQ = 0;
    static constexpr size_t kRaw = kQ + size_t(kHeadsPerCta) * kRow16 * 2;
    static constexpr size_t kKv = kRaw + size_t(2) * kT * kRawRow;        // FP8 only
    static constexpr size_t kP = kKv + (kFp8 ? size_t(kT) * kRow16 * 2 : 0);
    static constexpr size_t kRed = kP + size_t(kHeadsPerCta) * kPRow * 2;
    static constexpr size_t kL = kRed + size_t(kWarps) * kHeadsPerCta * 4;
    static constexpr size_t kCoef = kL + size_t(kWarps) * kHeadsPerCta * 4;
    static constexpr size_t kMask = kCoef + size_t(kHeadsPerCta) * 4;   // 4 tiles x 64 rows
    static constexpr size_t kBytes = kMask + size_t(4) * kT;
};



constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Slot of row (warp + 4*lane) of a tile, for lanes 0..15; -1 if masked.
__device__ __forceinline__ int64_t fetch_slot(const DecodeParams& p, const int32_t* pages,
                                              int32_t t_begin, int32_t t_end, int warp, int lane) {
    if (lane >= 16) return -1;
    const int32_t t = t_begin + warp + 4 * lane;
    if (t >= t_end) return -1;
    const int64_t page = pages[t / p.page_size];
    const int64_t slot = page * p.page_size + t % p.page_size;
    if (page < 0 || slot >= p.num_slots) {
        raise_flag(p.flags, MLA_FLAG_INDEX_OOB);
        return -1;
    }
    return slot;
}

// Gather the 16 rows of this warp (rows warp + 4k) into a raw stage and
// record which rows hold a real token (mask ring slot for this tile).
template <bool kFp8>
__device__ __forceinline__ void issue_rows(const DecodeParams& p, uint8_t* stage, int64_t slot_reg,
                                           uint8_t* mask, int warp, int lane) {
    using S = Smem<kFp8>;
    if (lane < 16) mask[warp + 4 * lane] = slot_reg >= 0 ? 1 : 0;
#pragma unroll 4
    for (int k = 0; k < 16; ++k) {
        const int64_t s = __shfl_sync(0xffffffffu, slot_reg, k);
        const uint32_t n = s >= 0 ? 16u : 0u;
        const int64_t ss = s >= 0 ? s : 0;
        uint8_t* dst = stage + (warp + 4 * k) * S::kRawRow;
        const uint8_t* ck = p.ckv + ss * p.ckv_stride;
        const uint8_t* kp = p.kpe + ss * p.kpe_stride;
        if constexpr (kFp8) {
            cp_async16(dst + 16 * lane, ck + 16 * lane, n);                  // 512 B c_kv
            if (lane < 4) cp_async16(dst + 512 + 16 * lane, kp + 16 * lane, n);  // 64 B k_pe
        } else {
            cp_async16(dst + 16 * lane, ck + 16 * lane, n);                  // 1024 B c_kv
            cp_async16(dst + 512 + 16 * lane, ck + 512 + 16 * lane, n);
            if (lane < 8) cp_async16(dst + 1024 + 16 * lane, kp + 16 * lane, n);  // 128 B k_pe
        }
    }
    cp_async_commit();
}

template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1) mla_decode_mma_kernel(const DecodeParams p) {
    using S = Smem<kFp8>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint16_t* sQ = reinterpret_cast<uint16_t*>(smem + S::kQ);
    uint8_t* sRaw = smem + S::kRaw;
    uint16_t* sKvF16 = reinterpret_cast<uint16_t*>(smem + S::kKv);
    uint16_t* sP = reinterpret_cast<uint16_t*>(smem + S::kP);
    float* sRed = reinterpret_cast<float*>(smem + S::kRed);
    float* sL = reinterpret_cast<float*>(smem + S::kL);
    float* sCoef = reinterpret_cast<float*>(smem + S::kCoef);
    uint8_t* sMask = smem + S::kMask;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, j = lane & 3;
    const int cta = blockIdx.x / p.head_groups;
    const int head0 = (blockIdx.x % p.head_groups) * kHeadsPerCta;

    for (int si = p.cta_ptr[cta]; si < p.cta_ptr[cta + 1]; ++si) {
        const int32_t b = p.segs[4 * si], t0 = p.segs[4 * si + 1], t1 = p.segs[4 * si + 2];
        const int32_t part = p.segs[4 * si + 3];
        if (t1 > p.seq_lens[b]) {                     // device page table != plan
            if (tid == 0) raise_flag(p.flags, MLA_FLAG_PLAN_MISMATCH);
            continue;
        }
        const int32_t* pages = p.indices + p.indptr[b];
        const int n_tiles = (t1 - t0 + kT - 1) / kT;

        // start the KV gather before touching q
        int64_t slot_next = fetch_slot(p, pages, t0, t1, warp, lane);
        issue_rows<kFp8>(p, sRaw, slot_next, sMask, warp, lane);
        slot_next = fetch_slot(p, pages, t0 + kT, t1, warp, lane);
        issue_rows<kFp8>(p, sRaw + kT * S::kRawRow, slot_next, sMask + kT, warp, lane);
        slot_next = fetch_slot(p, pages, t0 + 2 * kT, t1, warp, lane);

        // ---- q rows of this head group -> sQ (16-bit), score multipliers
        for (int r = warp * 4; r < warp * 4 + 4; ++r) {
            const int head = head0 + r;
            const bool valid = head < p.heads;
            const uint4* src = reinterpret_cast<const uint4*>(p.q + b * p.q_sb + head * p.q_sh);
            uint4 v[3];
            float amax = 0.f;
#pragma unroll
            for (int c = 0; c < 3; ++c) {
                const int idx = lane + 32 * c;
                v[c] = (valid && idx < kDQk / 8) ? src[idx] : make_uint4(0, 0, 0, 0);
                const uint32_t w4[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    amax = fmaxf(amax, fabsf(__uint_as_float(w4[e] << 16)));
                    amax = fmaxf(amax, fabsf(__uint_as_float(w4[e] & 0xffff0000u)));
                }
            }
            float coef = valid ? p.softmax_scale * p.k_scale * kLog2e : 0.f;
            float qscale = 1.f;
            if constexpr (kFp8) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                int e = 0;
                frexpf(amax, &e);                    // amax = m * 2^e, m in [0.5, 1)
                int sigma = amax > 0.f ? 15 - e : 0; // max |q| * 2^sigma in [2^14, 2^15)
                sigma = sigma > 100 ? 100 : (sigma < -100 ? -100 : sigma);
                qscale = ldexpf(1.f, sigma);
                coef = ldexpf(coef, -sigma);
            }
#pragma unroll
            for (int c = 0; c < 3; ++c) {
                const int idx = lane + 32 * c;
                if (idx >= kDQk / 8) continue;
                uint4 o = v[c];
                if constexpr (kFp8) {
                    const uint32_t w4[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
                    uint32_t h4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        h4[e] = pack_f16x2(__uint_as_float(w4[e] << 16) * qscale,
                                           __uint_as_float(w4[e] & 0xffff0000u) * qscale);
                    o = make_uint4(h4[0], h4[1], h4[2], h4[3]);
                }
                *reinterpret_cast<uint4*>(sQ + r * kRow16 + idx * 8) = o;
            }
            if (lane == 0) sCoef[r] = coef;
        }
        // (sQ / sCoef become visible at the first barrier of the tile loop)

        float o_acc[16][4];
#pragma unroll
        for (int n = 0; n < 16; ++n) o_acc[n][0] = o_acc[n][1] = o_acc[n][2] = o_acc[n][3] = 0.f;
        float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

        for (int it = 0; it < n_tiles; ++it) {
            const int stage = it & 1;
            uint8_t* raw = sRaw + stage * kT * S::kRawRow;
            cp_async_wait<1>();
            __syncthreads();                                         // (A) tile `it` landed
            const uint16_t* kv;
            if constexpr (kFp8) {
                // widen E4M3 -> f16: 16 bytes in, 32 bytes out per step
                for (int c = tid; c < kT * (kDQk / 16); c += kThreads) {
                    const int row = c / (kDQk / 16), col = c % (kDQk / 16);
                    const uint4 in = *reinterpret_cast<const uint4*>(raw + row * kDQk + col * 16);
                    const uint32_t w4[4] = {in.x, in.y, in.z, in.w};
                    uint32_t h[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        h[2 * e] = e4m3x2_to_f16x2(static_cast<uint16_t>(w4[e] & 0xffffu));
                        h[2 * e + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w4[e] >> 16));
                    }
                    uint4* d = reinterpret_cast<uint4*>(sKvF16 + row * kRow16 + col * 16);
                    d[0] = make_uint4(h[0], h[1], h[2], h[3]);
                    d[1] = make_uint4(h[4], h[5], h[6], h[7]);
                }
                __syncthreads();                                     // (B) f16 tile ready
                if (it + 2 < n_tiles)
                    issue_rows<kFp8>(p, raw, slot_next, sMask + ((it + 2) & 3) * kT, warp, lane);
                else
                    cp_async_commit();
                slot_next = fetch_slot(p, pages, t0 + (it + 3) * kT, t1, warp, lane);
                kv = sKvF16;
            } else {
                kv = reinterpret_cast<const uint16_t*>(raw);
            }

            // ---- S = Q K^T for this warp's 16 tokens (2 n-tiles of 8)
            float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            const uint16_t* qrow = sQ + ((lane & 7) + ((lane >> 3) & 1) * 8) * kRow16 + (lane >> 4) * 8;
            const uint16_t* krow = kv + (16 * warp + (lane & 7) + (lane >> 4) * 8) * kRow16 +
                                   ((lane >> 3) & 1) * 8;
#pragma unroll 4
            for (int kb = 0; kb < kDQk / 16; ++kb) {
                uint32_t a[4], b0, b1, b2, b3;
                ldmatrix_x4(a[0], a[1], a[2], a[3], qrow + kb * 16);
                ldmatrix_x4(b0, b1, b2, b3, krow + kb * 16);
                mma_16816<!kFp8>(sacc[0], a, b0, b1);
                mma_16816<!kFp8>(sacc[1], a, b2, b3);
            }

            // ---- online softmax (log2 domain)
            const int n_valid = min(kT, t1 - t0 - it * kT);
            const uint8_t* tile_mask = sMask + (it & 3) * kT;
            const float c_lo = sCoef[g], c_hi = sCoef[g + 8];
            float s_lo[4], s_hi[4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tok = 16 * warp + 8 * nt + 2 * j + e;
                    const bool ok = tok < n_valid && tile_mask[tok];
                    s_lo[2 * nt + e] = ok ? sacc[nt][e] * c_lo : -INFINITY;
                    s_hi[2 * nt + e] = ok ? sacc[nt][2 + e] * c_hi : -INFINITY;
                }
            }
            float mx_lo = fmaxf(fmaxf(s_lo[0], s_lo[1]), fmaxf(s_lo[2], s_lo[3]));
            float mx_hi = fmaxf(fmaxf(s_hi[0], s_hi[1]), fmaxf(s_hi[2], s_hi[3]));
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
                mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, o));
                mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, o));
            }
            if (j == 0) {
                sRed[warp * kHeadsPerCta + g] = mx_lo;
                sRed[warp * kHeadsPerCta + g + 8] = mx_hi;
            }
            __syncthreads();                                         // (C) tile maxima
            float t_lo = sRed[g], t_hi = sRed[g + 8];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) {
                t_lo = fmaxf(t_lo, sRed[w * kHeadsPerCta + g]);
                t_hi = fmaxf(t_hi, sRed[w * kHeadsPerCta + g + 8]);
            }
            const float mn_lo = fmaxf(m_lo, t_lo), mn_hi = fmaxf(m_hi, t_hi);
            const float al_lo = fast_exp2(m_lo - mn_lo), al_hi = fast_exp2(m_hi - mn_hi);
            m_lo = mn_lo;
            m_hi = mn_hi;
            float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const float p0 = fast_exp2(s_lo[2 * nt] - mn_lo), p1 = fast_exp2(s_lo[2 * nt + 1] - mn_lo);
                const float p2 = fast_exp2(s_hi[2 * nt] - mn_hi), p3 = fast_exp2(s_hi[2 * nt + 1] - mn_hi);
                ps_lo += p0 + p1;
                ps_hi += p2 + p3;
                const int col = 16 * warp + 8 * nt + 2 * j;
                *reinterpret_cast<uint32_t*>(sP + g * kPRow + col) =
                    kFp8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
                *reinterpret_cast<uint32_t*>(sP + (g + 8) * kPRow + col) =
                    kFp8 ? pack_f16x2(p2, p3) : pack_bf16x2(p2, p3);
            }
            l_lo = l_lo * al_lo + ps_lo;
            l_hi = l_hi * al_hi + ps_hi;
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                o_acc[n][0] *= al_lo;
                o_acc[n][1] *= al_lo;
                o_acc[n][2] *= al_hi;
                o_acc[n][3] *= al_hi;
            }
            __syncthreads();                                         // (D) P ready

            // ---- O += P V over this warp's 128 output channels
            const uint16_t* prow = sP + ((lane & 7) + ((lane >> 3) & 1) * 8) * kPRow + (lane >> 4) * 8;
#pragma unroll
            for (int kk = 0; kk < kT / 16; ++kk) {
                uint32_t a[4];
                ldmatrix_x4(a[0], a[1], a[2], a[3], prow + kk * 16);
                const uint16_t* vrow = kv + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * kRow16 +
                                       128 * warp + (lane >> 4) * 8;
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    uint32_t b0, b1, b2, b3;
                    ldmatrix_x4_trans(b0, b1, b2, b3, vrow + 16 * np);
                    mma_16816<!kFp8>(o_acc[2 * np], a, b0, b1);
                    mma_16816<!kFp8>(o_acc[2 * np + 1], a, b2, b3);
                }
            }
            if constexpr (!kFp8) {
                __syncthreads();                                     // (E) raw stage free
                if (it + 2 < n_tiles)
                    issue_rows<kFp8>(p, raw, slot_next, sMask + ((it + 2) & 3) * kT, warp, lane);
                else
                    cp_async_commit();
                slot_next = fetch_slot(p, pages, t0 + (it + 3) * kT, t1, warp, lane);
            }
        }
        cp_async_wait<0>();

        // ---- epilogue: total softmax denominators, normalise, store
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            l_lo += __shfl_xor_sync(0xffffffffu, l_lo, o);
            l_hi += __shfl_xor_sync(0xffffffffu, l_hi, o);
        }
        if (j == 0) {
            sL[warp * kHeadsPerCta + g] = l_lo;
            sL[warp * kHeadsPerCta + g + 8] = l_hi;
        }
        __syncthreads();
        float L_lo = 0.f, L_hi = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            L_lo += sL[w * kHeadsPerCta + g];
            L_hi += sL[w * kHeadsPerCta + g + 8];
        }
        const float vscale = p.k_scale;             // v_t = value * k_scale for both pool types
        const float inv_lo = L_lo > 0.f ? vscale / L_lo : 0.f;
        const float inv_hi = L_hi > 0.f ? vscale / L_hi : 0.f;
        const int h_lo = head0 + g, h_hi = head0 + g + 8;
        const float lse_lo = (m_lo + log2f(L_lo)) * kLn2, lse_hi = (m_hi + log2f(L_hi)) * kLn2;
        if (part < 0) {
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                const int d = 128 * warp + 8 * n + 2 * j;
                if (h_lo < p.heads)
                    *reinterpret_cast<uint32_t*>(p.out + (int64_t(b) * p.heads + h_lo) * kDCkv + d) =
                        pack_bf16x2(o_acc[n][0] * inv_lo, o_acc[n][1] * inv_lo);
                if (h_hi < p.heads)
                    *reinterpret_cast<uint32_t*>(p.out + (int64_t(b) * p.heads + h_hi) * kDCkv + d) =
                        pack_bf16x2(o_acc[n][2] * inv_hi, o_acc[n][3] * inv_hi);
            }
            if (warp == 0 && j == 0) {
                if (h_lo < p.heads) p.lse[int64_t(b) * p.heads + h_lo] = lse_lo;
                if (h_hi < p.heads) p.lse[int64_t(b) * p.heads + h_hi] = lse_hi;
            }
        } else {
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                const int d = 128 * warp + 8 * n + 2 * j;
                if (h_lo < p.heads)
                    *reinterpret_cast<float2*>(p.part_o + (int64_t(part) * p.heads + h_lo) * kDCkv + d) =
                        make_float2(o_acc[n][0] * inv_lo, o_acc[n][1] * inv_lo);
                if (h_hi < p.heads)
                    *reinterpret_cast<float2*>(p.part_o + (int64_t(part) * p.heads + h_hi) * kDCkv + d) =
                        make_float2(o_acc[n][2] * inv_hi, o_acc[n][3] * inv_hi);
            }
            if (warp == 0 && j == 0) {
                if (h_lo < p.heads) p.part_lse[int64_t(part) * p.heads + h_lo] = lse_lo;
                if (h_hi < p.heads) p.part_lse[int64_t(part) * p.heads + h_hi] = lse_hi;
            }
        }
        __syncthreads();                                             // smem reuse by the next segment
    }
}

// Combine split-KV partials.  One block of 128 threads per output row
// (request x head, or a query block's row), thread t owning channels
// 4t .. 4t + 3.  Entry e: output rows row0 .. row0 + rows - 1 from partials
// first .. first + n - 1, row h of each at partial row h (part_rows rows per
// partial).  Partials are taken kBatch at a time (their lse and o loads all
// in flight together), folded in with a running maximum:
//   m' = max(m, max_i lse_i);  acc = acc * e^(m - m') + sum_i e^(lse_i - m') o_i
// so a request split into n partials costs about n / kBatch memory round
// trips.  kBatch = 8 keeps a block small enough for a batch's rows to run in
// one wave; plans with more pieces per request (one long request spread over
// many CTAs) have few rows and take 16 at a time (measured on GB300 for a
// 4,096-token request in 33 pieces: 12.5 us per call, 12.8 with 8 at a time,
// 12.7 with 32).
template <int kBatch>
__global__ void __launch_bounds__(128)
mla_merge_kernel(const int32_t* __restrict__ merge, int n_merge, int part_rows,
                 const float* __restrict__ part_o, const float* __restrict__ part_lse,
                 uint16_t* __restrict__ out, float* __restrict__ lse) {
    const int e = blockIdx.x, h = blockIdx.y, t = threadIdx.x;
    // the merge table is the plan's, on the device before the call began:
    // read it while the decode kernel still runs
    int4 ent = make_int4(0, 0, 0, 0);
    if (e < n_merge) ent = reinterpret_cast<const int4*>(merge)[e];
    griddep_wait();                                 // the decode kernel's partials are complete
    const int row0 = ent.x, first = ent.y, n = ent.z, rows = ent.w;
    if (e >= n_merge || h >= rows) return;
    const int64_t row = int64_t(row0) + h;
    uint16_t* dst = out + row * kDCkv + 4 * t;
    if (n == 0) {                                   // empty context: o = 0, lse = -inf
        *reinterpret_cast<uint2*>(dst) = make_uint2(0, 0);
        if (t == 0) lse[row] = -INFINITY;
        return;
    }
    float m = -INFINITY, wsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const uint64_t once = l2_policy(false);         // each partial is read once
    for (int c = 0; c < n; c += kBatch) {
        float l[kBatch];
        float4 v[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const bool ok = c + i < n;
            const int64_t pr = int64_t(first + (ok ? c + i : 0)) * part_rows + h;
            // a partial whose tokens the row cannot see (extend) has lse = -inf
            // and o = 0: weight 0
            l[i] = ok ? ld_f32_hint(part_lse + pr, once) : -INFINITY;
            v[i] = ok ? ld_f32x4_hint(reinterpret_cast<const float4*>(part_o + pr * kDCkv) + t, once)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mc = m;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) mc = fmaxf(mc, l[i]);
        const float r = m == -INFINITY ? 0.f : expf(m - mc);
        acc.x *= r;
        acc.y *= r;
        acc.z *= r;
        acc.w *= r;
        wsum *= r;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const float w = l[i] == -INFINITY ? 0.f : expf(l[i] - mc);
            wsum += w;
            acc.x += w * v[i].x;
            acc.y += w * v[i].y;
            acc.z += w * v[i].z;
            acc.w += w * v[i].w;
        }
        m = mc;
    }
    const float inv = 1.f / wsum;
    *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
    if (t == 0) lse[row] = m + logf(wsum);
}

std::mutex g_attr_mu;
std::vector<int> g_attr_done;   // per device: bit0 fp8 kernel, bit1 bf16 kernel

template <bool kFp8>
cudaError_t ensure_smem_attr() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if ((int)g_attr_done.size() <= dev) g_attr_done.resize(dev + 1, 0);
    const int bit = kFp8 ? 1 : 2;
    if (!(g_attr_done[dev] & bit)) {
        e = cudaFuncSetAttribute(mla_decode_mma_kernel<kFp8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(Smem<kFp8>::kBytes));
        if (e != cudaSuccess) return e;
        g_attr_done[dev] |= bit;
    }
    return cudaSuccess;
}

}  // namespace
}  // namespace mla

namespace {

// The run() half shared by decode and extend plans: checks, then the q split
// + decode (+ merge) launches.  q_stride_b steps a request (decode) or a new
// token (extend).
mla_status_t run_plan(mla_plan_t plan, bool extend, const void* q, int64_t q_stride_b,
                      int64_t q_stride_h, const void* ckv_pool, int64_t ckv_row_stride_bytes,
                      const void* kpe_pool, int64_t kpe_row_stride_bytes, int64_t num_pool_slots,
                      const int32_t* kv_indptr_dev, const int32_t* kv_indices_dev,
                      const int32_t* seq_lens_dev, float k_scale, float softmax_scale, void* out,
                      float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    using namespace mla;
    if (!plan || !q || !ckv_pool || !kpe_pool || !kv_indptr_dev || !seq_lens_dev || !out || !lse)
        return MLA_ERR_INVALID_ARG;
    const Schedule& s = plan->sched;
    if (s.extend != extend) return MLA_ERR_INVALID_ARG;    // a decode plan for extend or back
    if (s.n_tokens > 0 && !kv_indices_dev) return MLA_ERR_INVALID_ARG;
    if (num_pool_slots < 0) return MLA_ERR_INVALID_ARG;
    if (!(k_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(softmax_scale))
        return MLA_ERR_INVALID_ARG;
    if (q_stride_h < kDQk || q_stride_b < 0) return MLA_ERR_INVALID_ARG;
    if (!aligned16(q) || (q_stride_b & 7) || (q_stride_h & 7) || !aligned16(ckv_pool) ||
        !aligned16(kpe_pool) || (ckv_row_stride_bytes & 15) || (kpe_row_stride_bytes & 15) ||
        ckv_row_stride_bytes <= 0 || kpe_row_stride_bytes <= 0 || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return MLA_ERR_UNSUPPORTED;
    if (s.workspace_bytes > 0) {
        if (!workspace || workspace_bytes < s.workspace_bytes) return MLA_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return MLA_ERR_WORKSPACE;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device) return MLA_ERR_INVALID_ARG;
    const bool fp8 = s.kv_dtype == MLA_KV_FP8_E4M3;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);

    DecodeParams p;
    p.q = static_cast<const uint16_t*>(q);
    p.q_sb = q_stride_b;
    p.q_sh = q_stride_h;
    p.ckv = static_cast<const uint8_t*>(ckv_pool);
    p.ckv_stride = ckv_row_stride_bytes;
    p.kpe = static_cast<const uint8_t*>(kpe_pool);
    p.kpe_stride = kpe_row_stride_bytes;
    p.num_slots = num_pool_slots;
    p.indptr = kv_indptr_dev;
    p.indices = kv_indices_dev;
    p.seq_lens = seq_lens_dev;
    p.page_size = s.page_size;
    set_page_divider(p);
    p.heads = s.heads;
    p.head_groups = s.head_groups;
    p.k_scale = k_scale;
    p.softmax_scale = softmax_scale;
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse;
    p.part_o = static_cast<float*>(workspace);
    p.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + s.partial_lse_offset);
    p.cta_ptr = plan->dev_meta + plan->off_cta;
    p.segs = plan->dev_meta + plan->off_segs;
    p.seg_pages = plan->dev_meta + plan->off_seg_pages;
    p.flags = device_flags_ptr();
    p.qimg = static_cast<uint8_t*>(workspace) + s.qimg_offset;
    p.batch = s.batch;
    p.group_heads = s.group_heads;
    p.part_rows = s.part_rows;
    p.blocks = s.extend ? plan->dev_meta + plan->off_blocks : nullptr;
    p.n_blocks = s.n_blocks();

    if (s.kernel == DecodeKernel::kTc && num_pool_slots >= INT32_MAX) return MLA_ERR_UNSUPPORTED;
    if (s.num_ctas > 0 && s.kernel == DecodeKernel::kTc) {
        // each range's segments and first segment travel with the launch
        // (kept in the plan: built once per plan, reused by every run)
        if (launch_decode_tc(p, plan->ranges, s.num_ctas, cs) != cudaSuccess) return MLA_ERR_CUDA;
    } else if (s.num_ctas > 0) {
        const dim3 grid(s.num_ctas * s.head_groups);
        cudaError_t e;
        if (fp8) {
            e = ensure_smem_attr<true>();
            if (e != cudaSuccess) return MLA_ERR_CUDA;
            mla_decode_mma_kernel<true><<<grid, kThreads, Smem<true>::kBytes, cs>>>(p);
        } else {
            e = ensure_smem_attr<false>();
            if (e != cudaSuccess) return MLA_ERR_CUDA;
            mla_decode_mma_kernel<false><<<grid, kThreads, Smem<false>::kBytes, cs>>>(p);
        }
        if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
    }
    if (s.n_merge() > 0) {
        // a programmatic dependent of the decode kernel: its launch is
        // processed while the decode's last CTAs finish, and its blocks wait
        // on the device for the decode's partials (released at CTA start
        // instead, blocks parked beside 16-head CTAs slowed the decode by
        // 1.4 us per call on GB300)
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(s.n_merge(), s.part_rows);
        cfg.blockDim = dim3(128);
        cfg.stream = cs;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, s.max_merge_parts > 8 ? mla_merge_kernel<16> : mla_merge_kernel<8>,
                               static_cast<const int32_t*>(plan->dev_meta + plan->off_merge),
                               static_cast<int>(s.n_merge()), static_cast<int>(s.part_rows),
                               static_cast<const float*>(p.part_o), static_cast<const float*>(p.part_lse), p.out,
                               p.lse) != cudaSuccess)
            return MLA_ERR_CUDA;
    }
    return MLA_OK;
}

}  // namespace

extern "C" mla_status_t mla_decode_run(mla_plan_t plan, const void* q, int64_t q_stride_b,
                                       int64_t q_stride_h, const void* ckv_pool,
                                       int64_t ckv_row_stride_bytes, const void* kpe_pool,
                                       int64_t kpe_row_stride_bytes, int64_t num_pool_slots,
                                       const int32_t* kv_indptr_dev, const int32_t* kv_indices_dev,
                                       const int32_t* seq_lens_dev, float k_scale,
                                       float softmax_scale, void* out, float* lse, void* workspace,
                                       size_t workspace_bytes, void* stream) {
    return run_plan(plan, false, q, q_stride_b, q_stride_h, ckv_pool, ckv_row_stride_bytes,
                    kpe_pool, kpe_row_stride_bytes, num_pool_slots, kv_indptr_dev, kv_indices_dev,
                    seq_lens_dev, k_scale, softmax_scale, out, lse, workspace, workspace_bytes,
                    stream);
}

extern "C" mla_status_t mla_extend_run(mla_plan_t plan, const void* q, int64_t q_stride_tok,
                                       int64_t q_stride_h, const void* ckv_pool,
                                       int64_t ckv_row_stride_bytes, const void* kpe_pool,
                                       int64_t kpe_row_stride_bytes, int64_t num_pool_slots,
                                       const int32_t* kv_indptr_dev, const int32_t* kv_indices_dev,
                                       const int32_t* seq_lens_dev, float k_scale,
                                       float softmax_scale, void* out, float* lse, void* workspace,
                                       size_t workspace_bytes, void* stream) {
    return run_plan(plan, true, q, q_stride_tok, q_stride_h, ckv_pool, ckv_row_stride_bytes,
                    kpe_pool, kpe_row_stride_bytes, num_pool_slots, kv_indptr_dev, kv_indices_dev,
                    seq_lens_dev, k_scale, softmax_scale, out, lse, workspace, workspace_bytes,
                    stream);
}

extern "C" mla_status_t mla_debug_set_wait_limit(uint64_t limit_ns) {
    return mla::set_decode_wait_limit(limit_ns) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
