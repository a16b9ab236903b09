// Paged MLA decode on Blackwell tensor cores, reading the E4M3 cache in place.
//
// Same computation as the mma.sync kernel (decode.cu): per request and head,
// s_t = softmax_scale * q . k_t over 576 channels with k_t = value(row_t) *
// k_scale, o = softmax(s) . v (512 channels), lse.  The pages' goal is that
// the attention kernel consume the FP8 cache directly instead of a BF16 copy
// ("The KV Cache Cast Bottleneck", section "The Message"; "The Gather-Then-Cast
// Pivot", section "The Subject Message").  Here the FP8 bytes are the tensor
// core operands themselves: nothing is converted.
//
// Exact operand splitting.  tcgen05.mma kind::f8f6f4 multiplies E4M3 by
// E4M3.  The BF16 query of each head is scaled by a power of two 2^sigma and
// written as the sum of two E4M3 numbers, q * 2^sigma = q1 + q2 (q1 the
// nearest E4M3, q2 the nearest E4M3 to the remainder); a BF16 value has 8
// significant bits and each term carries 4, so the sum is exact whenever both
// terms are normal -- anything smaller than 2^-14 of the head's largest entry
// may lose bits, far below the output's BF16 rounding.  Likewise the softmax
// weights p * 256 = p1 + p2 (8 significant bits, like a BF16 P).  The two
// terms are stacked along N, so one MMA computes both partial products and
// reads the cache tile once.
//
// Tile = 128 tokens = the MMA's M.  Per tile:
//   S^T[128 x 32]  = K_tile[128 x 576] . [q1;q2]^T    18 MMAs, K-major A/B
//   O^T[512 x 32] += V^T[512 x 128] . [P1;P2]^T       16 MMAs, MN-major A/B
// The same 128-byte-swizzled smem tile serves as K-major A (tokens x dims)
// and MN-major A (dims x tokens); S and O live in TMEM.
//
// Warp roles (one CTA per SM, persistent over its token range):
//   warps 0-1  gather the tile's rows with 16-byte cp.async into a 2-stage
//              ring (arrive on the stage's mbarrier when the copies land);
//   warp 2     one thread issues every tcgen05.mma and commit;
//   warp 3     prepares [q1;q2] and the per-head score multipliers for each
//              segment (double-buffered; lane = half a head row);
//   warps 4-7  one thread per TMEM lane: online softmax of a token's 16
//              heads, the E4M3 split of P, then the O correction (lane =
//              output channel) and the epilogue.
// Every mbarrier wait is bounded; on a timeout the CTA sets
// MLA_FLAG_WAIT_TIMEOUT, drains its MMAs and copies, frees TMEM and exits.
#include <mutex>
#include <vector>

#include "common.cuh"
#include "decode_params.h"
#include "plan.h"
#include "tc.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int kTT = kTcTileTokens;          // 128 tokens per tile (MMA M)
constexpr int kThreads = 256;
constexpr int kBlk = kTT * 128;             // one 128-row x 128-byte SW128 column block
constexpr int kNBlk = 5;                    // 4 c_kv blocks + the k_pe block (64 of 128 B)
constexpr int kStage = kNBlk * kBlk;        // 80 KB
constexpr int kQRows = 2 * kHeadsPerCta;    // B rows: q1 of heads 0..15, then q2
constexpr int kQBlk = kQRows * 128;         // 4 KB
constexpr int kQBytes = kNBlk * kQBlk;      // 20 KB
constexpr int kPUnit = kTT * 16;            // one E4M3 term of P^T: 128 tokens x 16 heads
constexpr int kPBytes = 2 * kPUnit;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;               // S[j]: columns 32j .. 32j+31
constexpr uint32_t kColO = 64;              // O[j]: 64 + 128j + 32mb (mb = 128-channel block)
constexpr int kKSteps = kDQk / 32;          // 18 k-steps of 32 channels for QK
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kOffStage = 0;
constexpr int kOffQ = kOffStage + 2 * kStage;
constexpr int kOffP = kOffQ + 2 * kQBytes;
constexpr int kOffBar = kOffP + 2 * kPBytes;
constexpr int kOffRed = kOffBar + 256;      // tile maxima: 2 x 4 warps x 16
constexpr int kOffLsum = kOffRed + 512;     // softmax denominators: 4 warps x 16
constexpr int kOffCoef = kOffLsum + 256;    // score multipliers: 2 x 16
constexpr int kOffMisc = kOffCoef + 128;    // TMEM base, abort flag
constexpr int kSmemBytes = kOffMisc + 16 + 1024;

enum : int {
    KV_FULL = 0, KV_EMPTY = 2, S_FULL = 4, S_FREE = 6, P_FULL = 8, O_FULL = 10, O_FREE = 12,
    Q_FULL = 14, Q_FREE = 16, DONE = 18, NUM_BARS = 19
};

struct Seg {
    int32_t b, t0, t1, part, ntiles;
};

__device__ __forceinline__ Seg load_seg(const DecodeParams& p, int si) {
    Seg s;
    s.b = p.segs[4 * si];
    s.t0 = p.segs[4 * si + 1];
    s.t1 = p.segs[4 * si + 2];
    s.part = p.segs[4 * si + 3];
    // a segment longer than the device-side context means the page table
    // changed after planning: it is skipped (and flagged by the MMA thread)
    s.ntiles = s.t1 <= p.seq_lens[s.b] ? (s.t1 - s.t0 + kTT - 1) / kTT : 0;
    return s;
}

__device__ __forceinline__ int64_t token_slot(const DecodeParams& p, const int32_t* pages, int32_t t,
                                              int32_t t_end, bool flag) {
    if (t >= t_end) return -1;
    const int64_t page = pages[p.page_size == 1 ? t : t / p.page_size];
    const int64_t slot = p.page_size == 1 ? page : page * p.page_size + t % p.page_size;
    if (page < 0 || slot >= p.num_slots) {
        if (flag) raise_flag(p.flags, MLA_FLAG_INDEX_OOB);
        return -1;
    }
    return slot;
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
    const uint32_t h = e4m3x2_to_f16x2(two);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__device__ __forceinline__ void wg_bar() { asm volatile("bar.sync 1, 128;\n" ::: "memory"); }

// ------------------------------------------------------------ producer warps

__device__ void producer(const DecodeParams& p, uint8_t* base, uint64_t* bars, volatile int* abort,
                         int seg_lo, int seg_hi, int pw, int lane) {
    int si = seg_lo, it = 0;
    Seg sg{};
    while (si < seg_hi && (sg = load_seg(p, si)).ntiles == 0) ++si;
    const int32_t* pages = si < seg_hi ? p.indices + p.indptr[sg.b] : nullptr;
    int64_t s0 = -1, s1 = -1;
    if (si < seg_hi) {
        const int32_t tb = sg.t0 + pw * 64;
        s0 = token_slot(p, pages, tb + lane, sg.t1, true);
        s1 = token_slot(p, pages, tb + 32 + lane, sg.t1, true);
    }
    for (int i = 0; si < seg_hi; ++i) {
        const int slot = i & 1;
        const uint32_t u = static_cast<uint32_t>(i) >> 1;
        if (!mbar_wait(&bars[KV_EMPTY + slot], (u & 1) ^ 1, abort, p.flags)) break;
        uint8_t* stage = base + kOffStage + slot * kStage;
#pragma unroll 4
        for (int r = 0; r < 64; ++r) {
            const int64_t s = __shfl_sync(0xffffffffu, r < 32 ? s0 : s1, r & 31);
            const int row = pw * 64 + r;
            const uint32_t n = s >= 0 ? 16u : 0u;
            const int64_t ss = s >= 0 ? s : 0;
            const int sw = row & 7;
            cp_async16(stage + (lane >> 3) * kBlk + row * 128 + (((lane & 7) ^ sw) << 4),
                       p.ckv + ss * p.ckv_stride + lane * 16, n);
            if (lane < 4)
                cp_async16(stage + 4 * kBlk + row * 128 + ((lane ^ sw) << 4),
                           p.kpe + ss * p.kpe_stride + lane * 16, n);
        }
        mbar_arrive_cp_async(&bars[KV_FULL + slot]);
        // next tile's slots, loaded while this tile's rows are in flight
        if (++it == sg.ntiles) {
            it = 0;
            ++si;
            while (si < seg_hi && (sg = load_seg(p, si)).ntiles == 0) ++si;
            if (si < seg_hi) pages = p.indices + p.indptr[sg.b];
        }
        if (si < seg_hi) {
            const int32_t tb = sg.t0 + it * kTT + pw * 64;
            s0 = token_slot(p, pages, tb + lane, sg.t1, true);
            s1 = token_slot(p, pages, tb + 32 + lane, sg.t1, true);
        }
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------- MMA issuer

struct MmaCtx {
    uint32_t sbase, tmem, idesc_qk, idesc_pv;
    uint64_t* bars;
    volatile int* abort;
    uint32_t* flags;
};

__device__ __forceinline__ bool issue_pv(const MmaCtx& c, int j) {
    const int slot = j & 1;
    const uint32_t u = static_cast<uint32_t>(j) >> 1;
    if (!mbar_wait(&c.bars[P_FULL + slot], u & 1, c.abort, c.flags)) return false;
    if (!mbar_wait(&c.bars[O_FREE + slot], (u & 1) ^ 1, c.abort, c.flags)) return false;
    fence_after_sync();
    fence_proxy_async_smem();
    const uint32_t stage = c.sbase + kOffStage + slot * kStage;
    const uint32_t pb = c.sbase + kOffP + slot * kPBytes;
#pragma unroll
    for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
        for (int ks = 0; ks < kTT / 32; ++ks) {
            // A = V^T: 128 channels (one column block) x 32 tokens, MN-major
            const uint64_t a = smem_desc(stage + mb * kBlk + ks * 32 * 128, kBlk, 1024, kSwizzle128B);
            // B = [P1;P2]^T: 32 tokens x 32 (term, head), MN-major, unswizzled
            const uint64_t b = smem_desc(pb + ks * 32 * 16, 128, kPUnit, kSwizzleNone);
            mma_e4m3(c.tmem + kColO + 128 * slot + 32 * mb, a, b, c.idesc_pv, ks > 0);
        }
    }
    mma_commit(&c.bars[O_FULL + slot]);
    mma_commit(&c.bars[KV_EMPTY + slot]);
    return true;
}

__device__ void mma_issuer(const DecodeParams& p, const MmaCtx& c, int seg_lo, int seg_hi) {
    // Order per tile i: PV(i-1) first, then QK(i).  PV(i-1) releases the
    // stage of tile i-1 as soon as its softmax is done, so the load of tile
    // i+1 overlaps tile i's compute and both stages can be in flight.
    int i = 0, k = 0, prev = -1;
    bool ok = true;
    for (int si = seg_lo; si < seg_hi && ok; ++si) {
        const Seg sg = load_seg(p, si);
        if (sg.ntiles == 0) {
            if (sg.t1 > sg.t0) raise_flag(p.flags, MLA_FLAG_PLAN_MISMATCH);
            continue;
        }
        const int qs = k & 1;
        const uint32_t qu = static_cast<uint32_t>(k) >> 1;
        const uint32_t qb = c.sbase + kOffQ + qs * kQBytes;
        for (int it = 0; it < sg.ntiles; ++it, ++i) {
            if (prev >= 0 && !issue_pv(c, prev)) { ok = false; break; }
            prev = -1;
            const int slot = i & 1;
            const uint32_t u = static_cast<uint32_t>(i) >> 1;
            if ((it == 0 && !mbar_wait(&c.bars[Q_FULL + qs], qu & 1, c.abort, c.flags)) ||
                !mbar_wait(&c.bars[KV_FULL + slot], u & 1, c.abort, c.flags) ||
                !mbar_wait(&c.bars[S_FREE + slot], (u & 1) ^ 1, c.abort, c.flags)) {
                ok = false;
                break;
            }
            fence_after_sync();
            fence_proxy_async_smem();
            const uint32_t stage = c.sbase + kOffStage + slot * kStage;
#pragma unroll
            for (int ks = 0; ks < kKSteps; ++ks) {
                const uint64_t a = smem_desc(stage + (ks >> 2) * kBlk + (ks & 3) * 32, 16, 1024,
                                             kSwizzle128B);
                const uint64_t b = smem_desc(qb + (ks >> 2) * kQBlk + (ks & 3) * 32, 16, 1024,
                                             kSwizzle128B);
                mma_e4m3(c.tmem + kColS + 32 * slot, a, b, c.idesc_qk, ks > 0);
            }
            mma_commit(&c.bars[S_FULL + slot]);
            if (it == sg.ntiles - 1) mma_commit(&c.bars[Q_FREE + qs]);
            prev = i;
        }
        ++k;
    }
    if (ok && prev >= 0) issue_pv(c, prev);
    // every MMA issued so far has completed before TMEM may be released
    mma_commit(&c.bars[DONE]);
    volatile int never = 0;
    mbar_wait(&c.bars[DONE], 0, &never, c.flags, 1000000000ull);
}

// ---------------------------------------------------------------- q prep

__device__ void q_prep(const DecodeParams& p, uint8_t* base, uint64_t* bars, volatile int* abort,
                       int seg_lo, int seg_hi, int head0, int lane) {
    // lane = (head, half row): head lane/2, 16-channel chunks 18*(lane&1) ..
    // +17, all loads issued before any is used (one memory latency per
    // segment instead of one per head)
    constexpr int kChunks = kDQk / 16 / 2;          // 18 chunks of 16 channels per lane
    float* coefs = reinterpret_cast<float*>(base + kOffCoef);
    const int r = lane >> 1, c0 = (lane & 1) * kChunks;
    const int head = head0 + r;
    const bool valid = head < p.heads;
    int k = 0;
    for (int si = seg_lo; si < seg_hi; ++si) {
        const Seg sg = load_seg(p, si);
        if (sg.ntiles == 0) continue;
        const int qs = k & 1;
        const uint32_t qu = static_cast<uint32_t>(k) >> 1;
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + int64_t(sg.b) * p.q_sb + int64_t(valid ? head : 0) * p.q_sh + 16 * c0);
        // pass 1: the head's largest magnitude (9 chunks in flight at a time)
        float amax = 0.f;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            uint4 v[kChunks];
#pragma unroll
            for (int j = 0; j < kChunks; ++j) v[j] = valid ? src[g * kChunks + j] : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int j = 0; j < kChunks; ++j) {
                const uint32_t w4[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w4[e] << 16)),
                                             fabsf(__uint_as_float(w4[e] & 0xffff0000u))));
            }
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        int e2 = 0;
        frexpf(amax, &e2);                              // amax = m * 2^e2, m in [0.5, 1)
        int sigma = amax > 0.f ? 8 - e2 : 0;            // max |q| * 2^sigma in [128, 256)
        sigma = sigma > 100 ? 100 : (sigma < -100 ? -100 : sigma);
        const float scale = ldexpf(1.f, sigma);
        if (!mbar_wait(&bars[Q_FREE + qs], (qu & 1) ^ 1, abort, p.flags)) break;
        uint8_t* qb = base + kOffQ + qs * kQBytes;
        // pass 2 (re-read, now cached): split each value into two E4M3 terms
#pragma unroll 1
        for (int cc16 = 0; cc16 < kChunks; ++cc16) {
            const uint4 va = valid ? src[2 * cc16] : make_uint4(0, 0, 0, 0);
            const uint4 vb = valid ? src[2 * cc16 + 1] : make_uint4(0, 0, 0, 0);
            const uint32_t w8[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
            uint32_t t1[4], t2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint32_t lo1 = 0, lo2 = 0;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t w = w8[2 * e + hh];
                    const float x0 = __uint_as_float(w << 16) * scale;
                    const float x1 = __uint_as_float(w & 0xffff0000u) * scale;
                    const uint16_t b1 = f32x2_to_e4m3x2(x0, x1);
                    const float2 d = e4m3x2_to_float2(b1);
                    const uint16_t b2 = f32x2_to_e4m3x2(x0 - d.x, x1 - d.y);
                    lo1 |= static_cast<uint32_t>(b1) << (16 * hh);
                    lo2 |= static_cast<uint32_t>(b2) << (16 * hh);
                }
                t1[e] = lo1;
                t2[e] = lo2;
            }
            const int c = c0 + cc16;
            const int cb = c >> 3, cc = c & 7;
            const int row1 = r, row2 = kHeadsPerCta + r;
            *reinterpret_cast<uint4*>(qb + cb * kQBlk + row1 * 128 + ((cc ^ (row1 & 7)) << 4)) =
                make_uint4(t1[0], t1[1], t1[2], t1[3]);
            *reinterpret_cast<uint4*>(qb + cb * kQBlk + row2 * 128 + ((cc ^ (row2 & 7)) << 4)) =
                make_uint4(t2[0], t2[1], t2[2], t2[3]);
        }
        if ((lane & 1) == 0)
            coefs[qs * kHeadsPerCta + r] =
                valid ? ldexpf(p.softmax_scale * p.k_scale * kLog2e, -sigma) : 0.f;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[Q_FULL + qs]);
        ++k;
    }
}

// ------------------------------------------------- softmax / correction WG

struct WgCtx {
    uint8_t* base;
    uint64_t* bars;
    uint32_t tmem_lane;     // TMEM base + this warp's lane quadrant
    volatile int* abort;
    uint32_t* flags;
    int t, wq, lane;        // thread 0..127, warp 0..3, lane
};

__device__ __forceinline__ bool correction(const WgCtx& w, int j, const float (&alpha)[16],
                                           float (&o)[4][16]) {
    const int slot = j & 1;
    const uint32_t u = static_cast<uint32_t>(j) >> 1;
    if (!mbar_wait(&w.bars[O_FULL + slot], u & 1, w.abort, w.flags)) return false;
    fence_after_sync();
#pragma unroll
    for (int mb = 0; mb < 4; ++mb) {
        uint32_t r1[16], r2[16];
        tmem_ld16(w.tmem_lane + kColO + 128 * slot + 32 * mb, r1);
        tmem_ld16(w.tmem_lane + kColO + 128 * slot + 32 * mb + 16, r2);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 16; ++h)
            o[mb][h] = fmaf(o[mb][h], alpha[h], __uint_as_float(r1[h]) + __uint_as_float(r2[h]));
    }
    fence_before_sync();
    mbar_arrive(&w.bars[O_FREE + slot]);
    return true;
}

__device__ void softmax_wg(const DecodeParams& p, const WgCtx& w, int seg_lo, int seg_hi, int head0) {
    float* red = reinterpret_cast<float*>(w.base + kOffRed);
    float* lsum = reinterpret_cast<float*>(w.base + kOffLsum);
    const float* coefs = reinterpret_cast<const float*>(w.base + kOffCoef);
    uint8_t* pbase = w.base + kOffP;
    int i = 0, k = 0;
    for (int si = seg_lo; si < seg_hi; ++si) {
        const Seg sg = load_seg(p, si);
        if (sg.ntiles == 0) continue;
        const int qs = k & 1;
        const uint32_t qu = static_cast<uint32_t>(k) >> 1;
        if (!mbar_wait(&w.bars[Q_FULL + qs], qu & 1, w.abort, w.flags)) return;
        float coef[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) coef[h] = coefs[qs * kHeadsPerCta + h];
        mbar_arrive(&w.bars[Q_FREE + qs]);
        const int32_t* pages = p.indices + p.indptr[sg.b];

        float m[16], l[16], alpha_pend[16], o[4][16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
            alpha_pend[h] = 0.f;
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) o[mb][h] = 0.f;
        }
        for (int it = 0; it < sg.ntiles; ++it, ++i) {
            const int slot = i & 1;
            const uint32_t u = static_cast<uint32_t>(i) >> 1;
            const bool valid = token_slot(p, pages, sg.t0 + it * kTT + w.t, sg.t1, false) >= 0;
            if (!mbar_wait(&w.bars[S_FULL + slot], u & 1, w.abort, w.flags)) return;
            fence_after_sync();
            uint32_t r1[16], r2[16];
            tmem_ld16(w.tmem_lane + kColS + 32 * slot, r1);
            tmem_ld16(w.tmem_lane + kColS + 32 * slot + 16, r2);
            tmem_wait_ld();
            fence_before_sync();
            mbar_arrive(&w.bars[S_FREE + slot]);

            float s[16], mx[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                s[h] = valid ? (__uint_as_float(r1[h]) + __uint_as_float(r2[h])) * coef[h] : -INFINITY;
                mx[h] = s[h];
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                for (int h = 0; h < 16; ++h) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], off));
            }
            float* rb = red + (i & 1) * 64;
            if (w.lane == 0) {
#pragma unroll
                for (int h = 0; h < 16; ++h) rb[w.wq * 16 + h] = mx[h];
            }
            wg_bar();
            float alpha[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                const float tmax = fmaxf(fmaxf(rb[h], rb[16 + h]), fmaxf(rb[32 + h], rb[48 + h]));
                const float mn = fmaxf(m[h], tmax);
                alpha[h] = mn == -INFINITY ? 1.f : fast_exp2(m[h] - mn);
                m[h] = mn;
            }
            // P = exp2(s - m) as two E4M3 terms of p * 256
            uint32_t pk1[4], pk2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint32_t w1 = 0, w2 = 0;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int h = 4 * e + 2 * hh;
                    const float x0 = m[h] == -INFINITY ? 0.f : fast_exp2(s[h] - m[h]) * 256.f;
                    const float x1 = m[h + 1] == -INFINITY ? 0.f : fast_exp2(s[h + 1] - m[h + 1]) * 256.f;
                    const uint16_t b1 = f32x2_to_e4m3x2(x0, x1);
                    const float2 d1 = e4m3x2_to_float2(b1);
                    const uint16_t b2 = f32x2_to_e4m3x2(x0 - d1.x, x1 - d1.y);
                    const float2 d2 = e4m3x2_to_float2(b2);
                    l[h] = fmaf(l[h], alpha[h], d1.x + d2.x);
                    l[h + 1] = fmaf(l[h + 1], alpha[h + 1], d1.y + d2.y);
                    w1 |= static_cast<uint32_t>(b1) << (16 * hh);
                    w2 |= static_cast<uint32_t>(b2) << (16 * hh);
                }
                pk1[e] = w1;
                pk2[e] = w2;
            }
            uint8_t* pb = pbase + slot * kPBytes + w.t * 16;
            *reinterpret_cast<uint4*>(pb) = make_uint4(pk1[0], pk1[1], pk1[2], pk1[3]);
            *reinterpret_cast<uint4*>(pb + kPUnit) = make_uint4(pk2[0], pk2[1], pk2[2], pk2[3]);
            fence_proxy_async_smem();
            mbar_arrive(&w.bars[P_FULL + slot]);

            if (it > 0 && !correction(w, i - 1, alpha_pend, o)) return;
#pragma unroll
            for (int h = 0; h < 16; ++h) alpha_pend[h] = alpha[h];
        }
        if (!correction(w, i - 1, alpha_pend, o)) return;

        // ---- epilogue: denominators over the 128 token lanes, normalise, store
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
            for (int h = 0; h < 16; ++h) l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
        }
        if (w.lane == 0) {
#pragma unroll
            for (int h = 0; h < 16; ++h) lsum[w.wq * 16 + h] = l[h];
        }
        wg_bar();
        float L[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) L[h] = lsum[h] + lsum[16 + h] + lsum[32 + h] + lsum[48 + h];
        wg_bar();                                   // lsum is reused by the next segment
        const int H = p.heads;
        if (sg.part < 0) {
            uint16_t* out = p.out + (int64_t(sg.b) * H + head0) * kDCkv + w.t;
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                if (head0 + h >= H) break;
                const float inv = L[h] > 0.f ? p.k_scale / L[h] : 0.f;
#pragma unroll
                for (int mb = 0; mb < 4; ++mb)
                    out[h * kDCkv + mb * 128] = __bfloat16_as_ushort(__float2bfloat16_rn(o[mb][h] * inv));
            }
            if (w.t == 0) {
#pragma unroll
                for (int h = 0; h < 16; ++h)
                    if (head0 + h < H)
                        p.lse[int64_t(sg.b) * H + head0 + h] = (m[h] + log2f(L[h]) - 8.f) * kLn2;
            }
        } else {
            float* po = p.part_o + (int64_t(sg.part) * H + head0) * kDCkv + w.t;
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                if (head0 + h >= H) break;
                const float inv = L[h] > 0.f ? p.k_scale / L[h] : 0.f;
#pragma unroll
                for (int mb = 0; mb < 4; ++mb) po[h * kDCkv + mb * 128] = o[mb][h] * inv;
            }
            if (w.t == 0) {
#pragma unroll
                for (int h = 0; h < 16; ++h)
                    if (head0 + h < H)
                        p.part_lse[int64_t(sg.part) * H + head0 + h] = (m[h] + log2f(L[h]) - 8.f) * kLn2;
            }
        }
        ++k;
    }
}

__global__ void __launch_bounds__(kThreads, 1) mla_decode_tc_kernel(const DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + kOffMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(base + kOffMisc + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        const uint32_t counts[NUM_BARS] = {64, 64, 1, 1, 1, 1, 128, 128, 128, 128,
                                           1,  1,  128, 128, 1, 1, 129, 129, 1};
        for (int b = 0; b < NUM_BARS; ++b) mbar_init(&bars[b], counts[b]);
        *abort = 0;
        mbar_fence_init();
    }
    if (warp == 2) tmem_alloc(tmem_slot, kTmemCols);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int seg_lo = p.cta_ptr[blockIdx.x], seg_hi = p.cta_ptr[blockIdx.x + 1];
    const int head0 = 0;                          // this kernel serves H <= 16

    if (warp < 2) {
        producer(p, base, bars, abort, seg_lo, seg_hi, warp, lane);
    } else if (warp == 2) {
        if (lane == 0) {
            MmaCtx c;
            c.sbase = smem_u32(base);
            c.tmem = tmem;
            c.idesc_qk = idesc_e4m3_f32(kTT, 32, false, false);
            c.idesc_pv = idesc_e4m3_f32(kTT, 32, true, true);
            c.bars = bars;
            c.abort = abort;
            c.flags = p.flags;
            mma_issuer(p, c, seg_lo, seg_hi);
        }
        __syncwarp();
    } else if (warp == 3) {
        q_prep(p, base, bars, abort, seg_lo, seg_hi, head0, lane);
    } else {
        WgCtx w;
        w.base = base;
        w.bars = bars;
        w.wq = warp - 4;
        w.tmem_lane = tmem + (static_cast<uint32_t>(w.wq * 32) << 16);
        w.abort = abort;
        w.flags = p.flags;
        w.t = tid - 128;
        w.lane = lane;
        softmax_wg(p, w, seg_lo, seg_hi, head0);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == 2) tmem_dealloc(tmem, kTmemCols);
}

std::mutex g_mu;
std::vector<char> g_attr;     // per device: max dynamic smem set

}  // namespace

cudaError_t launch_decode_tc(const DecodeParams& p, int grid, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if ((int)g_attr.size() <= dev) g_attr.resize(dev + 1, 0);
        if (!g_attr[dev]) {
            e = cudaFuncSetAttribute(mla_decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemBytes);
            if (e != cudaSuccess) return e;
            g_attr[dev] = 1;
        }
    }
    mla_decode_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace mla
