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
// weights p * 16 = p1 + p2 (8 significant bits, like a BF16 P).  The two
// terms are stacked along N, so one MMA computes both partial products and
// reads the cache tile once.
//
// Tile = 128 tokens = the MMA's M.  Per tile:
//   S^T[128 x 32]  = K_tile[128 x 576] . [q1;q2]^T    18 MMAs, K-major A/B
//   O^T[512 x 32] += V^T[512 x 128] . [P1;P2]^T       16 MMAs, MN-major A/B
// The same swizzled smem tile serves as K-major A (tokens x dims) and
// MN-major A (dims x tokens); S and O live in TMEM.
//
// Online softmax with lazy rescaling: the running maximum m only moves when
// some score exceeds it by more than 2^4 (in log2 units), so most tiles skip
// the cross-token maximum; p = 2^(s - m) <= 16 and p * 16 still fits E4M3.
//
// Warp roles (one CTA per SM, persistent over its token range):
//   warps 0-1  gather the tile's rows into a 2-stage ring, split between
//              two engines by their measured rates: warp 0 uses TMA
//              tile::gather4 (four pool rows per instruction, c_kv channels
//              0..127, 128-byte swizzle, out-of-range rows zero-filled),
//              warp 1 16-byte cp.async (c_kv channels 128..511 and the 64
//              k_pe channels, 64-byte swizzle); both complete on the stage's
//              mbarrier;
//   warp 2     one thread issues every tcgen05.mma and commit, polling so
//              that PV of one tile and QK^T of the next go out in whichever
//              order their inputs become ready;
//   warp 3     prepares [q1;q2] and the per-head score multipliers for each
//              segment (double-buffered; lane = half a head row);
//   warps 4-7  one thread per TMEM lane: online softmax of a token's 16
//              heads, the E4M3 split of P, then the O correction (lane =
//              output channel) and the epilogue.
// Every mbarrier wait is bounded; on a timeout the CTA sets
// MLA_FLAG_WAIT_TIMEOUT, drains its MMAs and copies, frees TMEM and exits.
#include <cuda.h>

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
constexpr int kM = 128;
constexpr int kStages = 2;
constexpr int kThreads = 256;
constexpr int kBlk = kTT * 128;             // 128 rows x 128 B, 128-byte swizzle (128 c_kv channels)
constexpr int kRope = kTT * 64;             // 128 rows x 64 B, 64-byte swizzle (the 64 k_pe channels)
constexpr int kStage = 4 * kBlk + kRope;    // 72 KB per tile
constexpr int kQRows = 2 * kHeadsPerCta;    // B rows: q1 of heads 0..15, then q2
constexpr int kQBlk = kQRows * 128;         // 4 KB per 128-channel block
constexpr int kQBytes = 4 * kQBlk + kQRows * 64;   // + the k_pe block: 18 KB
constexpr int kPUnit = kTT * 16;            // one E4M3 term of P^T: 128 tokens x 16 heads
constexpr int kPBytes = 2 * kPUnit;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;               // S[j]: columns 32j .. 32j+31
constexpr uint32_t kColO = 64;              // O[j]: 64 + 128j + 32mb (mb = 128-channel block)
constexpr int kKSteps = kDQk / 32;          // 18 k-steps of 32 channels for QK
constexpr float kTau = 4.f;                 // lazy-rescale threshold (log2 units)
constexpr float kPScale = 16.f;             // P is stored as p * 2^kTau
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kOffStage = 0;
constexpr int kOffQ = kOffStage + kStages * kStage;
constexpr int kOffP = kOffQ + 2 * kQBytes;
constexpr int kOffBar = kOffP + 2 * kPBytes;
constexpr int kOffRed = kOffBar + 256;      // tile maxima: 2 x 4 warps x 16
constexpr int kOffLsum = kOffRed + 512;     // softmax denominators: 4 warps x 16
constexpr int kOffCoef = kOffLsum + 256;    // score multipliers: 2 x 16
constexpr int kOffFlag = kOffCoef + 128;    // rescale votes: 2 x 4 warps
constexpr int kOffMisc = kOffFlag + 32;     // TMEM base, abort flag
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kBlk % 1024 == 0 && kStage % 1024 == 0 && kQBytes % 1024 == 0,
              "swizzle atoms need 1 KB alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kTT == kM, "a tile fills the MMA's M exactly");

enum : int {
    KV_FULL = 0, KV_EMPTY = kStages, S_FULL = 2 * kStages, S_FREE = S_FULL + 2, P_FULL = S_FREE + 2,
    O_FULL = P_FULL + 2, O_FREE = O_FULL + 2, Q_FULL = O_FREE + 2, Q_FREE = Q_FULL + 2,
    DONE = Q_FREE + 2, NUM_BARS = DONE + 1
};
static_assert(NUM_BARS == 19, "barrier count table below assumes two stages");

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
//
// Rows of a tile are gathered by two engines at once: the TMA unit (warp 0,
// tile::gather4: c_kv channels 0..127) and the LSU (warp 1, 16-byte
// cp.async: c_kv channels 128..511 and k_pe).  Each engine caps the gather
// requests an SM keeps in flight; measured on GB300, TMA gathers sustain
// about a quarter of the LSU's rate, so it takes 16 of the tile's 72 KB.

struct TmaMaps {
    CUtensorMap ckv;    // [rows][512] E4M3, box 128 x 1, 128-byte swizzle
    int32_t rows;       // tensor-map height; a row coordinate >= rows reads zeros
};

constexpr int kTmaBlocks = 1;                                   // c_kv block 0 by TMA
constexpr int32_t kNoRow = INT32_MIN;
constexpr uint32_t kTmaBytes = kTmaBlocks * kBlk;

// Cursor over the tiles of a CTA's segments, with the raw page entries of up
// to four rows per lane for one tile: rows lane + 32q (LSU warp) or 4 lane + q
// (TMA warp, whose gather4 takes four consecutive rows).
struct TileCursor {
    int si, seg_hi, it;
    Seg sg;
    const int32_t* pages;
    int32_t pg[4];                      // page entry, or kNoRow past the context / tile
    int32_t t[4];                       // token index of each row

    __device__ void init(const DecodeParams& p, int lo, int hi) {
        si = lo;
        seg_hi = hi;
        it = 0;
        while (si < seg_hi && (sg = load_seg(p, si)).ntiles == 0) ++si;
        if (si < seg_hi) pages = p.indices + p.indptr[sg.b];
    }
    __device__ bool valid() const { return si < seg_hi; }
    // issue the (independent) index loads of the current tile; nothing waits
    // on them until rows() is called
    __device__ void prefetch(const DecodeParams& p, int lane, bool consecutive) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int row = consecutive ? 4 * lane + q : lane + 32 * q;
            t[q] = sg.t0 + it * kTT + row;
            pg[q] = (row < kTT && t[q] < sg.t1) ? pages[p.page_size == 1 ? t[q] : t[q] / p.page_size]
                                                : kNoRow;
        }
    }
    // slot of each row, or -1 (past the context or the tile, or outside the pool)
    __device__ void rows(const DecodeParams& p, int32_t (&slot)[4], bool flag) const {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int64_t s = p.page_size == 1 ? int64_t(pg[q])
                                               : int64_t(pg[q]) * p.page_size + t[q] % p.page_size;
            const bool ok = pg[q] >= 0 && s < p.num_slots;
            if (!ok && pg[q] != kNoRow && flag) raise_flag(p.flags, MLA_FLAG_INDEX_OOB);
            slot[q] = ok ? static_cast<int32_t>(s) : -1;
        }
    }
    __device__ void advance(const DecodeParams& p) {
        if (++it == sg.ntiles) {
            it = 0;
            ++si;
            while (si < seg_hi && (sg = load_seg(p, si)).ntiles == 0) ++si;
            if (si < seg_hi) pages = p.indices + p.indptr[sg.b];
        }
    }
};

__device__ void producer_tma(const DecodeParams& p, const TmaMaps& maps, uint8_t* base,
                             uint64_t* bars, volatile int* abort, int seg_lo, int seg_hi, int lane) {
    TileCursor cur;
    cur.init(p, seg_lo, seg_hi);
    if (cur.valid()) cur.prefetch(p, lane, true);
    const uint32_t sbase = smem_u32(base);
    int i = 0;
    for (bool more = cur.valid(); more; ++i) {
        const int slot = i % kStages;
        const uint32_t u = static_cast<uint32_t>(i / kStages);
        int32_t sl[4];
        cur.rows(p, sl, true);
        // the next tile's index loads fly while this tile is issued
        cur.advance(p);
        more = cur.valid();
        if (more) cur.prefetch(p, lane, true);
        if (!mbar_wait(&bars[KV_EMPTY + slot], (u & 1) ^ 1, abort, p.flags)) break;
        if (lane == 0) mbar_arrive_expect_tx(&bars[KV_FULL + slot], kTmaBytes);
        __syncwarp();
        if (4 * lane < kTT) {                  // lane l gathers rows 4l .. 4l+3
            int32_t rc[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) rc[q] = sl[q] >= 0 ? sl[q] : maps.rows;
            const uint32_t stage = sbase + kOffStage + slot * kStage;
#pragma unroll
            for (int cb = 0; cb < kTmaBlocks; ++cb)
                tma_gather4(stage + cb * kBlk + 4 * lane * 128, &maps.ckv, cb * 128, rc[0], rc[1],
                            rc[2], rc[3], &bars[KV_FULL + slot]);
        }
    }
    // copies still in flight (only after an abort) land before the CTA exits
    volatile int never = 0;
    for (int j = i - kStages < 0 ? 0 : i - kStages; j < i; ++j)
        mbar_wait(&bars[KV_FULL + j % kStages], (static_cast<uint32_t>(j / kStages)) & 1, &never,
                  p.flags, 1000000000ull);
}

__device__ void producer_lsu(const DecodeParams& p, uint8_t* base, uint64_t* bars,
                             volatile int* abort, int seg_lo, int seg_hi, int lane) {
    TileCursor cur;
    cur.init(p, seg_lo, seg_hi);
    if (cur.valid()) cur.prefetch(p, lane, false);
    int i = 0;
    for (bool more = cur.valid(); more; ++i) {
        const int slot = i % kStages;
        const uint32_t u = static_cast<uint32_t>(i / kStages);
        int32_t sl[4];
        cur.rows(p, sl, false);
        cur.advance(p);
        more = cur.valid();
        if (more) cur.prefetch(p, lane, false);
        if (!mbar_wait(&bars[KV_EMPTY + slot], (u & 1) ^ 1, abort, p.flags)) break;
        uint8_t* stage = base + kOffStage + slot * kStage;
        // c_kv blocks kTmaBlocks..3: 8 chunks (128 B) per row, four rows per
        // instruction
        const int r4 = lane >> 3, c8 = lane & 7;
#pragma unroll
        for (int cb = kTmaBlocks; cb < 4; ++cb) {
#pragma unroll
            for (int j = 0; j < kTT / 4; ++j) {
                const int row = 4 * j + r4;
                const int32_t s = __shfl_sync(0xffffffffu, sl[j >> 3], row & 31);
                const int64_t ss = s >= 0 ? s : 0;
                cp_async16(stage + cb * kBlk + row * 128 + ((c8 ^ (row & 7)) << 4),
                           p.ckv + ss * p.ckv_stride + cb * 128 + c8 * 16, s >= 0 ? 16u : 0u);
            }
        }
        // k_pe: 4 chunks per row, eight rows per instruction (64-byte swizzle)
        const int r8 = lane >> 2, c4 = lane & 3;
#pragma unroll
        for (int g = 0; g < kTT / 8; ++g) {
            const int row = 8 * g + r8;
            const int32_t s = __shfl_sync(0xffffffffu, sl[g >> 2], row & 31);
            const int64_t ss = s >= 0 ? s : 0;
            cp_async16(stage + 4 * kBlk + row * 64 + ((c4 ^ ((row >> 1) & 3)) << 4),
                       p.kpe + ss * p.kpe_stride + c4 * 16, s >= 0 ? 16u : 0u);
        }
        mbar_arrive_cp_async(&bars[KV_FULL + slot]);
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

__device__ __forceinline__ void issue_qk(const MmaCtx& c, int i, int qs) {
    const int slot = i & 1;
    const uint32_t stage = c.sbase + kOffStage + (i % kStages) * kStage;
    const uint32_t qb = c.sbase + kOffQ + qs * kQBytes;
#pragma unroll
    for (int ks = 0; ks < kKSteps; ++ks) {
        uint64_t a, b;
        if (ks < 16) {           // c_kv channels: 128-byte swizzle, 8-row groups 1 KB apart
            a = smem_desc(stage + (ks >> 2) * kBlk + (ks & 3) * 32, 16, 1024, kSwizzle128B);
            b = smem_desc(qb + (ks >> 2) * kQBlk + (ks & 3) * 32, 16, 1024, kSwizzle128B);
        } else {                 // k_pe channels: 64-byte swizzle, 8-row groups 512 B apart
            a = smem_desc(stage + 4 * kBlk + (ks - 16) * 32, 16, 512, kSwizzle64B);
            b = smem_desc(qb + 4 * kQBlk + (ks - 16) * 32, 16, 512, kSwizzle64B);
        }
        mma_e4m3(c.tmem + kColS + 32 * slot, a, b, c.idesc_qk, ks > 0);
    }
    mma_commit(&c.bars[S_FULL + slot]);
}

__device__ __forceinline__ void issue_pv(const MmaCtx& c, int j) {
    const int slot = j & 1;
    const int kv = j % kStages;
    const uint32_t stage = c.sbase + kOffStage + kv * kStage;
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
    mma_commit(&c.bars[KV_EMPTY + kv]);       // the stage may be refilled
}

// QK^T of tile i and PV of tile j < i are independent once their inputs are
// ready; the issuer polls both and sends whichever is ready (PV first, since
// it frees a stage for the next load).  QK^T runs at most one tile ahead.
__device__ void mma_issuer(const DecodeParams& p, const MmaCtx& c, int seg_lo, int seg_hi) {
    int total = 0;
    for (int si = seg_lo; si < seg_hi; ++si) {
        const Seg sg = load_seg(p, si);
        if (sg.ntiles == 0 && sg.t1 > sg.t0) raise_flag(p.flags, MLA_FLAG_PLAN_MISMATCH);
        total += sg.ntiles;
    }
    int si = seg_lo, it = 0, k = 0;
    Seg sg{};
    while (si < seg_hi && (sg = load_seg(p, si)).ntiles == 0) ++si;
    int qk = 0, pv = 0;
    uint64_t last = global_ns();
    uint32_t spins = 0;
    while (pv < total) {
        bool did = false;
        if (pv < qk) {
            const int slot = pv & 1;
            const uint32_t u = static_cast<uint32_t>(pv) >> 1;
            if (mbar_test(&c.bars[P_FULL + slot], u & 1) &&
                mbar_test(&c.bars[O_FREE + slot], (u & 1) ^ 1)) {
                fence_after_sync();
                fence_proxy_async_smem();
                issue_pv(c, pv);
                ++pv;
                did = true;
            }
        }
        if (!did && qk < total && qk - pv < 2) {
            const int slot = qk & 1;
            const uint32_t u = static_cast<uint32_t>(qk) >> 1;
            const int qs = k & 1;
            const uint32_t qu = static_cast<uint32_t>(k) >> 1;
            const int kv = qk % kStages;
            const uint32_t kvu = static_cast<uint32_t>(qk / kStages);
            if ((it != 0 || mbar_test(&c.bars[Q_FULL + qs], qu & 1)) &&
                mbar_test(&c.bars[KV_FULL + kv], kvu & 1) &&
                mbar_test(&c.bars[S_FREE + slot], (u & 1) ^ 1)) {
                fence_after_sync();
                fence_proxy_async_smem();
                issue_qk(c, qk, qs);
                if (it == sg.ntiles - 1) {
                    mma_commit(&c.bars[Q_FREE + qs]);     // q buffer of this segment done
                    it = 0;
                    ++k;
                    ++si;
                    while (si < seg_hi && (sg = load_seg(p, si)).ntiles == 0) ++si;
                } else {
                    ++it;
                }
                ++qk;
                did = true;
            }
        }
        if (did) {
            spins = 0;
            last = global_ns();
        } else {
            __nanosleep(64);           // leave issue slots to the softmax warp on this SMSP
        }
        if (!did && (++spins & 63) == 0) {
            if (*c.abort) break;
            if (global_ns() - last > 2000000000ull) {
                *c.abort = 1;
                raise_flag(c.flags, MLA_FLAG_WAIT_TIMEOUT);
                break;
            }
        }
    }
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
            const int row1 = r, row2 = kHeadsPerCta + r;
            uint8_t *d1, *d2;
            if (c < 32) {                               // c_kv: 128-byte rows, 128-byte swizzle
                const int cb = c >> 3, cc = c & 7;
                d1 = qb + cb * kQBlk + row1 * 128 + ((cc ^ (row1 & 7)) << 4);
                d2 = qb + cb * kQBlk + row2 * 128 + ((cc ^ (row2 & 7)) << 4);
            } else {                                    // k_pe: 64-byte rows, 64-byte swizzle
                const int cc = c - 32;
                d1 = qb + 4 * kQBlk + row1 * 64 + ((cc ^ ((row1 >> 1) & 3)) << 4);
                d2 = qb + 4 * kQBlk + row2 * 64 + ((cc ^ ((row2 >> 1) & 3)) << 4);
            }
            *reinterpret_cast<uint4*>(d1) = make_uint4(t1[0], t1[1], t1[2], t1[3]);
            *reinterpret_cast<uint4*>(d2) = make_uint4(t2[0], t2[1], t2[2], t2[3]);
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

// Maximum over the 32 lanes of 16 values at once by halving exchanges
// (16 shuffles instead of 80): afterwards lane l holds head l >> 1.
__device__ __forceinline__ float warp_max16(const float (&v)[16], int lane) {
    float a8[8], a4[4], a2[2];
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        a8[j] = fmaxf(b4 ? v[j + 8] : v[j], __shfl_xor_sync(0xffffffffu, b4 ? v[j] : v[j + 8], 16));
#pragma unroll
    for (int j = 0; j < 4; ++j)
        a4[j] = fmaxf(b3 ? a8[j + 4] : a8[j], __shfl_xor_sync(0xffffffffu, b3 ? a8[j] : a8[j + 4], 8));
#pragma unroll
    for (int j = 0; j < 2; ++j)
        a2[j] = fmaxf(b2 ? a4[j + 2] : a4[j], __shfl_xor_sync(0xffffffffu, b2 ? a4[j] : a4[j + 2], 4));
    float a1 = fmaxf(b1 ? a2[1] : a2[0], __shfl_xor_sync(0xffffffffu, b1 ? a2[0] : a2[1], 2));
    return fmaxf(a1, __shfl_xor_sync(0xffffffffu, a1, 1));
}

__device__ void softmax_wg(const DecodeParams& p, const WgCtx& w, int seg_lo, int seg_hi, int head0) {
    float* red = reinterpret_cast<float*>(w.base + kOffRed);
    float* lsum = reinterpret_cast<float*>(w.base + kOffLsum);
    int* vote = reinterpret_cast<int*>(w.base + kOffFlag);
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

            float s[16];
            bool need = false;
#pragma unroll
            for (int h = 0; h < 16; ++h) {
                s[h] = valid ? (__uint_as_float(r1[h]) + __uint_as_float(r2[h])) * coef[h] : -INFINITY;
                need |= s[h] > m[h] + kTau;         // always true on a segment's first tile
            }
            // the running maximum moves only if some score got more than
            // 2^kTau above it (one vote per warp, then one barrier)
            need = __any_sync(0xffffffffu, need);
            int* vb = vote + (i & 1) * 4;
            if (w.lane == 0) vb[w.wq] = need;
            wg_bar();
            need = vb[0] | vb[1] | vb[2] | vb[3];
            float alpha[16];
            if (need) {
                const float wmax = warp_max16(s, w.lane);
                float* rb = red + (i & 1) * 64;
                if ((w.lane & 1) == 0) rb[w.wq * 16 + (w.lane >> 1)] = wmax;
                wg_bar();
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                    const float tmax = fmaxf(fmaxf(rb[h], rb[16 + h]), fmaxf(rb[32 + h], rb[48 + h]));
                    const float mn = fmaxf(m[h], tmax);
                    alpha[h] = mn == -INFINITY ? 1.f : fast_exp2(m[h] - mn);
                    m[h] = mn;
                }
            } else {
#pragma unroll
                for (int h = 0; h < 16; ++h) alpha[h] = 1.f;
            }
            // P = 2^(s - m) <= 2^kTau, stored as two E4M3 terms of p * kPScale
            uint32_t pk1[4], pk2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint32_t w1 = 0, w2 = 0;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int h = 4 * e + 2 * hh;
                    const float x0 = m[h] == -INFINITY ? 0.f : fast_exp2(s[h] - m[h]) * kPScale;
                    const float x1 = m[h + 1] == -INFINITY ? 0.f : fast_exp2(s[h + 1] - m[h + 1]) * kPScale;
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

        // ---- epilogue: denominators over the token lanes, normalise, store
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
        // o and L are both in units of p * kPScale; lse = m + log2(sum p)
        const float lse_off = -kTau;                 // kPScale = 2^kTau
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
                        p.lse[int64_t(sg.b) * H + head0 + h] = (m[h] + log2f(L[h]) + lse_off) * kLn2;
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
                        p.part_lse[int64_t(sg.part) * H + head0 + h] = (m[h] + log2f(L[h]) + lse_off) * kLn2;
            }
        }
        ++k;
    }
}

__global__ void __launch_bounds__(kThreads, 1)
mla_decode_tc_kernel(const DecodeParams p, const __grid_constant__ TmaMaps maps) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + kOffMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(base + kOffMisc + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        // KV_FULL: 1 TMA arrive (+ transaction bytes) and 32 cp.async arrivals
        const uint32_t counts[NUM_BARS] = {33, 33, 1, 1, 1, 1, 128, 128, 128, 128,
                                           1, 1, 128, 128, 1, 1, 129, 129, 1};
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

    if (warp == 0) {
        producer_tma(p, maps, base, bars, abort, seg_lo, seg_hi, lane);
    } else if (warp == 1) {
        producer_lsu(p, base, bars, abort, seg_lo, seg_hi, lane);
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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// Row-gather tensor map over a pool: `width` E4M3 channels per row, rows
// `stride` bytes apart, boxes of one row.
bool encode_rows(CUtensorMap* m, const void* base, uint64_t width, uint64_t rows, uint64_t stride,
                 uint32_t box, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {width, rows};
    const cuuint64_t strides[1] = {stride};
    const cuuint32_t boxd[2] = {box, 1};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, boxd, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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
    TmaMaps maps;
    // an empty pool still gets a one-row map: every token is then out of
    // range, gets row coordinate `rows` and reads zeros
    if (p.num_slots >= INT32_MAX) return cudaErrorInvalidValue;   // TMA row coordinates are int32
    const uint64_t rows = p.num_slots > 0 ? static_cast<uint64_t>(p.num_slots) : 1;
    maps.rows = static_cast<int32_t>(rows);
    if (!encode_rows(&maps.ckv, p.ckv, kDCkv, rows, p.ckv_stride, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    mla_decode_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace mla
