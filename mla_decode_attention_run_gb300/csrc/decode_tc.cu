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
// terms are normal, i.e. for every entry above 2^-14 of the head's largest.
// What those two terms miss of smaller entries (E4M3's range is only 2^17)
// goes into a third term q3 at its own, finer power-of-two scale, with 4
// significant bits.  Likewise the softmax weights p * 16 = p1 + p2 / 2^5 (8
// significant bits, like a BF16 P; the second term scaled up so that weights
// far below the maximum survive).  The terms are stacked along N, so one MMA
// computes all partial products and reads the cache tile once.
//
// Tile = 64 tokens = the QK^T MMA's M.  Per tile:
//   S^T[64 x 3G]   = K_tile[64 x 576] . [q1;q2;q3]^T  18 MMAs, K-major A/B
//   O^T[512 x 2G] += V^T[512 x 64] . [P1;P2]^T        8 MMAs, MN-major A/B
// A 64-token tile (36 KB) keeps four tiles in flight in 144 KB of shared
// memory, which hides a tile's fill -> QK^T -> softmax -> PV round trip.
// The same swizzled smem tile serves as K-major A (tokens x dims) and
// MN-major A (dims x tokens).  S (double-buffered per tile) and O (one
// accumulator per segment, double-buffered across segments) live in TMEM.
//
// Online softmax with lazy rescaling: the running maximum m only moves when
// some score exceeds it by more than 2^4 (in log2 units), so most tiles skip
// the cross-token maximum; p = 2^(s - m) <= 16 and p * 16 still fits E4M3.
// O accumulates in TMEM across a segment's tiles; when m does move, the
// softmax warps rescale it in place before the next PV may add to it.
//
// A CTA serves G = 16 or 32 heads of its token range (32 when H is a multiple
// of 32); more heads run as more CTAs (grid.y = head group).  The groups of a
// token range start together, so their repeated reads of the same rows
// mostly hit L2.
//
// Extend (several new tokens per request, causal) is the same kernel built
// with E = true: a CTA then serves a block of G query rows (token x head) of
// one request, each with its own causal limit; the softmax hides the tokens
// at or past a row's limit on the tiles that reach them.
//
// Warp roles (one CTA per SM, persistent over its token range; warp numbers
// for G = 16, 384 threads, with G = 32's in brackets, 512 threads):
//   warp 11 [7]  publishes tiles ahead of the stage fills: resolves each row's
//              pool slot (or -1: past the context, outside the pool) into a
//              small shared ring and has L2 prefetch the rows' cache lines,
//              so the fills below read L2 rather than wait on DRAM;
//   warps 0-3  fill a 4-stage ring with 16-byte cp.async: warp w copies
//              c_kv channels 128w .. 128w+127 (128-byte swizzle) and a
//              quarter of the k_pe rows (64-byte swizzle); an invalid row is
//              zero-filled.  Measured on GB300, four LSU warps fed from L2
//              gather at the HBM rate, which neither fewer warps nor TMA
//              tile::gather4 reach;
//   warp 4     issues the QK^T MMAs, tile after tile (G = 16: the whole
//              warp runs the loop and one elected lane issues; G = 32: one
//              thread);
//   warp 10 [6]  issues the PV MMAs the same way, so that PV of one tile
//              never waits behind QK^T of the next;
//   warp 5     fetches each segment's [q1;q2;q3] image, per-row score
//              multipliers and causal limits, written by the q split kernel
//              that precedes this one (double-buffered for G = 16);
//   warps 6-9 [8-11, 12-15]  one softmax warpgroup per 16 heads: online
//              softmax of a token's heads and the E4M3 split of P (an M = 64
//              accumulator puts a tile's rows in lanes 0-15 of each warp's
//              TMEM lane quadrant; threads 0-15 take 8 of the warpgroup's
//              heads, 16-31 the other 8), rescaling its heads' O columns when
//              their maximum moves, and the epilogue (all lanes: lane = output
//              channel).
// Every mbarrier wait is bounded; on a timeout the CTA sets
// MLA_FLAG_WAIT_TIMEOUT, drains its MMAs and copies, frees TMEM and exits.
// The 16-head and 32-head instantiations differ in several of these forms
// (issue, waits, epilogue), each chosen by measurement on GB300: the code a
// CTA runs cold at a segment's end and the instruction cache it shares with
// the other roles turned out to set much of the call's time.
#include <mutex>
#include <vector>

#include "common.cuh"
#include "decode_params.h"
#include "plan.h"
#include "tc.cuh"

namespace mla {
namespace {

using namespace tc;

// Tiles are 64 tokens (the QK^T MMA's M): segments start on multiples of the
// plan's 128-token granularity, so they also start on a tile.
constexpr int kTT = 64;
constexpr int kM = 64;
constexpr int kStages = 4;
constexpr int kFillWarps = 4;
constexpr int kWarpMma = 4, kWarpQ = 5;      // the other roles depend on G (Shape<G>)
constexpr int kBlk = kTT * 128;             // 64 rows x 128 B, 128-byte swizzle (128 c_kv channels)
constexpr int kRope = kTT * 64;             // 64 rows x 64 B, 64-byte swizzle (the 64 k_pe channels)
constexpr int kStage = 4 * kBlk + kRope;    // 36 KB per tile
constexpr int kPUnit = kTT * 16;            // 16 columns of P^T (one term, 16 heads) x 64 tokens
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;               // S[j]: columns kN j .. kN j + kN - 1
constexpr int kKSteps = kDQk / 32;          // 18 k-steps of 32 channels for QK
constexpr float kTau = 4.f;                 // lazy-rescale threshold (log2 units)
constexpr float kPScale = 16.f;             // P is stored as p * 2^kTau
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kP2Scale = 32.f;            // P's second term is stored x 2^5
constexpr uint32_t kP2ScaleF16x2 = 0x50005000u;   // 32.0 in both f16 halves
constexpr int kCoefBytesPerRow = 12;        // per q image row: two fp32 multipliers, one int32 limit
// Published tiles' slot lists (and L2 prefetches) in flight: the scheduler
// runs at most this many tiles ahead of the softmax.  Measured on GB300:
// 6 for 16-head CTAs (the batch-40 call 34.5 us, against 34.9 with 8 and
// with 5, 34.7 with 7: fewer outstanding prefetches queue less in DRAM and
// the tiles still land in time); for 32-head CTAs 8 in decode (12 made the
// 128-head call 1.4 % slower) and 12 in extend (256-token extend 657 vs 663
// us; 6 made the 4-token extend 1.4 % and the 256-token one 2 % slower).
constexpr int kRing = 12;                   // ring entries in shared memory (the deepest ring)
template <int G, bool E>
constexpr int ring_depth() { return G == 16 ? 6 : (E ? 12 : 8); }
static_assert(ring_depth<16, false>() > kStages && ring_depth<32, false>() > kStages &&
                  ring_depth<32, true>() <= kRing,
              "the ring covers the tiles the stages hold");

// 32-head decode CTAs store a segment's output in a rolled loop over
// 4-column TMEM loads, measured on GB300: 128-head call 2.07 vs 2.19 ms.  The
// others keep the unrolled store: the rolled one took 33.91 vs 33.66 us per
// batch-40 call at 16 heads, and 67.4 vs 65.2 us for the 4-token extend and
// 676 vs 656 us for the 256-token one at 32.
template <int G, bool E>
constexpr bool compact_epilogue() { return G == 32 && !E; }

// A CTA serves G = 16 or 32 heads (32 when H is a multiple of 32: one read of
// a tile then feeds twice the heads, and an N = 64 MMA costs what N = 32 does).
constexpr int kMaxG = 32;

template <int G>
struct Shape {
    static constexpr int kN = 2 * G;                  // PV MMA N: both E4M3 terms of P for G heads
    static constexpr int kNq = 3 * G;                 // QK^T MMA N: the three E4M3 terms of q
    static constexpr int kQBlk = kNq * 128;           // q rows x 128 B per 128-channel block
    static constexpr int kQBytes = 4 * kQBlk + kNq * 64;  // + the k_pe block
    static constexpr int kQBufs = G == 16 ? 2 : 1;    // q buffers in shared memory
    static constexpr int kOBufs = G == 16 ? 2 : 1;    // O accumulators in TMEM
    static constexpr int kPBytes = (kN / 16) * kPUnit;    // [P1;P2]^T of one tile
    // softmax: one warpgroup per 16 heads, 8 heads per lane (threads 0-15 the
    // first 8 of a token row, 16-31 the other 8)
    static constexpr int kWgs = G / 16;
    static constexpr int kThreads = 384 + 128 * (kWgs - 1);
    static constexpr int kWarpWg = G == 16 ? 6 : 8;   // first softmax warp
    static constexpr int kWarpPv = G == 16 ? 10 : 6;
    static constexpr int kWarpSched = G == 16 ? 11 : 7;
    // TMEM: S[0], S[1] (kNq columns each, starting on multiples of 32), then
    // O[b] at kColO + 4 kN b
    static constexpr uint32_t kSCols = (kNq + 31) / 32 * 32;
    static constexpr uint32_t kColO = 2 * kSCols;
    // q image + two score multipliers and a causal limit per row
    static constexpr int kImage = kQBytes + G * kCoefBytesPerRow;
    static_assert(kQBytes % 1024 == 0, "swizzle atoms need 1 KB alignment");
    static_assert(kColO + kOBufs * 4 * kN <= kTmemCols, "TMEM columns");
};

// shared memory map (offsets from a 1024-byte aligned base), the same for
// both head counts
constexpr int kQRegion = 2 * Shape<16>::kQBytes;
static_assert(Shape<16>::kQBufs * Shape<16>::kQBytes <= kQRegion &&
              Shape<32>::kQBufs * Shape<32>::kQBytes <= kQRegion, "q region");
constexpr int kOffStage = 0;
constexpr int kOffQ = kOffStage + kStages * kStage;
constexpr int kOffP = kOffQ + kQRegion;
constexpr int kOffRing = kOffP + 2 * Shape<kMaxG>::kPBytes;   // kRing x 64 slots (int32)
constexpr int kOffBar = kOffRing + kRing * kTT * 4;
constexpr int kOffRed = kOffBar + 512;      // tile maxima: 2 x 4 warps x G
constexpr int kOffLsum = kOffRed + 2 * 4 * kMaxG * 4;   // softmax denominators: 4 warps x G
constexpr int kOffCoef = kOffLsum + 4 * kMaxG * 4;      // per q buffer: 2 G multipliers, G limits
constexpr int kOffFlag = kOffCoef + 2 * 16 * kCoefBytesPerRow;   // rescale votes: per warpgroup 2 x 4 warps
constexpr int kOffMisc = kOffFlag + 64;     // TMEM base, abort flag
constexpr int kSegTab = 64;                 // segment records a CTA keeps in shared memory
constexpr int kOffSegTab = kOffMisc + 16;   // kSegTab x 32 B
constexpr int kOffInv = kOffSegTab + kSegTab * 32;   // epilogue: per warpgroup 16 inverse denominators
constexpr int kSmemBytes = kOffInv + kMaxG * 4 + 1024;
static_assert(Shape<16>::kQBufs * 16 * kCoefBytesPerRow <= 2 * 16 * kCoefBytesPerRow &&
                  Shape<32>::kQBufs * 32 * kCoefBytesPerRow <= 2 * 16 * kCoefBytesPerRow,
              "multiplier and limit space");
static_assert(Shape<16>::kImage == kTcQImageBytes && Shape<32>::kImage == 2 * kTcQImageBytes,
              "q image sizes the plan reserves");
static_assert(kBlk % 1024 == 0 && kStage % 1024 == 0, "swizzle atoms need 1 KB alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kTT == kM && kTcTileTokens % kTT == 0, "a tile fills the MMA's M; segments start on tiles");
static_assert(Shape<16>::kWarpPv == Shape<16>::kWarpWg + 4 && Shape<16>::kWarpSched == Shape<16>::kWarpPv + 1 &&
                  Shape<16>::kThreads == 32 * (Shape<16>::kWarpSched + 1),
              "warp roles, 16 heads");
static_assert(Shape<32>::kWarpPv == kWarpQ + 1 && Shape<32>::kWarpSched == Shape<32>::kWarpPv + 1 &&
                  Shape<32>::kWarpWg == 8 && Shape<32>::kThreads == 32 * (Shape<32>::kWarpWg + 8),
              "warp roles, 32 heads: warpgroups fill | issuers | softmax | softmax");

enum : int {
    KV_FULL = 0, KV_EMPTY = kStages, S_FULL = 2 * kStages, S_FREE = S_FULL + 2, P_FULL = S_FREE + 2,
    PV_DONE = P_FULL + 2, O_FREE = PV_DONE + 2, Q_FULL = O_FREE + 2, Q_FREE = Q_FULL + 2,
    DONE = Q_FREE + 2, SL_FULL = DONE + 1, SL_EMPTY = SL_FULL + kRing,
    NUM_BARS = SL_EMPTY + kRing
};
static_assert(NUM_BARS * 8 <= 512, "barrier space");

// b: the request, or (extend) the query block; req: the request whose pages
// and context the segment reads
struct Seg {
    int32_t b, req, t0, t1, part, ntiles;
};
// a segment table entry: the record and its request's first page-table entry
struct alignas(16) SegEntry {
    Seg s;
    int32_t pages, pad;
};
static_assert(sizeof(SegEntry) == 32, "segment table entries");

// E: extend plan (segments name query blocks); the decode kernels are
// compiled without the indirection
template <bool E>
__device__ __forceinline__ Seg load_seg(const DecodeParams& p, int si) {
    Seg s;
    s.b = p.segs[4 * si];
    s.t0 = p.segs[4 * si + 1];
    s.t1 = p.segs[4 * si + 2];
    s.part = p.segs[4 * si + 3];
    s.req = E ? p.blocks[4 * s.b] : s.b;
    // a segment longer than the device-side context means the page table
    // changed after planning: it is skipped (and flagged by the MMA thread)
    s.ntiles = s.t1 <= p.seq_lens[s.req] ? (s.t1 - s.t0 + kTT - 1) / kTT : 0;
    return s;
}

// The same read out of line, for the segments past a 16-head CTA's table
// (rarely reached; the tables it reads come by value so that no thread copies
// the launch parameters to local memory for the call).
template <bool E>
__device__ __noinline__ Seg load_seg_past_table(const int32_t* segs, const int32_t* blocks, const int32_t* seq_lens,
                                                int si) {
    Seg s;
    s.b = segs[4 * si];
    s.t0 = segs[4 * si + 1];
    s.t1 = segs[4 * si + 2];
    s.part = segs[4 * si + 3];
    s.req = E ? blocks[4 * s.b] : s.b;
    s.ntiles = s.t1 <= seq_lens[s.req] ? (s.t1 - s.t0 + kTT - 1) / kTT : 0;
    return s;
}

// The CTA's segments lo .. hi - 1.  The first N of them are loaded into
// shared memory once, before the roles start, so that no role waits on the
// plan's dependent loads (record, then context length) at a switch between
// segments; later ones are read from the plan.  16-head CTAs keep kSegTab
// (batch-40 call 33.94 vs 34.18 us on GB300); 32-head CTAs none: at 128
// registers a thread the table's code made that kernel spill more, and it
// ran 12 % slower (256-token extend 780 vs 656 us).
template <bool E, int N>
struct SegView {
    const SegEntry* tab;
    int lo, hi;
    __device__ __forceinline__ Seg at(const DecodeParams& p, int si) const {
        if constexpr (N > 0) {
            if (si - lo < N) return tab[si - lo].s;
            return load_seg_past_table<E>(p.segs, p.blocks, p.seq_lens, si);
        } else if constexpr (N < 0) {
            return load_seg_past_table<E>(p.segs, p.blocks, p.seq_lens, si);
        }
        return load_seg<E>(p, si);
    }
};

// Segment records a CTA keeps in shared memory: 16-head CTAs kSegTab; 32-head
// CTAs none, and 32-head decode CTAs (-1) read each record through one
// out-of-line call (128-head call 2.03 vs 2.07 ms on GB300; 32-head extend
// keeps the inlined read: out of line it measured 661 vs 636 us for the
// 256-token extend, and 16-head decode 30.30 vs 30.15 us).
template <int G, bool E>
constexpr int seg_tab_entries() { return G == 16 ? kSegTab : (E ? 0 : -1); }

template <bool E, int N>
__device__ __forceinline__ int count_tiles(const DecodeParams& p, const SegView<E, N>& sv) {
    int n = 0;
    for (int si = sv.lo; si < sv.hi; ++si) n += sv.at(p, si).ntiles;
    return n;
}

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
    const uint32_t h = e4m3x2_to_f16x2(two);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// named barrier of softmax warpgroup g (ids 1, 2; 0 is __syncthreads),
// immediate ids so that the kernel reserves only those
__device__ __forceinline__ void wg_bar(int g) {
    if (g == 0) asm volatile("bar.sync 1, 128;\n" ::: "memory");
    else asm volatile("bar.sync 2, 128;\n" ::: "memory");
}

// ------------------------------------------------------------ producer warps
//
// The scheduler warp walks the CTA's tiles ahead of the stage fills: it resolves
// the 128 rows of a tile to pool slots, publishes them in a shared ring
// (SL_FULL / SL_EMPTY) and has L2 prefetch each row's cache lines.  By the
// time a stage frees up, the rows it needs are on their way to (or already
// in) L2, so a stage is held for an L2 round trip rather than a DRAM one.

constexpr int32_t kNoRow = INT32_MIN;

// The bounded wait of the roles of a CTA of G heads.  16-head CTAs wait with
// whole warps, also in their MMA issuers, and use the polled form; 32-head
// CTAs (512 threads at 128 registers, whose speed moved by 5-18 % with the
// shape of their code) keep the single-lane issuers and mbar_wait.
template <int G>
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* flags) {
    if constexpr (G == 16) return mbar_wait_polled(bar, parity, abort, flags);
    else return mbar_wait(bar, parity, abort, flags);
}

// A wait made by every lane of a warp that then acts together (shuffles,
// warp barriers): the warp goes on only if every lane's wait succeeded, so
// that after an abort no lane leaves the loop while the others stay in it.
template <int G>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t* flags) {
    return __all_sync(0xffffffffu, bwait<G>(bar, parity, abort, flags));
}

// The page holding token t (t / page_size by the launch's multiply and shift).
__device__ __forceinline__ int32_t page_of(const DecodeParams& p, int32_t t) {
    return static_cast<int32_t>((static_cast<uint64_t>(static_cast<uint32_t>(t)) * p.page_magic) >> p.page_shift);
}

// Cursor over the tiles of a CTA's segments, with the raw page entries of
// rows 2 lane, 2 lane + 1 of one tile.
template <bool E, int N>
struct TileCursor {
    int si, seg_hi, it;
    Seg sg;
    const int32_t* pages;
    int32_t pg[2];                      // page entry, or kNoRow past the context
    int32_t t[2];                       // token index of each row
    SegView<E, N> sv;                   // the shared segment table (tab null until it is loaded)

    // first: the first segment's t0, t1 and page-table offset when the
    // launch carries them (its page entries are then requested before the
    // segment record arrives), else nullptr
    __device__ void init(const DecodeParams& p, int lo, int hi, const int4* first, int lane) {
        si = lo;
        seg_hi = hi;
        sv.tab = nullptr;
        if (first != nullptr && si < seg_hi) {
            pages = p.indices + first->z;
            sg.t0 = first->x;
            sg.t1 = first->y;
            it = 0;
            prefetch(p, lane);
            sg = N < 0 ? load_seg_past_table<E>(p.segs, p.blocks, p.seq_lens, si) : load_seg<E>(p, si);
            if (sg.ntiles > 0) return;
            ++si;
        }
        seek(p, lane);
    }
    // Moves to the first segment from si on that has tiles and requests its
    // first tile's page entries.  The plan carries each segment's page-table
    // offset, so those loads go out with the segment record, before the
    // context check (seq_lens) resolves; they stay inside the planned page
    // table either way.
    __device__ void seek(const DecodeParams& p, int lane) {
        while (si < seg_hi) {
            if (N > 0 && sv.tab != nullptr && si - sv.lo < N) {
                const SegEntry& e = sv.tab[si - sv.lo];
                sg = e.s;
                pages = p.indices + e.pages;
            } else {
                pages = p.indices + p.seg_pages[si];
                sg = (N > 0 && sv.tab != nullptr) || N < 0 ? load_seg_past_table<E>(p.segs, p.blocks, p.seq_lens, si)
                                                           : load_seg<E>(p, si);
            }
            it = 0;
            prefetch(p, lane);
            if (sg.ntiles > 0) break;
            ++si;
        }
    }
    __device__ bool valid() const { return si < seg_hi; }
    // issue the (independent) index loads of the current tile; nothing waits
    // on them until rows() is called
    __device__ void prefetch(const DecodeParams& p, int lane) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            t[q] = sg.t0 + it * kTT + 2 * lane + q;
            pg[q] = t[q] < sg.t1 ? pages[page_of(p, t[q])] : kNoRow;
        }
    }
    // slot of each row, or -1 (past the context or outside the pool: flagged)
    __device__ void rows(const DecodeParams& p, int32_t (&slot)[2]) const {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int64_t s = int64_t(pg[q]) * p.page_size + (t[q] - page_of(p, t[q]) * p.page_size);
            const bool ok = pg[q] >= 0 && s < p.num_slots;
            if (!ok && pg[q] != kNoRow) raise_flag(p.flags, MLA_FLAG_INDEX_OOB);
            slot[q] = ok ? static_cast<int32_t>(s) : -1;
        }
    }
    // next tile, its page entries requested
    __device__ void advance(const DecodeParams& p, int lane) {
        if (++it == sg.ntiles) {
            ++si;
            seek(p, lane);
        } else {
            prefetch(p, lane);
        }
    }
};

// Copies warp w's share of tile i into its stage: c_kv block w (8 chunks of
// 16 B per row, four rows per instruction) and k_pe rows 8g .. 8g+7 for
// g = w, w+4 (4 chunks per row, eight rows per instruction).
// `sl` holds the slots of rows lane + 32q.
__device__ __forceinline__ void fill_share(const DecodeParams& p, uint8_t* stage, const int32_t (&sl)[2],
                                           int w, int lane) {
    const int r4 = lane >> 3, c8 = lane & 7;
#pragma unroll
    for (int j = 0; j < kTT / 4; ++j) {
        const int row = 4 * j + r4;
        const int32_t s = __shfl_sync(0xffffffffu, sl[j >> 3], row & 31);
        const int64_t ss = s >= 0 ? s : 0;
        cp_async16(stage + w * kBlk + row * 128 + ((c8 ^ (row & 7)) << 4),
                   p.ckv + ss * p.ckv_stride + w * 128 + c8 * 16, s >= 0 ? 16u : 0u);
    }
    const int r8 = lane >> 2, c4 = lane & 3;
#pragma unroll
    for (int gq = 0; gq < kTT / 8 / kFillWarps; ++gq) {
        const int g = w + kFillWarps * gq;
        const int row = 8 * g + r8;
        const int32_t s = __shfl_sync(0xffffffffu, sl[g >> 2], row & 31);
        const int64_t ss = s >= 0 ? s : 0;
        cp_async16(stage + 4 * kBlk + row * 64 + ((c4 ^ ((row >> 1) & 3)) << 4),
                   p.kpe + ss * p.kpe_stride + c4 * 16, s >= 0 ? 16u : 0u);
    }
}

// cur: started by the caller (its first page entries already requested)
template <int G, bool E, int kR, int N>
__device__ void scheduler(const DecodeParams& p, uint8_t* base, uint64_t* bars, volatile int* abort,
                          TileCursor<E, N>& cur, const SegView<E, N>& sv, int lane) {
    int32_t* ring = reinterpret_cast<int32_t*>(base + kOffRing);
    cur.sv = sv;
    // one prefetch sweep per row when k_pe follows c_kv in the same row
    const bool joint = p.kpe == p.ckv + kDCkv && p.kpe_stride == p.ckv_stride;
    // publishes every tile as soon as its ring entry is free (the ring bounds
    // how far ahead of the softmax warps the prefetches run)
    for (int n = 0; cur.valid(); ++n) {
        const int e = n % kR;
        const uint32_t u = static_cast<uint32_t>(n / kR);
        int32_t sl[2];
        cur.rows(p, sl);
        cur.advance(p, lane);                         // the next tile's index loads fly meanwhile
        if (!warp_wait<G>(&bars[SL_EMPTY + e], (u & 1) ^ 1, abort, p.flags)) break;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            if (sl[q] < 0) continue;
            const uint8_t* row = p.ckv + int64_t(sl[q]) * p.ckv_stride;
            if (joint) {
                prefetch_row_l2<kDQk>(row);
            } else {
                prefetch_row_l2<kDCkv>(row);
                prefetch_row_l2<kDKpe>(p.kpe + int64_t(sl[q]) * p.kpe_stride);
            }
        }
        *reinterpret_cast<int2*>(ring + e * kTT + 2 * lane) = make_int2(sl[0], sl[1]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[SL_FULL + e]);
    }
}

template <int G, bool E, int kR, int N>
__device__ void fill_warp(const DecodeParams& p, uint8_t* base, uint64_t* bars, volatile int* abort,
                          const SegView<E, N>& sv, int w, int lane) {
    const int32_t* ring = reinterpret_cast<const int32_t*>(base + kOffRing);
    const int total = count_tiles<E>(p, sv);
    for (int i = 0; i < total; ++i) {
        const int slot = i % kStages;
        const uint32_t u = static_cast<uint32_t>(i / kStages);
        const int e = i % kR;
        if (!warp_wait<G>(&bars[SL_FULL + e], static_cast<uint32_t>(i / kR) & 1, abort, p.flags)) break;
        int32_t sl[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) sl[q] = ring[e * kTT + lane + 32 * q];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[SL_EMPTY + e]);
        if (!warp_wait<G>(&bars[KV_EMPTY + slot], (u & 1) ^ 1, abort, p.flags)) break;
        fill_share(p, base + kOffStage + slot * kStage, sl, w, lane);
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

// Descriptors are built once per operand region and advanced by adding the
// (compile-time) byte offset / 16 to the start-address field: the issuing
// thread then spends a 64-bit add per MMA instead of rebuilding the word,
// which on GB300 halves the time a thread takes to issue one MMA.  The field
// cannot carry: shared addresses stay below 256 KB.
__device__ __forceinline__ uint64_t desc_at(uint64_t base_desc, uint32_t byte_offset) {
    return base_desc + static_cast<uint64_t>(byte_offset >> 4);
}

// 16-head CTAs issue their MMAs from whole warps (one elected lane issues
// and commits; the operands, computed by the warp, stay warp-uniform): the
// batch-40 call 33.7 vs 34.2 us on GB300.  32-head CTAs issue from one lane.
template <int G>
constexpr bool warp_issue() { return G == 16; }

// q_done: the segment's last tile (its q buffer is released with it).
template <int G>
__device__ __forceinline__ void issue_qk(const MmaCtx& c, int i, int qs, bool q_done) {
    using S = Shape<G>;
    const int slot = i & 1;
    const uint32_t stage = c.sbase + kOffStage + (i % kStages) * kStage;
    const uint32_t qb = c.sbase + kOffQ + qs * S::kQBytes;
    // c_kv channels: 128-byte swizzle, 8-row groups 1 KB apart; k_pe
    // channels: 64-byte swizzle, 8-row groups 512 B apart
    const uint64_t a128 = smem_desc(stage, 16, 1024, kSwizzle128B);
    const uint64_t b128 = smem_desc(qb, 16, 1024, kSwizzle128B);
    const uint64_t a64 = smem_desc(stage + 4 * kBlk, 16, 512, kSwizzle64B);
    const uint64_t b64 = smem_desc(qb + 4 * S::kQBlk, 16, 512, kSwizzle64B);
    const uint32_t d = c.tmem + kColS + S::kSCols * slot;
    if (!warp_issue<G>() || elect_one()) {
#pragma unroll
        for (int ks = 0; ks < kKSteps; ++ks) {
            const uint64_t a = ks < 16 ? desc_at(a128, (ks >> 2) * kBlk + (ks & 3) * 32)
                                       : desc_at(a64, (ks - 16) * 32);
            const uint64_t b = ks < 16 ? desc_at(b128, (ks >> 2) * S::kQBlk + (ks & 3) * 32)
                                       : desc_at(b64, (ks - 16) * 32);
            mma_e4m3(d, a, b, c.idesc_qk, ks > 0);
        }
        mma_commit(&c.bars[S_FULL + slot]);
        if (q_done) mma_commit(&c.bars[Q_FREE + qs]);   // q buffer done
    }
    if constexpr (warp_issue<G>()) __syncwarp();
}

// PV of tile j into O buffer `ob`; the segment's first tile overwrites it.
template <int G>
__device__ __forceinline__ void issue_pv(const MmaCtx& c, int j, int ob, bool first) {
    using S = Shape<G>;
    const int kv = j % kStages;
    // A = V^T: 128 channels (one column block) x 32 tokens, MN-major;
    // B = [P1;P2]^T: 32 tokens x kN (term, head), MN-major, unswizzled, one
    // 16-column group (16 heads of one term) every kPUnit bytes
    const uint64_t a0 = smem_desc(c.sbase + kOffStage + kv * kStage, kBlk, 1024, kSwizzle128B);
    const uint64_t b0 = smem_desc(c.sbase + kOffP + (j & 1) * S::kPBytes, 128, kPUnit, kSwizzleNone);
    const uint32_t d = c.tmem + S::kColO + 4 * S::kN * ob;
    if (!warp_issue<G>() || elect_one()) {
#pragma unroll
        for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
            for (int ks = 0; ks < kTT / 32; ++ks)
                mma_e4m3(d + S::kN * mb, desc_at(a0, mb * kBlk + ks * 32 * 128), desc_at(b0, ks * 32 * 16),
                         c.idesc_pv, ks > 0 || !first);
        }
        mma_commit(&c.bars[PV_DONE + (j & 1)]);
        mma_commit(&c.bars[KV_EMPTY + kv]);   // the stage may be refilled
    }
    if constexpr (warp_issue<G>()) __syncwarp();
}

// Position in the CTA's tile sequence: segment ordinal k and tile it of it.
template <bool E, int N>
struct SegWalk {
    int si, it, k;
    Seg sg;
    __device__ void init(const DecodeParams& p, const SegView<E, N>& sv) {
        si = sv.lo;
        it = 0;
        k = 0;
        while (si < sv.hi && (sg = sv.at(p, si)).ntiles == 0) ++si;
    }
    __device__ void advance(const DecodeParams& p, const SegView<E, N>& sv) {
        if (++it == sg.ntiles) {
            it = 0;
            ++k;
            ++si;
            while (si < sv.hi && (sg = sv.at(p, si)).ntiles == 0) ++si;
        }
    }
};

// Two issuers: one sends QK^T of the tiles in order, the other PV.  A thread
// waits for each MMA it issues to be accepted, so with one issuer the PV of
// tile i queued behind QK^T of tile i + 1 (and freed its stage late); with
// two, each goes out as soon as its inputs are ready.  QK^T needs its stage
// full, so it runs at most a stage ahead of PV by construction.  A warp that
// issues as a whole waits with warp_wait, so that its lanes agree.
template <int G>
__device__ __forceinline__ bool issuer_wait(uint64_t* bar, uint32_t parity, const MmaCtx& c) {
    if constexpr (warp_issue<G>()) return warp_wait<G>(bar, parity, c.abort, c.flags);
    else return bwait<G>(bar, parity, c.abort, c.flags);
}

template <int G, bool E>
__device__ void qk_issuer(const DecodeParams& p, const MmaCtx& c, const SegView<E, seg_tab_entries<G, E>()>& sv) {
    using S = Shape<G>;
    int total = 0;
    for (int si = sv.lo; si < sv.hi; ++si) {
        const Seg sg = sv.at(p, si);
        if (sg.ntiles == 0 && sg.t1 > sg.t0 && (!warp_issue<G>() || (threadIdx.x & 31) == 0))
            raise_flag(p.flags, MLA_FLAG_PLAN_MISMATCH);
        total += sg.ntiles;
    }
    SegWalk<E, seg_tab_entries<G, E>()> wq;
    wq.init(p, sv);
    for (int qk = 0; qk < total; ++qk) {
        const int slot = qk & 1;
        const int qs = wq.k % S::kQBufs;
        if (wq.it == 0 && !issuer_wait<G>(&c.bars[Q_FULL + qs], static_cast<uint32_t>(wq.k / S::kQBufs) & 1, c))
            break;
        if (!issuer_wait<G>(&c.bars[KV_FULL + qk % kStages], static_cast<uint32_t>(qk / kStages) & 1, c)) break;
        if (!issuer_wait<G>(&c.bars[S_FREE + slot], ((static_cast<uint32_t>(qk) >> 1) & 1) ^ 1, c)) break;
        fence_after_sync();
        fence_proxy_async_smem();
        issue_qk<G>(c, qk, qs, wq.it == wq.sg.ntiles - 1);
        wq.advance(p, sv);
    }
    // every MMA issued so far has completed before TMEM may be released
    if (!warp_issue<G>() || elect_one()) mma_commit(&c.bars[DONE]);
    if constexpr (warp_issue<G>()) __syncwarp();
    volatile int never = 0;
    mbar_wait(&c.bars[DONE], 0, &never, c.flags, 1000000000ull);
}

template <int G, bool E>
__device__ void pv_issuer(const DecodeParams& p, const MmaCtx& c, const SegView<E, seg_tab_entries<G, E>()>& sv) {
    using S = Shape<G>;
    const int total = count_tiles<E>(p, sv);
    SegWalk<E, seg_tab_entries<G, E>()> wp;
    wp.init(p, sv);
    for (int pv = 0; pv < total; ++pv) {
        const int ob = wp.k % S::kOBufs;
        if (!issuer_wait<G>(&c.bars[P_FULL + (pv & 1)], (static_cast<uint32_t>(pv) >> 1) & 1, c)) break;
        // a segment's first PV overwrites its O buffer: the segment that used
        // it before has been read out
        if (wp.it == 0 && !issuer_wait<G>(&c.bars[O_FREE + ob], (static_cast<uint32_t>(wp.k / S::kOBufs) & 1) ^ 1, c))
            break;
        fence_after_sync();
        fence_proxy_async_smem();
        issue_pv<G>(c, pv, ob, wp.it == 0);
        wp.advance(p, sv);
    }
    if (!warp_issue<G>() || elect_one()) mma_commit(&c.bars[DONE]);
    if constexpr (warp_issue<G>()) __syncwarp();
    volatile int never = 0;
    mbar_wait(&c.bars[DONE], 0, &never, c.flags, 1000000000ull);
}

// ---------------------------------------------------------------- q prep
//
// q is split once per request by a small kernel that runs just before the
// decode kernel: it writes [q1;q2;q3] as the exact shared-memory image the
// QK^T MMA reads (128-byte swizzle for the 512 c_kv channels, 64-byte for the
// 64 k_pe channels) plus the per-head score multipliers.  A decode CTA then
// fetches a segment's q with two bulk copies.
//
// Per head, with x = q * 2^sigma (largest |x| in [128, 256)):
//   q1 = E4M3(x), q2 = E4M3(x - q1)           -- exact for every entry above
//                                                2^-14 of the head's largest
//   r  = x - q1 - q2 (exact in fp32),  q3 = E4M3(r * 2^tau)
//                                              (largest |r| 2^tau in [128, 256))
// so q = 2^-sigma (q1 + q2) + 2^-(sigma + tau) q3: entries the first two terms
// cannot hold (too small next to the head's largest) keep 4 significant bits
// in the third, down to 2^-14 of the largest such remainder.

// Splits 16 BF16 values (two uint4) scaled by `scale` into two E4M3 terms
// and returns the exact remainders in `rem`.
__device__ __forceinline__ void split_chunk(const uint4& va, const uint4& vb, float scale, uint4& t1,
                                            uint4& t2, float (&rem)[16]) {
    const uint32_t w8[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
    uint32_t o1[4], o2[4];
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
            const float y0 = x0 - d.x, y1 = x1 - d.y;    // exact
            const uint16_t b2 = f32x2_to_e4m3x2(y0, y1);
            const float2 d2 = e4m3x2_to_float2(b2);
            rem[4 * e + 2 * hh] = y0 - d2.x;             // exact
            rem[4 * e + 2 * hh + 1] = y1 - d2.y;
            lo1 |= static_cast<uint32_t>(b1) << (16 * hh);
            lo2 |= static_cast<uint32_t>(b2) << (16 * hh);
        }
        o1[e] = lo1;
        o2[e] = lo2;
    }
    t1 = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    t2 = make_uint4(o2[0], o2[1], o2[2], o2[3]);
}

// 16 remainders times `scale` -> one E4M3 term.
__device__ __forceinline__ uint4 third_term(const float (&rem)[16], float scale) {
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        o[e] = static_cast<uint32_t>(f32x2_to_e4m3x2(rem[4 * e] * scale, rem[4 * e + 1] * scale)) |
               (static_cast<uint32_t>(f32x2_to_e4m3x2(rem[4 * e + 2] * scale, rem[4 * e + 3] * scale)) << 16);
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float amax_bf16x8(const uint4& v, float a) {
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
        a = fmaxf(a, fmaxf(fabsf(__uint_as_float(w4[e] << 16)), fabsf(__uint_as_float(w4[e] & 0xffff0000u))));
    return a;
}

// true if one of the 8 BF16 values is an infinity or a NaN (exponent all ones)
__device__ __forceinline__ bool nonfinite_bf16x8(const uint4& v) {
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    bool bad = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) bad |= (w4[e] & 0x7F80u) == 0x7F80u || (w4[e] & 0x7F800000u) == 0x7F800000u;
    return bad;
}

__device__ __forceinline__ float amax_f32x16(const float (&r)[16], float a) {
#pragma unroll
    for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(r[i]));
    return a;
}

// 2^e with e clamped to [-100, 100] (scales of the q terms)
__device__ __forceinline__ int split_exponent(float amax) {
    int e2 = 0;
    frexpf(amax, &e2);                              // amax = m * 2^e2, m in [0.5, 1)
    const int s = amax > 0.f ? 8 - e2 : 0;          // amax * 2^s in [128, 256)
    return s > 100 ? 100 : (s < -100 ? -100 : s);
}

// Four warps (query rows) per split block: one warp per SM sub-partition,
// which still fits beside a 16-head decode CTA; measured on GB300 against
// two and one: batch-40 call 34.29 vs 34.41 and 34.63 us.
constexpr int kSplitThreads = 128;

// One warp per image row: lane c splits 16-channel chunk c of c_kv, lanes 0-3
// also chunk c of k_pe.  Decode: one image per (request, group of G heads);
// heads >= H get zero rows and multipliers 0.  Extend: one image per query
// block, row r = block row r (token row / H, head row % H); rows past the
// block's end are zero.  Each valid row also gets its causal limit.  A row
// holding an infinity or a NaN gets zero terms and NaN multipliers: its
// output row and lse come out NaN.
// At most 56 registers: one warp of it then fits on an SM sub-partition
// beside a 16-head decode CTA (3 warps of 152 registers), so the decode
// kernel's CTAs are placed while the split still runs.
template <int G>
__global__ void __maxnreg__(56) mla_q_split_kernel(const DecodeParams p) {
    using S = Shape<G>;
    griddep_launch_dependents();                // the decode kernel may start loading KV now
    const int wg = (blockIdx.x * kSplitThreads + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int image = wg / G, r = wg % G;
    if (image >= (p.blocks ? p.n_blocks : p.batch * p.head_groups)) return;
    int64_t tok;
    int head, lim = 0;
    bool valid;
    if (p.blocks) {
        const int32_t* blk = p.blocks + 4 * image;
        valid = r < blk[2];
        const int row = blk[1] + (valid ? r : 0);
        tok = row / p.heads;
        head = row % p.heads;
        lim = blk[3] + static_cast<int>(tok);
    } else {
        tok = image / p.head_groups;
        head = (image % p.head_groups) * G + r;
        valid = head < p.heads;
    }
    const uint4* src =
        reinterpret_cast<const uint4*>(p.q + tok * p.q_sb + int64_t(valid ? head : 0) * p.q_sh);
    const uint4 z = make_uint4(0, 0, 0, 0);
    uint4 va = valid ? src[2 * lane] : z, vb = valid ? src[2 * lane + 1] : z;
    const bool rope = lane < 4;
    uint4 ra = valid && rope ? src[64 + 2 * lane] : z, rb = valid && rope ? src[64 + 2 * lane + 1] : z;
    const bool bad = __any_sync(0xffffffffu, nonfinite_bf16x8(va) || nonfinite_bf16x8(vb) ||
                                                 nonfinite_bf16x8(ra) || nonfinite_bf16x8(rb));
    if (bad) va = vb = ra = rb = z;
    float amax = amax_bf16x8(rb, amax_bf16x8(ra, amax_bf16x8(vb, amax_bf16x8(va, 0.f))));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int sigma = split_exponent(amax);
    const float scale = ldexpf(1.f, sigma);
    uint4 c1, c2, k1, k2;
    float rc[16], rk[16];
    split_chunk(va, vb, scale, c1, c2, rc);
    split_chunk(ra, rb, scale, k1, k2, rk);          // zeros on lanes 4-31
    float amax3 = amax_f32x16(rk, amax_f32x16(rc, 0.f));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax3 = fmaxf(amax3, __shfl_xor_sync(0xffffffffu, amax3, o));
    const int tau = amax3 > 0.f ? split_exponent(amax3) : 0;
    const float scale3 = ldexpf(1.f, tau);
    const uint4 c3 = third_term(rc, scale3), k3 = third_term(rk, scale3);

    uint8_t* img = p.qimg + int64_t(image) * S::kImage;
    const int row1 = r, row2 = G + r, row3 = 2 * G + r;
    const uint64_t keep = l2_policy(true);          // read again at each segment of the image
    {                                               // c_kv: 128-byte rows, 128-byte swizzle
        const int cb = lane >> 3, cc = lane & 7;
        uint8_t* blk = img + cb * S::kQBlk;
        st_v4_hint(blk + row1 * 128 + ((cc ^ (row1 & 7)) << 4), c1, keep);
        st_v4_hint(blk + row2 * 128 + ((cc ^ (row2 & 7)) << 4), c2, keep);
        st_v4_hint(blk + row3 * 128 + ((cc ^ (row3 & 7)) << 4), c3, keep);
    }
    if (rope) {                                     // k_pe: 64-byte rows, 64-byte swizzle
        uint8_t* blk = img + 4 * S::kQBlk;
        st_v4_hint(blk + row1 * 64 + ((lane ^ ((row1 >> 1) & 3)) << 4), k1, keep);
        st_v4_hint(blk + row2 * 64 + ((lane ^ ((row2 >> 1) & 3)) << 4), k2, keep);
        st_v4_hint(blk + row3 * 64 + ((lane ^ ((row3 >> 1) & 3)) << 4), k3, keep);
    }
    if (lane == 0) {
        // multipliers of the first two terms and of the third (2^-tau finer)
        const float base = valid ? (bad ? __int_as_float(0x7FC00000) : p.softmax_scale * p.k_scale * kLog2e) : 0.f;
        float* coef = reinterpret_cast<float*>(img + S::kQBytes);
        coef[r] = ldexpf(base, -sigma);
        coef[G + r] = ldexpf(ldexpf(base, -sigma), -tau);
        reinterpret_cast<int32_t*>(coef + 2 * G)[r] = valid ? lim : 0;
    }
}

// Warp 5: fetches each segment's q image into its q buffer (and the
// multipliers) once the split kernel has finished.
template <int G, bool E>
__device__ void q_fetch(const DecodeParams& p, uint8_t* base, uint64_t* bars, volatile int* abort,
                        const SegView<E, seg_tab_entries<G, E>()>& sv, int lane) {
    using S = Shape<G>;
    if (lane != 0) return;
    griddep_wait();                                 // the q images are complete
    int k = 0;
    for (int si = sv.lo; si < sv.hi; ++si) {
        const Seg sg = sv.at(p, si);
        if (sg.ntiles == 0) continue;
        const int qs = k % S::kQBufs;
        const uint32_t qu = static_cast<uint32_t>(k / S::kQBufs);
        if (!bwait<G>(&bars[Q_FREE + qs], (qu & 1) ^ 1, abort, p.flags)) break;
        // After an abort the softmax warps keep arriving on Q_FREE without
        // the QK^T commit, so a phase can complete before the buffer's last
        // copy has landed; a second copy (and arrive.expect_tx) on Q_FULL
        // then would overrun its phase.  So no copy is issued once the CTA
        // has aborted, and none before the buffer's previous copy landed
        // (its own Q_FULL phase: immediate unless aborted).
        if (*abort) break;
        if (k >= S::kQBufs) {
            volatile int never = 0;
            if (!mbar_wait(&bars[Q_FULL + qs], (qu - 1) & 1, &never, p.flags, 1000000000ull)) break;
        }
        const int64_t image = E ? sg.b : int64_t(sg.b) * p.head_groups + blockIdx.y;
        const uint8_t* img = p.qimg + image * S::kImage;
        mbar_arrive_expect_tx(&bars[Q_FULL + qs], S::kImage);
        bulk_copy_g2s(smem_u32(base + kOffQ + qs * S::kQBytes), img, S::kQBytes, &bars[Q_FULL + qs]);
        bulk_copy_g2s(smem_u32(base + kOffCoef + qs * G * kCoefBytesPerRow), img + S::kQBytes,
                      G * kCoefBytesPerRow, &bars[Q_FULL + qs]);
        ++k;
    }
    // copies in flight (after an abort) land before the CTA exits
    volatile int never = 0;
    for (int j = k - S::kQBufs < 0 ? 0 : k - S::kQBufs; j < k; ++j)
        mbar_wait(&bars[Q_FULL + j % S::kQBufs], static_cast<uint32_t>(j / S::kQBufs) & 1, &never, p.flags,
                  1000000000ull);
}

// ------------------------------------------------- softmax / rescale WG

struct WgCtx {
    uint8_t* base;
    uint64_t* bars;
    uint32_t tmem_lane;     // TMEM base + this warp's lane quadrant
    volatile int* abort;
    uint32_t* flags;
    int row;                // TMEM lane of O = channel within a 128-channel block
    int srow;               // token of S (M = 64: lanes 0-15 of each lane quadrant)
    int h0;                 // this warpgroup's heads: h0 .. h0 + 15
    int hb;                 // heads hb .. hb + 7 of token srow are this lane's: lanes 0-15
                            // take h0 .. h0 + 7, 16-31 h0 + 8 .. h0 + 15
    int wg, wq, lane;       // softmax warpgroup, warp within it 0..3, lane
};

// O (one segment's accumulator) *= alpha per head, in TMEM, for the
// warpgroup's 16 heads.  Each 128-channel block holds kN columns: head h's two
// P terms in columns h and G + h.
template <int G>
__device__ __forceinline__ void rescale_o(const WgCtx& w, uint32_t ocol, const float (&alpha)[16]) {
    using S = Shape<G>;
#pragma unroll
    for (int mb = 0; mb < 4; ++mb) {
        uint32_t r[2][16];
        tmem_ld16(w.tmem_lane + ocol + S::kN * mb + w.h0, r[0]);
        tmem_ld16(w.tmem_lane + ocol + S::kN * mb + G + w.h0, r[1]);
        tmem_wait_ld();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
            for (int i = 0; i < 16; ++i) r[cc][i] = __float_as_uint(__uint_as_float(r[cc][i]) * alpha[i]);
        }
        tmem_st16(w.tmem_lane + ocol + S::kN * mb + w.h0, r[0]);
        tmem_st16(w.tmem_lane + ocol + S::kN * mb + G + w.h0, r[1]);
    }
    tmem_wait_st();
}

// Reduction over the 16 lanes of a half warp of V (8 or 16) values at once by
// halving exchanges (V shuffles instead of 4 V): afterwards lane l holds
// value idx(l) reduced over its half, idx = (l >> 1) & 7 for V = 8 (lanes l
// and l ^ 1 agree) and l & 15 for V = 16.
template <bool kMax, int V>
__device__ __forceinline__ float half_reduce(const float (&v)[V], int lane) {
    auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
    float a8[8], a4[4], a2[2];
    if constexpr (V == 16) {
        const bool b3 = lane & 8;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            a8[j] = op(b3 ? v[j + 8] : v[j], __shfl_xor_sync(0xffffffffu, b3 ? v[j] : v[j + 8], 8));
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) a8[j] = v[j];
    }
    const int s4 = V == 16 ? 4 : 8, s2 = V == 16 ? 2 : 4, s1 = V == 16 ? 1 : 2;
    const bool c4 = lane & s4, c2 = lane & s2, c1 = lane & s1;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        a4[j] = op(c4 ? a8[j + 4] : a8[j], __shfl_xor_sync(0xffffffffu, c4 ? a8[j] : a8[j + 4], s4));
#pragma unroll
    for (int j = 0; j < 2; ++j)
        a2[j] = op(c2 ? a4[j + 2] : a4[j], __shfl_xor_sync(0xffffffffu, c2 ? a4[j] : a4[j + 2], s2));
    const float a1 = op(c1 ? a2[1] : a2[0], __shfl_xor_sync(0xffffffffu, c1 ? a2[0] : a2[1], s1));
    return V == 16 ? a1 : op(a1, __shfl_xor_sync(0xffffffffu, a1, 1));
}

template <int V>
__device__ __forceinline__ int half_reduce_index(int lane) { return V == 16 ? (lane & 15) : ((lane >> 1) & 7); }

template <int V>
__device__ __forceinline__ bool half_reduce_writer(int lane) { return V == 16 || (lane & 1) == 0; }

template <int G, bool E>
__device__ void softmax_wg(const DecodeParams& p, const WgCtx& w, const SegView<E, seg_tab_entries<G, E>()>& sv,
                           int head0) {
    using S = Shape<G>;
    constexpr int kHL = 8;                          // heads per lane
    float* red = reinterpret_cast<float*>(w.base + kOffRed);
    float* lsum = reinterpret_cast<float*>(w.base + kOffLsum);
    int* vote = reinterpret_cast<int*>(w.base + kOffFlag);
    const float* coefs = reinterpret_cast<const float*>(w.base + kOffCoef);
    uint8_t* pbase = w.base + kOffP;
    const int32_t* ring = reinterpret_cast<const int32_t*>(w.base + kOffRing);
    // A failed (aborted) wait is not a reason to leave: the softmax warps meet
    // at named barriers, so all of them run the loops to the end; once the
    // abort flag is set every wait returns at once and the results are void.
    int i = 0, k = 0;
    for (int si = sv.lo; si < sv.hi; ++si) {
        const Seg sg = sv.at(p, si);
        if (sg.ntiles == 0) continue;
        const int qs = k % S::kQBufs;
        const uint32_t qu = static_cast<uint32_t>(k / S::kQBufs);
        const uint32_t ocol = S::kColO + 4 * S::kN * (k % S::kOBufs);
        bwait<G>(&w.bars[Q_FULL + qs], qu & 1, w.abort, w.flags);
        // the segment's score multipliers and causal limits stay in shared
        // memory (its q buffer is released at the end of the segment)
        const float* coef = coefs + qs * 3 * G;      // first two terms' multipliers
        const float* coef3 = coef + G;                  // the third term's
        const int32_t* lim = reinterpret_cast<const int32_t*>(coef + 2 * G);
        // extend: tiles reaching the first row's limit need the causal mask
        // (rows are in token order, so the first row's limit is the lowest)
        const int mask_from = E ? lim[0] : INT32_MAX;

        float m[kHL], l[kHL];                       // heads hb .. hb + kHL - 1
#pragma unroll
        for (int j = 0; j < kHL; ++j) {
            m[j] = -INFINITY;
            l[j] = 0.f;
        }
        for (int it = 0; it < sg.ntiles; ++it, ++i) {
            const int slot = i & 1;
            const uint32_t u = static_cast<uint32_t>(i) >> 1;
            // row validity from the scheduler's slot list (a -1 row is zero-filled)
            constexpr int kR = ring_depth<G, E>();
            const int e = i % kR;
            bwait<G>(&w.bars[SL_FULL + e], static_cast<uint32_t>(i / kR) & 1, w.abort, w.flags);
            const bool valid = ring[e * kTT + w.srow] >= 0;
            __syncwarp();
            if (w.lane == 0) mbar_arrive(&w.bars[SL_EMPTY + e]);
            bwait<G>(&w.bars[S_FULL + slot], u & 1, w.abort, w.flags);
            fence_after_sync();
            // the warp's 16 token rows sit in lanes 0-15 of its TMEM quadrant:
            // threads 0-15 read heads h0 .. h0 + 7 of their row, threads 16-31
            // heads h0 + 8 .. h0 + 15 of the same row (term 1 at column h,
            // term 2 at column G + h)
            float s[kHL];
            {
                uint32_t r1[kHL], r2[kHL], r3[kHL];
                const uint32_t sc = w.tmem_lane + kColS + S::kSCols * slot + w.h0;
                tmem_ld_half8<kHL>(sc, r1);
                tmem_ld_half8<kHL>(sc + G, r2);
                tmem_ld_half8<kHL>(sc + 2 * G, r3);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < kHL; ++j)
                    s[j] = valid ? fmaf(__uint_as_float(r1[j]) + __uint_as_float(r2[j]), coef[w.hb + j],
                                        __uint_as_float(r3[j]) * coef3[w.hb + j])
                                 : -INFINITY;
            }
            fence_before_sync();
            mbar_arrive(&w.bars[S_FREE + slot]);

            if constexpr (E) {
                const int tile_t0 = sg.t0 + it * kTT;
                if (tile_t0 + kTT > mask_from) {    // token tile_t0 + srow is hidden from rows
                    const int t = tile_t0 + w.srow; // whose limit it reaches
#pragma unroll
                    for (int j = 0; j < kHL; ++j)
                        if (t >= lim[w.hb + j]) s[j] = -INFINITY;
                }
            }
            bool need = false;
#pragma unroll
            for (int j = 0; j < kHL; ++j) need |= s[j] > m[j] + kTau;   // true on a segment's first tile
            // the running maximum moves only if some score got more than
            // 2^kTau above it (one vote per warp, then one barrier)
            need = __any_sync(0xffffffffu, need);
            int* vb = vote + w.wg * 8 + (i & 1) * 4;
            if (w.lane == 0) vb[w.wq] = need;
            wg_bar(w.wg);
            need = vb[0] | vb[1] | vb[2] | vb[3];
            if (need) {
                const float hmax = half_reduce<true, kHL>(s, w.lane);
                float* rb = red + (i & 1) * 4 * G;
                if (half_reduce_writer<kHL>(w.lane)) rb[w.wq * G + w.hb + half_reduce_index<kHL>(w.lane)] = hmax;
                wg_bar(w.wg);
                float alpha[kHL];
#pragma unroll
                for (int j = 0; j < kHL; ++j) {
                    const int h = w.hb + j;
                    const float tmax = fmaxf(fmaxf(rb[h], rb[G + h]), fmaxf(rb[2 * G + h], rb[3 * G + h]));
                    const float mn = fmaxf(m[j], tmax);
                    alpha[j] = m[j] == -INFINITY ? 0.f : fast_exp2(m[j] - mn);
                    m[j] = mn;
                    l[j] *= alpha[j];
                }
                if (it > 0) {
                    // O holds tiles up to i - 1: rescale once PV(i - 1) has landed;
                    // every lane needs the warpgroup's 16 factors (lanes 0 and 16
                    // have them)
                    float a_all[16];
#pragma unroll
                    for (int j = 0; j < kHL; ++j) {
                        a_all[j] = __shfl_sync(0xffffffffu, alpha[j], 0);
                        a_all[kHL + j] = __shfl_sync(0xffffffffu, alpha[j], 16);
                    }
                    const int j = i - 1;
                    bwait<G>(&w.bars[PV_DONE + (j & 1)], (static_cast<uint32_t>(j) >> 1) & 1, w.abort, w.flags);
                    fence_after_sync();
                    rescale_o<G>(w, ocol, a_all);
                }
            }
            // P = 2^(s - m) <= 2^kTau, stored as two E4M3 terms of p * kPScale;
            // its buffer was last read by PV(i - 2)
            if (i >= 2) bwait<G>(&w.bars[PV_DONE + slot], (u & 1) ^ 1, w.abort, w.flags);
            uint32_t pk1[kHL / 4], pk2[kHL / 4];
#pragma unroll
            for (int e2 = 0; e2 < kHL / 4; ++e2) {
                uint32_t w1 = 0, w2 = 0;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int j = 4 * e2 + 2 * hh;
                    const float x0 = m[j] == -INFINITY ? 0.f : fast_exp2(s[j] - m[j]) * kPScale;
                    const float x1 = m[j + 1] == -INFINITY ? 0.f : fast_exp2(s[j + 1] - m[j + 1]) * kPScale;
                    // x = p1 + p2 / 2^5: p1 the nearest E4M3, p2 the nearest
                    // E4M3 to 2^5 times the remainder, taken in f16 (x <= 256
                    // keeps 11 bits there, f16(x) - p1 is exact and at most 8,
                    // and the factor 2^5 is exact); the denominator sums x
                    // itself.  The factor keeps weights down to 2^-15 / 16
                    // of the running maximum's in the second term.
                    const uint16_t b1 = f32x2_to_e4m3x2(x0, x1);
                    const uint16_t b2 = f16x2_to_e4m3x2(
                        mul_f16x2(sub_f16x2(pack_f16x2(x0, x1), e4m3x2_to_f16x2(b1)), kP2ScaleF16x2));
                    l[j] += x0;
                    l[j + 1] += x1;
                    w1 |= static_cast<uint32_t>(b1) << (16 * hh);
                    w2 |= static_cast<uint32_t>(b2) << (16 * hh);
                }
                pk1[e2] = w1;
                pk2[e2] = w2;
            }
            // [P1;P2]^T: 16-head column group g = term * (G / 16) + head / 16
            uint8_t* pb = pbase + slot * S::kPBytes + (w.hb / 16) * kPUnit + w.srow * 16 + (w.hb % 16);
            uint8_t* pb2 = pb + (G / 16) * kPUnit;
            *reinterpret_cast<uint2*>(pb) = make_uint2(pk1[0], pk1[1]);
            *reinterpret_cast<uint2*>(pb2) = make_uint2(pk2[0], pk2[1]);
            fence_proxy_async_smem();
            fence_before_sync();                    // orders a rescale's TMEM stores too
            mbar_arrive(&w.bars[P_FULL + slot]);
        }

        // ---- epilogue: denominators over the token lanes, normalise, store
        {
            const float hsum = half_reduce<false, kHL>(l, w.lane);
            if (half_reduce_writer<kHL>(w.lane)) lsum[w.wq * G + w.hb + half_reduce_index<kHL>(w.lane)] = hsum;
        }
        wg_bar(w.wg);
        // inverse denominators of the warpgroup's heads h0 + t; a head whose q
        // held an infinity or a NaN has NaN multipliers: its output and lse
        // become NaN (nothing else of it is NaN).  One lane per head, through
        // shared memory, rather than all 16 in every thread (16 divisions of
        // code each): 16-head CTAs (batch-40 call 32.7 vs 33.3 us on GB300)
        // and the rolled store of 32-head decode; 32-head extend keeps them
        // in registers.
        constexpr bool kSharedInv = compact_epilogue<G, E>() || G == 16;
        float inv[kSharedInv ? 1 : 16];
        float* invs = reinterpret_cast<float*>(w.base + kOffInv) + w.h0;
        if constexpr (kSharedInv) {
            if (w.wq == 0 && w.lane < 16) {
                const int h = w.h0 + w.lane;
                const float L = lsum[h] + lsum[G + h] + lsum[2 * G + h] + lsum[3 * G + h];
                invs[w.lane] = (L > 0.f ? p.k_scale / L : 0.f) + (coef[h] - coef[h]);
            }
        } else {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
                const int h = w.h0 + t;
                const float L = lsum[h] + lsum[G + h] + lsum[2 * G + h] + lsum[3 * G + h];
                inv[t] = (L > 0.f ? p.k_scale / L : 0.f) + (coef[h] - coef[h]);
            }
        }
        // denominators for the lse: 16-head CTAs one per lane (head hb + (lane
        // & 7), stored by lanes 0-7 and 16-23 of the first warp), the others
        // all kHL of the lane's heads (stored by lanes 0 and 16)
        constexpr int kLse = G == 16 ? 1 : kHL;
        float Lmine[kLse];
#pragma unroll
        for (int j = 0; j < kLse; ++j) {
            const int h = w.hb + (kLse == 1 ? (w.lane & 7) : j);
            Lmine[j] = lsum[h] + lsum[G + h] + lsum[2 * G + h] + lsum[3 * G + h] + (coef[h] - coef[h]);
        }
        wg_bar(w.wg);                               // lsum is reused by the next segment; invs is written
        // output rows row0 .. row0 + nrows - 1; a partial slot holds
        // p.part_rows rows, this CTA's from prow0
        int64_t row0;
        int nrows, prow0;
        if constexpr (E) {
            row0 = p.blocks[4 * sg.b + 1];
            nrows = p.blocks[4 * sg.b + 2];
            prow0 = 0;
        } else {
            row0 = int64_t(sg.b) * p.heads + head0;
            nrows = p.heads - head0 < G ? p.heads - head0 : G;
            prow0 = head0;
        }
        // o and l are both in units of p * kPScale; lse = m + log2(sum p)
        const float lse_off = -kTau;                 // kPScale = 2^kTau
        if constexpr (G == 16) {
            // one lane per head, so that the code holds one log2f, not kHL: the
            // batch-40 call 30.4-31.1 vs 32.6 us on GB300 (two boxes; in 32-head
            // CTAs the same change measured slower: 128-head call 2.27 vs 2.07 ms);
            // stored before the wait for the segment's last PV, which it overlaps
            if (w.wq == 0 && (w.lane & 15) < kHL) {
                const int j = w.lane & 7;
                float mj = m[0];
#pragma unroll
                for (int jj = 1; jj < kHL; ++jj)
                    if (jj == j) mj = m[jj];
                float* dst = sg.part < 0 ? p.lse + row0 : p.part_lse + int64_t(sg.part) * p.part_rows + prow0;
                if (w.hb + j < nrows) {
                    const float v = (mj + log2f(Lmine[0]) + lse_off) * kLn2;
                    if (sg.part < 0) dst[w.hb + j] = v;
                    else st_f32_hint(dst + w.hb + j, v, l2_policy(true));
                }
            }
        }
        if constexpr (G != 16 && !E) {
            // 32-head decode: lanes 0 and 16 store heads hb .. hb + kHL - 1, also
            // before the wait (128-head call 2.05 vs 2.07 ms on GB300; one lane
            // per head measured 2.34).  32-head extend stores after the O: before
            // the wait it took 689 vs 652 us for the 256-token extend.
            if (w.wq == 0 && (w.lane & 15) == 0) {
                float* dst = sg.part < 0 ? p.lse + row0 : p.part_lse + int64_t(sg.part) * p.part_rows + prow0;
#pragma unroll
                for (int j = 0; j < kHL; ++j)
                    if (w.hb + j < nrows) {
                        const float v = (m[j] + log2f(Lmine[j]) + lse_off) * kLn2;
                        if (sg.part < 0) dst[w.hb + j] = v;
                        else st_f32_hint(dst + w.hb + j, v, l2_policy(true));
                    }
            }
        }
        const int jl = i - 1;                       // the segment's last tile
        bwait<G>(&w.bars[PV_DONE + (jl & 1)], (static_cast<uint32_t>(jl) >> 1) & 1, w.abort, w.flags);
        fence_after_sync();
        if constexpr (compact_epilogue<G, E>()) {
            // 128-channel block mb, heads h0 + 4 (st & 3) .. + 3 per step
            const int nh = nrows - w.h0 < 16 ? nrows - w.h0 : 16;   // this warpgroup's rows
#pragma unroll 1
            for (int st = 0; st < 16; ++st) {
                const int mb = st >> 2, t0 = 4 * (st & 3);
                if (t0 >= nh) continue;
                uint32_t r1[4], r2[4];
                tmem_ld4(w.tmem_lane + ocol + S::kN * mb + w.h0 + t0, r1);
                tmem_ld4(w.tmem_lane + ocol + S::kN * mb + G + w.h0 + t0, r2);
                tmem_wait_ld();
                const int ch = mb * 128 + w.row;
                const int64_t r0 = sg.part < 0 ? row0 : int64_t(sg.part) * p.part_rows + prow0;
                const int64_t off = (r0 + w.h0 + t0) * kDCkv + ch;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (t0 + u >= nh) break;
                    const float o = fmaf(__uint_as_float(r2[u]), 1.f / kP2Scale, __uint_as_float(r1[u])) *
                                    invs[t0 + u];
                    if (sg.part < 0) p.out[off + u * kDCkv] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
                    else st_f32_hint(p.part_o + off + u * kDCkv, o, l2_policy(true));
                }
            }
        } else if constexpr (G == 16) {
            // the next block's TMEM loads go out before this block's stores,
            // so that the stores cover their latency
            uint32_t r[2][16];
            tmem_ld16(w.tmem_lane + ocol + w.h0, r[0]);
            tmem_ld16(w.tmem_lane + ocol + G + w.h0, r[1]);
            tmem_wait_ld();
#pragma unroll 1
            for (int mb = 0; mb < 4; ++mb) {
                float o[16];                        // heads h0 .. h0 + 15
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    o[t] = fmaf(__uint_as_float(r[1][t]), 1.f / kP2Scale, __uint_as_float(r[0][t]));
                if (mb + 1 < 4) {
                    tmem_ld16(w.tmem_lane + ocol + S::kN * (mb + 1) + w.h0, r[0]);
                    tmem_ld16(w.tmem_lane + ocol + S::kN * (mb + 1) + G + w.h0, r[1]);
                }
                const int ch = mb * 128 + w.row;
                if (sg.part < 0) {
                    uint16_t* out = p.out + (int64_t(row0) + w.h0) * kDCkv + ch;
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        if (w.h0 + t >= nrows) break;
                        out[t * kDCkv] = __bfloat16_as_ushort(__float2bfloat16_rn(o[t] * invs[t]));
                    }
                } else {
                    float* po = p.part_o + (int64_t(sg.part) * p.part_rows + prow0 + w.h0) * kDCkv + ch;
                    const uint64_t keep = l2_policy(true);
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        if (w.h0 + t >= nrows) break;
                        st_f32_hint(po + t * kDCkv, o[t] * invs[t], keep);
                    }
                }
                if (mb + 1 < 4) tmem_wait_ld();
            }
        } else {
#pragma unroll 1
        for (int mb = 0; mb < 4; ++mb) {
            float o[16];                            // heads h0 .. h0 + 15
            {
                uint32_t r[2][16];
                tmem_ld16(w.tmem_lane + ocol + S::kN * mb + w.h0, r[0]);
                tmem_ld16(w.tmem_lane + ocol + S::kN * mb + G + w.h0, r[1]);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    o[t] = fmaf(__uint_as_float(r[1][t]), 1.f / kP2Scale, __uint_as_float(r[0][t]));
            }
            const int ch = mb * 128 + w.row;
            if (sg.part < 0) {
                uint16_t* out = p.out + (int64_t(row0) + w.h0) * kDCkv + ch;
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    if (w.h0 + t >= nrows) break;
                    out[t * kDCkv] = __bfloat16_as_ushort(__float2bfloat16_rn(o[t] * (kSharedInv ? invs[t] : inv[t])));
                }
            } else {
                float* po = p.part_o + (int64_t(sg.part) * p.part_rows + prow0 + w.h0) * kDCkv + ch;
                const uint64_t keep = l2_policy(true);
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    if (w.h0 + t >= nrows) break;
                    st_f32_hint(po + t * kDCkv, o[t] * (kSharedInv ? invs[t] : inv[t]), keep);
                }
            }
        }
        }
        fence_before_sync();
        mbar_arrive(&w.bars[O_FREE + (k % S::kOBufs)]);   // a later segment may overwrite O
        mbar_arrive(&w.bars[Q_FREE + qs]);
        if constexpr (G != 16 && E) {
            if (w.wq == 0 && (w.lane & 15) == 0) {    // lanes 0 and 16: heads hb .. hb + kHL - 1
                float* dst = sg.part < 0 ? p.lse + row0 : p.part_lse + int64_t(sg.part) * p.part_rows + prow0;
#pragma unroll
                for (int j = 0; j < kHL; ++j)
                    if (w.hb + j < nrows) {
                        const float v = (m[j] + log2f(Lmine[j]) + lse_off) * kLn2;
                        if (sg.part < 0) dst[w.hb + j] = v;
                        else st_f32_hint(dst + w.hb + j, v, l2_policy(true));
                    }
            }
        }
        ++k;
    }
}

// 152 registers at G = 16 (no spills): with 3 warps per SM sub-partition
// that leaves room for one warp of the q split kernel beside the CTA, so the
// programmatic launch places decode CTAs while the split still runs (at 160
// registers they waited for the split to drain; measured on GB300).  At
// G = 32 the CTA runs 512 threads (two softmax warpgroups) at 128 registers.
template <int G, bool E>
__global__ void __maxnreg__(G == 16 ? 152 : 128)
    mla_decode_tc_kernel(const DecodeParams p, const __grid_constant__ TcRanges ranges) {
    using S = Shape<G>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + kOffMisc);
    volatile int* abort = reinterpret_cast<volatile int*>(base + kOffMisc + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool ranged = static_cast<int>(blockIdx.x) < ranges.n;
    const int seg_lo = ranged ? ranges.seg[blockIdx.x] : p.cta_ptr[blockIdx.x];
    const int seg_hi = ranged ? ranges.seg[blockIdx.x + 1] : p.cta_ptr[blockIdx.x + 1];
    // the segment table: one thread per segment, visible after the barrier below
    constexpr int kTab = seg_tab_entries<G, E>();
    SegEntry* segtab = reinterpret_cast<SegEntry*>(base + kOffSegTab);
    if (tid < kTab && seg_lo + tid < seg_hi)
        segtab[tid] = SegEntry{load_seg<E>(p, seg_lo + tid), p.seg_pages[seg_lo + tid], 0};
    const SegView<E, kTab> sv{segtab, seg_lo, seg_hi};
    // the scheduler requests its first page entries while the CTA sets up
    TileCursor<E, kTab> cur;
    if (warp == S::kWarpSched) cur.init(p, seg_lo, seg_hi, ranged ? &ranges.first[blockIdx.x] : nullptr, lane);

    if (tid == 0) {
        // KV_FULL: 32 cp.async arrivals from each fill warp; KV_EMPTY, S_FULL,
        // PV_DONE, Q_FULL: one commit or bulk-copy arrival; S_FREE, P_FULL,
        // O_FREE: every softmax thread; Q_FREE: those and the QK commit; DONE:
        // both MMA threads; SL_EMPTY: the fill warps and the softmax warps
        constexpr uint32_t kSm = 128 * S::kWgs;
        for (int b = 0; b < kStages; ++b) {
            mbar_init(&bars[KV_FULL + b], 32 * kFillWarps);
            mbar_init(&bars[KV_EMPTY + b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars[S_FULL + b], 1);
            mbar_init(&bars[S_FREE + b], kSm);
            mbar_init(&bars[P_FULL + b], kSm);
            mbar_init(&bars[PV_DONE + b], 1);
            mbar_init(&bars[O_FREE + b], kSm);
            mbar_init(&bars[Q_FULL + b], 1);
            mbar_init(&bars[Q_FREE + b], kSm + 1);
        }
        mbar_init(&bars[DONE], 2);
        for (int e = 0; e < ring_depth<G, E>(); ++e) {
            mbar_init(&bars[SL_FULL + e], 1);
            mbar_init(&bars[SL_EMPTY + e], kFillWarps + 4 * S::kWgs);
        }
        *abort = 0;
        mbar_fence_init();
    }
    if (warp == kWarpMma) tmem_alloc(tmem_slot, kTmemCols);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int head0 = blockIdx.y * G;             // heads head0 .. head0 + G - 1 of every request

    if (warp == S::kWarpSched) {
        scheduler<G, E, ring_depth<G, E>()>(p, base, bars, abort, cur, sv, lane);
    } else if (warp < kFillWarps) {
        fill_warp<G, E, ring_depth<G, E>()>(p, base, bars, abort, sv, warp, lane);
    } else if (warp == kWarpMma || warp == S::kWarpPv) {
        if (warp_issue<G>() || lane == 0) {
            MmaCtx c;
            c.sbase = smem_u32(base);
            c.tmem = tmem;
            c.idesc_qk = idesc_e4m3_f32(kTT, S::kNq, false, false);
            c.idesc_pv = idesc_e4m3_f32(128, S::kN, true, true);   // M = 128 channels of a block
            c.bars = bars;
            c.abort = abort;
            c.flags = p.flags;
            if (warp == kWarpMma) qk_issuer<G, E>(p, c, sv);
            else pv_issuer<G, E>(p, c, sv);
        }
        if constexpr (!warp_issue<G>()) __syncwarp();
    } else if (warp == kWarpQ) {
        q_fetch<G, E>(p, base, bars, abort, sv, lane);
    } else {                                      // warps S::kWarpWg ..: softmax warpgroups
        WgCtx w;
        w.base = base;
        w.bars = bars;
        const int quad = warp & 3;                // a warp reaches TMEM lanes 32 (warp % 4) .. + 31
        w.tmem_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        w.abort = abort;
        w.flags = p.flags;
        w.row = quad * 32 + lane;
        w.srow = quad * 16 + (lane & 15);
        w.wg = G == 16 ? 0 : (warp - S::kWarpWg) >> 2;
        w.wq = (warp - S::kWarpWg) & 3;
        w.h0 = 16 * w.wg;
        w.hb = w.h0 + (lane >> 4) * 8;
        w.lane = lane;
        softmax_wg<G, E>(p, w, sv, head0);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
    // this CTA's work is done: the merge kernel may be launched once every
    // CTA got here
    if (tid == 0) griddep_launch_dependents();
}

std::mutex g_mu;
std::vector<char> g_attr;     // per device: bit (G / 16 - 1) + 2 E: max dynamic smem set

template <int G, bool E>
cudaError_t launch_g(const DecodeParams& p, const TcRanges& ranges, int grid, cudaStream_t stream,
                     int dev) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if ((int)g_attr.size() <= dev) g_attr.resize(dev + 1, 0);
        const char bit = static_cast<char>(1 << ((G / 16 - 1) + 2 * E));
        if (!(g_attr[dev] & bit)) {
            const cudaError_t e = cudaFuncSetAttribute(mla_decode_tc_kernel<G, E>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
            if (e != cudaSuccess) return e;
            // the split uses no shared memory; an SM configured for it with a
            // small carveout could not take a decode CTA until it drained
            const cudaError_t e2 = cudaFuncSetAttribute(mla_q_split_kernel<G>,
                                                        cudaFuncAttributePreferredSharedMemoryCarveout,
                                                        cudaSharedmemCarveoutMaxShared);
            if (e2 != cudaSuccess) return e2;
            g_attr[dev] |= bit;
        }
    }
    const int64_t images = E ? p.n_blocks : int64_t(p.batch) * p.head_groups;
    const int split_blocks = static_cast<int>((images * G * 32 + kSplitThreads - 1) / kSplitThreads);
    mla_q_split_kernel<G><<<split_blocks, kSplitThreads, 0, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the decode kernel starts while the split runs: only its q warp waits
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, p.head_groups);         // token ranges x head groups
    cfg.blockDim = dim3(Shape<G>::kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mla_decode_tc_kernel<G, E>, p, ranges);
}

}  // namespace

cudaError_t set_decode_wait_limit(uint64_t limit_ns) {
    const uint64_t v = limit_ns ? limit_ns : kDefaultWaitLimitNs;
    const cudaError_t e = cudaMemcpyToSymbol(g_wait_limit_ns, &v, sizeof(v));
    return e != cudaSuccess ? e : cudaMemcpyToSymbol(c_wait_limit_ns, &v, sizeof(v));
}

cudaError_t launch_decode_tc(const DecodeParams& p, const TcRanges& ranges, int grid,
                             cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    // slots are held as int32 in the kernel's shared slot lists
    if (p.num_slots >= INT32_MAX) return cudaErrorInvalidValue;
    const bool ext = p.blocks != nullptr;
    if (p.group_heads == 32) return ext ? launch_g<32, true>(p, ranges, grid, stream, dev) : launch_g<32, false>(p, ranges, grid, stream, dev);
    if (p.group_heads == 16) return ext ? launch_g<16, true>(p, ranges, grid, stream, dev) : launch_g<16, false>(p, ranges, grid, stream, dev);
    return cudaErrorInvalidValue;
}

}  // namespace mla
