// Host planner shared by plan.cu (construction) and decode.cu (launch).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "../../include/mla_decode.h"
#include "decode_params.h"

namespace mla {

// Tokens per KV tile of the mma.sync decode kernel, of the tcgen05 decode
// kernel, and heads per CTA.
constexpr int kTileTokens = 64;
constexpr int kTcTileTokens = 64;
// tcgen05 kernel: the schedule balances tiles + this many tiles per segment
// (its q fetch, pipeline refill and epilogue) across CTAs.  Measured on
// GB300: 2 for decode (the batch-40 call 34.3 us against 35.2-35.5 at 4 or
// 5), 4 for extend (4-token extend 65.3 vs 66.5 us).
constexpr int kTcSegmentCost = 2;
constexpr int kTcExtendSegmentCost = 4;
constexpr int kHeadsPerCta = 16;
// tcgen05 path: per request and group of 16 heads, [q1;q2;q3] as the
// shared-memory image the MMA reads (3 x 16 rows x 576 E4M3, swizzled)
// followed by 2 x 16 fp32 score multipliers and 16 int32 causal limits
// (extend: a row sees the tokens before its limit)
constexpr int kTcQImageBytes = 3 * kHeadsPerCta * 576 + kHeadsPerCta * 12;

// Which decode kernel a plan launches.
enum class DecodeKernel : int32_t {
    kMma = 0,   // mma.sync, E4M3 widened to f16 in smem; also the BF16-pool kernel
    kTc = 1,    // tcgen05 kind::f8f6f4 on the E4M3 bytes in place (FP8, H <= 16)
};

// The split-KV schedule.  The concatenation of all requests' tiles is cut
// into `num_ctas` contiguous, equal-sized (+-1 tile) ranges; each range is a
// CTA (per head group), and each piece of a range that lies in one request
// is a segment.  A request covered by one segment is written directly; the
// segments of a request covered by several write fp32 partials (normalised
// o and lse) that the merge kernel combines.
struct Schedule {
    int32_t batch = 0, heads = 0, page_size = 0;
    mla_kv_dtype_t kv_dtype = MLA_KV_FP8_E4M3;
    DecodeKernel kernel = DecodeKernel::kMma;
    int32_t tile_tokens = kTileTokens;
    int32_t head_groups = 0;         // CTAs per token range (grid.y)
    int32_t group_heads = 16;        // heads per CTA: 16, or 32 on the tcgen05 path when H % 32 == 0
    int32_t num_ctas = 0;            // token ranges; grid = num_ctas * head_groups
    std::vector<int32_t> cta_ptr;    // [num_ctas + 1] -> segment index
    std::vector<int32_t> segs;       // 4 per segment: request (extend: query block), t0, t1,
                                     // partial (-1 = final)
    std::vector<int32_t> merge;      // 4 per entry: first output row, first partial,
                                     // n partials, rows
    std::vector<int32_t> seg_pages;  // per segment: its request's first page-table entry
                                     // (kv_indptr[request]), so the kernel need not look it up
    int32_t part_rows = 0;           // rows per partial slot: H (decode), group_heads (extend)
    int32_t max_merge_parts = 0;     // the most partials one merge entry folds
    int32_t n_partials = 0;
    // extend: the query rows (new token x head, row = token * H + head) of
    // each request cut into blocks of group_heads rows; 4 ints per block:
    // request, first row, rows, causal base (row r sees the tokens before
    // base + r / H)
    bool extend = false;
    int32_t n_q = 0;                 // extend: query tokens (rows / H)
    std::vector<int32_t> blocks;
    int64_t n_tokens = 0;
    size_t partial_lse_offset = 0;   // bytes into the workspace
    size_t qimg_offset = 0;          // tcgen05 path: q images, batch x kTcQImageBytes
    size_t workspace_bytes = 0;

    int32_t n_segs() const { return static_cast<int32_t>(segs.size() / 4); }
    int32_t n_merge() const { return static_cast<int32_t>(merge.size() / 4); }
    void count_merge_parts() {
        max_merge_parts = 0;
        for (size_t e = 0; e + 3 < merge.size(); e += 4)
            max_merge_parts = merge[e + 2] > max_merge_parts ? merge[e + 2] : max_merge_parts;
    }
    int32_t n_blocks() const { return static_cast<int32_t>(blocks.size() / 4); }
};

mla_status_t validate_plan_inputs(const int32_t* kv_indptr, const int32_t* seq_lens,
                                  int32_t batch, int32_t heads, int32_t page_size,
                                  mla_kv_dtype_t kv_dtype);

mla_status_t build_schedule(const int32_t* kv_indptr, const int32_t* seq_lens, int32_t batch,
                            int32_t heads, int32_t page_size, mla_kv_dtype_t kv_dtype,
                            int32_t num_sms, Schedule& out);

mla_status_t validate_extend_inputs(const int32_t* qo_indptr, const int32_t* kv_indptr,
                                    const int32_t* seq_lens, int32_t batch, int32_t heads,
                                    int32_t page_size, mla_kv_dtype_t kv_dtype);

mla_status_t build_extend_schedule(const int32_t* qo_indptr, const int32_t* kv_indptr,
                                   const int32_t* seq_lens, int32_t batch, int32_t heads,
                                   int32_t page_size, mla_kv_dtype_t kv_dtype, int32_t num_sms,
                                   Schedule& out);

}  // namespace mla

struct mla_plan {
    mla::Schedule sched;
    int device = -1;
    int32_t* dev_meta = nullptr;      // merge | segs | blocks | cta_ptr | seg_pages (int32)
    size_t dev_meta_cap = 0;          // elements
    int32_t* pinned = nullptr;        // staging for the upload
    size_t pinned_cap = 0;
    cudaEvent_t upload_done = nullptr;
    size_t off_cta = 0, off_segs = 0, off_merge = 0, off_blocks = 0, off_seg_pages = 0;   // in dev_meta
    mla::TcRanges ranges;             // tcgen05 path: the token ranges, passed with each launch
};
