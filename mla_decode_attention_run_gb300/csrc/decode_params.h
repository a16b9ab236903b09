// Launch parameters shared by the decode kernels (decode.cu, decode_tc.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

struct DecodeParams {
    const uint16_t* q;          // BF16 [B][H][576] with strides q_sb / q_sh (elements)
    int64_t q_sb, q_sh;
    const uint8_t* ckv;         // row `slot` at ckv + slot * ckv_stride
    int64_t ckv_stride;
    const uint8_t* kpe;
    int64_t kpe_stride;
    int64_t num_slots;
    const int32_t* indptr;
    const int32_t* indices;
    const int32_t* seq_lens;
    int32_t page_size, heads, head_groups;
    // t / page_size == (t * page_magic) >> page_shift for 0 <= t < 2^31
    // (set_page_divider)
    uint32_t page_magic;
    int32_t page_shift;
    float k_scale, softmax_scale;
    uint16_t* out;              // BF16 [B][H][512]
    float* lse;                 // [B][H], natural log
    float* part_o;              // split-KV partials: [partials][H][512] fp32 (normalised)
    float* part_lse;            // [partials][H]
    const int32_t* cta_ptr;     // plan: segments of CTA c are [cta_ptr[c], cta_ptr[c+1])
    const int32_t* segs;        // plan: 4 ints per segment: request, t0, t1, partial (-1 final)
    const int32_t* seg_pages;   // plan: per segment, kv_indptr of its request
    uint32_t* flags;            // library flag word
    uint8_t* qimg;              // tcgen05 path: per-request q images (workspace)
    int32_t batch;
    int32_t group_heads;        // tcgen05 path: heads per CTA (16 or 32); grid.y = head_groups
    int32_t part_rows;          // rows per partial slot (H; extend: group_heads)
    // extend (causal, several new tokens per request): q / out / lse rows are
    // token * H + head over all requests' new tokens, and the plan's segments
    // name query blocks, 4 ints each: request, first row, rows, causal base
    // (row r sees the tokens before base + r / H).  nullptr for decode.
    const int32_t* blocks;
    int32_t n_blocks;
};

// Division by the page size as a multiply and a shift, exact for every
// dividend 0 <= t < 2^31 (the round-up method of Granlund and Montgomery,
// "Division by Invariant Integers using Multiplication"): with 2^s >= d,
// m = floor(2^(31+s) / d) + 1 gives 2^(31+s) < m d <= 2^(31+s) + 2^s, so
// floor(t m / 2^(31+s)) = floor(t / d); m < 2^32 and t m < 2^63.
inline void set_page_divider(DecodeParams& p) {
    const uint64_t d = static_cast<uint64_t>(p.page_size > 0 ? p.page_size : 1);
    int s = 0;
    while ((uint64_t(1) << s) < d) ++s;
    p.page_magic = static_cast<uint32_t>((uint64_t(1) << (31 + s)) / d + 1);
    p.page_shift = 31 + s;
}

// The tcgen05 decode's token ranges (its CTAs, per head group), passed by
// value as a kernel parameter: a CTA then knows its segments and issues its
// first page-table loads at once instead of after two dependent global loads
// (range -> segment record -> page entries).  Ranges past kMaxTcRanges read
// the plan's device tables instead.
constexpr int kMaxTcRanges = 256;
struct TcRanges {
    int32_t n;                          // ranges described here
    int32_t seg[kMaxTcRanges + 1];      // range c: segments [seg[c], seg[c + 1])
    int4 first[kMaxTcRanges];           // range c's first segment: t0, t1, page-table offset, 0
};

// Launches the q split kernel and then, as its programmatic dependent, the
// tcgen05 FP8 decode kernel (decode_tc.cu) on `grid` token ranges x
// p.head_groups.
cudaError_t launch_decode_tc(const DecodeParams& p, const TcRanges& ranges, int grid,
                             cudaStream_t stream);

// Sets the time limit of the tcgen05 decode kernels' bounded waits on the
// current device (0: the default); synchronous.
cudaError_t set_decode_wait_limit(uint64_t limit_ns);

}  // namespace mla
