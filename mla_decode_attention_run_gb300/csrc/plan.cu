// mla_decode_plan / mla_decode_schedule: the plan() half of the plan/run
// split ("The KV Cache Cast Bottleneck", section "The Message": plan() is
// told the query and KV data types; "The Gather-Then-Cast Pivot", section
// "The Subject Message": plan() fixes which pool slots run() reads).
//
// The schedule balances work by tokens, not by requests: with contexts drawn
// from [1024, 8192] a per-request split leaves SMs idle, so the tile list of
// all requests is cut into equal contiguous ranges (one per CTA).
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>

#include "common.cuh"
#include "plan.h"

namespace mla {
namespace {

bool heads_supported(int32_t h) { return (h >= 1 && h <= 16) || (h > 16 && h <= 128 && h % 16 == 0); }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Resident decode CTAs per SM (both kernels' shared-memory budgets allow one).
int ctas_per_sm(DecodeKernel) { return 1; }

// The tcgen05 kernel covers FP8 pools (16 heads per CTA, more heads as more
// CTAs); the mma.sync kernel BF16 pools.
DecodeKernel pick_kernel(mla_kv_dtype_t dtype, int32_t) {
    return dtype == MLA_KV_FP8_E4M3 ? DecodeKernel::kTc : DecodeKernel::kMma;
}

// A CTA gets at least this many tiles when there is enough work (every
// split of a request adds a partial to merge).  Two for the tcgen05 kernel:
// a single 4,096-token request then runs on 33 CTAs (12.5 us per call on
// GB300) rather than 22 at three (13.1) or 17 at four (13.5).
int64_t min_tiles_per_cta(DecodeKernel) { return 2; }

// tcgen05 schedule: requests' tiles in order, cut into CTA ranges so that the
// largest CTA cost (tiles + seg_cost per segment) is as small as
// possible: binary search on the cost cap, greedy fill under it.
int64_t fill_under_cap(const int32_t* seq, int32_t B, int64_t tile, int64_t seg_cost, int64_t cap,
                       int64_t max_ctas, Schedule* out, std::vector<int32_t>* segs_per_req) {
    int64_t c = 0, cost = 0;
    bool any = false;
    if (out) out->cta_ptr.assign(1, 0);
    for (int32_t b = 0; b < B; ++b) {
        int64_t done = 0;
        const int64_t tiles = (seq[b] + tile - 1) / tile;
        while (done < tiles) {
            const int64_t room = cap - cost - seg_cost;
            if (room < 1) {
                if (cost == 0) return INT64_MAX;            // cap below one tile + segment
                if (++c >= max_ctas) return INT64_MAX;
                cost = 0;
                if (out) out->cta_ptr.push_back(static_cast<int32_t>(out->segs.size() / 4));
                continue;
            }
            const int64_t k = tiles - done < room ? tiles - done : room;
            if (out) {
                int64_t t1 = (done + k) * tile;
                if (t1 > seq[b]) t1 = seq[b];
                out->segs.insert(out->segs.end(), {b, static_cast<int32_t>(done * tile),
                                                   static_cast<int32_t>(t1), -1});
                ++(*segs_per_req)[b];
            }
            cost += seg_cost + k;
            done += k;
            any = true;
        }
    }
    return any ? c + 1 : 0;
}

// The greedy fill at the smallest cap can leave CTAs unused (at a larger
// segment cost it packs the ranges tighter).  More ranges never raise a
// range's cost, so the ranges of highest cost are split at their middle tile
// (a segment cut there becomes two segments of its request) until every CTA
// has one: the largest cost stays the same or drops, and no SM idles.
void split_costliest(Schedule& s, int64_t tile, int64_t seg_cost, int64_t max_ctas,
                     std::vector<int32_t>& segs_per_req) {
    std::vector<std::vector<int32_t>> ranges(s.num_ctas);
    for (int32_t c = 0; c < s.num_ctas; ++c)
        ranges[c].assign(s.segs.begin() + 4 * s.cta_ptr[c], s.segs.begin() + 4 * s.cta_ptr[c + 1]);
    auto tiles_of = [&](const std::vector<int32_t>& r) {
        int64_t t = 0;
        for (size_t i = 0; i < r.size(); i += 4) t += (r[i + 2] - r[i + 1] + tile - 1) / tile;
        return t;
    };
    auto cost_of = [&](const std::vector<int32_t>& r) {
        return tiles_of(r) + seg_cost * static_cast<int64_t>(r.size() / 4);
    };
    while (static_cast<int64_t>(ranges.size()) < max_ctas) {
        size_t top = 0;
        for (size_t c = 1; c < ranges.size(); ++c)
            if (cost_of(ranges[c]) > cost_of(ranges[top])) top = c;
        const std::vector<int32_t> r = ranges[top];
        const int64_t half = tiles_of(r) / 2;
        if (half < 1) break;
        std::vector<int32_t> left, right;
        int64_t acc = 0;
        for (size_t i = 0; i < r.size(); i += 4) {
            const int32_t b = r[i], t0 = r[i + 1], t1 = r[i + 2];
            const int64_t n = (t1 - t0 + tile - 1) / tile;
            if (acc + n <= half) {
                left.insert(left.end(), {b, t0, t1, -1});
            } else if (acc >= half) {
                right.insert(right.end(), {b, t0, t1, -1});
            } else {                                   // cut this segment on a tile boundary
                const int32_t cut = static_cast<int32_t>(t0 + (half - acc) * tile);
                left.insert(left.end(), {b, t0, cut, -1});
                right.insert(right.end(), {b, cut, t1, -1});
                ++segs_per_req[b];
            }
            acc += n;
        }
        ranges[top] = left;
        ranges.insert(ranges.begin() + static_cast<int64_t>(top) + 1, right);
    }
    s.segs.clear();
    s.cta_ptr.assign(1, 0);
    for (const auto& r : ranges) {
        s.segs.insert(s.segs.end(), r.begin(), r.end());
        s.cta_ptr.push_back(static_cast<int32_t>(s.segs.size() / 4));
    }
    s.num_ctas = static_cast<int32_t>(ranges.size());
}

void build_cost_balanced(const int32_t* seq, int32_t B, int64_t tile, int64_t seg_cost, int64_t max_ctas,
                         Schedule& s, std::vector<int32_t>& segs_per_req) {
    int64_t n_tiles = 0, n_req = 0;
    for (int32_t b = 0; b < B; ++b) {
        n_tiles += (seq[b] + tile - 1) / tile;
        n_req += seq[b] > 0;
    }
    s.segs.clear();
    if (n_tiles == 0 || max_ctas < 1) {
        s.num_ctas = 0;
        s.cta_ptr.assign(1, 0);
        return;
    }
    int64_t lo = (n_tiles + seg_cost * n_req + max_ctas - 1) / max_ctas;
    if (lo < seg_cost + 1) lo = seg_cost + 1;
    // everything in one CTA: every request one segment (always feasible)
    int64_t hi = n_tiles + seg_cost * n_req;
    if (hi < lo) hi = lo;
    while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (fill_under_cap(seq, B, tile, seg_cost, mid, max_ctas, nullptr, nullptr) != INT64_MAX) hi = mid;
        else lo = mid + 1;
    }
    const int64_t used = fill_under_cap(seq, B, tile, seg_cost, lo, max_ctas, &s, &segs_per_req);
    if (used == INT64_MAX) {                                   // cannot happen with the bounds above
        s.segs.clear();
        s.num_ctas = 0;
        s.cta_ptr.assign(1, 0);
        std::fill(segs_per_req.begin(), segs_per_req.end(), 0);
        return;
    }
    s.num_ctas = static_cast<int32_t>(used);
    s.cta_ptr.resize(s.num_ctas + 1);
    s.cta_ptr[s.num_ctas] = static_cast<int32_t>(s.segs.size() / 4);
    if (used < max_ctas) split_costliest(s, tile, seg_cost, max_ctas, segs_per_req);
}

// Workspace: partials (o, then lse) for part_rows rows each, then, on the
// tcgen05 path, one q image per (request, head group) or query block.
void size_workspace(Schedule& s, int64_t images) {
    const size_t o_bytes = static_cast<size_t>(s.n_partials) * s.part_rows * kDCkv * sizeof(float);
    s.partial_lse_offset = align256(o_bytes);
    s.workspace_bytes =
        s.n_partials ? align256(s.partial_lse_offset + static_cast<size_t>(s.n_partials) * s.part_rows * 4)
                     : 0;
    if (s.kernel == DecodeKernel::kTc && s.num_ctas > 0) {
        s.qimg_offset = s.workspace_bytes;
        s.workspace_bytes =
            align256(s.qimg_offset + static_cast<size_t>(images) * (s.group_heads / 16) * kTcQImageBytes);
    }
}

}  // namespace

mla_status_t validate_plan_inputs(const int32_t* indptr, const int32_t* seq, int32_t B,
                                  int32_t H, int32_t ps, mla_kv_dtype_t dtype) {
    if (!indptr || !seq) return MLA_ERR_INVALID_ARG;
    if (B < 1 || B > (1 << 24) || ps < 1 || ps > (1 << 20)) return MLA_ERR_INVALID_ARG;
    if (dtype != MLA_KV_FP8_E4M3 && dtype != MLA_KV_BF16) return MLA_ERR_INVALID_ARG;
    if (!heads_supported(H)) return MLA_ERR_UNSUPPORTED;
    if (indptr[0] < 0) return MLA_ERR_INVALID_ARG;
    for (int32_t b = 0; b < B; ++b) {
        if (seq[b] < 0) return MLA_ERR_INVALID_ARG;
        const int64_t pages = static_cast<int64_t>(indptr[b + 1]) - indptr[b];
        if (pages != (static_cast<int64_t>(seq[b]) + ps - 1) / ps) return MLA_ERR_INVALID_ARG;
    }
    return MLA_OK;
}

mla_status_t build_schedule(const int32_t* indptr, const int32_t* seq, int32_t B, int32_t H,
                            int32_t ps, mla_kv_dtype_t dtype, int32_t num_sms, Schedule& s) {
    const mla_status_t st = validate_plan_inputs(indptr, seq, B, H, ps, dtype);
    if (st != MLA_OK) return st;
    if (num_sms < 1) return MLA_ERR_INVALID_ARG;
    const DecodeKernel kernel = pick_kernel(dtype, H);
    const int64_t tile = kernel == DecodeKernel::kTc ? kTcTileTokens : kTileTokens;
    int64_t n_tokens = 0, n_tiles = 0;
    for (int32_t b = 0; b < B; ++b) {
        n_tokens += seq[b];
        n_tiles += (seq[b] + tile - 1) / tile;
    }

    s = Schedule();
    s.batch = B;
    s.heads = H;
    s.page_size = ps;
    s.kv_dtype = dtype;
    s.kernel = kernel;
    s.tile_tokens = static_cast<int32_t>(tile);
    s.n_tokens = n_tokens;
    // the tcgen05 kernel takes 32 heads per CTA when it can: one read of a tile
    // then serves twice the heads
    s.group_heads = (kernel == DecodeKernel::kTc && H % 32 == 0) ? 32 : kHeadsPerCta;
    s.head_groups = (H + s.group_heads - 1) / s.group_heads;

    int64_t ctas = static_cast<int64_t>(num_sms) * ctas_per_sm(kernel) / s.head_groups;
    if (ctas < 1) ctas = 1;
    const int64_t by_work = (n_tiles + min_tiles_per_cta(kernel) - 1) / min_tiles_per_cta(kernel);
    if (ctas > by_work) ctas = by_work;
    s.num_ctas = static_cast<int32_t>(ctas);

    std::vector<int32_t> segs_per_req(B, 0);
    if (kernel == DecodeKernel::kTc) {
        build_cost_balanced(seq, B, tile, kTcSegmentCost, ctas, s, segs_per_req);
    } else {
        // request tile offsets in the concatenated tile list
        std::vector<int64_t> first_tile(B + 1, 0);
        for (int32_t b = 0; b < B; ++b)
            first_tile[b + 1] = first_tile[b] + (seq[b] + tile - 1) / tile;

        s.cta_ptr.assign(s.num_ctas + 1, 0);
        int32_t b = 0;
        for (int32_t c = 0; c < s.num_ctas; ++c) {
            s.cta_ptr[c] = static_cast<int32_t>(s.segs.size() / 4);
            const int64_t lo = n_tiles * c / s.num_ctas, hi = n_tiles * (c + 1) / s.num_ctas;
            int64_t pos = lo;
            while (pos < hi) {
                while (first_tile[b + 1] <= pos) ++b;       // skips empty requests too
                const int64_t end = hi < first_tile[b + 1] ? hi : first_tile[b + 1];
                const int64_t t0 = (pos - first_tile[b]) * tile;
                int64_t t1 = (end - first_tile[b]) * tile;
                if (t1 > seq[b]) t1 = seq[b];
                s.segs.insert(s.segs.end(), {b, static_cast<int32_t>(t0), static_cast<int32_t>(t1), -1});
                ++segs_per_req[b];
                pos = end;
            }
        }
        s.cta_ptr[s.num_ctas] = static_cast<int32_t>(s.segs.size() / 4);
    }

    // partial slots: consecutive per request, in launch order
    std::vector<int32_t> first_partial(B, -1);
    for (int32_t i = 0; i < s.n_segs(); ++i) {
        const int32_t r = s.segs[4 * i];
        if (segs_per_req[r] > 1) {
            if (first_partial[r] < 0) first_partial[r] = s.n_partials;
            s.segs[4 * i + 3] = s.n_partials++;
        }
    }
    for (int32_t r = 0; r < B; ++r) {
        if (segs_per_req[r] > 1) s.merge.insert(s.merge.end(), {r * H, first_partial[r], segs_per_req[r], H});
        else if (seq[r] == 0) s.merge.insert(s.merge.end(), {r * H, 0, 0, H});
    }
    s.part_rows = H;
    s.seg_pages.resize(s.n_segs());
    for (int32_t i = 0; i < s.n_segs(); ++i) s.seg_pages[i] = indptr[s.segs[4 * i]];
    s.count_merge_parts();
    size_workspace(s, static_cast<int64_t>(B) * s.head_groups);
    return MLA_OK;
}

mla_status_t validate_extend_inputs(const int32_t* qo, const int32_t* indptr, const int32_t* seq,
                                    int32_t B, int32_t H, int32_t ps, mla_kv_dtype_t dtype) {
    if (!qo) return MLA_ERR_INVALID_ARG;
    const mla_status_t st = validate_plan_inputs(indptr, seq, B, H, ps, dtype);
    if (st != MLA_OK) return st;
    // the extend kernel reads E4M3 pools only (the BF16-pool kernel is decode only)
    if (dtype != MLA_KV_FP8_E4M3) return MLA_ERR_UNSUPPORTED;
    if (qo[0] != 0) return MLA_ERR_INVALID_ARG;
    for (int32_t b = 0; b < B; ++b) {
        const int64_t n = static_cast<int64_t>(qo[b + 1]) - qo[b];
        if (n < 0 || n > seq[b]) return MLA_ERR_INVALID_ARG;
    }
    // rows (token x head) are int32 on the device
    if (static_cast<int64_t>(qo[B]) * H >= INT32_MAX) return MLA_ERR_UNSUPPORTED;
    return MLA_OK;
}

mla_status_t build_extend_schedule(const int32_t* qo, const int32_t* indptr, const int32_t* seq,
                                   int32_t B, int32_t H, int32_t ps, mla_kv_dtype_t dtype,
                                   int32_t num_sms, Schedule& s) {
    const mla_status_t st = validate_extend_inputs(qo, indptr, seq, B, H, ps, dtype);
    if (st != MLA_OK) return st;
    if (num_sms < 1) return MLA_ERR_INVALID_ARG;
    s = Schedule();
    s.batch = B;
    s.heads = H;
    s.page_size = ps;
    s.kv_dtype = dtype;
    s.kernel = DecodeKernel::kTc;
    s.tile_tokens = kTcTileTokens;
    s.extend = true;
    s.n_q = qo[B];
    s.head_groups = 1;

    // Query rows of request b: row = token * H + head over its new tokens.
    // Blocks of 32 rows when that needs clearly fewer blocks than 16 (an
    // N = 64 MMA costs what N = 32 does; the softmax pays per row)
    int64_t blocks16 = 0, blocks32 = 0;
    for (int32_t b = 0; b < B; ++b) {
        const int64_t rows = (static_cast<int64_t>(qo[b + 1]) - qo[b]) * H;
        blocks16 += (rows + 15) / 16;
        blocks32 += (rows + 31) / 32;
    }
    s.group_heads = 4 * blocks32 <= 3 * blocks16 ? 32 : kHeadsPerCta;
    const int64_t G = s.group_heads;

    // each block is scheduled like a request whose context ends at the
    // causal limit of its last row
    std::vector<int32_t> len;
    for (int32_t b = 0; b < B; ++b) {
        const int64_t r_lo = static_cast<int64_t>(qo[b]) * H, r_hi = static_cast<int64_t>(qo[b + 1]) * H;
        // row r (token r / H) sees the tokens before base + r / H: the last
        // new token sees the whole context
        const int64_t base = static_cast<int64_t>(seq[b]) + 1 - qo[b + 1];
        for (int64_t r0 = r_lo; r0 < r_hi; r0 += G) {
            const int64_t rows = r_hi - r0 < G ? r_hi - r0 : G;
            s.blocks.insert(s.blocks.end(), {b, static_cast<int32_t>(r0), static_cast<int32_t>(rows),
                                             static_cast<int32_t>(base)});
            len.push_back(static_cast<int32_t>(base + (r0 + rows - 1) / H));
        }
    }
    const int32_t nb = s.n_blocks();
    int64_t n_tiles = 0;
    for (int32_t v = 0; v < nb; ++v) {
        s.n_tokens += len[v];
        n_tiles += (len[v] + kTcTileTokens - 1) / kTcTileTokens;
    }
    int64_t ctas = num_sms;
    const int64_t by_work = (n_tiles + min_tiles_per_cta(DecodeKernel::kTc) - 1) /
                            min_tiles_per_cta(DecodeKernel::kTc);
    if (ctas > by_work) ctas = by_work;
    // Blocks are scheduled by their place within their request first: every
    // request's first block, then every second block, and so on.  A
    // request's blocks read the same context; ordered this way they sit at
    // about the same relative place in different parts of the CTA list and
    // run at about the same time, so the later reads of each row come from L2
    // (in request order they are neighbours in one CTA range, read one after
    // the other, far apart in time).
    std::vector<int32_t> order(nb), place(nb);
    for (int32_t v = 0; v < nb; ++v) {
        order[v] = v;
        place[v] = v > 0 && s.blocks[4 * v] == s.blocks[4 * (v - 1)] ? place[v - 1] + 1 : 0;
    }
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return place[a] < place[b]; });
    std::vector<int32_t> len_o(nb), segs_o(nb, 0);
    for (int32_t j = 0; j < nb; ++j) len_o[j] = len[order[j]];
    build_cost_balanced(len_o.data(), nb, kTcTileTokens, kTcExtendSegmentCost, ctas, s, segs_o);
    for (int32_t i = 0; i < s.n_segs(); ++i) s.segs[4 * i] = order[s.segs[4 * i]];
    std::vector<int32_t> segs_per_block(nb, 0);
    for (int32_t j = 0; j < nb; ++j) segs_per_block[order[j]] = segs_o[j];

    std::vector<int32_t> first_partial(nb, -1);
    for (int32_t i = 0; i < s.n_segs(); ++i) {
        const int32_t v = s.segs[4 * i];
        if (segs_per_block[v] > 1) {
            if (first_partial[v] < 0) first_partial[v] = s.n_partials;
            s.segs[4 * i + 3] = s.n_partials++;
        }
    }
    for (int32_t v = 0; v < nb; ++v)
        if (segs_per_block[v] > 1)
            s.merge.insert(s.merge.end(), {s.blocks[4 * v + 1], first_partial[v], segs_per_block[v],
                                           s.blocks[4 * v + 2]});
    s.part_rows = static_cast<int32_t>(G);
    s.seg_pages.resize(s.n_segs());
    for (int32_t i = 0; i < s.n_segs(); ++i) s.seg_pages[i] = indptr[s.blocks[4 * s.segs[4 * i]]];
    s.count_merge_parts();
    size_workspace(s, nb);
    return MLA_OK;
}

}  // namespace mla

using mla::Schedule;

extern "C" mla_status_t mla_decode_schedule(const int32_t* kv_indptr_host,
                                            const int32_t* seq_lens_host, int32_t batch,
                                            int32_t num_heads, int32_t page_size,
                                            mla_kv_dtype_t kv_dtype, int32_t num_sms,
                                            int32_t* segments_out, int32_t capacity,
                                            int32_t* num_segments, int32_t* num_partials,
                                            int32_t* num_ctas, int32_t* tile_tokens,
                                            int32_t* kernel, size_t* workspace_bytes) {
    Schedule s;
    const mla_status_t st = mla::build_schedule(kv_indptr_host, seq_lens_host, batch, num_heads,
                                                page_size, kv_dtype, num_sms, s);
    if (st != MLA_OK) return st;
    if (segments_out) {
        int32_t k = 0;
        for (int32_t c = 0; c < s.num_ctas; ++c) {
            for (int32_t i = s.cta_ptr[c]; i < s.cta_ptr[c + 1] && k < capacity; ++i, ++k) {
                int32_t* d = segments_out + 5 * k;
                d[0] = c;
                std::memcpy(d + 1, &s.segs[4 * i], 4 * sizeof(int32_t));
            }
        }
    }
    if (num_segments) *num_segments = s.n_segs();
    if (num_partials) *num_partials = s.n_partials;
    if (num_ctas) *num_ctas = s.num_ctas;
    if (tile_tokens) *tile_tokens = s.tile_tokens;
    if (kernel) *kernel = static_cast<int32_t>(s.kernel);
    if (workspace_bytes) *workspace_bytes = s.workspace_bytes;
    return MLA_OK;
}

extern "C" mla_status_t mla_extend_schedule(const int32_t* qo_indptr_host,
                                            const int32_t* kv_indptr_host,
                                            const int32_t* seq_lens_host, int32_t batch,
                                            int32_t num_heads, int32_t page_size,
                                            mla_kv_dtype_t kv_dtype, int32_t num_sms,
                                            int32_t* segments_out, int32_t seg_capacity,
                                            int32_t* blocks_out, int32_t block_capacity,
                                            int32_t* counts_out, size_t* workspace_bytes) {
    Schedule s;
    const mla_status_t st = mla::build_extend_schedule(qo_indptr_host, kv_indptr_host,
                                                       seq_lens_host, batch, num_heads, page_size,
                                                       kv_dtype, num_sms, s);
    if (st != MLA_OK) return st;
    if (segments_out) {
        int32_t k = 0;
        for (int32_t c = 0; c < s.num_ctas; ++c) {
            for (int32_t i = s.cta_ptr[c]; i < s.cta_ptr[c + 1] && k < seg_capacity; ++i, ++k) {
                int32_t* d = segments_out + 5 * k;
                d[0] = c;
                std::memcpy(d + 1, &s.segs[4 * i], 4 * sizeof(int32_t));
            }
        }
    }
    if (blocks_out) {
        const int32_t n = s.n_blocks() < block_capacity ? s.n_blocks() : block_capacity;
        if (n > 0) std::memcpy(blocks_out, s.blocks.data(), 4 * sizeof(int32_t) * n);
    }
    if (counts_out) {
        counts_out[0] = s.n_segs();
        counts_out[1] = s.n_partials;
        counts_out[2] = s.num_ctas;
        counts_out[3] = s.n_blocks();
        counts_out[4] = s.group_heads;
    }
    if (workspace_bytes) *workspace_bytes = s.workspace_bytes;
    return MLA_OK;
}

namespace {

void release_buffers(mla_plan* p) {
    if (p->dev_meta) cudaFree(p->dev_meta);
    if (p->pinned) cudaFreeHost(p->pinned);
    if (p->upload_done) cudaEventDestroy(p->upload_done);
    p->dev_meta = nullptr;
    p->pinned = nullptr;
    p->upload_done = nullptr;
    p->dev_meta_cap = p->pinned_cap = 0;
}

}  // namespace

namespace {

// Makes (or refills) the plan handle and uploads the schedule's device tables
// (CTA ranges, segments, merge entries, query blocks) with one async copy.
mla_status_t install(mla_plan_t* plan, Schedule&& s, size_t* workspace_bytes, void* stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    mla_plan* p = *plan;
    const bool fresh = (p == nullptr);
    if (fresh) {
        p = new (std::nothrow) mla_plan();
        if (!p) return MLA_ERR_CUDA;
    } else if (p->device != dev) {
        return MLA_ERR_INVALID_ARG;       // a plan belongs to one device
    }
    p->device = dev;
    const size_t need = static_cast<size_t>(s.num_ctas + 1) + s.segs.size() + s.merge.size() +
                        s.blocks.size() + s.seg_pages.size();
    cudaStream_t cs = static_cast<cudaStream_t>(stream);

    if (!p->upload_done &&
        cudaEventCreateWithFlags(&p->upload_done, cudaEventDisableTiming) != cudaSuccess) {
        if (fresh) { release_buffers(p); delete p; }
        return MLA_ERR_CUDA;
    }
    // the previous upload must be finished before the staging buffer is reused
    if (cudaEventSynchronize(p->upload_done) != cudaSuccess) {
        if (fresh) { release_buffers(p); delete p; }
        return MLA_ERR_CUDA;
    }
    if (p->pinned_cap < need) {
        if (p->pinned) cudaFreeHost(p->pinned);
        p->pinned = nullptr;
        p->pinned_cap = 0;
        size_t cap = need < 1024 ? 1024 : need * 2;
        if (cudaHostAlloc(reinterpret_cast<void**>(&p->pinned), cap * sizeof(int32_t),
                          cudaHostAllocDefault) != cudaSuccess) {
            if (fresh) { release_buffers(p); delete p; }
            return MLA_ERR_CUDA;
        }
        p->pinned_cap = cap;
    }
    if (p->dev_meta_cap < need) {
        // growing: earlier runs may still read the old buffer; cudaFree waits
        // for the device before releasing it
        if (p->dev_meta) cudaFree(p->dev_meta);
        p->dev_meta = nullptr;
        p->dev_meta_cap = 0;
        size_t cap = need < 1024 ? 1024 : need * 2;
        if (cudaMalloc(reinterpret_cast<void**>(&p->dev_meta), cap * sizeof(int32_t)) !=
            cudaSuccess) {
            if (fresh) { release_buffers(p); delete p; }
            return MLA_ERR_CUDA;
        }
        p->dev_meta_cap = cap;
    }
    // the 4-int records first, so that each starts on 16 bytes (one vector
    // load per record on the device); cudaMalloc memory is 256-byte aligned
    p->off_merge = 0;
    p->off_segs = p->off_merge + s.merge.size();
    p->off_blocks = p->off_segs + s.segs.size();
    p->off_cta = p->off_blocks + s.blocks.size();
    p->off_seg_pages = p->off_cta + s.num_ctas + 1;
    std::memcpy(p->pinned + p->off_cta, s.cta_ptr.data(), (s.num_ctas + 1) * sizeof(int32_t));
    if (!s.segs.empty())
        std::memcpy(p->pinned + p->off_segs, s.segs.data(), s.segs.size() * sizeof(int32_t));
    if (!s.merge.empty())
        std::memcpy(p->pinned + p->off_merge, s.merge.data(), s.merge.size() * sizeof(int32_t));
    if (!s.blocks.empty())
        std::memcpy(p->pinned + p->off_blocks, s.blocks.data(), s.blocks.size() * sizeof(int32_t));
    if (!s.seg_pages.empty())
        std::memcpy(p->pinned + p->off_seg_pages, s.seg_pages.data(), s.seg_pages.size() * sizeof(int32_t));
    if (cudaMemcpyAsync(p->dev_meta, p->pinned, need * sizeof(int32_t), cudaMemcpyHostToDevice,
                        cs) != cudaSuccess ||
        cudaEventRecord(p->upload_done, cs) != cudaSuccess) {
        if (fresh) { release_buffers(p); delete p; }
        return MLA_ERR_CUDA;
    }
    p->sched = std::move(s);
    // the tcgen05 kernel's token ranges as a launch parameter: each range's
    // segments and its first segment's t0, t1 and page-table offset
    {
        const Schedule& sc = p->sched;
        mla::TcRanges& r = p->ranges;
        r.n = sc.kernel == mla::DecodeKernel::kTc ? std::min(sc.num_ctas, mla::kMaxTcRanges) : 0;
        for (int32_t c = 0; c < r.n; ++c) {
            const int32_t lo = sc.cta_ptr[c], hi = sc.cta_ptr[c + 1];
            r.seg[c] = lo;
            r.seg[c + 1] = hi;
            r.first[c] = lo < hi ? make_int4(sc.segs[4 * lo + 1], sc.segs[4 * lo + 2], sc.seg_pages[lo], 0)
                                 : make_int4(0, 0, 0, 0);
        }
    }
    *workspace_bytes = p->sched.workspace_bytes;
    *plan = p;
    return MLA_OK;
}

}  // namespace

extern "C" mla_status_t mla_decode_plan(mla_plan_t* plan, const int32_t* kv_indptr_host,
                                        const int32_t* seq_lens_host, int32_t batch,
                                        int32_t num_heads, int32_t page_size,
                                        mla_kv_dtype_t kv_dtype, size_t* workspace_bytes,
                                        void* stream) {
    if (!plan || !workspace_bytes) return MLA_ERR_INVALID_ARG;
    mla_status_t st = mla::validate_plan_inputs(kv_indptr_host, seq_lens_host, batch, num_heads,
                                                page_size, kv_dtype);
    if (st != MLA_OK) return st;
    const int sms = mla::device_sm_count();
    if (sms <= 0) return MLA_ERR_CUDA;
    Schedule s;
    st = mla::build_schedule(kv_indptr_host, seq_lens_host, batch, num_heads, page_size,
                             kv_dtype, sms, s);
    if (st != MLA_OK) return st;
    return install(plan, std::move(s), workspace_bytes, stream);
}

extern "C" mla_status_t mla_extend_plan(mla_plan_t* plan, const int32_t* qo_indptr_host,
                                        const int32_t* kv_indptr_host,
                                        const int32_t* seq_lens_host, int32_t batch,
                                        int32_t num_heads, int32_t page_size,
                                        mla_kv_dtype_t kv_dtype, size_t* workspace_bytes,
                                        void* stream) {
    if (!plan || !workspace_bytes) return MLA_ERR_INVALID_ARG;
    mla_status_t st = mla::validate_extend_inputs(qo_indptr_host, kv_indptr_host, seq_lens_host,
                                                  batch, num_heads, page_size, kv_dtype);
    if (st != MLA_OK) return st;
    const int sms = mla::device_sm_count();
    if (sms <= 0) return MLA_ERR_CUDA;
    Schedule s;
    st = mla::build_extend_schedule(qo_indptr_host, kv_indptr_host, seq_lens_host, batch,
                                    num_heads, page_size, kv_dtype, sms, s);
    if (st != MLA_OK) return st;
    return install(plan, std::move(s), workspace_bytes, stream);
}

extern "C" mla_status_t mla_decode_plan_destroy(mla_plan_t plan) {
    if (!plan) return MLA_OK;
    if (plan->upload_done) cudaEventSynchronize(plan->upload_done);
    release_buffers(plan);
    delete plan;
    return MLA_OK;
}

extern "C" mla_status_t mla_decode_plan_info(mla_plan_t plan, int32_t* num_ctas,
                                             int32_t* num_segments, int32_t* num_partials,
                                             size_t* workspace_bytes) {
    if (!plan) return MLA_ERR_INVALID_ARG;
    if (num_ctas) *num_ctas = plan->sched.num_ctas;
    if (num_segments) *num_segments = plan->sched.n_segs();
    if (num_partials) *num_partials = plan->sched.n_partials;
    if (workspace_bytes) *workspace_bytes = plan->sched.workspace_bytes;
    return MLA_OK;
}
