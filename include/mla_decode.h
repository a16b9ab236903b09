/*
 * mla_decode.h -- C ABI of libmla_decode.so: paged MLA decode attention that
 * reads an FP8 E4M3 KV cache directly, plus its two companion kernels
 * (quantize-on-store and active-slot gather-then-cast).  One GPU (sm_103a).
 *
 * Sources (web pages, by title and section):
 *  [P1] "When a Faster Kernel Doesn't Speed Up Serving: Profiling FP8 KV
 *       Cache on AMD Instinct MI308X": "Setup" (--kv-cache-dtype fp8_e4m3,
 *       a 16-head q_len-1 MLA decode kernel), "Step 3: Source Validation"
 *       (CastFromFP8 / CastToFP8: the FP8<->BF16 casts on the cache read and
 *       write paths).
 *  [P2] "The KV Cache Cast Bottleneck: A Surgical Fix for 69% Decode
 *       Overhead": "The Context" (cache rows [495552, 1, 576] of
 *       Float8_e4m3fn; 576 = kv_lora_rank 512 + qk_rope_head_dim 64),
 *       "The Message" (plan() takes separate query and KV data types; the
 *       attention kernel reads FP8 rows and computes in higher precision).
 *  [P3] "The Gather-Then-Cast Pivot": "The Subject Message" (run() reads
 *       page-indexed ckv/kpe buffers; kv_indices from plan() say which slots),
 *       "The Reasoning Process" (gather the active FP8 rows into a compact
 *       buffer, cast it, replan with sequential indices).
 *
 * Conventions for every entry point:
 *  - Pointers named *_host are host memory; every other data pointer is
 *    device memory owned by the caller.  The library owns only plan handles.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call that launches work is asynchronous on it.
 *  - Host-detectable errors (NULL pointers, bad sizes, misalignment, an
 *    inconsistent page table, a small workspace) return a status before any
 *    launch and leave every output untouched.
 *  - Device-detected problems (a slot or page index outside the pool) never
 *    trap: the offending row is skipped (store / gather: its destination is
 *    left unwritten; decode: the token is excluded from the softmax) and a
 *    bit is OR-ed into a device flag word that mla_get_last_error() reads.
 *  - FP8 means OCP E4M3: bias 7, largest finite 448, 0x7F / 0xFF are NaN, no
 *    infinities.  BF16 tensors hold raw bfloat16 values.
 *  - Pool layout: row `slot` of the c_kv pool starts at
 *    ckv_pool + slot * ckv_row_stride_bytes and holds 512 channels; row
 *    `slot` of the k_pe pool starts at kpe_pool + slot * kpe_row_stride_bytes
 *    and holds 64 channels.  The pages' combined [slots, 576] layout is
 *    kpe_pool = ckv_pool + 512 elements with both strides = one 576-row.
 *    Pool base pointers and row strides must be multiples of 16 bytes.
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,  /* NULL pointer, bad size, bad page table     */
    MLA_ERR_UNSUPPORTED = 2,  /* head count / alignment the kernels lack    */
    MLA_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than planned     */
    MLA_ERR_INDEX_OOB = 4,    /* reported by mla_get_last_error()           */
    MLA_ERR_CUDA = 5          /* a CUDA runtime call failed                 */
} mla_status_t;

typedef enum {
    MLA_KV_FP8_E4M3 = 0,      /* the product path: pools hold E4M3 bytes    */
    MLA_KV_BF16 = 1           /* pools hold BF16 (cast-then-attend baselines) */
} mla_kv_dtype_t;

/* Bits of the device flag word read by mla_get_last_error(). */
#define MLA_FLAG_INDEX_OOB      0x1u  /* a slot / page index was outside the pool */
#define MLA_FLAG_PLAN_MISMATCH  0x2u  /* device seq_lens disagree with the plan  */
#define MLA_FLAG_WAIT_TIMEOUT   0x4u  /* a bounded in-kernel wait gave up        */

typedef struct mla_plan* mla_plan_t;

#define MLA_D_CKV 512   /* kv_lora_rank   ([P2] "The Context") */
#define MLA_D_KPE 64    /* qk_rope_head_dim ([P2] "The Context") */
#define MLA_D_QK  576   /* score width = 512 + 64 */

/*
 * mla_decode_plan -- the plan() half of the plan/run split ([P2] "The
 * Message"; [P3] "The Subject Message").  Runs on the host once per decode
 * step, shared by all layers of that step.
 *
 *  plan             in/out.  If *plan is NULL a new plan is created;
 *                   otherwise that plan is rebuilt in place (its device and
 *                   pinned buffers are reused when large enough).
 *  kv_indptr_host   int32 [batch+1]: request b owns page-table entries
 *                   kv_indices[kv_indptr[b] .. kv_indptr[b+1]).  Must be
 *                   non-decreasing, kv_indptr[0] >= 0, and each request must
 *                   own exactly ceil(seq_lens[b] / page_size) pages.
 *  seq_lens_host    int32 [batch]: context length of each request (>= 0).
 *  num_heads        query heads H: 1..16, or a multiple of 16 up to 128.
 *  page_size        tokens per page (>= 1).  Token t of request b is slot
 *                   kv_indices[kv_indptr[b] + t / page_size] * page_size
 *                   + t % page_size.
 *  kv_dtype         element type of the pools run() will read.
 *  workspace_bytes  out: device scratch run() needs: the split-KV partials
 *                   and, on the tensor-core FP8 path, one 27,840-byte image
 *                   of the split query per request and group of 16 heads.
 *  stream           the plan's device metadata is uploaded on this stream
 *                   (stream-ordered before later runs on it).
 * Errors: MLA_ERR_INVALID_ARG / MLA_ERR_UNSUPPORTED before any allocation;
 * MLA_ERR_CUDA if an allocation or copy fails (the plan stays valid if it
 * existed).  The plan must be rebuilt whenever kv_indptr or seq_lens change.
 */
mla_status_t mla_decode_plan(mla_plan_t* plan, const int32_t* kv_indptr_host,
                             const int32_t* seq_lens_host, int32_t batch,
                             int32_t num_heads, int32_t page_size,
                             mla_kv_dtype_t kv_dtype, size_t* workspace_bytes,
                             void* stream);

/*
 * mla_decode_run -- the run() half: decode attention for every request of
 * the plan, reading the cache rows in place (no BF16 copy of the cache is
 * made).  Per request b and head h, with k_t = value(row_t) * k_scale over
 * all 576 channels (c_kv then k_pe) and v_t = the 512 c_kv channels:
 *     s_t = softmax_scale * sum_d q[b][h][d] * k_t[d]
 *     out[b][h] = sum_t softmax(s)_t * v_t        (BF16)
 *     lse[b][h] = ln sum_t exp(s_t)               (fp32, natural log)
 * A request with seq_len 0 gets out = 0 and lse = -inf; a head whose query
 * row holds an infinity or a NaN gets out = NaN and lse = NaN.
 * Arithmetic of FP8 plans: the E4M3 cache bytes are the tensor-core operands
 * as they are; each query row enters as three E4M3 terms (exactly for every
 * entry above 2^-14 of the row's largest, with 4 significant bits below) and
 * the softmax weights as two (8 significant bits; a token more than 19 log2
 * units, about 13 nats, below the running maximum score may be dropped from
 * the output sum, one more than 23 always is); products accumulate in fp32.
 *
 *  q                BF16, element (b, h, d) at q + b*q_stride_b + h*q_stride_h
 *                   + d (strides in elements; d < 576 contiguous).
 *  ckv_pool, ...    see the pool layout above; E4M3 bytes for
 *                   MLA_KV_FP8_E4M3 plans, BF16 for MLA_KV_BF16 plans.
 *  num_pool_slots   rows in each pool; indices reaching past it are skipped.
 *  kv_indptr_dev, kv_indices_dev, seq_lens_dev
 *                   device copies of the page table given to the plan
 *                   (kv_indptr / seq_lens must equal the plan's host arrays).
 *  k_scale          per-tensor dequantization scale (use 1 for BF16 pools
 *                   that already hold real values).
 *  out              BF16 [batch][H][512], contiguous.
 *  lse              fp32 [batch][H], contiguous.
 *  workspace        device scratch of at least the planned workspace_bytes,
 *                   256-byte aligned; its contents are not preserved.
 * No host synchronisation, allocation or host<->device copy happens here.
 * The call enqueues up to three kernels on `stream` (query split, decode,
 * split-KV merge); on the tensor-core path the decode kernel is launched as a
 * programmatic dependent of the query split, so it may start early and waits
 * on the device for the split's results.  Work enqueued before the call is
 * complete before any of them reads it.
 * Errors: MLA_ERR_INVALID_ARG (NULL / misaligned / plan mismatch),
 * MLA_ERR_WORKSPACE, MLA_ERR_CUDA (launch failure).
 */
mla_status_t mla_decode_run(mla_plan_t plan, const void* q, int64_t q_stride_b,
                            int64_t q_stride_h, const void* ckv_pool,
                            int64_t ckv_row_stride_bytes, const void* kpe_pool,
                            int64_t kpe_row_stride_bytes, int64_t num_pool_slots,
                            const int32_t* kv_indptr_dev,
                            const int32_t* kv_indices_dev,
                            const int32_t* seq_lens_dev, float k_scale,
                            float softmax_scale, void* out, float* lse,
                            void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * mla_decode_run_static_scratch -- mla_decode_run for callers that cannot
 * allocate device memory.  The pages have no counterpart to this call.
 *
 * Some callers have no way to hand the decode a workspace: a plugin inside a
 * framework that owns every GPU allocation, a real-time loop that must not
 * pay cudaMalloc's implicit device synchronisation, code that must not touch
 * the allocator between steps.  This call takes the same arguments as
 * mla_decode_run minus the workspace and keeps its scratch (split-KV
 * partials, query images) in a
 * fixed array of MLA_STATIC_SCRATCH_BYTES compiled into the library; the
 * call allocates nothing (the plan is built beforehand by mla_decode_plan).
 *  - The array exists once per GPU that loads the library and stays
 *    allocated until the process exits.
 *  - The first call on a device looks up the array's device address; make
 *    that first call before any stream capture begins.  The address is kept
 *    until exit: after a cudaDeviceReset of that device, do not use this
 *    call on it again.
 *  - Every call shares the array: calls whose GPU work overlaps (other
 *    streams, other host threads) race on it.  Calls on one stream are
 *    ordered.  Nothing in the array needs to start at zero.
 * Errors: as mla_decode_run; MLA_ERR_WORKSPACE if the plan needs more than
 * MLA_STATIC_SCRATCH_BYTES of scratch (see mla_decode_plan_info).
 */
#define MLA_STATIC_SCRATCH_BYTES (8u << 20)
mla_status_t mla_decode_run_static_scratch(mla_plan_t plan, const void* q,
                                           int64_t q_stride_b, int64_t q_stride_h,
                                           const void* ckv_pool,
                                           int64_t ckv_row_stride_bytes,
                                           const void* kpe_pool,
                                           int64_t kpe_row_stride_bytes,
                                           int64_t num_pool_slots,
                                           const int32_t* kv_indptr_dev,
                                           const int32_t* kv_indices_dev,
                                           const int32_t* seq_lens_dev, float k_scale,
                                           float softmax_scale, void* out, float* lse,
                                           void* stream);

/*
 * mla_extend_plan -- plan() for causal extend attention over an FP8 cache:
 * several new tokens per request (a prefill chunk on top of a cached prefix,
 * or several speculative tokens), each attending to the request's cached
 * history and to the new tokens before it.  This is the attention whose BF16
 * requirement makes the FP8 configuration cast the whole history back to
 * BF16 on every extend step ([P1] "Step 3: Source Validation", CastFromFP8);
 * [P1] "From Attribution to Optimization Targets" asks for a prefill
 * attention that reads the FP8 cache instead, which is what this plan runs.
 * The pages do not spell the extend attention out; the reading implemented:
 * request b has q_len_b = qo_indptr[b+1] - qo_indptr[b] new tokens, already
 * stored in the cache (so seq_lens[b] counts them, q_len_b <= seq_lens[b]);
 * new token i (0-based) sits at position seq_lens[b] - q_len_b + i and sees
 * the tokens at positions 0 .. seq_lens[b] - q_len_b + i.  With every q_len
 * equal to 1 this is exactly decode.
 *  qo_indptr_host   int32 [batch+1], qo_indptr[0] = 0, non-decreasing: the
 *                   new tokens of request b are query rows
 *                   qo_indptr[b] .. qo_indptr[b+1]-1.
 *  kv_indptr_host, seq_lens_host, num_heads, page_size
 *                   as for mla_decode_plan.
 *  kv_dtype         MLA_KV_FP8_E4M3 only (MLA_ERR_UNSUPPORTED otherwise).
 *  workspace_bytes  out: scratch mla_extend_run needs (split partials and
 *                   one split-query image per block of query rows).
 * The query rows (new token x head, row = token * H + head) of each request
 * are cut into blocks of 16 or 32 rows; each block runs like a decode
 * request whose context ends at its last row's causal limit, rows of the
 * block that see fewer tokens are masked.  Errors and plan lifetime as for
 * mla_decode_plan (the plan must be rebuilt when qo_indptr changes too).  A
 * plan made here is run with mla_extend_run only.
 */
mla_status_t mla_extend_plan(mla_plan_t* plan, const int32_t* qo_indptr_host,
                             const int32_t* kv_indptr_host,
                             const int32_t* seq_lens_host, int32_t batch,
                             int32_t num_heads, int32_t page_size,
                             mla_kv_dtype_t kv_dtype, size_t* workspace_bytes,
                             void* stream);

/*
 * mla_extend_run -- run() for an extend plan.  For query row (n, h), n a new
 * token of request b at position pos_n (see mla_extend_plan):
 *     s_t = softmax_scale * sum_d q[n][h][d] * k_t[d],   t <= pos_n
 *     out[n][h] = sum_{t <= pos_n} softmax(s)_t * v_t    (BF16)
 *     lse[n][h] = ln sum_{t <= pos_n} exp(s_t)          (fp32)
 * with k_t, v_t as in mla_decode_run.
 *  q                BF16, element (n, h, d) at q + n*q_stride_tok +
 *                   h*q_stride_h + d (elements; d < 576 contiguous), n <
 *                   qo_indptr[batch].
 *  out              BF16 [qo_indptr[batch]][H][512], contiguous.
 *  lse              fp32 [qo_indptr[batch]][H], contiguous.
 * Every other argument, the launches (query split, tcgen05 kernel, merge)
 * and the errors are as for mla_decode_run; a decode plan is rejected
 * (MLA_ERR_INVALID_ARG), as is an extend plan passed to mla_decode_run.
 */
mla_status_t mla_extend_run(mla_plan_t plan, const void* q, int64_t q_stride_tok,
                            int64_t q_stride_h, const void* ckv_pool,
                            int64_t ckv_row_stride_bytes, const void* kpe_pool,
                            int64_t kpe_row_stride_bytes, int64_t num_pool_slots,
                            const int32_t* kv_indptr_dev,
                            const int32_t* kv_indices_dev,
                            const int32_t* seq_lens_dev, float k_scale,
                            float softmax_scale, void* out, float* lse,
                            void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * mla_extend_schedule -- host only: the schedule mla_extend_plan would build
 * on a GPU with num_sms SMs.  segments_out (may be NULL): up to seg_capacity
 * int32 quintuples (cta, block, token_begin, token_end, partial or -1);
 * blocks_out (may be NULL): up to block_capacity int32 quadruples (request,
 * first query row, rows, causal base: row r sees the tokens before
 * base + r / H); counts_out (may be NULL): int32 [5] = segments, partials,
 * CTAs, blocks, rows per block.  Validates exactly like mla_extend_plan.
 */
mla_status_t mla_extend_schedule(const int32_t* qo_indptr_host,
                                 const int32_t* kv_indptr_host,
                                 const int32_t* seq_lens_host, int32_t batch,
                                 int32_t num_heads, int32_t page_size,
                                 mla_kv_dtype_t kv_dtype, int32_t num_sms,
                                 int32_t* segments_out, int32_t seg_capacity,
                                 int32_t* blocks_out, int32_t block_capacity,
                                 int32_t* counts_out, size_t* workspace_bytes);

/* Releases a plan and its device / pinned buffers (after the caller has
 * synchronised any stream still using it).  NULL is accepted. */
mla_status_t mla_decode_plan_destroy(mla_plan_t plan);

/* Plan summary: CTAs launched, (cta, request, token range) segments, split
 * partials written to the workspace, and the workspace size.  Host only. */
mla_status_t mla_decode_plan_info(mla_plan_t plan, int32_t* num_ctas,
                                  int32_t* num_segments, int32_t* num_partials,
                                  size_t* workspace_bytes);

/*
 * mla_decode_schedule -- host only, no GPU needed: the split-KV schedule a
 * plan with these arguments would use on a GPU with `num_sms` SMs.  Writes
 * up to `capacity` segments as int32 quintuples
 *     (cta, request, token_begin, token_end, partial_index or -1)
 * into segments_out (may be NULL), in launch order; tile_tokens receives the
 * kernel's tile (segments start on tile boundaries) and kernel the decode
 * kernel the plan would launch: 0 = mma.sync (BF16 pools), 1 = tcgen05 on
 * the E4M3 bytes (FP8 pools; 16 heads per CTA, 32 when H is a multiple of
 * 32, more heads as more CTAs).  The
 * mma.sync schedule gives each CTA an equal share of tiles; the tcgen05 one
 * balances tiles plus a fixed cost per segment.  Validates exactly like
 * mla_decode_plan.  Output pointers may be NULL.
 */
mla_status_t mla_decode_schedule(const int32_t* kv_indptr_host,
                                 const int32_t* seq_lens_host, int32_t batch,
                                 int32_t num_heads, int32_t page_size,
                                 mla_kv_dtype_t kv_dtype, int32_t num_sms,
                                 int32_t* segments_out, int32_t capacity,
                                 int32_t* num_segments, int32_t* num_partials,
                                 int32_t* num_ctas, int32_t* tile_tokens,
                                 int32_t* kernel, size_t* workspace_bytes);

/*
 * kv_store_fp8 -- quantize-on-store scatter ([P1] "Step 3", CastToFP8 in
 * set_kv_buffer), fused into one pass: for each new token i,
 *     ckv_pool[slots[i]][d] = E4M3(float(ckv_new[i][d]) / k_scale), d < 512
 *     kpe_pool[slots[i]][d] = E4M3(float(kpe_new[i][d]) / k_scale), d < 64
 * with one IEEE fp32 division, round to nearest (ties to even), saturation
 * of |x| > 448 (and +-inf) to +-448, NaN -> 0x7F, sign kept.
 *  ckv_new  BF16 [n][512] contiguous;  kpe_new  BF16 [n][64] contiguous.
 *  slots    int64 [n], device.  Duplicate slots give an unspecified row.
 * n = 0 is a no-op.  Errors: MLA_ERR_INVALID_ARG, MLA_ERR_CUDA.
 */
mla_status_t kv_store_fp8(const void* ckv_new, const void* kpe_new,
                          const int64_t* slots, int64_t n, float k_scale,
                          void* ckv_pool, int64_t ckv_row_stride_bytes,
                          void* kpe_pool, int64_t kpe_row_stride_bytes,
                          int64_t num_pool_slots, void* stream);

/*
 * kv_proj_store_fp8 -- the KV projection with the FP8 cache write fused into
 * its epilogue ([P1] "Step 3", CastToFP8: the new BF16 KV comes out of the
 * attention projection and set_kv_buffer quantizes it as a separate copy;
 * [P1] "From Attribution to Optimization Targets": let the projection
 * kernel emit FP8 directly).  The pages give no shape for the projection;
 * the reading implemented: one linear map of each new token's hidden state
 * to the 576 latent channels (512 c_kv, then 64 k_pe),
 *     latent[i][j] = BF16_rne( sum_k x[i][k] * w[j][k] )   (fp32 accumulation)
 * and then, per token, exactly kv_store_fp8 of that BF16 row into pool row
 * slots[i].  One kernel: BF16 tensor-core GEMM, rounding, quantization and
 * scatter; no BF16 latent is written unless latent_out is given.
 *  x           BF16 [n][d_model], row stride x_row_stride elements (a multiple
 *              of 8, >= d_model), 16-byte aligned.
 *  w           BF16 [576][d_model]: row j holds the weights of latent channel
 *              j (the transposed weight matrix), row stride w_row_stride.
 *  d_model     a multiple of 64, 64 .. 65536.
 *  slots       int64 [n], device; an out-of-range slot skips its row and
 *              sets MLA_FLAG_INDEX_OOB.  Duplicate slots give an unspecified row.
 *  k_scale, pools, num_pool_slots   as for kv_store_fp8.
 *  latent_out  optional BF16 [n][576], contiguous, 16-byte aligned: the
 *              rounded latents the bytes were made from.
 * n = 0 is a no-op.  Asynchronous on `stream`; no allocation, no workspace.
 * Errors: MLA_ERR_INVALID_ARG (NULL / bad size / scale), MLA_ERR_UNSUPPORTED
 * (alignment), MLA_ERR_CUDA (launch).
 */
mla_status_t kv_proj_store_fp8(const void* x, int64_t x_row_stride, const void* w,
                               int64_t w_row_stride, int64_t n, int32_t d_model,
                               const int64_t* slots, float k_scale, void* ckv_pool,
                               int64_t ckv_row_stride_bytes, void* kpe_pool,
                               int64_t kpe_row_stride_bytes, int64_t num_pool_slots,
                               void* latent_out, void* stream);

/*
 * kv_gather_cast -- gather-then-cast of the active pages ([P3] "The
 * Reasoning Process"): row j*page_size + r of the outputs is pool slot
 * kv_indices[j]*page_size + r, converted as
 *     BF16_rne(float(value(byte)) * k_scale)
 * (one fp32 multiply; with k_scale = 1 this is exactly the pages' unscaled
 * .to(bfloat16)).  The two NaN codes 0x7F / 0xFF become the quiet NaN
 * 0x7FC0 (sign dropped, as PyTorch's float8_e4m3fn -> bfloat16 cast gives
 * them).  A caller then replans with indices 0..n_pages-1 and runs a
 * MLA_KV_BF16 decode on the compact buffers.
 *  kv_indices  int32 [n_pages], device.
 *  ckv_out     BF16 [n_pages*page_size][512];  kpe_out  BF16 [..][64].
 * n_pages = 0 is a no-op.  Errors: MLA_ERR_INVALID_ARG, MLA_ERR_CUDA.
 */
mla_status_t kv_gather_cast(const void* ckv_pool, int64_t ckv_row_stride_bytes,
                            const void* kpe_pool, int64_t kpe_row_stride_bytes,
                            int64_t num_pool_slots, const int32_t* kv_indices,
                            int64_t n_pages, int32_t page_size, float k_scale,
                            void* ckv_out, void* kpe_out, void* stream);

/*
 * mla_get_last_error -- synchronises `stream`, then reads and clears the
 * current device's flag word (MLA_FLAG_* bits, OR-ed by every kernel since
 * the last call).  Returns MLA_ERR_INDEX_OOB if any flag was set,
 * MLA_ERR_CUDA if the synchronisation failed, else MLA_OK.
 */
mla_status_t mla_get_last_error(void* stream, uint32_t* device_flags_out);

/*
 * mla_debug_set_wait_limit -- test hook for the decode kernels' failure
 * handling.  Every wait of the FP8 decode / extend kernels on an in-kernel
 * barrier is bounded: after the limit the CTA sets MLA_FLAG_WAIT_TIMEOUT,
 * abandons its work (its outputs are void), lets its copies and MMAs
 * finish, frees its tensor memory and exits, so a stuck pipeline never
 * hangs the GPU ("When a Faster Kernel Doesn't Speed Up Serving" runs the
 * decode inside CUDA graphs of a serving loop, where a hung kernel stalls
 * every request).  The limit is 2 s; this call sets it, in nanoseconds, for
 * the current device (0 restores 2 s).  A tiny limit makes the next calls
 * give up early, which is how the timeout path is tested: under 1 ms,
 * 16-head CTAs poll their barriers without suspending and give up at the
 * first wait that finds its barrier not ready; 32-head CTAs give up at the
 * first wait that outlasts one suspended try_wait.
 * Synchronous: call it between launches, with no decode kernel running.
 * Errors: MLA_ERR_CUDA.
 */
mla_status_t mla_debug_set_wait_limit(uint64_t limit_ns);

/* Static description of a status code. */
const char* mla_status_string(mla_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H */
