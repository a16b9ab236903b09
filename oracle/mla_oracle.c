/*
 * Oracle for paged MLA decode over an FP8 E4M3 KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * CPU statement of what the GPU library computes.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or constant with the CUDA library, and the CUDA library
 * never calls it.
 *
 * Sources (web pages, by title and section):
 *  [P1] "When a Faster Kernel Doesn't Speed Up Serving: Profiling FP8 KV Cache
 *       on AMD Instinct MI308X", sections "Step 3: Source Validation"
 *       (CastFromFP8: kvc.to(dtype) / k_pe.to(dtype) are plain FP8->BF16
 *       casts; CastToFP8: set_kv_buffer quantizes new BF16 KV into the FP8
 *       cache).
 *  [P2] "The KV Cache Cast Bottleneck: A Surgical Fix for 69% Decode
 *       Overhead", section "The Context" (cache rows of 576 = kv_lora_rank 512
 *       + qk_rope_head_dim 64, Float8_e4m3fn) and "The Message" (the decode
 *       kernel reads FP8 rows and computes in higher precision).
 *  [P3] "The Gather-Then-Cast Pivot", sections "The Subject Message" (run()
 *       reads page-indexed ckv/kpe buffers through kv_indices) and "The
 *       Reasoning Process" (gather the active FP8 rows, cast them, replan
 *       with sequential indices).
 *
 * The pages name the E4M3 format and the MLA shapes but define neither the
 * format's bits nor the attention formula.  The readings used here:
 *  - E4M3 (OCP FP8): byte s|eeee|mmm, exponent bias 7; e = 0 is subnormal
 *    (m/8 * 2^-6); 0x7F and 0xFF are NaN; no infinities; largest finite 448.
 *  - Encoding rounds to the nearest finite value, ties to the even mantissa
 *    code, and saturates any |x| > 448 (including +-inf) to +-448; NaN
 *    encodes as 0x7F; the sign is always kept (-0 -> 0x80).
 *  - Store: byte = enc(float(bf16) / k_scale), one IEEE fp32 division.
 *  - Gather-cast: bf16 = RNE_bf16(float(dec(byte)) * k_scale), one fp32
 *    multiply, then round to nearest even BF16.  With k_scale = 1 this is the
 *    pages' unscaled .to(bfloat16).
 *  - Attention, per request b and head h, with k_t = dec(row_t) * k_scale
 *    over all 576 channels and v_t = k_t[0:512]:
 *        s_t  = softmax_scale * sum_d q[h][d] k_t[d]
 *        p_t  = exp(s_t - m) / sum_u exp(s_u - m),   m = max_t s_t
 *        o[h] = sum_t p_t v_t ,   lse[h] = m + ln(sum_u exp(s_u - m))
 *    (natural logarithm).  An empty context gives o = 0 and lse = -inf.
 *  - Page table: token t of request b lives in slot
 *        kv_indices[kv_indptr[b] + t / page_size] * page_size + t % page_size.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fopenmp -shared -fPIC.  No fast
 * math: every fp32 step above is a single IEEE operation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define D_CKV 512
#define D_KPE 64
#define D_ALL (D_CKV + D_KPE)

/* ---------------------------------------------------------------- E4M3 */

/* Value of one E4M3 byte, straight from the bit fields (OCP FP8 E4M3). */
static double e4m3_value(uint8_t b) {
    int s = b >> 7, e = (b >> 3) & 0xF, m = b & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) mag = ldexp((double)m / 8.0, -6);
    else mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

void oracle_e4m3_table(double out[256]) {
    for (int b = 0; b < 256; ++b) out[b] = e4m3_value((uint8_t)b);
}

/* Nearest finite E4M3 code to x, ties to the even mantissa code, saturating.
 * The magnitudes of codes 0x00..0x7E are strictly increasing, so the nearest
 * value is found by locating x between two neighbours and comparing it with
 * their midpoint (exact in double: both neighbours have 4 significant bits). */
uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a > 448.0) return sign | 0x7E;
    int lo = 0, hi = 0x7E;              /* value(lo) <= a < value(hi+1) */
    while (lo < hi) {                    /* largest code with value <= a */
        int mid = (lo + hi + 1) / 2;
        if (e4m3_value((uint8_t)mid) <= a) lo = mid; else hi = mid - 1;
    }
    if (lo == 0x7E || e4m3_value((uint8_t)lo) == a) return sign | (uint8_t)lo;
    double v0 = e4m3_value((uint8_t)lo), v1 = e4m3_value((uint8_t)(lo + 1));
    double midpoint = 0.5 * (v0 + v1);
    int code;
    if (a < midpoint) code = lo;
    else if (a > midpoint) code = lo + 1;
    else code = (lo & 1) ? lo + 1 : lo; /* mantissa lsb is the code lsb */
    return sign | (uint8_t)code;
}

static float bf16_to_float(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a float to the nearest BF16, ties to even.  The two BF16 neighbours
 * of f bracket it; the midpoint between them decides, in exact double. */
static uint16_t float_to_bf16_rne(float f) {
    if (isnan(f)) return 0x7FC0;
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t lo = (uint16_t)(u >> 16);           /* truncation toward zero */
    if ((u & 0xFFFF) == 0) return lo;
    uint16_t up = (uint16_t)(lo + 1);            /* next magnitude */
    double dlo = fabs((double)bf16_to_float(lo));
    double dup = fabs((double)bf16_to_float(up)); /* may be +-inf: fine */
    double a = fabs((double)f);
    double midpoint = 0.5 * (dlo + dup);
    if (isinf(dup)) midpoint = dlo + (dlo - fabs((double)bf16_to_float((uint16_t)(lo - 1)))) / 2.0;
    if (a < midpoint) return lo;
    if (a > midpoint) return up;
    return (lo & 1) ? up : lo;
}

uint16_t oracle_float_to_bf16(float f) { return float_to_bf16_rne(f); }

void oracle_e4m3_encode_array(const float* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

/* ------------------------------------------------------------- store */

/* Quantize-on-store ([P1] "Step 3", CastToFP8 in set_kv_buffer): each new
 * token's BF16 c_kv[512] and k_pe[64] are divided by k_scale in fp32 and
 * encoded into pool row `slots[i]`.  Returns the number of slots that were
 * out of range (those rows are skipped). */
int64_t oracle_kv_store_fp8(const uint16_t* ckv_new, const uint16_t* kpe_new,
                            const int64_t* slots, int64_t n, float k_scale,
                            uint8_t* ckv_pool, int64_t ckv_stride,
                            uint8_t* kpe_pool, int64_t kpe_stride,
                            int64_t num_slots) {
    int64_t bad = 0;
    /* tokens are independent: one per iteration */
#pragma omp parallel for schedule(static) reduction(+ : bad)
    for (int64_t i = 0; i < n; ++i) {
        int64_t s = slots[i];
        if (s < 0 || s >= num_slots) { ++bad; continue; }
        for (int d = 0; d < D_CKV; ++d) {
            float v = bf16_to_float(ckv_new[i * D_CKV + d]) / k_scale;
            ckv_pool[s * ckv_stride + d] = oracle_e4m3_encode(v);
        }
        for (int d = 0; d < D_KPE; ++d) {
            float v = bf16_to_float(kpe_new[i * D_KPE + d]) / k_scale;
            kpe_pool[s * kpe_stride + d] = oracle_e4m3_encode(v);
        }
    }
    return bad;
}

/* ------------------------------------------- fused KV projection store */

/* Round a double to the nearest BF16 value, ties to even (one rounding of
 * the double itself, not through float).  BF16: 8 significant bits, the
 * float exponent range, subnormal spacing 2^-133; beyond the largest finite
 * value (2^128 - 2^120) the result is +-inf. */
static uint16_t double_to_bf16_rne(double x) {
    if (x != x) return 0x7FC0;
    if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
    int e = 0;
    frexp(x, &e);                       /* |x| = m * 2^e, m in [0.5, 1) */
    int q = e - 8;                      /* spacing of 8-bit significands */
    if (q < -133) q = -133;             /* subnormal spacing */
    double r = nearbyint(ldexp(x, -q)); /* default rounding: nearest, ties even */
    double v = ldexp(r, q);
    if (fabs(v) >= ldexp(1.0, 128)) return signbit(x) ? 0xFF80 : 0x7F80;
    float f = (float)v;                 /* exact: v has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

uint16_t oracle_double_to_bf16(double x) { return double_to_bf16_rne(x); }

/* The KV projection with the cache write fused into it ([P1] "Step 3",
 * CastToFP8: every step's new KV comes out of the attention projection in
 * BF16 and set_kv_buffer quantizes it into the FP8 cache as a separate copy;
 * "From Attribution to Optimization Targets": the projection kernel should
 * emit FP8 itself).  The pages give neither the projection's shape nor its
 * weights; the reading: one linear map of the hidden state to the 576 latent
 * channels (512 c_kv, then 64 k_pe), weights w[j][k] for output channel j,
 * whose BF16 output is what the unfused path stores:
 *   latent[i][j] = BF16_rne( sum_k x[i][k] * w[j][k] )   (exact sum, one rounding)
 *   pool rows slots[i] = kv_store_fp8(latent[i])          (as above)
 * The products of BF16 values are exact in double and the sums of up to a
 * few thousand of them carry far more than the 8 bits the rounding keeps.
 * x: BF16 [n][d], w: BF16 [576][d]; latent_out (optional): BF16 [n][576].
 * Returns the number of out-of-range slots (their rows are left alone). */
int64_t oracle_kv_proj_fp8(const uint16_t* x, const uint16_t* w, int64_t n, int32_t d,
                           const int64_t* slots, float k_scale, uint8_t* ckv_pool,
                           int64_t ckv_stride, uint8_t* kpe_pool, int64_t kpe_stride,
                           int64_t num_slots, uint16_t* latent_out) {
    uint16_t* lat = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(n > 0 ? n : 1) * D_ALL);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        for (int j = 0; j < D_ALL; ++j) {
            double acc = 0.0;
            for (int32_t k = 0; k < d; ++k)
                acc += (double)bf16_to_float(x[i * d + k]) * (double)bf16_to_float(w[(int64_t)j * d + k]);
            lat[i * D_ALL + j] = double_to_bf16_rne(acc);
        }
    }
    if (latent_out) memcpy(latent_out, lat, sizeof(uint16_t) * (size_t)n * D_ALL);
    /* the store reads c_kv and k_pe as separate [n][512] / [n][64] arrays */
    uint16_t* ckv = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(n > 0 ? n : 1) * D_CKV);
    uint16_t* kpe = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(n > 0 ? n : 1) * D_KPE);
    for (int64_t i = 0; i < n; ++i) {
        memcpy(ckv + i * D_CKV, lat + i * D_ALL, sizeof(uint16_t) * D_CKV);
        memcpy(kpe + i * D_KPE, lat + i * D_ALL + D_CKV, sizeof(uint16_t) * D_KPE);
    }
    int64_t bad = oracle_kv_store_fp8(ckv, kpe, slots, n, k_scale, ckv_pool, ckv_stride,
                                      kpe_pool, kpe_stride, num_slots);
    free(lat);
    free(ckv);
    free(kpe);
    return bad;
}

/* -------------------------------------------------------- gather-cast */

/* Gather-then-cast ([P3] "The Reasoning Process"): the rows of the listed
 * pages are copied, in page-list order, into a compact BF16 buffer so that
 * a BF16 attention kernel can run on them with sequential indices.  Row
 * j*page_size + r of the output is slot kv_indices[j]*page_size + r.
 * Returns the number of out-of-range pages (their rows are left untouched). */
int64_t oracle_kv_gather_cast(const uint8_t* ckv_pool, int64_t ckv_stride,
                              const uint8_t* kpe_pool, int64_t kpe_stride,
                              int64_t num_slots, const int32_t* kv_indices,
                              int64_t n_pages, int32_t page_size, float k_scale,
                              uint16_t* ckv_out, uint16_t* kpe_out) {
    int64_t bad = 0;
    for (int64_t j = 0; j < n_pages; ++j) {
        int64_t first = (int64_t)kv_indices[j] * page_size;
        if (kv_indices[j] < 0 || first + page_size > num_slots) { ++bad; continue; }
        for (int32_t r = 0; r < page_size; ++r) {
            int64_t s = first + r, row = j * page_size + r;
            for (int d = 0; d < D_CKV; ++d) {
                float v = (float)e4m3_value(ckv_pool[s * ckv_stride + d]) * k_scale;
                ckv_out[row * D_CKV + d] = float_to_bf16_rne(v);
            }
            for (int d = 0; d < D_KPE; ++d) {
                float v = (float)e4m3_value(kpe_pool[s * kpe_stride + d]) * k_scale;
                kpe_out[row * D_KPE + d] = float_to_bf16_rne(v);
            }
        }
    }
    return bad;
}

/* ---------------------------------------------------------- attention */

/* Softmax attention of H query rows against L key rows, all in fp64.
 * q: [H][576]; k: [L][576] (v = the first 512 channels of k).
 * o: [H][512]; lse: [H]; p (optional): [H][L] softmax weights. */
static void attention_one_request(const double* q, const double* k, int64_t L,
                                  int32_t H, double softmax_scale, double* o,
                                  double* lse, double* p, double* s_buf) {
    for (int32_t h = 0; h < H; ++h) {
        const double* qh = q + (int64_t)h * D_ALL;
        double* oh = o + (int64_t)h * D_CKV;
        for (int d = 0; d < D_CKV; ++d) oh[d] = 0.0;
        if (L == 0) { lse[h] = -INFINITY; continue; }
        double m = -INFINITY;
        for (int64_t t = 0; t < L; ++t) {
            const double* kt = k + t * D_ALL;
            double acc = 0.0;
            for (int d = 0; d < D_ALL; ++d) acc += qh[d] * kt[d];
            s_buf[t] = softmax_scale * acc;
            if (s_buf[t] > m) m = s_buf[t];
        }
        double sum = 0.0;
        for (int64_t t = 0; t < L; ++t) sum += exp(s_buf[t] - m);
        for (int64_t t = 0; t < L; ++t) {
            double pt = exp(s_buf[t] - m) / sum;
            if (p) p[(int64_t)h * L + t] = pt;
            const double* vt = k + t * D_ALL;
            for (int d = 0; d < D_CKV; ++d) oh[d] += pt * vt[d];
        }
        lse[h] = m + log(sum);
    }
}

/* Slot of token t of a request whose page list starts at `pages`. */
static int64_t token_slot(const int32_t* pages, int64_t t, int32_t page_size) {
    return (int64_t)pages[t / page_size] * page_size + t % page_size;
}

/* One channel of one pool row, dequantized and multiplied by k_scale.
 * kind 0 = E4M3 bytes, kind 1 = BF16 values. */
static double pool_value(int kind, const void* pool, int64_t stride_bytes,
                         int64_t slot, int d, double k_scale) {
    const uint8_t* row = (const uint8_t*)pool + slot * stride_bytes;
    if (kind == 0) return e4m3_value(row[d]) * k_scale;
    uint16_t h;
    memcpy(&h, row + 2 * d, 2);
    return (double)bf16_to_float(h) * k_scale;
}

/* Paged MLA decode.  q: BF16 bits [B][H][576] (contiguous).  Pools are byte
 * addressed with row strides in bytes; kind selects E4M3 (0) or BF16 (1)
 * rows.  o: [B][H][512], lse: [B][H], p (optional): [B][H][max_len] with
 * p[b][h][t] for t < seq_lens[b].  Returns -1 on an out-of-range slot or a
 * page table too short for a sequence, else 0. */
static int decode_common(int kind, const uint16_t* q_bf16, const void* ckv_pool,
                         int64_t ckv_stride, const void* kpe_pool,
                         int64_t kpe_stride, int64_t num_slots,
                         const int32_t* kv_indptr, const int32_t* kv_indices,
                         const int32_t* seq_lens, int32_t B, int32_t H,
                         int32_t page_size, double k_scale, double softmax_scale,
                         double* o, double* lse, double* p, int64_t p_stride,
                         int nthreads) {
    for (int32_t b = 0; b < B; ++b) {
        int64_t L = seq_lens[b];
        int64_t pages = kv_indptr[b + 1] - kv_indptr[b];
        if (L < 0 || pages * page_size < L) return -1;
        for (int64_t t = 0; t < L; ++t) {
            int64_t s = token_slot(kv_indices + kv_indptr[b], t, page_size);
            if (s < 0 || s >= num_slots) return -1;
        }
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    /* one (request, head) pair per iteration; each is fully independent */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        int32_t b = (int32_t)(bh / H), h = (int32_t)(bh % H);
        int64_t L = seq_lens[b];
        const int32_t* pages = kv_indices + kv_indptr[b];
        double qh[D_ALL];
        for (int d = 0; d < D_ALL; ++d)
            qh[d] = bf16_to_float(q_bf16[((int64_t)b * H + h) * D_ALL + d]);
        double* k = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * D_ALL);
        double* s_buf = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        for (int64_t t = 0; t < L; ++t) {
            int64_t slot = token_slot(pages, t, page_size);
            for (int d = 0; d < D_CKV; ++d)
                k[t * D_ALL + d] = pool_value(kind, ckv_pool, ckv_stride, slot, d, k_scale);
            for (int d = 0; d < D_KPE; ++d)
                k[t * D_ALL + D_CKV + d] = pool_value(kind, kpe_pool, kpe_stride, slot, d, k_scale);
        }
        attention_one_request(qh, k, L, 1, softmax_scale,
                              o + ((int64_t)b * H + h) * D_CKV,
                              lse + (int64_t)b * H + h,
                              p ? p + ((int64_t)b * H + h) * p_stride : NULL, s_buf);
        free(k);
        free(s_buf);
    }
    return 0;
}

int oracle_decode_fp8(const uint16_t* q_bf16, const uint8_t* ckv_pool,
                      int64_t ckv_stride, const uint8_t* kpe_pool,
                      int64_t kpe_stride, int64_t num_slots,
                      const int32_t* kv_indptr, const int32_t* kv_indices,
                      const int32_t* seq_lens, int32_t B, int32_t H,
                      int32_t page_size, double k_scale, double softmax_scale,
                      double* o, double* lse, double* p, int64_t p_stride,
                      int nthreads) {
    return decode_common(0, q_bf16, ckv_pool, ckv_stride, kpe_pool, kpe_stride,
                         num_slots, kv_indptr, kv_indices, seq_lens, B, H,
                         page_size, k_scale, softmax_scale, o, lse, p, p_stride,
                         nthreads);
}

/* Same attention over BF16 pool rows (the cast-then-attend baselines); the
 * row values are multiplied by k_scale exactly as E4M3 rows are. */
int oracle_decode_bf16(const uint16_t* q_bf16, const uint16_t* ckv_pool,
                       int64_t ckv_stride_bytes, const uint16_t* kpe_pool,
                       int64_t kpe_stride_bytes, int64_t num_slots,
                       const int32_t* kv_indptr, const int32_t* kv_indices,
                       const int32_t* seq_lens, int32_t B, int32_t H,
                       int32_t page_size, double k_scale, double softmax_scale,
                       double* o, double* lse, double* p, int64_t p_stride,
                       int nthreads) {
    return decode_common(1, q_bf16, ckv_pool, ckv_stride_bytes, kpe_pool,
                         kpe_stride_bytes, num_slots, kv_indptr, kv_indices,
                         seq_lens, B, H, page_size, k_scale, softmax_scale, o,
                         lse, p, p_stride, nthreads);
}

/* Causal extend (prefill with a cached prefix) over E4M3 pool rows.
 *
 * [P1] "Step 3: Source Validation", CastFromFP8: on every extend step the
 * prefill attention reads the request's whole cached history, which the FP8
 * configuration first casts back to BF16; "From Attribution to Optimization
 * Targets" names the fix, a prefill attention that reads the FP8 cache
 * itself.  The pages do not write the extend attention out; the reading used
 * here is the usual causal one, in the same latent (576-channel query, 512-
 * channel value) form as decode:
 *  - request b has q_len_b = qo_indptr[b+1] - qo_indptr[b] new tokens, whose
 *    query rows are rows qo_indptr[b] .. qo_indptr[b+1]-1 of q; they are
 *    already in the cache (the store precedes attention), so its context
 *    L_b = seq_lens[b] counts them, and 0 <= q_len_b <= L_b;
 *  - new token i (0-based) sits at sequence position L_b - q_len_b + i and
 *    attends to the tokens at positions 0 .. L_b - q_len_b + i, inclusive:
 *    the decode attention above over the first L_b - q_len_b + i + 1 tokens.
 * q: BF16 bits [n_q][H][576] (contiguous, n_q = qo_indptr[B]); o: [n_q][H][512];
 * lse: [n_q][H].  Returns -1 when a q_len is negative or above its context,
 * a page table is too short, or a slot is outside the pool; else 0. */
int oracle_extend_fp8(const uint16_t* q_bf16, const uint8_t* ckv_pool,
                      int64_t ckv_stride, const uint8_t* kpe_pool,
                      int64_t kpe_stride, int64_t num_slots,
                      const int32_t* qo_indptr, const int32_t* kv_indptr,
                      const int32_t* kv_indices, const int32_t* seq_lens,
                      int32_t B, int32_t H, int32_t page_size, double k_scale,
                      double softmax_scale, double* o, double* lse, int nthreads) {
    if (qo_indptr[0] != 0) return -1;
    for (int32_t b = 0; b < B; ++b) {
        int64_t L = seq_lens[b];
        int64_t q_len = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
        int64_t pages = kv_indptr[b + 1] - kv_indptr[b];
        if (L < 0 || q_len < 0 || q_len > L || pages * page_size < L) return -1;
        for (int64_t t = 0; t < L; ++t) {
            int64_t s = token_slot(kv_indices + kv_indptr[b], t, page_size);
            if (s < 0 || s >= num_slots) return -1;
        }
    }
    const int64_t n_q = qo_indptr[B];
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    /* one (query token, head) pair per iteration */
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t nh = 0; nh < n_q * H; ++nh) {
        int64_t n = nh / H;
        int32_t h = (int32_t)(nh % H);
        int32_t b = 0;
        while (qo_indptr[b + 1] <= n) ++b;
        int64_t q_len = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
        int64_t i = n - qo_indptr[b];
        int64_t visible = (int64_t)seq_lens[b] - q_len + i + 1;
        const int32_t* pages = kv_indices + kv_indptr[b];
        double qh[D_ALL];
        for (int d = 0; d < D_ALL; ++d)
            qh[d] = bf16_to_float(q_bf16[(n * H + h) * D_ALL + d]);
        double* k = (double*)malloc(sizeof(double) * (size_t)visible * D_ALL);
        double* s_buf = (double*)malloc(sizeof(double) * (size_t)visible);
        for (int64_t t = 0; t < visible; ++t) {
            int64_t slot = token_slot(pages, t, page_size);
            for (int d = 0; d < D_CKV; ++d)
                k[t * D_ALL + d] = pool_value(0, ckv_pool, ckv_stride, slot, d, k_scale);
            for (int d = 0; d < D_KPE; ++d)
                k[t * D_ALL + D_CKV + d] = pool_value(0, kpe_pool, kpe_stride, slot, d, k_scale);
        }
        attention_one_request(qh, k, visible, 1, softmax_scale, o + (n * H + h) * D_CKV,
                              lse + n * H + h, NULL, s_buf);
        free(k);
        free(s_buf);
    }
    return 0;
}

/* The attention core alone, on explicit fp64 rows: q [H][576], k [L][576]. */
void oracle_attention_f64(const double* q, const double* k, int64_t L, int32_t H,
                          double softmax_scale, double* o, double* lse, double* p) {
    double* s_buf = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    for (int32_t h = 0; h < H; ++h)
        attention_one_request(q + (int64_t)h * D_ALL, k, L, 1, softmax_scale,
                              o + (int64_t)h * D_CKV, lse + h,
                              p ? p + (int64_t)h * L : NULL, s_buf);
    free(s_buf);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
