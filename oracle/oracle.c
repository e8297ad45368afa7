/*
 * oracle.c -- plain, slow, fp64 CPU reference for paged grouped-query attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file; only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (page titles; sections cited as [P1 §x.y] etc.):
 *   [P1] "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎，C++/CUDA 实现性能追平 98%"
 *        (a from-scratch Qwen3-8B inference engine in C++/CUDA)
 *   [P2] "从零手搓AI推理引擎：避开调包陷阱的工程实践指南"
 *        (hand-building an inference engine: engineering practice guide)
 *   [P3] "从零搭建AI工程能力：手写KV Cache与动态批处理实战"
 *        (hand-writing a KV cache and dynamic batching)
 *
 * What is computed (the plain definition, no tiling, no online softmax, no splits):
 *
 *   attention = softmax(Q K^T / sqrt(d)) V                              [P2 §2.2]
 *   with the max subtracted before exponentiation                       [P2 §2.2]
 *   a query sees only itself and earlier positions (causal)             [P2 §2.2]
 *   query head h reads KV group g = h / (Hq / Hkv)                      [P1 §4.4.2]
 *   KV lives in fixed 256-token blocks filled in order; token j of a
 *   sequence is slot j % 256 of block block_table[j / 256]              [P1 §4.3.1]
 *   new K/V are appended to the cache before attention runs            [P3 §4.2]
 *
 * For sequence s with q_len = cu_q_lens[s+1] - cu_q_lens[s] new tokens and total
 * context seq_lens[s] (which already counts the new tokens), new token i sits at
 * absolute position p = seq_lens[s] - q_len + i and attends to keys 0..p.  A decode
 * step is the case q_len = 1 (p = seq_len - 1); a chunked prefill is q_len > 1 with
 * earlier context in the cache.  Scores, softmax, the weighted sum and the
 * log-sum-exp are all evaluated in double precision on the exact bf16 input values.
 *
 * Memory layouts (row-major, all contiguous):
 *   q        [total_tokens][Hq][D]                 bf16 bit patterns (uint16)
 *   k_pool   [num_blocks][block_size][Hkv][D]      bf16 bit patterns
 *   v_pool   same as k_pool
 *   out      [total_tokens][Hq][D]                 double
 *   lse      [total_tokens][Hq]                    double (natural log)
 *   block_table [num_seqs][max_blocks_per_seq]     int32
 * The 8-bit cache (E4M3 codes with one fp32 scale per row; its definition is given at
 * oracle_kv_append_fp8 below):
 *   k_codes  [num_blocks][block_size][Hkv][D]      uint8, v_codes likewise
 *   k_scale  [num_blocks][Hkv][block_size]         float, v_scale likewise
 *
 * The merged Q/K/V projection (its definition is given at oracle_qkv_project below):
 *   x        [tokens][hidden]                      bf16 bit patterns
 *   w        [n_out][hidden]                       bf16 bit patterns (a linear layer's weight)
 *   y        [tokens][n_out]                       double
 *
 * Rotary position embedding of q and k heads (not on the pages; RoFormer's definition,
 * given at oracle_rope below) acts on the projection's output in place, and so does the
 * per-head RMS normalisation of q and k (QK-norm; not on the pages either, defined at
 * oracle_rms_norm_heads below).
 *
 * Functions return 0 on success and a negative code on inconsistent input.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the top half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* Sequence that owns new-token row t: the s with cu[s] <= t < cu[s+1]. */
static int owner_sequence(const int32_t *cu_q_lens, int num_seqs, int t)
{
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (cu_q_lens[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

static int check_common(const int32_t *block_table, int max_blocks_per_seq, int num_blocks,
                        const int32_t *cu_q_lens, const int32_t *seq_lens, int num_seqs,
                        int block_size)
{
    if (num_seqs < 0 || max_blocks_per_seq < 0 || num_blocks < 0 || block_size <= 0) return -1;
    if (num_seqs > 0 && cu_q_lens[0] != 0) return -2;
    for (int s = 0; s < num_seqs; ++s) {
        int q_len = cu_q_lens[s + 1] - cu_q_lens[s];
        if (q_len < 0) return -3;
        if (q_len == 0) continue;
        if (seq_lens[s] < q_len) return -4;
        int nblk = (seq_lens[s] + block_size - 1) / block_size;
        if (nblk > max_blocks_per_seq) return -5;
        for (int j = 0; j < nblk; ++j) {
            int b = block_table[(size_t)s * max_blocks_per_seq + j];
            if (b < 0 || b >= num_blocks) return -6;
        }
    }
    return 0;
}

/*
 * Append: write the new K/V rows of every sequence into their cache slots
 * [P1 §4.3.1, KVBlockManager::append; P3 §4.2].
 * k_new, v_new: [total_tokens][Hkv][D] bf16 bits, rows grouped by sequence via cu_q_lens.
 */
int oracle_kv_append(uint16_t *k_pool, uint16_t *v_pool,
                     const uint16_t *k_new, const uint16_t *v_new,
                     const int32_t *block_table, int max_blocks_per_seq, int num_blocks,
                     const int32_t *cu_q_lens, const int32_t *seq_lens, int num_seqs,
                     int num_kv_heads, int head_dim, int block_size)
{
    int rc = check_common(block_table, max_blocks_per_seq, num_blocks, cu_q_lens, seq_lens,
                          num_seqs, block_size);
    if (rc) return rc;
    const size_t row = (size_t)num_kv_heads * head_dim; /* elements per token */
    for (int s = 0; s < num_seqs; ++s) {
        int q_len = cu_q_lens[s + 1] - cu_q_lens[s];
        for (int i = 0; i < q_len; ++i) {
            int t = cu_q_lens[s] + i;
            int p = seq_lens[s] - q_len + i;            /* absolute position */
            int blk = block_table[(size_t)s * max_blocks_per_seq + p / block_size];
            int slot = p % block_size;
            size_t dst = ((size_t)blk * block_size + slot) * row;
            for (size_t e = 0; e < row; ++e) {
                k_pool[dst + e] = k_new[(size_t)t * row + e];
                v_pool[dst + e] = v_new[(size_t)t * row + e];
            }
        }
    }
    return 0;
}

/*
 * The KV cache an attention call reads: the bf16 pools, or the 8-bit cache (codes and
 * row scales, see below).  Exactly one of the two pairs is set.
 */
typedef struct {
    const uint16_t *k_pool, *v_pool;     /* bf16 [num_blocks][block_size][Hkv][D] */
    const uint8_t *k_codes, *v_codes;    /* E4M3 [num_blocks][block_size][Hkv][D] */
    const float *k_scale, *v_scale;      /* [num_blocks][Hkv][block_size] */
    int num_kv_heads, head_dim, block_size;
} kv_cache;

static double e4m3_to_double(uint8_t c);

/* Element offset of the row of KV head g for token j (block bt[j/bs], slot j%bs). */
static size_t kv_row(const kv_cache *c, const int32_t *bt, int j, int g)
{
    return (((size_t)bt[j / c->block_size] * c->block_size + j % c->block_size) * c->num_kv_heads + g)
           * c->head_dim;
}

/* The row's scale in the 8-bit cache; the bf16 cache has none (1). */
static double kv_row_scale(const kv_cache *c, const float *scales, const int32_t *bt, int j, int g)
{
    if (!scales) return 1.0;
    return (double)scales[((size_t)bt[j / c->block_size] * c->num_kv_heads + g) * c->block_size
                          + (size_t)(j % c->block_size)];
}

/* Element d of the row at offset base: the bf16 value, or code * row scale. */
static double kv_elem(const uint16_t *pool, const uint8_t *codes, size_t base, int d, double row_scale)
{
    return pool ? bf16_to_double(pool[base + d]) : e4m3_to_double(codes[base + d]) * row_scale;
}

/*
 * One output row: query token t, query head h.  Writes out_row[0..D) and *lse_out.
 * scores: caller-provided scratch of at least (p + 1) doubles.
 */
static void attend_one(double *out_row, double *lse_out, double *scores,
                       const uint16_t *q, const kv_cache *c,
                       const int32_t *block_table, int max_blocks_per_seq,
                       const int32_t *cu_q_lens, const int32_t *seq_lens, int num_seqs,
                       int num_q_heads, double scale, int t, int h)
{
    const int num_kv_heads = c->num_kv_heads, head_dim = c->head_dim;
    int s = owner_sequence(cu_q_lens, num_seqs, t);
    int q_len = cu_q_lens[s + 1] - cu_q_lens[s];
    int i = t - cu_q_lens[s];
    int p = seq_lens[s] - q_len + i;                    /* this query's absolute position */
    int g = h / (num_q_heads / num_kv_heads);           /* GQA: consecutive q-heads share a group */
    const uint16_t *qrow = q + ((size_t)t * num_q_heads + h) * head_dim;
    const int32_t *bt = block_table + (size_t)s * max_blocks_per_seq;

    /* x_j = scale * <q, k_j> for every visible key j <= p (causal, diagonal included) */
    double m = -INFINITY;
    for (int j = 0; j <= p; ++j) {
        size_t base = kv_row(c, bt, j, g);
        double ks = kv_row_scale(c, c->k_scale, bt, j, g);
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += bf16_to_double(qrow[d]) * kv_elem(c->k_pool, c->k_codes, base, d, ks);
        scores[j] = scale * dot;
        if (scores[j] > m) m = scores[j];
    }
    /* softmax weights e^{x_j - m} / sum, then the weighted sum of V rows */
    double denom = 0.0;
    for (int j = 0; j <= p; ++j) {
        scores[j] = exp(scores[j] - m);
        denom += scores[j];
    }
    for (int d = 0; d < head_dim; ++d) out_row[d] = 0.0;
    for (int j = 0; j <= p; ++j) {
        size_t base = kv_row(c, bt, j, g);
        double vs = kv_row_scale(c, c->v_scale, bt, j, g);
        double w = scores[j];
        for (int d = 0; d < head_dim; ++d) out_row[d] += w * kv_elem(c->v_pool, c->v_codes, base, d, vs);
    }
    for (int d = 0; d < head_dim; ++d) out_row[d] /= denom;
    *lse_out = m + log(denom);
}

/* Rows (token, head) over either cache, spread over OpenMP threads. */
static int attention_rows(double *out, double *lse, const int32_t *row_tokens, const int32_t *row_heads,
                          int n, const uint16_t *q, const kv_cache *c,
                          const int32_t *block_table, int max_blocks_per_seq, int num_blocks,
                          const int32_t *cu_q_lens, const int32_t *seq_lens, int num_seqs,
                          int num_q_heads, double scale, int num_threads)
{
    if (num_q_heads <= 0 || c->num_kv_heads <= 0 || num_q_heads % c->num_kv_heads) return -10;
    int rc = check_common(block_table, max_blocks_per_seq, num_blocks, cu_q_lens, seq_lens,
                          num_seqs, c->block_size);
    if (rc) return rc;
    int total_tokens = num_seqs > 0 ? cu_q_lens[num_seqs] : 0;
    int max_ctx = 1;
    for (int s = 0; s < num_seqs; ++s)
        if (cu_q_lens[s + 1] > cu_q_lens[s] && seq_lens[s] > max_ctx) max_ctx = seq_lens[s];
    for (int r = 0; r < n; ++r)
        if (row_tokens[r] < 0 || row_tokens[r] >= total_tokens || row_heads[r] < 0 ||
            row_heads[r] >= num_q_heads)
            return -11;

    int failed = 0;
#ifdef _OPENMP
    /* a thread count for this region only: the process-wide default stays as it was */
    const int team = num_threads > 0 ? num_threads : omp_get_max_threads();
#pragma omp parallel num_threads(team)
#endif
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)max_ctx);
        if (!scores) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int r = 0; r < n; ++r) {
            if (!scores) continue;
            attend_one(out + (size_t)r * c->head_dim, lse + r, scores, q, c, block_table,
                       max_blocks_per_seq, cu_q_lens, seq_lens, num_seqs, num_q_heads, scale,
                       row_tokens[r], row_heads[r]);
        }
        free(scores);
    }
    return failed ? -12 : 0;
}

/* Every row of every new token: out [total_tokens][Hq][D], lse [total_tokens][Hq]. */
static int attention_all(double *out, double *lse, const uint16_t *q, const kv_cache *c,
                         const int32_t *block_table, int max_blocks_per_seq, int num_blocks,
                         const int32_t *cu_q_lens, const int32_t *seq_lens, int num_seqs,
                         int num_q_heads, double scale, int num_threads)
{
    int total_tokens = num_seqs > 0 ? cu_q_lens[num_seqs] : 0;
    int n = total_tokens * num_q_heads;
    if (n == 0) return 0;
    int32_t *tok = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int32_t *hd = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    if (!tok || !hd) { free(tok); free(hd); return -12; }
    for (int r = 0; r < n; ++r) { tok[r] = r / num_q_heads; hd[r] = r % num_q_heads; }
    int rc = attention_rows(out, lse, tok, hd, n, q, c, block_table, max_blocks_per_seq, num_blocks,
                            cu_q_lens, seq_lens, num_seqs, num_q_heads, scale, num_threads);
    free(tok);
    free(hd);
    return rc;
}

/*
 * Attention for a list of (token, head) output rows over the bf16 cache.
 * out: [n][D], lse: [n].  num_threads > 0 fixes the OpenMP thread count (0 = default).
 */
int oracle_attention_rows(double *out, double *lse,
                          const int32_t *row_tokens, const int32_t *row_heads, int n,
                          const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                          const int32_t *block_table, int max_blocks_per_seq, int num_blocks,
                          const int32_t *cu_q_lens, const int32_t *seq_lens, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          double scale, int num_threads)
{
    kv_cache c = {k_pool, v_pool, NULL, NULL, NULL, NULL, num_kv_heads, head_dim, block_size};
    return attention_rows(out, lse, row_tokens, row_heads, n, q, &c, block_table, max_blocks_per_seq,
                          num_blocks, cu_q_lens, seq_lens, num_seqs, num_q_heads, scale, num_threads);
}

/* Every row of every new token over the bf16 cache. */
int oracle_paged_attention(double *out, double *lse,
                           const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                           const int32_t *block_table, int max_blocks_per_seq, int num_blocks,
                           const int32_t *cu_q_lens, const int32_t *seq_lens, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           double scale, int num_threads)
{
    kv_cache c = {k_pool, v_pool, NULL, NULL, NULL, NULL, num_kv_heads, head_dim, block_size};
    return attention_all(out, lse, q, &c, block_table, max_blocks_per_seq, num_blocks, cu_q_lens,
                         seq_lens, num_seqs, num_q_heads, scale, num_threads);
}

/* ======================================================================== 8-bit KV cache
 *
 * [P3 §3.2]: keeping the KV cache in 8 bits instead of 16 halves its memory (the page
 * quantises to INT8 and warns that the error accumulates over decode steps).  Reading
 * taken here: the 8-bit code is the E4M3 float of the OCP FP8 format, with one fp32
 * scale per (token, KV head) row.
 *
 * E4M3: bit 7 sign, bits 6..3 exponent field e (bias 7), bits 2..0 mantissa m.
 *   e = 0:            value (-1)^s * m * 2^-9          (zero and subnormals)
 *   1 <= e <= 15:     value (-1)^s * (1 + m/8) * 2^(e-7)
 *   e = 15, m = 7:    NaN (there is no infinity); the largest finite value is 448.
 * Quantising a row x[0..D) of new K (or V) for one KV head:
 *   amax  = max_d |x_d|                                   (exact)
 *   scale = amax / 448 in fp32 (round to nearest even), or 1 when amax == 0
 *   c_d   = E4M3(x_d / scale): the fp32 quotient rounded to the nearest E4M3 value
 *           (ties to even mantissa); magnitudes beyond 448 become 448
 * and the stored row stands for c_d * scale.
 *
 * Layouts: codes  [num_blocks][block_size][Hkv][D] uint8 (as the bf16 pools)
 *          scales [num_blocks][Hkv][block_size] float (one row of scales per block and head)
 */
static double e4m3_to_double(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

static uint8_t e4m3_from_float(float x)
{
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a > 448.0) return sign | 0x7E;                    /* saturate to the largest finite */
    if (a < ldexp(1.0, -6)) {                             /* subnormal range: quantum 2^-9 */
        double m = nearbyint(a * 512.0);                  /* ties to even (default mode) */
        return sign | (uint8_t)m;                         /* m = 8 is 2^-6, code 0x08: correct */
    }
    int k;
    frexp(a, &k);                                         /* a = f * 2^k, f in [0.5, 1) */
    int e = k - 1;                                        /* a in [2^e, 2^(e+1)) */
    double m = nearbyint(ldexp(a, 3 - e));                /* 8 <= m <= 16, exact scaling */
    if (m == 16.0) { m = 8.0; e += 1; }
    if (e > 8 || (e == 8 && m > 14.0)) return sign | 0x7E;
    return sign | (uint8_t)(((e + 7) << 3) | ((int)m - 8));
}

/* Element-wise codec, exposed for the oracle's own pins. */
void oracle_e4m3_encode(const float *x, uint8_t *c, long n)
{
    for (long i = 0; i < n; ++i) c[i] = e4m3_from_float(x[i]);
}

void oracle_e4m3_decode(const uint8_t *c, double *x, long n)
{
    for (long i = 0; i < n; ++i) x[i] = e4m3_to_double(c[i]);
}

static float bf16_to_float(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return f;
}

/* Quantise one row of D bf16 values into D codes and its scale. */
static void quantise_row(const uint16_t *x, int d_len, uint8_t *codes, float *scale_out)
{
    float amax = 0.0f;
    for (int d = 0; d < d_len; ++d) {
        float v = fabsf(bf16_to_float(x[d]));
        if (v > amax) amax = v;
    }
    float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int d = 0; d < d_len; ++d) {
        float q = bf16_to_float(x[d]) / scale;
        codes[d] = e4m3_from_float(q);
    }
    *scale_out = scale;
}

/*
 * Append into the 8-bit cache: the placement of oracle_kv_append [P1 §4.3.1] with each
 * (token, KV head) row quantised as above.
 */
int oracle_kv_append_fp8(uint8_t *k_codes, uint8_t *v_codes, float *k_scale, float *v_scale,
                         const uint16_t *k_new, const uint16_t *v_new,
                         const int32_t *block_table, int max_blocks_per_seq, int num_blocks,
                         const int32_t *cu_q_lens, const int32_t *seq_lens, int num_seqs,
                         int num_kv_heads, int head_dim, int block_size)
{
    int rc = check_common(block_table, max_blocks_per_seq, num_blocks, cu_q_lens, seq_lens,
                          num_seqs, block_size);
    if (rc) return rc;
    for (int s = 0; s < num_seqs; ++s) {
        int q_len = cu_q_lens[s + 1] - cu_q_lens[s];
        for (int i = 0; i < q_len; ++i) {
            int t = cu_q_lens[s] + i;
            int p = seq_lens[s] - q_len + i;
            int blk = block_table[(size_t)s * max_blocks_per_seq + p / block_size];
            int slot = p % block_size;
            for (int g = 0; g < num_kv_heads; ++g) {
                size_t src = ((size_t)t * num_kv_heads + g) * head_dim;
                size_t dst = (((size_t)blk * block_size + slot) * num_kv_heads + g) * head_dim;
                size_t sc = ((size_t)blk * num_kv_heads + g) * block_size + slot;
                quantise_row(k_new + src, head_dim, k_codes + dst, k_scale + sc);
                quantise_row(v_new + src, head_dim, v_codes + dst, v_scale + sc);
            }
        }
    }
    return 0;
}

/* Every row of every new token over the 8-bit cache (K/V element = code * row scale). */
int oracle_paged_attention_fp8(double *out, double *lse,
                               const uint16_t *q, const uint8_t *k_codes, const uint8_t *v_codes,
                               const float *k_scale, const float *v_scale,
                               const int32_t *block_table, int max_blocks_per_seq, int num_blocks,
                               const int32_t *cu_q_lens, const int32_t *seq_lens, int num_seqs,
                               int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                               double scale, int num_threads)
{
    kv_cache c = {NULL, NULL, k_codes, v_codes, k_scale, v_scale, num_kv_heads, head_dim, block_size};
    return attention_all(out, lse, q, &c, block_table, max_blocks_per_seq, num_blocks, cu_q_lens,
                         seq_lens, num_seqs, num_q_heads, scale, num_threads);
}

/*
 * The merged Q/K/V projection [P1 §4.4.3 QKV fusion]: the q, k and v weights stacked
 * into one matrix, one product, the output sliced by columns.  For each listed token
 * row t (rows[r], or r itself when rows is NULL) and output column n:
 *     y[r][n] = sum_k x[t][k] * w[n][k]
 * in double precision on the exact bf16 values, summed in order of k.
 */
int oracle_qkv_project(double *y, const uint16_t *x, const uint16_t *w, const int32_t *rows, int n_rows,
                       int tokens, int hidden, int n_out, int num_threads)
{
    if (n_rows < 0 || tokens < 0 || hidden < 1 || n_out < 1) return -1;
    for (int r = 0; r < n_rows; ++r)
        if (rows && (rows[r] < 0 || rows[r] >= tokens)) return -2;
#ifdef _OPENMP
    const int team = num_threads > 0 ? num_threads : omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(team)
#endif
    for (long rn = 0; rn < (long)n_rows * n_out; ++rn) {
        const int r = (int)(rn / n_out), n = (int)(rn % n_out);
        const int t = rows ? rows[r] : r;
        double acc = 0.0;
        for (int k = 0; k < hidden; ++k)
            acc += bf16_to_double(x[(size_t)t * hidden + k]) * bf16_to_double(w[(size_t)n * hidden + k]);
        y[(size_t)r * n_out + n] = acc;
    }
    return 0;
}

/*
 * Round doubles to the nearest bf16 (ties to even), as bit patterns: a result that
 * fits the bf16 grid exactly, with the format's subnormals and overflow to infinity.
 * bf16 keeps 8 significant bits; a value in [2^e, 2^(e+1)) with e >= -126 is a
 * multiple of 2^(e-7), below 2^-126 a multiple of 2^-133.
 */
void oracle_bf16_round(const double *v, uint16_t *out, long n)
{
    for (long i = 0; i < n; ++i) {
        const double x = v[i];
        if (isnan(x)) { out[i] = 0x7FC0; continue; }
        const uint16_t sign = signbit(x) ? 0x8000 : 0;
        const double a = fabs(x);
        if (a == 0.0) { out[i] = sign; continue; }
        int e;
        frexp(a, &e);              /* a = m * 2^e, m in [0.5, 1): a in [2^(e-1), 2^e) */
        int lo = e - 1;
        if (lo < -126) lo = -126;
        const double quantum = ldexp(1.0, lo - 7);
        double m = floor(a / quantum);   /* a / quantum is exact: a power-of-two scaling */
        const double frac = a / quantum - m;
        if (frac > 0.5 || (frac == 0.5 && fmod(m, 2.0) != 0.0)) m += 1.0;
        const double r = m * quantum;
        if (r >= 0x1p128) { out[i] = sign | 0x7F80; continue; }   /* beyond the largest finite */
        /* r is on the bf16 grid, hence exactly a float whose low 16 bits are zero */
        const float f = (float)r;
        uint32_t bits;
        memcpy(&bits, &f, sizeof bits);
        out[i] = sign | (uint16_t)(bits >> 16);
    }
}

/*
 * Absolute position of every new token: new token i of sequence s sits at
 * p = seq_lens[s] - q_len + i, the rule the append and the attention use [P1 §4.3.1;
 * P3 §3.3 chunked prefill].  pos: [cu_q_lens[num_seqs]].
 */
int oracle_token_positions(int32_t *pos, const int32_t *cu_q_lens, const int32_t *seq_lens, int num_seqs)
{
    if (num_seqs < 0 || (num_seqs > 0 && cu_q_lens[0] != 0)) return -1;
    for (int s = 0; s < num_seqs; ++s) {
        int q_len = cu_q_lens[s + 1] - cu_q_lens[s];
        if (q_len < 0 || seq_lens[s] < q_len) return -2;
        for (int i = 0; i < q_len; ++i) pos[cu_q_lens[s] + i] = seq_lens[s] - q_len + i;
    }
    return 0;
}

/*
 * Rotary position embedding.  The pages do not define it; the definition here is that of
 * RoFormer (Su et al., 2021, "RoFormer: Enhanced Transformer with Rotary Position
 * Embedding"), in the pairing Qwen3 and the Llama family use ("rotate half"): in a head
 * vector of D values, dims i and i + D/2 (0 <= i < D/2) form a pair, turned by the angle
 * p * theta^(-2i/D) at position p:
 *     x'[i]       = x[i] cos(a) - x[i + D/2] sin(a)
 *     x'[i + D/2] = x[i + D/2] cos(a) + x[i] sin(a),      a = p * theta^(-2i/D)
 * (Qwen3: theta = 1 000 000).  y: [tokens][row_stride] doubles; the n_heads head vectors
 * of head_dim values from column first_col on are rotated in place, token t at
 * positions[t].  Double precision throughout.
 */
int oracle_rope(double *y, int tokens, int row_stride, int first_col, int n_heads, int head_dim,
                const int32_t *positions, double theta)
{
    if (tokens < 0 || head_dim < 2 || head_dim % 2 || n_heads < 0 || first_col < 0 ||
        first_col + n_heads * head_dim > row_stride || !(theta > 1.0))
        return -1;
    const int half = head_dim / 2;
    for (int t = 0; t < tokens; ++t) {
        for (int h = 0; h < n_heads; ++h) {
            double *v = y + (size_t)t * row_stride + first_col + (size_t)h * head_dim;
            for (int i = 0; i < half; ++i) {
                const double a = (double)positions[t] * pow(theta, -2.0 * i / head_dim);
                const double c = cos(a), s = sin(a);
                const double lo = v[i], hi = v[i + half];
                v[i] = lo * c - hi * s;
                v[i + half] = hi * c + lo * s;
            }
        }
    }
    return 0;
}

/*
 * Per-head RMS normalisation (QK-norm).  The pages do not define it; Qwen3 normalises each
 * q and k head before the rotary embedding (the Qwen3 technical report, 2025, §2: QK-Norm)
 * with RMSNorm (Zhang and Sennrich, 2019, "Root Mean Square Layer Normalization", §3): a
 * head vector x of D values, divided by its root mean square, times a learned gain g of D
 * values, with Qwen3's eps inside the square root (its configuration: 1e-6):
 *     y[d] = g[d] * x[d] / sqrt((x[0]^2 + ... + x[D-1]^2) / D + eps)
 * y: [tokens][row_stride] doubles; the n_heads head vectors of head_dim values from column
 * first_col on are normalised in place, each on its own.  gain: head_dim bf16 bit patterns
 * (one gain for all the heads).  Double precision throughout.
 */
int oracle_rms_norm_heads(double *y, int tokens, int row_stride, int first_col, int n_heads, int head_dim,
                          const uint16_t *gain, double eps)
{
    if (tokens < 0 || head_dim < 1 || n_heads < 0 || first_col < 0 ||
        first_col + n_heads * head_dim > row_stride || !(eps >= 0.0))
        return -1;
    for (int t = 0; t < tokens; ++t) {
        for (int h = 0; h < n_heads; ++h) {
            double *v = y + (size_t)t * row_stride + first_col + (size_t)h * head_dim;
            double sum_sq = 0.0;
            for (int d = 0; d < head_dim; ++d) sum_sq += v[d] * v[d];
            const double rms = sqrt(sum_sq / head_dim + eps);
            for (int d = 0; d < head_dim; ++d) v[d] = bf16_to_double(gain[d]) * v[d] / rms;
        }
    }
    return 0;
}

/* Threads the OpenMP runtime would use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
