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
 * One output row: query token t, query head h.  Writes out_row[0..D) and *lse_out.
 * scores: caller-provided scratch of at least (p + 1) doubles.
 */
static void attend_one(double *out_row, double *lse_out, double *scores,
                       const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                       const int32_t *block_table, int max_blocks_per_seq,
                       const int32_t *cu_q_lens, const int32_t *seq_lens, int num_seqs,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       double scale, int t, int h)
{
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
        size_t base = (((size_t)bt[j / block_size] * block_size + j % block_size) * num_kv_heads + g)
                      * head_dim;
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += bf16_to_double(qrow[d]) * bf16_to_double(k_pool[base + d]);
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
        size_t base = (((size_t)bt[j / block_size] * block_size + j % block_size) * num_kv_heads + g)
                      * head_dim;
        double w = scores[j];
        for (int d = 0; d < head_dim; ++d) out_row[d] += w * bf16_to_double(v_pool[base + d]);
    }
    for (int d = 0; d < head_dim; ++d) out_row[d] /= denom;
    *lse_out = m + log(denom);
}

/*
 * Attention for a list of (token, head) output rows.  out: [n][D], lse: [n].
 * The rows are independent; they are distributed over OpenMP threads when
 * num_threads > 0 (0 = the OpenMP default).
 */
int oracle_attention_rows(double *out, double *lse,
                          const int32_t *row_tokens, const int32_t *row_heads, int n,
                          const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                          const int32_t *block_table, int max_blocks_per_seq, int num_blocks,
                          const int32_t *cu_q_lens, const int32_t *seq_lens, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          double scale, int num_threads)
{
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return -10;
    int rc = check_common(block_table, max_blocks_per_seq, num_blocks, cu_q_lens, seq_lens,
                          num_seqs, block_size);
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
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel
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
            attend_one(out + (size_t)r * head_dim, lse + r, scores, q, k_pool, v_pool,
                       block_table, max_blocks_per_seq, cu_q_lens, seq_lens, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, scale,
                       row_tokens[r], row_heads[r]);
        }
        free(scores);
    }
    return failed ? -12 : 0;
}

/* Every row of every new token: out [total_tokens][Hq][D], lse [total_tokens][Hq]. */
int oracle_paged_attention(double *out, double *lse,
                           const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                           const int32_t *block_table, int max_blocks_per_seq, int num_blocks,
                           const int32_t *cu_q_lens, const int32_t *seq_lens, int num_seqs,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           double scale, int num_threads)
{
    int total_tokens = num_seqs > 0 ? cu_q_lens[num_seqs] : 0;
    int n = total_tokens * num_q_heads;
    if (n == 0) return 0;
    int32_t *tok = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    int32_t *hd = (int32_t *)malloc(sizeof(int32_t) * (size_t)n);
    if (!tok || !hd) { free(tok); free(hd); return -12; }
    for (int r = 0; r < n; ++r) { tok[r] = r / num_q_heads; hd[r] = r % num_q_heads; }
    int rc = oracle_attention_rows(out, lse, tok, hd, n, q, k_pool, v_pool, block_table,
                                   max_blocks_per_seq, num_blocks, cu_q_lens, seq_lens, num_seqs,
                                   num_q_heads, num_kv_heads, head_dim, block_size, scale,
                                   num_threads);
    free(tok);
    free(hd);
    return rc;
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
