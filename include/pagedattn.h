/*
 * pagedattn.h -- C ABI of libpagedattn.so: grouped-query attention over a paged
 * KV cache on one GB300 (sm_103a).
 *
 * Sources (page titles; sections cited as [P1 §x.y] etc.):
 *   [P1] "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎，C++/CUDA 实现性能追平 98%"
 *   [P2] "从零手搓AI推理引擎：避开调包陷阱的工程实践指南"
 *   [P3] "从零搭建AI工程能力：手写KV Cache与动态批处理实战"
 *
 * The three compute calls are the per-layer attention work behind the engine's
 * Prefill / DecodeStep requests [P1 §4.1.2]:
 *   kv_append           writes the new tokens' K/V into their cache blocks
 *                       [P1 §4.3.1 KVBlockManager::append]
 *   paged_attn_decode   one query token per sequence over its whole cached context,
 *                       the four query heads of a KV group sharing each KV read
 *                       [P1 §4.4.2 gqa_decode_attn]
 *   paged_attn_prefill  causal attention of a chunk of new tokens over the earlier
 *                       context plus itself [P1 §4.4.1 flash_attn_prefill; P3 §3.3
 *                       chunked prefill]
 * and, before them, paged_qkv_append computes the new tokens' q, k and v in one merged
 * projection [P1 §4.4.3 QKV fusion] with k and v written straight into the cache.
 * The attention calls compute softmax(Q K^T * scale) V [P2 §2.2] with the causal rule "a
 * position sees itself and earlier positions" [P2 §2.2]; the caller appends before
 * attending, so a context length always counts the new tokens [P3 §4.2].
 *
 * Shapes.  Only {num_q_heads 32, num_kv_heads 8, head_dim 128, block_size 256} is
 * built; anything else returns PA_ERR_UNSUPPORTED.  Query head h reads KV head
 * h / 4 [P1 §4.4.2].  Token j of a sequence lives in slot j % 256 of physical block
 * block_table[s][j / 256] [P1 §4.3.1].
 *
 * Layouts (row-major, contiguous, device memory, 16-byte aligned):
 *   q, out        bf16 [tokens][32][128]
 *   k_new, v_new  bf16 [tokens][8][128]
 *   k_pool,v_pool bf16 [num_blocks][256][8][128]
 *   lse           fp32 [tokens][32], natural-log log-sum-exp of the scaled scores
 *   block_table   int32 [num_seqs][max_blocks_per_seq]
 *   seq_lens      int32 [num_seqs]     context length including the new tokens
 *   cu_q_lens     int32 [num_seqs + 1] offsets of each sequence's new tokens
 *
 * Ownership.  Every pointer is caller-owned device memory; the library allocates
 * nothing and keeps no per-call state outside the caller's workspace (except
 * paged_attn_decode_static, which uses a fixed array of its own instead).
 *
 * Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 * are asynchronous and stream-ordered; PA_OK means "validated and launched".  The
 * decode, prefill and projection kernels are launched as programmatic dependents of the
 * kernel before them on the stream: they may start before it has finished, and wait for
 * it before touching q, x, k_new, v_new, the pools, out or lse.  block_table, seq_lens and
 * cu_q_lens may be read earlier, so a kernel that writes them immediately before a
 * call must not let its dependents start early (griddepcontrol.launch_dependents).
 *
 * Errors.  Scalar arguments and pointers are checked on the host (PA_ERR_INVALID_ARG,
 * PA_ERR_UNSUPPORTED) before anything is launched.  Device arrays the host does not
 * read (block_table, seq_lens, cu_q_lens) are checked by the kernels: a block id
 * outside [0, num_blocks), a length outside its bound or an inconsistent cu_q_lens
 * makes the affected work skip its memory accesses and records PA_ERR_DEVICE in the
 * workspace error word; a bounded device wait that expires records PA_ERR_TIMEOUT.
 * Kernels never trap.  pa_check_error() reports and clears the word.
 *
 * Workspace.  Caller-allocated device memory of pa_workspace_bytes() bytes, zeroed
 * once by pa_workspace_init() (or cudaMemset to 0) before its first use.  It holds
 * the error word, split-K partial results and self-resetting counters.  One
 * workspace must not be used by two calls that may run at the same time.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* bad scalar argument, null or misaligned pointer */
    PA_ERR_UNSUPPORTED = 2, /* shape other than 32/8/128/256 */
    PA_ERR_CUDA = 3,        /* a CUDA runtime call failed */
    PA_ERR_DEVICE = 4,      /* a device-side check of block_table/seq_lens/cu_q_lens failed */
    PA_ERR_TIMEOUT = 5,     /* a bounded device wait expired */
    PA_ERR_WORKSPACE = 6    /* workspace smaller than pa_workspace_bytes() requires */
} pa_status;

typedef struct {
    int32_t num_q_heads;  /* 32 */
    int32_t num_kv_heads; /* 8 */
    int32_t head_dim;     /* 128 */
    int32_t block_size;   /* 256 */
} pa_shape;

/* Human-readable name of a status code (static string). */
const char *pa_status_string(pa_status status);

/* Library version as major*10000 + minor*100 + patch. */
int32_t pa_version(void);

/*
 * Workspace bytes enough for any of the three calls with up to max_batch sequences
 * and block tables max_blocks_per_seq wide.  Returns 0 for an unsupported shape or
 * non-positive sizes.
 */
size_t pa_workspace_bytes(pa_shape shape, int32_t max_batch, int32_t max_blocks_per_seq);

/* Zero a workspace on `stream` (asynchronous). */
pa_status pa_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/*
 * Synchronise `stream`, read the workspace error word, clear it and return its
 * status: PA_OK, PA_ERR_DEVICE or PA_ERR_TIMEOUT (PA_ERR_TIMEOUT wins when both
 * were recorded).  If detail is non-NULL it receives the raw word
 * (bit 0 device check, bit 1 timeout, bits 8.. the kind of device check).
 */
pa_status pa_check_error(void *workspace, void *stream, uint32_t *detail);

/*
 * kv_append: K/V of the new tokens into their cache slots [P1 §4.3.1].
 * For sequence s with q_len = cu_q_lens[s+1] - cu_q_lens[s], new token i (row
 * cu_q_lens[s] + i of k_new/v_new) goes to absolute position
 * p = seq_lens[s] - q_len + i, i.e. slot p % 256 of block block_table[s][p / 256].
 * Bit-exact copy; no other pool byte is written.  The blocks written must belong
 * to one sequence only, and no two new tokens may map to the same slot.
 *   total_tokens = cu_q_lens[num_seqs]; q_len 0 is allowed (nothing to write).
 */
pa_status kv_append(pa_shape shape, void *k_pool, void *v_pool,
                    const void *k_new, const void *v_new,
                    const int32_t *block_table, int32_t max_blocks_per_seq, int32_t num_blocks,
                    const int32_t *cu_q_lens, const int32_t *seq_lens, int32_t num_seqs,
                    int32_t total_tokens, void *workspace, size_t workspace_bytes,
                    void *stream);

/*
 * paged_qkv_append: the merged Q/K/V projection of the new tokens [P1 §4.4.3 QKV fusion:
 * one matrix product with the three weights stacked, output sliced into q, k, v], with
 * k and v written straight into their cache slots by the kv_append rule above (no
 * round trip of K/V through memory).  For token t (row t of x):
 *   y[n] = sum_k x[t][k] * w_qkv[n][k],  n = 0 .. 6143, fp32 accumulation, bf16 result;
 *   columns 0..4095 -> q_out[t][n / 128][n % 128];
 *   columns 4096..5119 -> K of KV head (n - 4096) / 128, dim n % 128, at the token's
 *   cache slot; columns 5120..6143 -> V likewise [P1 §4.4.2: 8 KV heads].
 * rope_theta > 1 applies the rotary position embedding to the 32 q heads and the 8 k heads
 * before the bf16 rounding (v is not rotated).  The pages define no position encoding; the
 * definition is RoFormer's (Su et al. 2021) in the pairing Qwen3 uses (Qwen3: theta = 1e6):
 * at the token's absolute position p = seq_len - q_len + i, dims d and d + 64 of a head
 * (d < 64) become
 *   y'[d] = y[d] cos(a) - y[d+64] sin(a),  y'[d+64] = y[d+64] cos(a) + y[d] sin(a),
 *   a = p * rope_theta^(-d/64),
 * in fp32 with the angle reduced to about 1e-6 rad.  rope_theta = 0 applies no rotation;
 * with a rotation max_blocks_per_seq * 256 must not exceed 2^24 (positions exact in fp32),
 * else PA_ERR_INVALID_ARG.  No per-head normalisation is applied (paged_qkv_append_qknorm
 * below applies it).
 *   x [total_tokens][hidden] bf16, hidden a multiple of 256 (4096 for Qwen3-8B);
 *   w_qkv [6144][hidden] bf16: rows 0-4095 the q weight, 4096-5119 k, 5120-6143 v, each
 *   [out][in] as a linear layer stores it; q_out [total_tokens][32][128] bf16.
 * Pools, block_table, cu_q_lens, seq_lens and the workspace as for kv_append; a token
 * whose block id is outside the pool gets no K/V write and records PA_ERR_DEVICE (its q
 * row is still written); a token whose sequence data are inconsistent gets no K/V write
 * either and, with a rotation, a NaN q row (its position is unknown).
 */
pa_status paged_qkv_append(pa_shape shape, int32_t hidden, float rope_theta, void *q_out, const void *x,
                           const void *w_qkv, void *k_pool, void *v_pool,
                           const int32_t *block_table, int32_t max_blocks_per_seq,
                           int32_t num_blocks, const int32_t *cu_q_lens,
                           const int32_t *seq_lens, int32_t num_seqs, int32_t total_tokens,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * paged_qkv_append_qknorm: paged_qkv_append with the per-head normalisation of q and k that
 * Qwen3 applies before the rotary embedding (QK-norm; the pages define none: RMSNorm,
 * Zhang and Sennrich 2019, §3).  The projection's q and k heads are rounded to bf16 (its
 * output format), then each 128-dim q head and k head x becomes
 *   y[d] = g[d] * x[d] / sqrt((x[0]^2 + ... + x[127]^2) / 128 + norm_eps)
 * in fp32, g = q_norm_weight for q heads and k_norm_weight for k heads; then, with
 * rope_theta > 1, y is rotated as above, and the result is rounded to bf16 into q_out and the
 * token's cache slot.  v is neither normalised nor rotated.  Qwen3: norm_eps = 1e-6.
 *   q_norm_weight, k_norm_weight: [128] bf16 device arrays, 16-byte aligned, read only;
 *   norm_eps: finite, >= 0.  Otherwise PA_ERR_INVALID_ARG.
 * Two launches on `stream` (the projection, then an in-place pass over the new q and k
 * rows); every other argument, layout, error and rule as paged_qkv_append.
 */
pa_status paged_qkv_append_qknorm(pa_shape shape, int32_t hidden, float rope_theta,
                                  const void *q_norm_weight, const void *k_norm_weight, float norm_eps,
                                  void *q_out, const void *x, const void *w_qkv, void *k_pool,
                                  void *v_pool, const int32_t *block_table, int32_t max_blocks_per_seq,
                                  int32_t num_blocks, const int32_t *cu_q_lens, const int32_t *seq_lens,
                                  int32_t num_seqs, int32_t total_tokens, void *workspace,
                                  size_t workspace_bytes, void *stream);

/*
 * paged_attn_decode: one query token per sequence [P1 §4.4.2].
 * out[b][h] = sum_{j < seq_lens[b]} softmax_j(scale * q[b][h] . K_b[j][h/4]) V_b[j][h/4]
 * where K_b[j] is slot j % 256 of block block_table[b][j / 256].  seq_lens[b] >= 1
 * counts the current token (appended before the call).  lse may be NULL.
 * The context is split over CTAs (split-K over KV blocks) and the partial results
 * are merged by log-sum-exp; the split depends only on batch, max_blocks_per_seq
 * and the device's SM count, never on the physical block ids.
 */
pa_status paged_attn_decode(pa_shape shape, void *out, float *lse, const void *q,
                            const void *k_pool, const void *v_pool,
                            const int32_t *block_table, int32_t max_blocks_per_seq,
                            int32_t num_blocks, const int32_t *seq_lens, int32_t batch,
                            float scale, void *workspace, size_t workspace_bytes, void *stream);

/*
 * As paged_attn_decode, with the split length fixed by the caller: split_tokens is
 * the number of context tokens one CTA handles (a positive multiple of 64), or 0
 * for the library's own choice.  Exposed for tuning and for split-invariance tests.
 * A split shorter than the library's choice needs more partial results than
 * pa_workspace_bytes() provides for: batch * 8 * ceil(max_blocks_per_seq * 256 /
 * split_tokens) entries of 2080 bytes past the fixed part; a smaller workspace
 * returns PA_ERR_WORKSPACE and launches nothing.
 */
pa_status paged_attn_decode_split(pa_shape shape, void *out, float *lse, const void *q,
                                  const void *k_pool, const void *v_pool,
                                  const int32_t *block_table, int32_t max_blocks_per_seq,
                                  int32_t num_blocks, const int32_t *seq_lens, int32_t batch,
                                  float scale, int32_t split_tokens, void *workspace,
                                  size_t workspace_bytes, void *stream);

/*
 * The 8-bit KV cache [P3 §3.2: storing the KV cache in 8 bits instead of 16 halves its
 * memory].  A K or V row (one token, one KV head) is 128 E4M3 codes (sign, 4 exponent
 * bits with bias 7, 3 mantissa bits; largest finite value 448) and one fp32 scale; the row
 * stands for code * scale.  Layouts (device memory, 16-byte aligned):
 *   k_codes, v_codes  uint8 [num_blocks][256][8][128]  (the bf16 pool layout, 1 byte a value)
 *   k_scale, v_scale  fp32  [num_blocks][8][256]        (one scale per row, slots contiguous)
 * A decode step then reads 264 bytes per token and KV head instead of 512.
 *
 * kv_append_fp8 quantises every new row: scale = amax / 448 in fp32 (amax = the largest
 * magnitude of the row; 1 for an all-zero row) and code = E4M3(x / scale), the fp32
 * quotient rounded to the nearest code (ties to even), magnitudes beyond 448 clamped to
 * 448.  Placement, arguments and errors are those of kv_append.
 * paged_attn_decode_fp8 is paged_attn_decode over the 8-bit cache.  Its tensor-core
 * products run in f16 (the codes convert exactly), so q must stay within f16's range
 * (|q| < 65504); outputs are bf16 as for paged_attn_decode.
 */
pa_status kv_append_fp8(pa_shape shape, void *k_codes, void *v_codes, float *k_scale,
                        float *v_scale, const void *k_new, const void *v_new,
                        const int32_t *block_table, int32_t max_blocks_per_seq,
                        int32_t num_blocks, const int32_t *cu_q_lens, const int32_t *seq_lens,
                        int32_t num_seqs, int32_t total_tokens, void *workspace,
                        size_t workspace_bytes, void *stream);

pa_status paged_attn_decode_fp8(pa_shape shape, void *out, float *lse, const void *q,
                                const void *k_codes, const void *v_codes, const float *k_scale,
                                const float *v_scale, const int32_t *block_table,
                                int32_t max_blocks_per_seq, int32_t num_blocks,
                                const int32_t *seq_lens, int32_t batch, float scale,
                                void *workspace, size_t workspace_bytes, void *stream);

/* The decode step over the 8-bit cache in one kernel: kv_append_fp8 of each sequence's new
 * token (row b of k_new / v_new [batch][8][128] bf16, at position seq_lens[b] - 1) fused
 * with paged_attn_decode_fp8.  Caches and outputs are those of the two separate calls. */
pa_status paged_attn_decode_append_fp8(pa_shape shape, void *out, float *lse, const void *q,
                                       const void *k_new, const void *v_new, void *k_codes,
                                       void *v_codes, float *k_scale, float *v_scale,
                                       const int32_t *block_table, int32_t max_blocks_per_seq,
                                       int32_t num_blocks, const int32_t *seq_lens, int32_t batch,
                                       float scale, void *workspace, size_t workspace_bytes,
                                       void *stream);

/* As paged_attn_decode_fp8 with the split length fixed by the caller: a positive multiple
 * of 128 tokens (the kernel's stage), or 0 for the library's choice. */
pa_status paged_attn_decode_fp8_split(pa_shape shape, void *out, float *lse, const void *q,
                                      const void *k_codes, const void *v_codes,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *block_table, int32_t max_blocks_per_seq,
                                      int32_t num_blocks, const int32_t *seq_lens, int32_t batch,
                                      float scale, int32_t split_tokens, void *workspace,
                                      size_t workspace_bytes, void *stream);

/*
 * paged_attn_decode_append: kv_append of one new token per sequence followed by
 * paged_attn_decode, in one kernel [P1 §4.3.1 append, §4.4.2 decode; P3 §4.2 "append,
 * then attend"].  Row b of k_new / v_new ([batch][8][128] bf16) is written to position
 * seq_lens[b] - 1 of sequence b (slot (seq_lens[b]-1) % 256 of block
 * block_table[b][(seq_lens[b]-1) / 256]) and takes part in the attention of the same
 * call.  Results (pools and outputs) are those of the two separate calls.
 */
pa_status paged_attn_decode_append(pa_shape shape, void *out, float *lse, const void *q,
                                   const void *k_new, const void *v_new, void *k_pool,
                                   void *v_pool, const int32_t *block_table,
                                   int32_t max_blocks_per_seq, int32_t num_blocks,
                                   const int32_t *seq_lens, int32_t batch, float scale,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * One decode step driven from host memory: runs paged_attn_decode_append (append of each
 * sequence's new token + decode) on host inputs and leaves the output (and lse, when
 * lse_host is non-NULL) in host memory -- all enqueued on `stream` without synchronising;
 * the results are in host memory once the stream has reached that point.  A host buffer
 * the GPU can address in place (pinned, mapped host memory: on GB300 over NVLink-C2C, as
 * reported by cudaHostGetDevicePointer) is read or written by the kernel directly; any
 * other buffer is copied through the caller-provided device staging buffer.  Host layouts are those of the device calls: q [batch][32][128] bf16,
 * k_new / v_new [batch][8][128] bf16, block_table [batch][max_blocks_per_seq] int32,
 * seq_lens [batch] int32, out [batch][32][128] bf16, lse [batch][32] fp32.  The pools
 * stay in device memory.  staging: device memory of pa_decode_step_host_staging_bytes()
 * bytes (16-byte aligned).  Not on the source pages: the engine's DecodeStep request
 * [P1 §4.1.2] carries token ids; this is the per-layer data movement around it.
 */
size_t pa_decode_step_host_staging_bytes(pa_shape shape, int32_t max_batch,
                                         int32_t max_blocks_per_seq);

pa_status pa_decode_step_host(pa_shape shape, void *out_host, float *lse_host,
                              const void *q_host, const void *k_new_host, const void *v_new_host,
                              const int32_t *block_table_host, const int32_t *seq_lens_host,
                              int32_t batch, int32_t max_blocks_per_seq, void *k_pool,
                              void *v_pool, int32_t num_blocks, float scale, void *staging,
                              size_t staging_bytes, void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * paged_attn_decode_cascade: paged_attn_decode for a batch whose sequences share a prefix
 * [P1 §2.3 prefix cache: requests with the same prefix reuse its KV state].  The first
 * shared_blocks entries of every sequence's block table are the same physical blocks
 * (checked on the device: a sequence whose entries differ from row 0's gets a NaN output
 * and PA_ERR_DEVICE).  The result is that of paged_attn_decode; the work is split in two:
 * all batch x 32 queries attend to the shared prefix at once on the tensor cores (the
 * prefix is read once per KV head instead of once per sequence, split over keys), then
 * the decode kernel attends each sequence's private suffix and merges the two by
 * log-sum-exp.  Every seq_lens[b] must exceed shared_blocks * 256 (else PA_ERR_DEVICE).
 * 1 <= shared_blocks < max_blocks_per_seq.  workspace: pa_cascade_workspace_bytes() bytes,
 * zeroed once like any workspace.
 */
size_t pa_cascade_workspace_bytes(pa_shape shape, int32_t max_batch, int32_t max_blocks_per_seq,
                                  int32_t shared_blocks);

pa_status paged_attn_decode_cascade(pa_shape shape, void *out, float *lse, const void *q,
                                    const void *k_pool, const void *v_pool,
                                    const int32_t *block_table, int32_t max_blocks_per_seq,
                                    int32_t num_blocks, const int32_t *seq_lens, int32_t batch,
                                    int32_t shared_blocks, float scale, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * A decode step over several layers captured once as a CUDA graph and replayed per
 * step: the launch-gap remedy the pages name for a GPU kept idle between kernel
 * launches [P2 §4.2 troubleshooting table: "use CUDA Graph"], decode being dominated by
 * many small launches [P1 §2.2].  Each replay runs, for layer l = 0 .. layers-1 in
 * order, paged_attn_decode_append on layer l's slices of layer-major tensors:
 *   q, out          bf16 [layers][batch][32][128]
 *   k_new, v_new    bf16 [layers][batch][8][128]
 *   lse             fp32 [layers][batch][32], or NULL
 *   k_pool, v_pool  bf16 [layers][num_blocks][256][8][128]
 * with one block_table / seq_lens shared by all layers (the sequences are the same in
 * every layer) and one workspace (the layers run one after another).  The graph holds
 * the pointers given here: between replays the caller updates the contents in place
 * (new q / k_new / v_new, seq_lens + 1, grown tables), never the pointers.  Results
 * are those of the same calls made one by one.
 *
 * pa_decode_graph_create  validates as paged_attn_decode_append does, captures the
 *                         layers on a private stream (nothing runs) and instantiates
 *                         the graph; *graph receives a handle (NULL on failure).
 *                         batch must be >= 1; the graph is tied to the current device.
 * pa_decode_graph_launch  enqueues one replay on `stream`.
 * pa_decode_graph_destroy releases the handle (NULL is accepted).
 */
typedef struct pa_decode_graph pa_decode_graph;

pa_status pa_decode_graph_create(pa_shape shape, int32_t layers, void *out, float *lse,
                                 const void *q, const void *k_new, const void *v_new,
                                 void *k_pool, void *v_pool, const int32_t *block_table,
                                 int32_t max_blocks_per_seq, int32_t num_blocks,
                                 const int32_t *seq_lens, int32_t batch, float scale,
                                 void *workspace, size_t workspace_bytes,
                                 pa_decode_graph **graph);

pa_status pa_decode_graph_launch(pa_decode_graph *graph, void *stream);

pa_status pa_decode_graph_destroy(pa_decode_graph *graph);

/*
 * paged_attn_decode_static: paged_attn_decode for callers that cannot allocate device
 * memory -- code that runs where cudaMalloc is not allowed or not available and that is
 * handed only its input and output buffers, never a scratch workspace (for example a
 * plug-in called inside another runtime that owns all device memory).  There is no
 * counterpart on the source pages; it is a deployment convenience.
 *
 * The split-K partial results and merge counters live in a fixed array inside the
 * library (13 MiB per GPU, reserved on every GPU that loads the library until the
 * process exits).  The call allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.  Limits: batch <= 256 sequences; a larger batch returns
 * PA_ERR_WORKSPACE and launches nothing.
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, and looks it up again if the device's
 * context has been destroyed and created anew since (cudaDeviceReset); make that first
 * call before any stream capture.  Every call shares the one array and first clears, on `stream`, the
 * parts that must start at zero; calls whose executions may overlap on the GPU (other
 * streams, other host threads) race on it and must be serialised by the caller.
 *
 * error_word: optional caller-owned device word that receives the error bits of
 * pa_check_error (pass it to pa_check_error as the "workspace"); NULL discards them.
 * All other arguments, layouts and results are those of paged_attn_decode.
 */
pa_status paged_attn_decode_static(pa_shape shape, void *out, float *lse, const void *q,
                                   const void *k_pool, const void *v_pool,
                                   const int32_t *block_table, int32_t max_blocks_per_seq,
                                   int32_t num_blocks, const int32_t *seq_lens, int32_t batch,
                                   float scale, uint32_t *error_word, void *stream);

/*
 * paged_attn_prefill: causal attention of each sequence's new tokens
 * [P1 §4.4.1; P3 §3.3].  New token i of sequence s sits at absolute position
 * p = seq_lens[s] - q_len + i and attends to context positions 0..p (its own key
 * included).  A sequence with q_len 0 is skipped.  max_q_len must bound every
 * q_len (checked on the device).  lse may be NULL.
 * The workspace needs only its error word (256 bytes).  With several sequences and a
 * workspace of pa_workspace_bytes() size, a planning kernel first sorts the work
 * units (64 positions x one KV head) by the number of key tiles they visit, into the
 * workspace's split-K area, so that the longest are started first; a workspace too
 * small for that list gets the natural order.  Results do not depend on the order.
 * out must be 32-byte aligned (the kernel writes whole 32-byte sectors), else
 * PA_ERR_INVALID_ARG; a view starting at any token of a larger tensor qualifies.
 */
pa_status paged_attn_prefill(pa_shape shape, void *out, float *lse, const void *q,
                             const void *k_pool, const void *v_pool,
                             const int32_t *block_table, int32_t max_blocks_per_seq,
                             int32_t num_blocks, const int32_t *cu_q_lens,
                             const int32_t *seq_lens, int32_t num_seqs, int32_t total_tokens,
                             int32_t max_q_len, float scale, void *workspace,
                             size_t workspace_bytes, void *stream);

/*
 * paged_attn_prefill_append: kv_append of each sequence's new tokens followed by
 * paged_attn_prefill, in one kernel [P1 §4.3.1 append, §4.4.1 prefill; P3 §4.2 "append,
 * then attend"].  k_new / v_new are [total_tokens][8][128] bf16 rows grouped by sequence as
 * in kv_append.  The attention reads the new tokens' keys and values straight from k_new /
 * v_new (their key tiles start at each sequence's first new token) and the cache for the
 * positions before them; a warp of every CTA meanwhile writes the new rows into their cache
 * slots, which nothing in the call reads.  Pools are bit-identical to kv_append's; outputs
 * are those of the two calls up to rounding (bit-identical when every sequence's earlier
 * context is a multiple of 128 tokens, where both calls cut the keys into the same tiles).
 * Arguments, workspace and errors as for kv_append and paged_attn_prefill (out
 * 32-byte aligned).
 */
pa_status paged_attn_prefill_append(pa_shape shape, void *out, float *lse, const void *q,
                                    const void *k_new, const void *v_new, void *k_pool,
                                    void *v_pool, const int32_t *block_table,
                                    int32_t max_blocks_per_seq, int32_t num_blocks,
                                    const int32_t *cu_q_lens, const int32_t *seq_lens,
                                    int32_t num_seqs, int32_t total_tokens, int32_t max_q_len,
                                    float scale, void *workspace, size_t workspace_bytes,
                                    void *stream);

/*
 * Self-test of the bounded-wait machinery: launches one CTA that waits on a
 * barrier nothing will ever complete, with a limit of timeout_us microseconds.
 * The kernel gives up, records PA_ERR_TIMEOUT in the workspace and exits; the GPU
 * context stays usable.  Used by the tests of the failure path.
 */
pa_status pa_selftest_wait_timeout(void *workspace, size_t workspace_bytes, uint32_t timeout_us,
                                   void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
