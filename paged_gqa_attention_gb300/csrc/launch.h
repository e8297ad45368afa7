// launch.h -- internal interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

struct AppendArgs {
    void *k_pool;          // bf16 pools, or the 8-bit code pools when k_scale is set
    void *v_pool;
    float *k_scale;        // 8-bit cache only: [num_blocks][8][256] row scales (else null)
    float *v_scale;
    const void *k_new;
    const void *v_new;
    const int32_t *block_table;
    int32_t max_blocks_per_seq;
    int32_t num_blocks;
    const int32_t *cu_q_lens;
    const int32_t *seq_lens;
    int32_t num_seqs;
    int32_t total_tokens;
    uint32_t *err;
};

struct DecodeArgs {
    void *out;
    float *lse;
    const void *q;
    // fused append (optional): the new token of every sequence, [batch][8][128] bf16, and
    // the pools it is written into; k_new == nullptr means the pools already hold it
    const void *k_new;
    const void *v_new;
    void *k_pool_w;
    void *v_pool_w;
    const int32_t *block_table;
    int32_t max_blocks_per_seq;
    int32_t num_blocks;
    const int32_t *seq_lens;
    int32_t batch;
    int32_t split_tokens;  // context tokens per CTA (multiple of 64)
    int32_t nsplit;        // splits per (sequence, KV head) at the maximum context
    float scale_log2;      // softmax scale * log2(e)
    const float *k_scale;  // 8-bit cache only: row scales [num_blocks][8][256]
    const float *v_scale;
    // Cascade over a shared prefix (decode kernel only): attend to tokens kv_begin ..
    // seq_len-1 and fold in pre_n partials of the prefix, pre_o [k][batch][32][128] fp32
    // normalised and pre_lse [k][batch][32] (natural log); the first shared_blocks table
    // entries of every sequence must equal row 0's.  kv_begin = pre_n = shared_blocks = 0
    // otherwise.
    int32_t kv_begin;
    const float *pre_o;
    const float *pre_lse;
    int32_t pre_n;
    int32_t shared_blocks;
    int32_t *counters;     // [batch * 8], zero on entry, zero again on exit
    float *part_o;         // [batch * 8 * nsplit][4][128]
    float *part_ml;        // [batch * 8 * nsplit][4][2]
    uint32_t *err;
    // Decode kernel only: 1 = the splits of a (sequence, KV head) form a cluster (nsplit <= 8)
    // and merge through its shared memory; the counters and partials are not used.
    int32_t cluster_merge;
};

struct PrefillArgs {
    void *out;
    float *lse;
    const int32_t *block_table;
    int32_t max_blocks_per_seq;
    int32_t num_blocks;
    const int32_t *cu_q_lens;
    const int32_t *seq_lens;
    int32_t num_seqs;
    int32_t total_tokens;
    int32_t max_q_len;
    float scale_log2;
    uint32_t *err;
    // Shared-prefix mode (launch_prefill_prefix): the total_tokens queries all attend to
    // keys 0 .. prefix_len-1 of block_table row 0 (no causal mask), split over keys into
    // n_kv_splits ranges of kv_split_tiles 128-key tiles; out receives fp32 normalised
    // partial outputs [split][token][32][128] and lse [split][token][32] (natural log).
    int32_t prefix_len;
    int32_t kv_split_tiles;
    int32_t n_kv_splits;
    // Several sequences: order[rank] = unit dealt at rank (units sorted by key tiles, most
    // first), written by a planning kernel launched just before the prefill; nullptr: the
    // units are dealt in their natural order (latest query blocks first).
    int32_t *order;
    // Fused append (k_new != nullptr): the new tokens' K/V rows [total_tokens][8][128] bf16 are
    // attended straight from k_new / v_new (key tiles of the new positions start at each
    // sequence's first new token) and written into the pools by the kernel itself.
    const void *k_new;
    const void *v_new;
    void *k_pool_w;
    void *v_pool_w;
};

constexpr int kRopePairs = 64;   // rotated pairs of a 128-dim head
// Merged Q/K/V projection with K and V written into the cache (qkv.cu).
struct QkvArgs {
    void *q_out;            // [total_tokens][32][128] bf16
    void *k_pool;           // [num_blocks][256][8][128] bf16
    void *v_pool;
    const int32_t *block_table;
    int32_t max_blocks_per_seq;
    int32_t num_blocks;
    const int32_t *cu_q_lens;
    const int32_t *seq_lens;
    int32_t num_seqs;
    int32_t total_tokens;
    int32_t hidden;         // a multiple of 256
    uint32_t *err;
    // Rotary position embedding of the q and k heads (rope != 0): the frequency of pair i
    // (dims i and i + 64 of a head) as a float-float value hi + lo = theta^(-i/64).
    int32_t rope;
    float rope_freq_hi[kRopePairs];
    float rope_freq_lo[kRopePairs];
    // Per-head RMS normalisation of q and k (launch_qk_norm only): bf16 gains [128] for the
    // q heads and for the k heads, and the eps under the square root.
    const void *q_norm;
    const void *k_norm;
    float norm_eps;
};

cudaError_t launch_kv_append(const AppendArgs &a, cudaStream_t stream);

// x_map: x [total_tokens][hidden] bf16, box {64, qkv_tile_rows_loaded(total_tokens)}; w_map:
// w [6144][hidden] bf16, box {64, qkv_weight_box_rows()}; both 128-byte swizzle.
int qkv_tile_cols(int total_tokens);
int qkv_weight_box_rows();
int qkv_tile_rows_loaded(int total_tokens);
cudaError_t launch_qkv(const QkvArgs &a, const CUtensorMap &x_map, const CUtensorMap &w_map, int num_sms,
                       cudaStream_t stream);
// In place over q_out and the new tokens' k rows in the cache, after launch_qkv without a
// rotation: each q and k head normalised by its RMS and gain, then rotated when a.rope is set.
cudaError_t launch_qk_norm(const QkvArgs &a, int num_sms, cudaStream_t stream);

// k_map / v_map: 4-D tensor maps over the pools (see api.cu for the boxes).
// One-time per-device kernel setup (dynamic shared memory size) of the decode kernel;
// launch_decode does it on first use, callers about to capture launches do it first.
cudaError_t configure_decode();

cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &k_map,
                          const CUtensorMap &v_map, int num_sms, cudaStream_t stream);

// q_map: 3-D map over q; k_map / v_map: 4-D maps over the pools.
// Decode over the 8-bit cache (code pools as k_map / v_map, scales in the args); its
// stages are 128 tokens, so its split length is a multiple of 128.
constexpr int kDecodeFp8TileTokens = 128;
// Decode over the 8-bit cache (code pools as k_map / v_map, scales in the args).
cudaError_t launch_decode_fp8(const DecodeArgs &a, const CUtensorMap &k_map, const CUtensorMap &v_map,
                              cudaStream_t stream);

cudaError_t launch_prefill_prefix(const PrefillArgs &a, const CUtensorMap &q_map, const CUtensorMap &k_map,
                                  const CUtensorMap &v_map, int num_sms, cudaStream_t stream);

// Units the planning kernel orders (several sequences), 0 when the natural order is
// used; a non-null PrefillArgs::order must hold this many int32 entries.
long long prefill_plan_units(const PrefillArgs &a);

cudaError_t launch_prefill(const PrefillArgs &a, const CUtensorMap &q_map,
                           const CUtensorMap &k_map, const CUtensorMap &v_map, int num_sms,
                           cudaStream_t stream);

// The prefill with the append of the new tokens fused in (a.k_new set): kn_map / vn_map are
// 3-D maps (dim, head, token) over k_new / v_new with box {64, 1, 128}.
cudaError_t launch_prefill_append(const PrefillArgs &a, const CUtensorMap &q_map, const CUtensorMap &k_map,
                                  const CUtensorMap &v_map, const CUtensorMap &kn_map, const CUtensorMap &vn_map,
                                  int num_sms, cudaStream_t stream);

cudaError_t launch_wait_selftest(uint32_t *err, uint64_t limit_ns, cudaStream_t stream);

// Device address of the file-scope scratch of paged_attn_decode_static on the current
// device (looked up on the first call per device and context); nullptr and *status set on
// failure.
void *static_scratch_address(cudaError_t *status);

// Tile sizes the tensor maps must be encoded with.
constexpr int kDecodeTileTokens = 64;    // decode: rows per TMA box
constexpr int kPrefillKvTile = 128;      // prefill: K/V rows per TMA box
constexpr int kPrefillQPositions = 32;   // prefill: query positions per tile (x4 heads)

}  // namespace pa
