// api.cu -- the extern "C" entry points declared in include/pagedattn.h: argument
// validation, tensor-map encoding, the decode split choice and kernel launches.
#include <atomic>
#include <cmath>
#include <mutex>
#include <new>

#include <cudaTypedefs.h>

#include "pagedattn.h"
#include "common.cuh"
#include "launch.h"

// Handle of pa_decode_graph_create: the captured graph, its executable form and the
// device it was captured on.
struct pa_decode_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    int device = -1;
};

namespace {

using namespace pa;

constexpr int32_t kVersion = 1 * 10000 + 0 * 100 + 0;

bool shape_ok(const pa_shape &s) {
    return s.num_q_heads == kHq && s.num_kv_heads == kHkv && s.head_dim == kD && s.block_size == kBlock;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// ------------------------------------------------------------------ driver entry point
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// Pool [num_blocks][256][8][128] bf16 seen as a 4-D tensor (dim, head, slot, block),
// box {64 dims, 1 head, rows slots, 1 block}, 128-byte swizzle.
bool encode_pool_map(CUtensorMap *map, const void *pool, int num_blocks, int rows) {
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)kHkv, (cuuint64_t)kBlock, (cuuint64_t)num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)kRowBytes, (cuuint64_t)kTokenBytes,
                                   (cuuint64_t)kTokenBytes * kBlock};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(pool), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An 8-bit code pool [num_blocks][256][8][128] uint8 as a 4-D tensor (dim, head, slot,
// block), box {128, 1, rows, 1}: one 128-byte row per token, 128-byte swizzle.
bool encode_code_map(CUtensorMap *map, const void *codes, int num_blocks, int rows) {
    const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)kHkv, (cuuint64_t)kBlock, (cuuint64_t)num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)kD, (cuuint64_t)kD * kHkv, (cuuint64_t)kD * kHkv * kBlock};
    const cuuint32_t box[4] = {(cuuint32_t)kD, 1, (cuuint32_t)rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(codes), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q [tokens][32][128] bf16 as a 3-D tensor (dim, head, token), box {64, 4, 32}.
bool encode_q_map(CUtensorMap *map, const void *q, int tokens) {
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)kHq, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)kRowBytes, (cuuint64_t)kRowBytes * kHq};
    const cuuint32_t box[3] = {64, (cuuint32_t)kGroup, (cuuint32_t)kPrefillQPositions};
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// New K or V rows [tokens][8][128] bf16 as a 3-D tensor (dim, head, token), box {64, 1, 128}:
// the same shared-memory tile as a pool map with 128-slot boxes.
bool encode_new_rows_map(CUtensorMap *map, const void *rows, int tokens) {
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)kHkv, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)kRowBytes, (cuuint64_t)kTokenBytes};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kPrefillKvTile};
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(rows), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major bf16 matrix [rows][cols] as a 2-D tensor (col, row), box {64, box_rows},
// 128-byte swizzle (cols a multiple of 8 so that the row stride is 16-byte aligned).
bool encode_matrix_map(CUtensorMap *map, const void *base, int rows, int cols, int box_rows) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ device facts
std::atomic<int> g_sms[64];

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
        int v = g_sms[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) g_sms[dev].store(n, std::memory_order_relaxed);
    return n;
}

// ------------------------------------------------------------------ decode split
// Context tokens per CTA.  Enough CTAs to keep every SM streaming (about 16 per SM
// over the widest table), capped; a multiple of the 64-token tile.  Depends only on
// batch, table width and SM count.
// Split size when the caller leaves it to the library.  Two regimes, measured on GB300:
// a small problem (few sequences x KV heads) wants many short splits for parallelism
// (about 16 CTAs per SM); once there is enough work, each CTA's fixed cost (its first tile
// arrives ~2 us after it starts) favours splits of at least 1024 tokens, as long as that
// still leaves 4 or more CTAs per SM (batch 32 x U{128..4096}: 46.0 us with 1024-token
// splits against 50.5 us with 448).
int auto_split_tokens(int batch, int max_blocks_per_seq, int num_sms) {
    const long long max_tokens = (long long)max_blocks_per_seq * kBlock;
    const long long pairs = (long long)batch * kHkv;
    long long target = (long long)num_sms * 16;
    if (target > kDecodeCtaCap) target = kDecodeCtaCap;
    long long nsplit = (target + pairs - 1) / pairs;
    const long long n_big = (max_tokens + 1023) / 1024;
    if (pairs * n_big >= 4LL * num_sms && n_big < nsplit) nsplit = n_big;
    if (nsplit < 1) nsplit = 1;
    long long split = (max_tokens + nsplit - 1) / nsplit;
    split = (split + kDecodeTileTokens - 1) / kDecodeTileTokens * kDecodeTileTokens;
    return (int)split;
}

size_t partial_entries_bound(int max_batch, int max_blocks_per_seq) {
    // auto split: pairs * ceil(target / pairs) <= target + pairs; never more than one
    // entry per 64-token tile of the widest context either.
    const long long pairs = (long long)max_batch * kHkv;
    const long long by_target = kDecodeCtaCap + pairs;
    const long long by_tiles = pairs * (((long long)max_blocks_per_seq * kBlock + kDecodeTileTokens - 1) /
                                        kDecodeTileTokens);
    return (size_t)(by_target < by_tiles ? by_target : by_tiles);
}

size_t workspace_bytes_for(size_t entries) {
    return kPartialOffset + entries * (kPartialOBytes + kPartialMLBytes);
}

// Staging layout of pa_decode_step_host, per batch of B sequences and tables W wide (each
// part rounded up to 256 bytes): q [B][32][128] bf16 | k_new [B][8][128] | v_new | out
// [B][32][128] bf16 | lse [B][32] fp32 | block_table [B][W] int32 | seq_lens [B] int32.
struct HostStepLayout {
    size_t q, k_new, v_new, out, lse, bt, sl, total;
};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

HostStepLayout host_step_layout(int batch, int max_blocks_per_seq) {
    HostStepLayout L;
    size_t o = 0;
    L.q = o;     o += round256((size_t)batch * kHq * kD * 2);
    L.k_new = o; o += round256((size_t)batch * kHkv * kD * 2);
    L.v_new = o; o += round256((size_t)batch * kHkv * kD * 2);
    L.out = o;   o += round256((size_t)batch * kHq * kD * 2);
    L.lse = o;   o += round256((size_t)batch * kHq * 4);
    L.bt = o;    o += round256((size_t)batch * max_blocks_per_seq * 4);
    L.sl = o;    o += round256((size_t)batch * 4);
    L.total = o;
    return L;
}

// Cascade extras of a decode over a shared prefix (see DecodeArgs): the first attended
// token, the prefix partials and the number of shared table entries.
struct CascadeExtras {
    int32_t kv_begin;
    const float *pre_o;
    const float *pre_lse;
    int32_t pre_n;
    int32_t shared_blocks;
};

pa_status decode_impl(pa_shape shape, void *out, float *lse, const void *q, const void *k_new,
                      const void *v_new, const void *k_pool, const void *v_pool, const int32_t *block_table,
                      int32_t max_blocks_per_seq, int32_t num_blocks, const int32_t *seq_lens, int32_t batch,
                      float scale, int32_t split_tokens, void *workspace, size_t workspace_bytes, void *stream,
                      const CascadeExtras *cx = nullptr) {
    if (!shape_ok(shape)) return PA_ERR_UNSUPPORTED;
    if (batch < 0 || batch > kMaxBatch || max_blocks_per_seq < 1 || num_blocks < 1 || !std::isfinite(scale) ||
        split_tokens < 0 || split_tokens % kDecodeTileTokens != 0)
        return PA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kPartialOffset || !aligned16(workspace)) return PA_ERR_INVALID_ARG;
    if (batch == 0) return PA_OK;
    if (!out || !q || !k_pool || !v_pool || !block_table || !seq_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned4(block_table) ||
        !aligned4(seq_lens) || (lse && !aligned4(lse)))
        return PA_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr) || (k_new && (!aligned16(k_new) || !aligned16(v_new))))
        return PA_ERR_INVALID_ARG;
    if ((long long)max_blocks_per_seq * kBlock > (1ll << 30)) return PA_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms <= 0) return PA_ERR_CUDA;
    if (!get_encoder()) return PA_ERR_CUDA;
    const int skip_blocks = cx ? cx->kv_begin / kBlock : 0;   // a cascade splits only the suffix
    const int split = split_tokens ? split_tokens : auto_split_tokens(batch, max_blocks_per_seq - skip_blocks, sms);
    const long long max_tokens = (long long)(max_blocks_per_seq - skip_blocks) * kBlock;
    const long long nsplit = (max_tokens + split - 1) / split;
    if (nsplit > 65535) return PA_ERR_INVALID_ARG;
    const size_t entries = (size_t)batch * kHkv * (size_t)nsplit;
    if (workspace_bytes_for(entries) > workspace_bytes) return PA_ERR_WORKSPACE;

    CUtensorMap k_map, v_map;
    if (!encode_pool_map(&k_map, k_pool, num_blocks, kDecodeTileTokens) ||
        !encode_pool_map(&v_map, v_pool, num_blocks, kDecodeTileTokens))
        return PA_ERR_INVALID_ARG;

    char *ws = static_cast<char *>(workspace);
    DecodeArgs a = {};
    a.out = out;
    a.lse = lse;
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_pool_w = const_cast<void *>(k_pool);
    a.v_pool_w = const_cast<void *>(v_pool);
    a.block_table = block_table;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.seq_lens = seq_lens;
    a.batch = batch;
    a.split_tokens = split;
    a.nsplit = (int)nsplit;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.k_scale = nullptr;
    a.v_scale = nullptr;
    a.kv_begin = cx ? cx->kv_begin : 0;
    a.pre_o = cx ? cx->pre_o : nullptr;
    a.pre_lse = cx ? cx->pre_lse : nullptr;
    a.pre_n = cx ? cx->pre_n : 0;
    a.shared_blocks = cx ? cx->shared_blocks : 0;
    a.counters = reinterpret_cast<int32_t *>(ws + kCounterOffset);
    a.part_o = reinterpret_cast<float *>(ws + kPartialOffset);
    a.part_ml = reinterpret_cast<float *>(ws + kPartialOffset + entries * kPartialOBytes);
    a.err = reinterpret_cast<uint32_t *>(ws);
    // A grid that fits in one wave (two CTAs per SM) with at most 8 splits a pair: the splits
    // of a pair merge as a cluster, through its shared memory.
    a.cluster_merge = nsplit > 1 && nsplit <= 8 && (long long)batch * kHkv * nsplit <= 2LL * sms ? 1 : 0;
    return launch_decode(a, k_map, v_map, sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                                 : PA_ERR_CUDA;
}

// Cascade plan for batch B over tables max_blocks_per_seq wide with shared_blocks shared
// entries: the prefix keys split into n_kv_splits ranges of kv_split_tiles 128-key tiles
// (about one prefill unit per SM), and the workspace carved as [decode part | pre_o |
// pre_lse], each part 256-byte aligned.
struct CascadePlan {
    int kv_split_tiles, n_kv_splits;
    size_t decode_bytes, pre_o_offset, pre_lse_offset, total;
};

CascadePlan cascade_plan(int batch, int max_blocks_per_seq, int shared_blocks, int sms) {
    CascadePlan p;
    const int tiles = shared_blocks * (kBlock / kPrefillKvTile);
    const int qblocks = (batch + 2 * kPrefillQPositions - 1) / (2 * kPrefillQPositions);
    int nks = (sms + kHkv * qblocks / 2) / (kHkv * qblocks);
    nks = nks < 1 ? 1 : (nks > tiles ? tiles : nks);
    p.kv_split_tiles = (tiles + nks - 1) / nks;
    p.n_kv_splits = (tiles + p.kv_split_tiles - 1) / p.kv_split_tiles;
    p.decode_bytes = round256(workspace_bytes_for(partial_entries_bound(batch, max_blocks_per_seq - shared_blocks)));
    p.pre_o_offset = p.decode_bytes;
    p.pre_lse_offset = p.pre_o_offset + round256((size_t)p.n_kv_splits * batch * kHq * kD * sizeof(float));
    p.total = p.pre_lse_offset + round256((size_t)p.n_kv_splits * batch * kHq * sizeof(float));
    return p;
}

// paged_qkv_append with or without the per-head normalisation of q and k (q_norm, k_norm:
// the bf16 gains, or null for none; the caller has checked them).
pa_status qkv_impl(pa_shape shape, int32_t hidden, float rope_theta, const void *q_norm, const void *k_norm,
                   float norm_eps, void *q_out, const void *x, const void *w_qkv, void *k_pool, void *v_pool,
                   const int32_t *block_table, int32_t max_blocks_per_seq, int32_t num_blocks,
                   const int32_t *cu_q_lens, const int32_t *seq_lens, int32_t num_seqs, int32_t total_tokens,
                   void *workspace, size_t workspace_bytes, void *stream) {
    if (!shape_ok(shape)) return PA_ERR_UNSUPPORTED;
    if (hidden < 256 || hidden % 256 != 0 || hidden > (1 << 16)) return PA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || total_tokens < 0 || max_blocks_per_seq < 1 || num_blocks < 1 ||
        (num_seqs == 0 && total_tokens != 0))
        return PA_ERR_INVALID_ARG;
    // the rotation: off (0) or a base above 1; positions must stay below 2^24 (exact in fp32)
    if (rope_theta != 0.f && !(std::isfinite(rope_theta) && rope_theta > 1.f)) return PA_ERR_INVALID_ARG;
    if (rope_theta != 0.f && (long long)max_blocks_per_seq * kBlock > (1ll << 24)) return PA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kHeaderBytes || !aligned16(workspace)) return PA_ERR_INVALID_ARG;
    if (total_tokens == 0) return PA_OK;
    if (!q_out || !x || !w_qkv || !k_pool || !v_pool || !block_table || !cu_q_lens || !seq_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(q_out) || !aligned16(x) || !aligned16(w_qkv) || !aligned16(k_pool) || !aligned16(v_pool) ||
        !aligned4(block_table) || !aligned4(cu_q_lens) || !aligned4(seq_lens))
        return PA_ERR_INVALID_ARG;
    if ((long long)max_blocks_per_seq * kBlock > (1ll << 30)) return PA_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms <= 0) return PA_ERR_CUDA;
    if (!get_encoder()) return PA_ERR_CUDA;
    CUtensorMap x_map, w_map;
    if (!encode_matrix_map(&x_map, x, total_tokens, hidden, qkv_tile_rows_loaded(total_tokens)) ||
        !encode_matrix_map(&w_map, w_qkv, kHq * kD + 2 * kHkv * kD, hidden, qkv_weight_box_rows()))
        return PA_ERR_INVALID_ARG;
    QkvArgs a = {};
    a.q_out = q_out;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.block_table = block_table;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.cu_q_lens = cu_q_lens;
    a.seq_lens = seq_lens;
    a.num_seqs = num_seqs;
    a.total_tokens = total_tokens;
    a.hidden = hidden;
    a.err = static_cast<uint32_t *>(workspace);
    a.rope = rope_theta != 0.f ? 1 : 0;
    for (int i = 0; i < kRopePairs; ++i) {
        // frequency of pair i: theta^(-2i/128), kept as a float-float pair hi + lo
        const double f = a.rope ? std::pow((double)rope_theta, -2.0 * i / kD) : 0.0;
        a.rope_freq_hi[i] = (float)f;
        a.rope_freq_lo[i] = (float)(f - (double)a.rope_freq_hi[i]);
    }
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!q_norm) return launch_qkv(a, x_map, w_map, sms, st) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    // QK-norm: the projection without the rotation, then every q and k head normalised and
    // rotated in place by a second kernel (the norm needs whole heads)
    a.q_norm = q_norm;
    a.k_norm = k_norm;
    a.norm_eps = norm_eps;
    QkvArgs plain = a;
    plain.rope = 0;
    if (launch_qkv(plain, x_map, w_map, sms, st) != cudaSuccess) return PA_ERR_CUDA;
    return launch_qk_norm(a, sms, st) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}


}  // namespace

extern "C" {

const char *pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_DEVICE: return "PA_ERR_DEVICE";
        case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    }
    return "PA_ERR_UNKNOWN";
}

int32_t pa_version(void) { return kVersion; }

size_t pa_workspace_bytes(pa_shape shape, int32_t max_batch, int32_t max_blocks_per_seq) {
    if (!shape_ok(shape) || max_batch < 1 || max_batch > kMaxBatch || max_blocks_per_seq < 1) return 0;
    return workspace_bytes_for(partial_entries_bound(max_batch, max_blocks_per_seq));
}

pa_status pa_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
    if (!workspace || workspace_bytes < kPartialOffset) return PA_ERR_INVALID_ARG;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_check_error(void *workspace, void *stream, uint32_t *detail) {
    if (!workspace) return PA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(workspace, 0, sizeof word, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return PA_ERR_CUDA;
    if (detail) *detail = word;
    if (word & kErrTimeout) return PA_ERR_TIMEOUT;
    if (word & kErrDevice) return PA_ERR_DEVICE;
    return PA_OK;
}

pa_status kv_append(pa_shape shape, void *k_pool, void *v_pool, const void *k_new, const void *v_new,
                    const int32_t *block_table, int32_t max_blocks_per_seq, int32_t num_blocks,
                    const int32_t *cu_q_lens, const int32_t *seq_lens, int32_t num_seqs, int32_t total_tokens,
                    void *workspace, size_t workspace_bytes, void *stream) {
    if (!shape_ok(shape)) return PA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || total_tokens < 0 || max_blocks_per_seq < 1 || num_blocks < 1 ||
        (num_seqs == 0 && total_tokens != 0))
        return PA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kHeaderBytes || !aligned16(workspace)) return PA_ERR_INVALID_ARG;
    if (total_tokens == 0) return PA_OK;
    if (!k_pool || !v_pool || !k_new || !v_new || !block_table || !cu_q_lens || !seq_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new) ||
        !aligned4(block_table) || !aligned4(cu_q_lens) || !aligned4(seq_lens))
        return PA_ERR_INVALID_ARG;
    AppendArgs a = {};
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.k_scale = nullptr;
    a.v_scale = nullptr;
    a.k_new = k_new;
    a.v_new = v_new;
    a.block_table = block_table;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.cu_q_lens = cu_q_lens;
    a.seq_lens = seq_lens;
    a.num_seqs = num_seqs;
    a.total_tokens = total_tokens;
    a.err = static_cast<uint32_t *>(workspace);
    return launch_kv_append(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status paged_qkv_append(pa_shape shape, int32_t hidden, float rope_theta, void *q_out, const void *x,
                           const void *w_qkv, void *k_pool, void *v_pool, const int32_t *block_table,
                           int32_t max_blocks_per_seq, int32_t num_blocks, const int32_t *cu_q_lens,
                           const int32_t *seq_lens, int32_t num_seqs, int32_t total_tokens, void *workspace,
                           size_t workspace_bytes, void *stream) {
    return qkv_impl(shape, hidden, rope_theta, nullptr, nullptr, 0.f, q_out, x, w_qkv, k_pool, v_pool, block_table,
                    max_blocks_per_seq, num_blocks, cu_q_lens, seq_lens, num_seqs, total_tokens, workspace,
                    workspace_bytes, stream);
}

pa_status paged_qkv_append_qknorm(pa_shape shape, int32_t hidden, float rope_theta, const void *q_norm_weight,
                                  const void *k_norm_weight, float norm_eps, void *q_out, const void *x,
                                  const void *w_qkv, void *k_pool, void *v_pool, const int32_t *block_table,
                                  int32_t max_blocks_per_seq, int32_t num_blocks, const int32_t *cu_q_lens,
                                  const int32_t *seq_lens, int32_t num_seqs, int32_t total_tokens,
                                  void *workspace, size_t workspace_bytes, void *stream) {
    if (!q_norm_weight || !k_norm_weight || !aligned16(q_norm_weight) || !aligned16(k_norm_weight) ||
        !(std::isfinite(norm_eps) && norm_eps >= 0.f))
        return PA_ERR_INVALID_ARG;
    return qkv_impl(shape, hidden, rope_theta, q_norm_weight, k_norm_weight, norm_eps, q_out, x, w_qkv, k_pool,
                    v_pool, block_table, max_blocks_per_seq, num_blocks, cu_q_lens, seq_lens, num_seqs,
                    total_tokens, workspace, workspace_bytes, stream);
}

pa_status kv_append_fp8(pa_shape shape, void *k_codes, void *v_codes, float *k_scale, float *v_scale,
                        const void *k_new, const void *v_new, const int32_t *block_table,
                        int32_t max_blocks_per_seq, int32_t num_blocks, const int32_t *cu_q_lens,
                        const int32_t *seq_lens, int32_t num_seqs, int32_t total_tokens, void *workspace,
                        size_t workspace_bytes, void *stream) {
    if (!shape_ok(shape)) return PA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || total_tokens < 0 || max_blocks_per_seq < 1 || num_blocks < 1 ||
        (num_seqs == 0 && total_tokens != 0))
        return PA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kHeaderBytes || !aligned16(workspace)) return PA_ERR_INVALID_ARG;
    if (total_tokens == 0) return PA_OK;
    if (!k_codes || !v_codes || !k_scale || !v_scale || !k_new || !v_new || !block_table || !cu_q_lens ||
        !seq_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scale) || !aligned16(v_scale) ||
        !aligned16(k_new) || !aligned16(v_new) || !aligned4(block_table) || !aligned4(cu_q_lens) ||
        !aligned4(seq_lens))
        return PA_ERR_INVALID_ARG;
    AppendArgs a = {};
    a.k_pool = k_codes;
    a.v_pool = v_codes;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.k_new = k_new;
    a.v_new = v_new;
    a.block_table = block_table;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.cu_q_lens = cu_q_lens;
    a.seq_lens = seq_lens;
    a.num_seqs = num_seqs;
    a.total_tokens = total_tokens;
    a.err = static_cast<uint32_t *>(workspace);
    return launch_kv_append(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

static pa_status decode_fp8_impl(pa_shape shape, void *out, float *lse, const void *q, const void *k_new, const void *v_new,
                          const void *k_codes, const void *v_codes, const float *k_scale, const float *v_scale,
                          const int32_t *block_table, int32_t max_blocks_per_seq, int32_t num_blocks,
                          const int32_t *seq_lens, int32_t batch, float scale, int32_t split_tokens,
                          void *workspace, size_t workspace_bytes, void *stream) {
    if ((k_new == nullptr) != (v_new == nullptr) || (k_new && (!aligned16(k_new) || !aligned16(v_new))))
        return PA_ERR_INVALID_ARG;
    if (!shape_ok(shape)) return PA_ERR_UNSUPPORTED;
    if (batch < 0 || batch > kMaxBatch || max_blocks_per_seq < 1 || num_blocks < 1 || !std::isfinite(scale) ||
        split_tokens < 0 || split_tokens % kDecodeFp8TileTokens != 0)
        return PA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kPartialOffset || !aligned16(workspace)) return PA_ERR_INVALID_ARG;
    if (batch == 0) return PA_OK;
    if (!out || !q || !k_codes || !v_codes || !k_scale || !v_scale || !block_table || !seq_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scale) ||
        !aligned16(v_scale) || !aligned4(block_table) || !aligned4(seq_lens) || (lse && !aligned4(lse)))
        return PA_ERR_INVALID_ARG;
    if ((long long)max_blocks_per_seq * kBlock > (1ll << 30)) return PA_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms <= 0) return PA_ERR_CUDA;
    if (!get_encoder()) return PA_ERR_CUDA;
    // the library's split rounded up to whole 128-token stages
    const int split = split_tokens ? split_tokens
                                   : (auto_split_tokens(batch, max_blocks_per_seq, sms) + kDecodeFp8TileTokens - 1) /
                                         kDecodeFp8TileTokens * kDecodeFp8TileTokens;
    const long long max_tokens = (long long)max_blocks_per_seq * kBlock;
    const long long nsplit = (max_tokens + split - 1) / split;
    if (nsplit > 65535) return PA_ERR_INVALID_ARG;
    const size_t entries = (size_t)batch * kHkv * (size_t)nsplit;
    if (workspace_bytes_for(entries) > workspace_bytes) return PA_ERR_WORKSPACE;
    CUtensorMap k_map, v_map;
    if (!encode_code_map(&k_map, k_codes, num_blocks, kDecodeFp8TileTokens) ||
        !encode_code_map(&v_map, v_codes, num_blocks, kDecodeFp8TileTokens))
        return PA_ERR_INVALID_ARG;
    char *ws = static_cast<char *>(workspace);
    DecodeArgs a = {};
    a.out = out;
    a.lse = lse;
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_pool_w = const_cast<void *>(k_codes);
    a.v_pool_w = const_cast<void *>(v_codes);
    a.block_table = block_table;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.seq_lens = seq_lens;
    a.batch = batch;
    a.split_tokens = split;
    a.nsplit = (int)nsplit;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.kv_begin = 0;
    a.pre_o = nullptr;
    a.pre_lse = nullptr;
    a.pre_n = 0;
    a.shared_blocks = 0;
    a.counters = reinterpret_cast<int32_t *>(ws + kCounterOffset);
    a.part_o = reinterpret_cast<float *>(ws + kPartialOffset);
    a.part_ml = reinterpret_cast<float *>(ws + kPartialOffset + entries * kPartialOBytes);
    a.err = reinterpret_cast<uint32_t *>(ws);
    return launch_decode_fp8(a, k_map, v_map, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                             : PA_ERR_CUDA;
}

pa_status paged_attn_decode_fp8_split(pa_shape shape, void *out, float *lse, const void *q, const void *k_codes,
                                      const void *v_codes, const float *k_scale, const float *v_scale,
                                      const int32_t *block_table, int32_t max_blocks_per_seq, int32_t num_blocks,
                                      const int32_t *seq_lens, int32_t batch, float scale, int32_t split_tokens,
                                      void *workspace, size_t workspace_bytes, void *stream) {
    return decode_fp8_impl(shape, out, lse, q, nullptr, nullptr, k_codes, v_codes, k_scale, v_scale, block_table,
                           max_blocks_per_seq, num_blocks, seq_lens, batch, scale, split_tokens, workspace,
                           workspace_bytes, stream);
}

pa_status paged_attn_decode_fp8(pa_shape shape, void *out, float *lse, const void *q, const void *k_codes,
                                const void *v_codes, const float *k_scale, const float *v_scale,
                                const int32_t *block_table, int32_t max_blocks_per_seq, int32_t num_blocks,
                                const int32_t *seq_lens, int32_t batch, float scale, void *workspace,
                                size_t workspace_bytes, void *stream) {
    return decode_fp8_impl(shape, out, lse, q, nullptr, nullptr, k_codes, v_codes, k_scale, v_scale, block_table,
                           max_blocks_per_seq, num_blocks, seq_lens, batch, scale, 0, workspace, workspace_bytes,
                           stream);
}

pa_status paged_attn_decode_append_fp8(pa_shape shape, void *out, float *lse, const void *q, const void *k_new,
                                       const void *v_new, void *k_codes, void *v_codes, float *k_scale,
                                       float *v_scale, const int32_t *block_table, int32_t max_blocks_per_seq,
                                       int32_t num_blocks, const int32_t *seq_lens, int32_t batch, float scale,
                                       void *workspace, size_t workspace_bytes, void *stream) {
    if (batch > 0 && (!k_new || !v_new)) return PA_ERR_INVALID_ARG;
    return decode_fp8_impl(shape, out, lse, q, k_new, v_new, k_codes, v_codes, k_scale, v_scale, block_table,
                           max_blocks_per_seq, num_blocks, seq_lens, batch, scale, 0, workspace, workspace_bytes,
                           stream);
}

pa_status paged_attn_decode(pa_shape shape, void *out, float *lse, const void *q, const void *k_pool,
                            const void *v_pool, const int32_t *block_table, int32_t max_blocks_per_seq,
                            int32_t num_blocks, const int32_t *seq_lens, int32_t batch, float scale,
                            void *workspace, size_t workspace_bytes, void *stream) {
    return decode_impl(shape, out, lse, q, nullptr, nullptr, k_pool, v_pool, block_table, max_blocks_per_seq,
                       num_blocks, seq_lens, batch, scale, 0, workspace, workspace_bytes, stream);
}

pa_status paged_attn_decode_split(pa_shape shape, void *out, float *lse, const void *q, const void *k_pool,
                                  const void *v_pool, const int32_t *block_table, int32_t max_blocks_per_seq,
                                  int32_t num_blocks, const int32_t *seq_lens, int32_t batch, float scale,
                                  int32_t split_tokens, void *workspace, size_t workspace_bytes, void *stream) {
    return decode_impl(shape, out, lse, q, nullptr, nullptr, k_pool, v_pool, block_table, max_blocks_per_seq,
                       num_blocks, seq_lens, batch, scale, split_tokens, workspace, workspace_bytes, stream);
}

pa_status paged_attn_decode_append(pa_shape shape, void *out, float *lse, const void *q, const void *k_new,
                                   const void *v_new, void *k_pool, void *v_pool, const int32_t *block_table,
                                   int32_t max_blocks_per_seq, int32_t num_blocks, const int32_t *seq_lens,
                                   int32_t batch, float scale, void *workspace, size_t workspace_bytes,
                                   void *stream) {
    if (batch > 0 && (!k_new || !v_new)) return PA_ERR_INVALID_ARG;
    return decode_impl(shape, out, lse, q, k_new, v_new, k_pool, v_pool, block_table, max_blocks_per_seq,
                       num_blocks, seq_lens, batch, scale, 0, workspace, workspace_bytes, stream);
}

size_t pa_decode_step_host_staging_bytes(pa_shape shape, int32_t max_batch, int32_t max_blocks_per_seq) {
    if (!shape_ok(shape) || max_batch < 1 || max_batch > kMaxBatch || max_blocks_per_seq < 1) return 0;
    return host_step_layout(max_batch, max_blocks_per_seq).total;
}

// Device address under which the GPU reaches host buffer p in place (pinned, mapped host
// memory: on GB300 over NVLink-C2C), or nullptr when the runtime reports none -- then the
// buffer is staged with a copy instead.
const void *mapped(const void *p) {
    void *d = nullptr;
    if (cudaHostGetDevicePointer(&d, const_cast<void *>(p), 0) != cudaSuccess) {
        cudaGetLastError();   // reset the runtime's last-error state after the failed query
        return nullptr;
    }
    return d;
}

pa_status pa_decode_step_host(pa_shape shape, void *out_host, float *lse_host, const void *q_host,
                              const void *k_new_host, const void *v_new_host, const int32_t *block_table_host,
                              const int32_t *seq_lens_host, int32_t batch, int32_t max_blocks_per_seq,
                              void *k_pool, void *v_pool, int32_t num_blocks, float scale, void *staging,
                              size_t staging_bytes, void *workspace, size_t workspace_bytes, void *stream) {
    if (!shape_ok(shape)) return PA_ERR_UNSUPPORTED;
    if (batch < 0 || batch > kMaxBatch || max_blocks_per_seq < 1) return PA_ERR_INVALID_ARG;
    if (batch == 0) return PA_OK;
    if (!out_host || !q_host || !k_new_host || !v_new_host || !block_table_host || !seq_lens_host || !staging ||
        !aligned16(staging))
        return PA_ERR_INVALID_ARG;
    const HostStepLayout L = host_step_layout(batch, max_blocks_per_seq);
    if (staging_bytes < L.total) return PA_ERR_WORKSPACE;
    char *st = static_cast<char *>(staging);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t q_bytes = (size_t)batch * kHq * kD * 2, kv_bytes = (size_t)batch * kHkv * kD * 2;
    const size_t bt_bytes = (size_t)batch * max_blocks_per_seq * 4, sl_bytes = (size_t)batch * 4;
    const size_t lse_bytes = (size_t)batch * kHq * 4;
    // Inputs: read in place when mapped, else copied into the staging buffer.
    auto input = [&](const void *h, size_t off, size_t bytes, const void **d) -> bool {
        *d = mapped(h);
        if (*d && aligned16(*d)) return true;
        *d = st + off;
        return cudaMemcpyAsync(st + off, h, bytes, cudaMemcpyHostToDevice, s) == cudaSuccess;
    };
    const void *q, *kn, *vn, *bt, *sl;
    if (!input(q_host, L.q, q_bytes, &q) || !input(k_new_host, L.k_new, kv_bytes, &kn) ||
        !input(v_new_host, L.v_new, kv_bytes, &vn) || !input(block_table_host, L.bt, bt_bytes, &bt) ||
        !input(seq_lens_host, L.sl, sl_bytes, &sl))
        return PA_ERR_CUDA;
    // Outputs: written in place when mapped, else staged and copied back.
    void *out = const_cast<void *>(mapped(out_host));
    const bool out_direct = out && aligned16(out);
    if (!out_direct) out = st + L.out;
    float *lse = nullptr;
    bool lse_direct = false;
    if (lse_host) {
        lse = static_cast<float *>(const_cast<void *>(mapped(lse_host)));
        lse_direct = lse && aligned4(lse);
        if (!lse_direct) lse = reinterpret_cast<float *>(st + L.lse);
    }
    const pa_status r = decode_impl(shape, out, lse, q, kn, vn, k_pool, v_pool, static_cast<const int32_t *>(bt),
                                    max_blocks_per_seq, num_blocks, static_cast<const int32_t *>(sl), batch, scale,
                                    0, workspace, workspace_bytes, stream);
    if (r != PA_OK) return r;
    if (!out_direct && cudaMemcpyAsync(out_host, out, q_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PA_ERR_CUDA;
    if (lse_host && !lse_direct && cudaMemcpyAsync(lse_host, lse, lse_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

pa_status paged_attn_decode_static(pa_shape shape, void *out, float *lse, const void *q, const void *k_pool,
                                   const void *v_pool, const int32_t *block_table, int32_t max_blocks_per_seq,
                                   int32_t num_blocks, const int32_t *seq_lens, int32_t batch, float scale,
                                   uint32_t *error_word, void *stream) {
    // Same computation as paged_attn_decode, but the split-K scratch is the library's own
    // fixed device array, so the caller allocates nothing (see pagedattn.h).
    if (!shape_ok(shape)) return PA_ERR_UNSUPPORTED;
    if (batch < 0 || max_blocks_per_seq < 1 || num_blocks < 1 || !std::isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (batch > kStaticMaxBatch) return PA_ERR_WORKSPACE;   // beyond what the fixed scratch holds
    if (batch == 0) return PA_OK;
    if (!out || !q || !k_pool || !v_pool || !block_table || !seq_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned4(block_table) ||
        !aligned4(seq_lens) || (lse && !aligned4(lse)) || (error_word && !aligned4(error_word)))
        return PA_ERR_INVALID_ARG;
    if ((long long)max_blocks_per_seq * kBlock > (1ll << 30)) return PA_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms <= 0) return PA_ERR_CUDA;
    if (!get_encoder()) return PA_ERR_CUDA;
    const int split = auto_split_tokens(batch, max_blocks_per_seq, sms);
    const long long nsplit = ((long long)max_blocks_per_seq * kBlock + split - 1) / split;
    if (nsplit > 65535) return PA_ERR_INVALID_ARG;
    const size_t entries = (size_t)batch * kHkv * (size_t)nsplit;
    if (workspace_bytes_for(entries) > kStaticScratchBytes) return PA_ERR_WORKSPACE;
    cudaError_t e = cudaSuccess;
    char *ws = static_cast<char *>(static_scratch_address(&e));   // first call per device: symbol lookup
    if (!ws) return PA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The scratch keeps whatever the previous call left: zero its error word and this
    // call's merge counters (a call that was cut short may have left them non-zero).
    if (cudaMemsetAsync(ws, 0, kCounterOffset + sizeof(int32_t) * (size_t)batch * kHkv, st) != cudaSuccess)
        return PA_ERR_CUDA;
    CUtensorMap k_map, v_map;
    if (!encode_pool_map(&k_map, k_pool, num_blocks, kDecodeTileTokens) ||
        !encode_pool_map(&v_map, v_pool, num_blocks, kDecodeTileTokens))
        return PA_ERR_INVALID_ARG;
    DecodeArgs a = {};
    a.out = out;
    a.lse = lse;
    a.q = q;
    a.k_new = nullptr;
    a.v_new = nullptr;
    a.k_pool_w = nullptr;
    a.v_pool_w = nullptr;
    a.block_table = block_table;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.seq_lens = seq_lens;
    a.batch = batch;
    a.split_tokens = split;
    a.nsplit = (int)nsplit;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.k_scale = nullptr;
    a.v_scale = nullptr;
    a.kv_begin = 0;        // no shared prefix: the whole context, no partials to fold in
    a.pre_o = nullptr;
    a.pre_lse = nullptr;
    a.pre_n = 0;
    a.shared_blocks = 0;
    a.counters = reinterpret_cast<int32_t *>(ws + kCounterOffset);
    a.part_o = reinterpret_cast<float *>(ws + kPartialOffset);
    a.part_ml = reinterpret_cast<float *>(ws + kPartialOffset + entries * kPartialOBytes);
    a.err = error_word ? error_word : reinterpret_cast<uint32_t *>(ws);
    return launch_decode(a, k_map, v_map, sms, st) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

static pa_status prefill_impl(pa_shape shape, void *out, float *lse, const void *q, const void *k_new,
                              const void *v_new, const void *k_pool, const void *v_pool, const int32_t *block_table,
                              int32_t max_blocks_per_seq, int32_t num_blocks, const int32_t *cu_q_lens,
                              const int32_t *seq_lens, int32_t num_seqs, int32_t total_tokens, int32_t max_q_len,
                              float scale, void *workspace, size_t workspace_bytes, void *stream) {
    if (!shape_ok(shape)) return PA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || total_tokens < 0 || max_q_len < 0 || max_blocks_per_seq < 1 || num_blocks < 1 ||
        !std::isfinite(scale) || (num_seqs == 0 && total_tokens != 0) || max_q_len > total_tokens ||
        (total_tokens > 0 && max_q_len == 0))
        return PA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kHeaderBytes || !aligned16(workspace)) return PA_ERR_INVALID_ARG;
    if (total_tokens == 0) return PA_OK;
    if ((long long)num_seqs * kHkv * ((max_q_len + kPrefillQPositions - 1) / kPrefillQPositions) > (1ll << 30) ||
        (long long)max_blocks_per_seq * kBlock > (1ll << 30))
        return PA_ERR_INVALID_ARG;
    if (!out || !q || !k_pool || !v_pool || !block_table || !cu_q_lens || !seq_lens) return PA_ERR_INVALID_ARG;
    if (!aligned32(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned4(block_table) ||
        !aligned4(cu_q_lens) || !aligned4(seq_lens) || (lse && !aligned4(lse)))
        return PA_ERR_INVALID_ARG;
    if ((k_new == nullptr) != (v_new == nullptr) || (k_new && (!aligned16(k_new) || !aligned16(v_new))))
        return PA_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms <= 0) return PA_ERR_CUDA;
    if (!get_encoder()) return PA_ERR_CUDA;
    CUtensorMap q_map, k_map, v_map, kn_map, vn_map;
    if (!encode_q_map(&q_map, q, total_tokens) || !encode_pool_map(&k_map, k_pool, num_blocks, kPrefillKvTile) ||
        !encode_pool_map(&v_map, v_pool, num_blocks, kPrefillKvTile))
        return PA_ERR_INVALID_ARG;
    if (k_new && (!encode_new_rows_map(&kn_map, k_new, total_tokens) || !encode_new_rows_map(&vn_map, v_new, total_tokens)))
        return PA_ERR_INVALID_ARG;
    PrefillArgs a = {};
    a.out = out;
    a.lse = lse;
    a.block_table = block_table;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.cu_q_lens = cu_q_lens;
    a.seq_lens = seq_lens;
    a.num_seqs = num_seqs;
    a.total_tokens = total_tokens;
    a.max_q_len = max_q_len;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.err = static_cast<uint32_t *>(workspace);
    a.prefix_len = 0;
    a.kv_split_tiles = 0;
    a.n_kv_splits = 1;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_pool_w = const_cast<void *>(k_pool);
    a.v_pool_w = const_cast<void *>(v_pool);
    // Several sequences: the units are sorted by work first, into the workspace's partial
    // area (decode scratch, unused by the prefill) when it is large enough.
    a.order = nullptr;
    const long long plan_units = prefill_plan_units(a);
    if (plan_units > 0 && workspace_bytes >= kPartialOffset + (size_t)plan_units * sizeof(int32_t))
        a.order = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + kPartialOffset);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = k_new ? launch_prefill_append(a, q_map, k_map, v_map, kn_map, vn_map, sms, st)
                                : launch_prefill(a, q_map, k_map, v_map, sms, st);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status paged_attn_prefill(pa_shape shape, void *out, float *lse, const void *q, const void *k_pool,
                             const void *v_pool, const int32_t *block_table, int32_t max_blocks_per_seq,
                             int32_t num_blocks, const int32_t *cu_q_lens, const int32_t *seq_lens, int32_t num_seqs,
                             int32_t total_tokens, int32_t max_q_len, float scale, void *workspace,
                             size_t workspace_bytes, void *stream) {
    return prefill_impl(shape, out, lse, q, nullptr, nullptr, k_pool, v_pool, block_table, max_blocks_per_seq,
                        num_blocks, cu_q_lens, seq_lens, num_seqs, total_tokens, max_q_len, scale, workspace,
                        workspace_bytes, stream);
}

pa_status paged_attn_prefill_append(pa_shape shape, void *out, float *lse, const void *q, const void *k_new,
                                    const void *v_new, void *k_pool, void *v_pool, const int32_t *block_table,
                                    int32_t max_blocks_per_seq, int32_t num_blocks, const int32_t *cu_q_lens,
                                    const int32_t *seq_lens, int32_t num_seqs, int32_t total_tokens,
                                    int32_t max_q_len, float scale, void *workspace, size_t workspace_bytes,
                                    void *stream) {
    if (total_tokens > 0 && (!k_new || !v_new)) return PA_ERR_INVALID_ARG;
    return prefill_impl(shape, out, lse, q, k_new, v_new, k_pool, v_pool, block_table, max_blocks_per_seq,
                        num_blocks, cu_q_lens, seq_lens, num_seqs, total_tokens, max_q_len, scale, workspace,
                        workspace_bytes, stream);
}

pa_status pa_decode_graph_create(pa_shape shape, int32_t layers, void *out, float *lse, const void *q,
                                 const void *k_new, const void *v_new, void *k_pool, void *v_pool,
                                 const int32_t *block_table, int32_t max_blocks_per_seq, int32_t num_blocks,
                                 const int32_t *seq_lens, int32_t batch, float scale, void *workspace,
                                 size_t workspace_bytes, pa_decode_graph **graph) {
    if (!graph) return PA_ERR_INVALID_ARG;
    *graph = nullptr;
    if (!shape_ok(shape)) return PA_ERR_UNSUPPORTED;
    if (layers < 1 || batch < 1 || num_blocks < 1 || !k_new || !v_new || !out || !q || !k_pool || !v_pool)
        return PA_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    // Everything that is not a launch happens before the capture: kernel attributes,
    // the SM count and the tensor-map encoder are set up once here.
    if (configure_decode() != cudaSuccess || sm_count() <= 0 || !get_encoder()) return PA_ERR_CUDA;

    const size_t q_bytes = (size_t)batch * kHq * kD * sizeof(__nv_bfloat16);     // per layer
    const size_t kv_bytes = (size_t)batch * kHkv * kD * sizeof(__nv_bfloat16);
    const size_t lse_floats = (size_t)batch * kHq;
    const size_t pool_bytes = (size_t)num_blocks * kBlock * kHkv * kD * sizeof(__nv_bfloat16);
    cudaStream_t cs = nullptr;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        cudaStreamDestroy(cs);
        return PA_ERR_CUDA;
    }
    pa_status st = PA_OK;
    for (int32_t l = 0; l < layers && st == PA_OK; ++l) {
        st = decode_impl(shape, static_cast<char *>(out) + l * q_bytes, lse ? lse + l * lse_floats : nullptr,
                         static_cast<const char *>(q) + l * q_bytes, static_cast<const char *>(k_new) + l * kv_bytes,
                         static_cast<const char *>(v_new) + l * kv_bytes, static_cast<char *>(k_pool) + l * pool_bytes,
                         static_cast<char *>(v_pool) + l * pool_bytes, block_table, max_blocks_per_seq, num_blocks,
                         seq_lens, batch, scale, 0, workspace, workspace_bytes, cs);
    }
    cudaGraph_t g = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(cs, &g);
    cudaStreamDestroy(cs);
    if (st != PA_OK || ce != cudaSuccess || !g) {
        if (g) cudaGraphDestroy(g);
        cudaGetLastError();
        return st != PA_OK ? st : PA_ERR_CUDA;
    }
    cudaGraphExec_t x = nullptr;
    if (cudaGraphInstantiate(&x, g, 0) != cudaSuccess) {
        cudaGraphDestroy(g);
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    pa_decode_graph *h = new (std::nothrow) pa_decode_graph;
    if (!h) {
        cudaGraphExecDestroy(x);
        cudaGraphDestroy(g);
        return PA_ERR_CUDA;
    }
    h->graph = g;
    h->exec = x;
    h->device = dev;
    *graph = h;
    return PA_OK;
}

pa_status pa_decode_graph_launch(pa_decode_graph *graph, void *stream) {
    if (!graph || !graph->exec) return PA_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev != graph->device) return PA_ERR_INVALID_ARG;
    return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_decode_graph_destroy(pa_decode_graph *graph) {
    if (!graph) return PA_OK;
    const bool ok = (!graph->exec || cudaGraphExecDestroy(graph->exec) == cudaSuccess) &
                    (!graph->graph || cudaGraphDestroy(graph->graph) == cudaSuccess);
    delete graph;
    return ok ? PA_OK : PA_ERR_CUDA;
}

size_t pa_cascade_workspace_bytes(pa_shape shape, int32_t max_batch, int32_t max_blocks_per_seq,
                                  int32_t shared_blocks) {
    if (!shape_ok(shape) || max_batch < 1 || max_batch > kMaxBatch || shared_blocks < 1 ||
        shared_blocks >= max_blocks_per_seq)
        return 0;
    const int sms = sm_count();
    if (sms <= 0) return 0;
    return cascade_plan(max_batch, max_blocks_per_seq, shared_blocks, sms).total;
}

pa_status paged_attn_decode_cascade(pa_shape shape, void *out, float *lse, const void *q, const void *k_pool,
                                    const void *v_pool, const int32_t *block_table, int32_t max_blocks_per_seq,
                                    int32_t num_blocks, const int32_t *seq_lens, int32_t batch,
                                    int32_t shared_blocks, float scale, void *workspace, size_t workspace_bytes,
                                    void *stream) {
    if (!shape_ok(shape)) return PA_ERR_UNSUPPORTED;
    if (batch < 0 || batch > kMaxBatch || max_blocks_per_seq < 2 || num_blocks < 1 || shared_blocks < 1 ||
        shared_blocks >= max_blocks_per_seq || !std::isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < kPartialOffset || !aligned16(workspace)) return PA_ERR_INVALID_ARG;
    if (batch == 0) return PA_OK;
    if (!out || !q || !k_pool || !v_pool || !block_table || !seq_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned4(block_table) ||
        !aligned4(seq_lens) || (lse && !aligned4(lse)))
        return PA_ERR_INVALID_ARG;
    const int sms = sm_count();
    if (sms <= 0 || !get_encoder()) return PA_ERR_CUDA;
    const CascadePlan plan = cascade_plan(batch, max_blocks_per_seq, shared_blocks, sms);
    if (workspace_bytes < plan.total) return PA_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    float *pre_o = reinterpret_cast<float *>(ws + plan.pre_o_offset);
    float *pre_lse = reinterpret_cast<float *>(ws + plan.pre_lse_offset);

    // 1. every query over the shared prefix (block_table row 0), split over keys, on the
    //    tensor cores: normalised fp32 partials and their lse
    CUtensorMap q_map, kp_map, vp_map;
    if (!encode_q_map(&q_map, q, batch) || !encode_pool_map(&kp_map, k_pool, num_blocks, kPrefillKvTile) ||
        !encode_pool_map(&vp_map, v_pool, num_blocks, kPrefillKvTile))
        return PA_ERR_INVALID_ARG;
    PrefillArgs p = {};
    p.out = pre_o;
    p.lse = pre_lse;
    p.block_table = block_table;
    p.max_blocks_per_seq = shared_blocks;
    p.num_blocks = num_blocks;
    p.cu_q_lens = nullptr;
    p.seq_lens = nullptr;
    p.num_seqs = 1;
    p.total_tokens = batch;
    p.max_q_len = batch;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.err = reinterpret_cast<uint32_t *>(ws);
    p.prefix_len = shared_blocks * kBlock;
    p.kv_split_tiles = plan.kv_split_tiles;
    p.n_kv_splits = plan.n_kv_splits;
    p.order = nullptr;
    if (launch_prefill_prefix(p, q_map, kp_map, vp_map, sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_CUDA;
    // 2. each sequence's private suffix, merged with the prefix partials
    const CascadeExtras cx = {shared_blocks * kBlock, pre_o, pre_lse, plan.n_kv_splits, shared_blocks};
    return decode_impl(shape, out, lse, q, nullptr, nullptr, k_pool, v_pool, block_table, max_blocks_per_seq,
                       num_blocks, seq_lens, batch, scale, 0, workspace, plan.decode_bytes, stream, &cx);
}

pa_status pa_selftest_wait_timeout(void *workspace, size_t workspace_bytes, uint32_t timeout_us, void *stream) {
    if (!workspace || workspace_bytes < kHeaderBytes || timeout_us == 0 || timeout_us > 10000000u)
        return PA_ERR_INVALID_ARG;
    return launch_wait_selftest(static_cast<uint32_t *>(workspace), (uint64_t)timeout_us * 1000ull,
                                static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

}  // extern "C"
