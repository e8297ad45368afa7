// decode.cu -- batched single-token GQA attention over the paged KV cache.
//
// Page "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎，C++/CUDA 实现性能追平 98%":
//   §4.4.2 gqa_decode_attn  the query heads of one group share one KV read: the 4
//                           query heads of KV group g are 4g .. 4g + 3;
//   §4.3.1                  KV in 256-token blocks reached through a block table.
// Page "从零手搓AI推理引擎：避开调包陷阱的工程实践指南" §2.2: softmax(QK^T/sqrt(d))V with
// the maximum subtracted first.
//
// Decode reads every context byte once and does ~4 flops per byte, so it is bound by
// HBM bandwidth.  Design:
//   * grid (sequence x KV head, split): one CTA streams a contiguous range of the
//     context (split-K over KV blocks) for ONE KV head and serves all 4 query heads of
//     that group, so each K/V byte is read once;
//   * a producer warp issues TMA tile loads (64 tokens x 128 dims of one KV head,
//     128-byte swizzle) straight from the paged pool: the block-table walk is the TMA
//     coordinate; a 3-stage mbarrier ring keeps ~64 KiB per CTA in flight;
//   * 4 consumer warps each take 16 tokens of a tile: S^T = K Q^T and O^T += V^T P^T
//     on mma.sync (bf16 in, fp32 accumulate) -- the tensor cores here only save
//     issue slots, the bound is HBM -- with an online softmax in fp32 (exp2 with
//     scale*log2(e) folded in) and warp-shuffle row reductions;
//   * the warps' partial states merge in shared memory; with several splits each CTA
//     writes (O, m, l) to the workspace and the last CTA of the (sequence, KV head)
//     merges them by log-sum-exp and writes bf16 output (+ optional lse).
// Tokens past the context end inside the last tile are masked in the scores and
// their V rows are zeroed in registers, so uninitialised (even NaN) slots never
// reach the result.  A block id outside the pool is replaced by block 0 for the read,
// recorded in the error word and makes the (sequence, KV head)'s output NaN.
// The kernel is launched as a programmatic dependent of the previous kernel on the
// stream, so its launch and prologue overlap e.g. the kv_append that precedes it.
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

namespace pa {
namespace {

constexpr int kTile = kDecodeTileTokens;      // 64 tokens per stage
#ifndef PA_DECODE_STAGES
#define PA_DECODE_STAGES 3
#endif
constexpr int kStages = PA_DECODE_STAGES;      // pipeline depth (a compile-time tuning knob)
constexpr int kConsumerWarps = kTile / 16;    // 4
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kHalfBytes = kTile * 128;       // 64 tokens x 64 dims x 2 B
constexpr int kStageBytes = 4 * kHalfBytes;   // K lo/hi + V lo/hi = 32 KiB
constexpr float kLn2 = 0.693147180559945309f;

struct DecodeSmem {
    uint8_t tiles[kStages][4][kHalfBytes];    // [stage][K lo, K hi, V lo, V hi]
    float o[kConsumerWarps][kGroup][kD];
    float m[kConsumerWarps][kGroup];
    float l[kConsumerWarps][kGroup];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int last_cta;
    int poison;                                // a block id of this split was out of range
    float cl_ml[kGroup][2];                    // cluster merge: this split's (m, l) per head
};

constexpr size_t kSmemBytes = sizeof(DecodeSmem) + 1024;  // + alignment slack

// One log-sum-exp merge step: fold a split's (m, l, o) into the running (M, L, o4).  Written
// once, with explicit fused multiply-adds, so that every merge path rounds identically.
__device__ __forceinline__ void merge_split(float &M, float &L, float (&o)[4], float mk, float lk, float4 ok) {
    const float mn = fmaxf(M, mk);
    const float e_old = fast_exp2(M - mn), e_k = fast_exp2(mk - mn);
    L = __fmaf_rn(lk, e_k, L * e_old);
    o[0] = __fmaf_rn(ok.x, e_k, o[0] * e_old);
    o[1] = __fmaf_rn(ok.y, e_k, o[1] * e_old);
    o[2] = __fmaf_rn(ok.z, e_k, o[2] * e_old);
    o[3] = __fmaf_rn(ok.w, e_k, o[3] * e_old);
    M = mn;
}

// Fold the shared-prefix partials of output row (b, qh) into (M, L, o): M in log2 units,
// o unnormalised; each partial is a normalised output with weight e^lse.
__device__ __forceinline__ void fold_prefix(const DecodeArgs &a, int b, int qh, int d0, float &M, float &L,
                                            float (&o)[4]) {
    for (int k = 0; k < a.pre_n; ++k) {
        const size_t row = ((size_t)k * a.batch + b) * kHq + qh;
        const float mk = __ldcg(a.pre_lse + row) * 1.4426950408889634f;
        const float4 ok = __ldcg(reinterpret_cast<const float4 *>(a.pre_o + row * kD + d0));
        merge_split(M, L, o, mk, 1.f, ok);   // a normalised partial: weight e^lse
    }
}

// A cascade is only valid if this sequence's first shared_blocks table entries are row 0's
// (the prefix partials were computed from row 0): checked by each warp writing an output.
__device__ __forceinline__ bool shared_table_mismatch(const DecodeArgs &a, const int32_t *bt, int lane) {
    bool bad = false;
    for (int j = lane; j < a.shared_blocks; j += 32) bad |= __ldg(bt + j) != __ldg(a.block_table + j);
    return __any_sync(0xffffffffu, bad);
}

__device__ __forceinline__ void store_out4(__nv_bfloat16 *dst, const float (&v)[4], float inv) {
    uint2 w;
    w.x = pack_bf16x2(v[0] * inv, v[1] * inv);
    w.y = pack_bf16x2(v[2] * inv, v[3] * inv);
    *reinterpret_cast<uint2 *>(dst) = w;
}

// ------------------------------------------------------------------ cluster merge
// Every thread of every CTA of the cluster (a pair's splits).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// kCluster: the splits of one (sequence, KV head) form a thread-block cluster (at most 8,
// launched when the whole grid fits in one wave).  Split 0 merges the pair's partials straight
// from its peers' shared memory after a cluster barrier, instead of through the workspace and
// an atomic counter; splits past the context do no work but still meet the others at both
// cluster barriers (so no barrier waits on a CTA that has left).  Same merge order and
// arithmetic as the workspace path, so the results are bit-identical.
template <bool kCluster>
__global__ void __launch_bounds__(kThreads, 2)
decode_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
              const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    DecodeSmem &sm = *reinterpret_cast<DecodeSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int pair = blockIdx.x;          // sequence * 8 + kv head
    const int b = pair / kHkv;
    const int g = pair % kHkv;
    // CTAs start in the order of their linear index (x fastest).  Without a cluster the
    // highest splits go first: only long contexts have them and their splits are the longest,
    // so the long work starts early and the short single splits of short contexts fill the
    // tail (close to longest-first, at no cost: the split index alone decides).
    const int split = kCluster ? (int)blockIdx.y : (int)(gridDim.y - 1 - blockIdx.y);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // A sequence's n context tokens are cut into nsplit_b = ceil(n / split_tokens) splits
    // of equal length (rounded up to the tile), so the CTAs of one wave end at different
    // times and no split is a small remainder.  Each split starts at or after
    // split * split_tokens / 2 (for nsplit_b >= 2 the length exceeds split_tokens / 2):
    // the producer warp fetches the 32 block-table entries from there on (and the tensor
    // maps) while everyone fetches seq_len, so the first tile load is usually one memory
    // round trip from the kernel's start.
    const int32_t *bt = a.block_table + (size_t)b * a.max_blocks_per_seq;
    const int wlo = (a.kv_begin + split * (a.split_tokens >> 1)) / kBlock;
    int bwin = 0;
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            tma_prefetch_map(&k_map);
            tma_prefetch_map(&v_map);
        }
        if (wlo + lane < a.max_blocks_per_seq) bwin = __ldg(bt + wlo + lane);
    }
    const int seq_len = __ldg(a.seq_lens + b);
    // (a cascade attends only past the shared prefix: the context must extend beyond it)
    if (seq_len < 1 || seq_len > a.max_blocks_per_seq * kBlock || seq_len <= a.kv_begin) {
        if (split == 0 && g == 0 && threadIdx.x == 0) record_error(a.err, kErrDevice | kErrBadSeqLen);
        if constexpr (kCluster) {
            cluster_sync_all();
            cluster_sync_all();
        }
        return;  // every CTA of this sequence takes the same exit: counters untouched
    }
    const int n_ctx = seq_len - a.kv_begin;
    const int nsplit_b = (n_ctx + a.split_tokens - 1) / a.split_tokens;
    if (split >= nsplit_b) {              // this split lies past the context
        if constexpr (kCluster) {
            cluster_sync_all();
            cluster_sync_all();
        }
        return;
    }
    const int len_b = ((n_ctx + nsplit_b - 1) / nsplit_b + kTile - 1) / kTile * kTile;
    const int t_begin = a.kv_begin + split * len_b;
    const int t_end = min(t_begin + len_b, seq_len);
    const int n_tiles = (t_end - t_begin + kTile - 1) / kTile;

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sm.full[s]), 1);
            mbar_init(smem_u32(&sm.empty[s]), kConsumerWarps);
        }
        sm.poison = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ TMA producer
        const int wi = t_begin / kBlock - wlo;   // >= 0; beyond the window: fetch it now
        int blk0 = __shfl_sync(0xffffffffu, bwin, wi & 31);
        if (wi < 0 || wi >= 32) blk0 = __ldg(bt + t_begin / kBlock);
        if (lane == 0) {
            // The pools may be written by the kernel just before this one on the stream
            // (kv_append lets us launch early): wait for it before the first pool read.
            // The consumer warps wait too, before reading q or k_new / v_new.
            asm volatile("griddepcontrol.wait;" ::: "memory");
            int issued = 0;
            for (int i = 0; i < n_tiles; ++i) {
                const int st = i % kStages;
                if (i >= kStages && !mbar_wait(smem_u32(&sm.empty[st]), ((i / kStages) - 1) & 1)) {
                    record_error(a.err, kErrTimeout);
                    break;
                }
                const int tok = t_begin + i * kTile;
                int blk = i == 0 ? blk0 : __ldg(bt + tok / kBlock);
                if (blk < 0 || blk >= a.num_blocks) {
                    // a block id outside the pool: read block 0 instead and poison the result
                    record_error(a.err, kErrDevice | kErrBadBlock);
                    sm.poison = 1;
                    blk = 0;
                }
                const int off = tok % kBlock;
                const uint32_t bar = smem_u32(&sm.full[st]);
                mbar_arrive_expect_tx(bar, kStageBytes);
                tma_load_4d(smem_u32(sm.tiles[st][0]), &k_map, bar, 0, g, off, blk);
                tma_load_4d(smem_u32(sm.tiles[st][1]), &k_map, bar, 64, g, off, blk);
                tma_load_4d(smem_u32(sm.tiles[st][2]), &v_map, bar, 0, g, off, blk);
                tma_load_4d(smem_u32(sm.tiles[st][3]), &v_map, bar, 64, g, off, blk);
                issued = i + 1;
            }
            // No copy may still be landing in shared memory when the CTA exits.
            for (int i = max(0, issued - kStages); i < issued; ++i)
                mbar_wait(smem_u32(&sm.full[i % kStages]), (i / kStages) & 1);
        }
        if constexpr (kCluster) {
            __syncwarp();
            cluster_sync_all();
            cluster_sync_all();
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int w = warp;
    const int gq = lane >> 2;   // fragment row group
    const int tq = lane & 3;    // fragment column pair
    const int mi = lane >> 3;   // ldmatrix: which 8x8 matrix this lane addresses
    const int ri = lane & 7;    // ldmatrix: row within it

    // q, k_new and v_new may come from the kernel just before this one on the stream, and
    // the pools may still be read by it: wait for it before the first access to any of them
    // (only block_table and seq_lens are read earlier).
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // Q^T as the B operand of S^T = K Q^T: [k = 16 dims] x [n = 8 heads], heads 4..7 zero.
    uint32_t qb[8][2];
    {
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
            static_cast<const __nv_bfloat16 *>(a.q) + ((size_t)b * kHq + g * kGroup + (gq & 3)) * kD);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            qb[kk][0] = gq < kGroup ? __ldg(qrow + kk * 8 + tq) : 0u;
            qb[kk][1] = gq < kGroup ? __ldg(qrow + kk * 8 + 4 + tq) : 0u;
        }
    }

    float m0 = -INFINITY, m1 = -INFINITY;   // running max (log2 units) of heads 2tq, 2tq+1
    float l0 = 0.f, l1 = 0.f;               // this thread's share of the running sums
    float acc[8][4];                        // O^T tiles: 16 dims x 8 heads each
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;

    const int row_qk = w * 16 + ri + ((mi & 1) << 3);   // token row for the K fragment
    const int row_pv = w * 16 + ri + ((mi >> 1) << 3);  // token row for the V^T fragment

    // Fused append (k_new / v_new given): the CTA whose range ends the context owns the new
    // token at position seq_len-1.  The warp whose 16 rows hold it fetches the token's K and
    // V row of this KV head now (lanes 0-15: K, 16-31: V, 16 bytes each), stores them into the
    // pool and patches them over the (stale) row of the landed tile before using it.
    const int p_new = seq_len - 1;
    const int i_new = (a.k_new && t_end == seq_len) ? (p_new - t_begin) / kTile : -1;
    const int r_new = (p_new - t_begin) % kTile;        // row within that tile
    const bool new_here = i_new >= 0 && (r_new >> 4) == w;
    uint4 new_chunk = make_uint4(0u, 0u, 0u, 0u);
    if (new_here) {
        const int kv = lane >> 4, chunk = lane & 15;
        const uint4 *src = reinterpret_cast<const uint4 *>(
            static_cast<const char *>(kv ? a.v_new : a.k_new) + ((size_t)b * kHkv + g) * kRowBytes);
        new_chunk = __ldg(src + chunk);
        const int blk = __ldg(bt + p_new / kBlock);
        if (blk >= 0 && blk < a.num_blocks) {
            uint4 *dst = reinterpret_cast<uint4 *>(
                static_cast<char *>(kv ? a.v_pool_w : a.k_pool_w) +
                (((size_t)blk * kBlock + p_new % kBlock) * kHkv + g) * kRowBytes);
            dst[chunk] = new_chunk;
        }   // a bad block id is reported by the producer and poisons the result
    }

    for (int i = 0; i < n_tiles; ++i) {
        const int st = i % kStages;
        if (!mbar_wait(smem_u32(&sm.full[st]), (i / kStages) & 1)) {
            if (lane == 0) record_error(a.err, kErrTimeout);
            break;
        }
        if (new_here && i == i_new) {
            // the new token's row: 16-byte chunk c of the K (V) row goes to half c / 8,
            // swizzled chunk c % 8 of row r_new
            const int kv = lane >> 4, chunk = lane & 15;
            uint8_t *tile = sm.tiles[st][kv * 2 + (chunk >> 3)];
            *reinterpret_cast<uint4 *>(tile + sw128(r_new, chunk & 7)) = new_chunk;
            fence_proxy_async_smem();   // generic writes before the stage is refilled by TMA
            __syncwarp();
        }
        const int my_valid = min(max(t_end - (t_begin + i * kTile) - w * 16, 0), 16);
        if (my_valid > 0) {
            const uint32_t k_lo = smem_u32(sm.tiles[st][0]);
            const uint32_t k_hi = smem_u32(sm.tiles[st][1]);
            const uint32_t v_lo = smem_u32(sm.tiles[st][2]);
            const uint32_t v_hi = smem_u32(sm.tiles[st][3]);

            // S^T[16 tokens x 8 heads] = K[16 x 128] . Q^T[128 x 8]
            float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t af[4];
                const uint32_t base = kk < 4 ? k_lo : k_hi;
                ldsm_x4(af, base + sw128(row_qk, ((kk & 3) << 1) + (mi >> 1)));
                mma_16816(s, af, qb[kk][0], qb[kk][1]);
            }
            // s[0]: (token gq, head 2tq)   s[1]: (token gq, head 2tq+1)
            // s[2]: (token gq+8, head 2tq) s[3]: (token gq+8, head 2tq+1)
            float x0, x1, x2, x3;
            if (tq < 2) {
                const bool v_lo_ok = gq < my_valid;
                const bool v_hi_ok = gq + 8 < my_valid;
                x0 = v_lo_ok ? s[0] * a.scale_log2 : -INFINITY;
                x1 = v_lo_ok ? s[1] * a.scale_log2 : -INFINITY;
                x2 = v_hi_ok ? s[2] * a.scale_log2 : -INFINITY;
                x3 = v_hi_ok ? s[3] * a.scale_log2 : -INFINITY;
            } else {  // padding heads 4..7: finite dummies, results discarded
                x0 = x1 = x2 = x3 = 0.f;
            }
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float alpha0 = fast_exp2(m0 - mn0), alpha1 = fast_exp2(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            const float p0 = fast_exp2(x0 - m0), p1 = fast_exp2(x1 - m1);
            const float p2 = fast_exp2(x2 - m0), p3 = fast_exp2(x3 - m1);
            // P enters the PV product as bf16; the sums use those same rounded weights.
            const uint32_t pp_lo = pack_bf16x2(p0, p1);   // token gq:   heads 2tq, 2tq+1
            const uint32_t pp_hi = pack_bf16x2(p2, p3);   // token gq+8: heads 2tq, 2tq+1
            l0 = l0 * alpha0 + bf16_lo(pp_lo) + bf16_lo(pp_hi);
            l1 = l1 * alpha1 + bf16_hi(pp_lo) + bf16_hi(pp_hi);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                acc[mt][0] *= alpha0;
                acc[mt][1] *= alpha1;
                acc[mt][2] *= alpha0;
                acc[mt][3] *= alpha1;
            }
            // P^T as the B operand of O^T += V^T P^T: transpose the 8x8 bf16 blocks.
            const uint32_t pb0 = movmatrix_trans(pp_lo);
            const uint32_t pb1 = movmatrix_trans(pp_hi);
            // V rows past the context end are zeroed in the fragment (0 * NaN = NaN).
            const uint32_t keep_lo = (2 * tq < my_valid ? 0x0000ffffu : 0u) |
                                     (2 * tq + 1 < my_valid ? 0xffff0000u : 0u);
            const uint32_t keep_hi = (2 * tq + 8 < my_valid ? 0x0000ffffu : 0u) |
                                     (2 * tq + 9 < my_valid ? 0xffff0000u : 0u);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                uint32_t af[4];
                const uint32_t base = mt < 4 ? v_lo : v_hi;
                ldsm_x4_trans(af, base + sw128(row_pv, ((mt & 3) << 1) + (mi & 1)));
                af[0] &= keep_lo;
                af[1] &= keep_lo;
                af[2] &= keep_hi;
                af[3] &= keep_hi;
                mma_16816(acc[mt], af, pb0, pb1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.empty[st]));
    }

    // ------------------------------------------------------------ merge the 4 warps
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    if (tq < 2) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int d = mt * 16 + gq;
            sm.o[w][2 * tq][d] = acc[mt][0];
            sm.o[w][2 * tq + 1][d] = acc[mt][1];
            sm.o[w][2 * tq][d + 8] = acc[mt][2];
            sm.o[w][2 * tq + 1][d + 8] = acc[mt][3];
        }
        if (gq == 0) {
            sm.m[w][2 * tq] = m0;
            sm.m[w][2 * tq + 1] = m1;
            sm.l[w][2 * tq] = l0;
            sm.l[w][2 * tq + 1] = l1;
        }
    }
    named_barrier(1, kConsumerWarps * 32);
    const bool bad = *reinterpret_cast<volatile int *>(&sm.poison) != 0;

    const int c = threadIdx.x;          // 0..127
    const int h = c >> 5;               // query head within the group
    const int d0 = (c & 31) * 4;        // 4 dims per thread
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kConsumerWarps; ++ww) M = fmaxf(M, sm.m[ww][h]);
    float L = 0.f, o4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ww = 0; ww < kConsumerWarps; ++ww) {
        const float e = fast_exp2(sm.m[ww][h] - M);
        L += sm.l[ww][h] * e;
#pragma unroll
        for (int k = 0; k < 4; ++k) o4[k] += sm.o[ww][h][d0 + k] * e;
    }
    if (bad) {
        M = L = __int_as_float(0x7fc00000);
#pragma unroll
        for (int k = 0; k < 4; ++k) o4[k] = __int_as_float(0x7fc00000);
    }
    const int qh = g * kGroup + h;      // query head
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + ((size_t)b * kHq + qh) * kD + d0;

    if constexpr (kCluster) {
        // This split's partial into its own shared memory: thread c alone read entries
        // [.][h][d0 .. d0+3] of the merge area, so it may overwrite warp 0's without a barrier.
        *reinterpret_cast<float4 *>(&sm.o[0][h][d0]) = make_float4(o4[0], o4[1], o4[2], o4[3]);
        if ((c & 31) == 0) {
            sm.cl_ml[h][0] = M;
            sm.cl_ml[h][1] = L;
        }
        cluster_sync_all();   // every split's partial is in place
        if (split == 0) {
            float GM = M, GL = L, go[4] = {o4[0], o4[1], o4[2], o4[3]};
            if (nsplit_b > 1) {
                // by log-sum-exp in split order, as the workspace merge (split 0 from registers)
                GM = -INFINITY;
                GL = 0.f;
#pragma unroll
                for (int k = 0; k < 4; ++k) go[k] = 0.f;
                for (int k = 0; k < nsplit_b; ++k) {
                    float mk = M, lk = L;
                    float4 ok = make_float4(o4[0], o4[1], o4[2], o4[3]);
                    if (k > 0) {
                        mk = ld_cluster_f32(peer_addr(smem_u32(&sm.cl_ml[h][0]), (uint32_t)k));
                        lk = ld_cluster_f32(peer_addr(smem_u32(&sm.cl_ml[h][1]), (uint32_t)k));
                        ok = ld_cluster_f4(peer_addr(smem_u32(&sm.o[0][h][d0]), (uint32_t)k));
                    }
                    merge_split(GM, GL, go, mk, lk, ok);
                }
            }
            if (a.pre_n > 0) {
                fold_prefix(a, b, qh, d0, GM, GL, go);
                if (shared_table_mismatch(a, bt, c & 31)) {
                    if ((c & 31) == 0) record_error(a.err, kErrDevice | kErrBadBlock);
                    GM = GL = __int_as_float(0x7fc00000);
                }
            }
            store_out4(out, go, 1.f / GL);
            if (a.lse && (c & 31) == 0) a.lse[(size_t)b * kHq + qh] = (GM + __log2f(GL)) * kLn2;
        }
        cluster_sync_all();   // the peers' shared memory stays until split 0 has read it
        return;
    }

    if (nsplit_b == 1) {
        if (a.pre_n > 0) {
            fold_prefix(a, b, qh, d0, M, L, o4);
            if (shared_table_mismatch(a, bt, c & 31)) {
                if ((c & 31) == 0) record_error(a.err, kErrDevice | kErrBadBlock);
                M = L = __int_as_float(0x7fc00000);
            }
        }
        store_out4(out, o4, 1.f / L);
        if (a.lse && (c & 31) == 0) a.lse[(size_t)b * kHq + qh] = (M + __log2f(L)) * kLn2;
        return;
    }

    // ------------------------------------------------------------ split-K partials
    const size_t entry = (size_t)pair * a.nsplit + split;
    *reinterpret_cast<float4 *>(a.part_o + (entry * kGroup + h) * kD + d0) =
        make_float4(o4[0], o4[1], o4[2], o4[3]);
    if ((c & 31) == 0) {
        a.part_ml[(entry * kGroup + h) * 2 + 0] = M;
        a.part_ml[(entry * kGroup + h) * 2 + 1] = L;
    }
    // Count this split in with one release/acquire atomic: the barrier orders every
    // thread's partial stores before thread 0's release, and the acquire of the CTA that
    // counts last (then the barrier) orders its loads of the others' partials after them.
    named_barrier(1, kConsumerWarps * 32);
    if (c == 0) {
        int prev;
        asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(a.counters + pair) : "memory");
        sm.last_cta = (prev == nsplit_b - 1);
    }
    named_barrier(1, kConsumerWarps * 32);
    if (!sm.last_cta) return;

    // The last CTA of this (sequence, KV head) merges every split by log-sum-exp, in split
    // order whichever CTA it is (its own split from registers: the same values), with the
    // loads of four splits issued together.
    if (c == 0) a.counters[pair] = 0;   // ready for the next call
    const size_t e0 = (size_t)pair * a.nsplit;
    float GM = -INFINITY, GL = 0.f, go[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < nsplit_b; k0 += 4) {
        float mk[4], lk[4];
        float4 ok[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = k0 + u;
            if (k == split) {
                mk[u] = M;
                lk[u] = L;
                ok[u] = make_float4(o4[0], o4[1], o4[2], o4[3]);
            } else if (k < nsplit_b) {
                mk[u] = __ldcg(a.part_ml + ((e0 + k) * kGroup + h) * 2);
                lk[u] = __ldcg(a.part_ml + ((e0 + k) * kGroup + h) * 2 + 1);
                ok[u] = __ldcg(reinterpret_cast<const float4 *>(a.part_o + ((e0 + k) * kGroup + h) * kD + d0));
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (k0 + u >= nsplit_b) break;
            merge_split(GM, GL, go, mk[u], lk[u], ok[u]);
        }
    }
    if (a.pre_n > 0) {
        fold_prefix(a, b, qh, d0, GM, GL, go);
        if (shared_table_mismatch(a, bt, c & 31)) {
            if ((c & 31) == 0) record_error(a.err, kErrDevice | kErrBadBlock);
            GM = GL = __int_as_float(0x7fc00000);
        }
    }
    store_out4(out, go, 1.f / GL);
    if (a.lse && (c & 31) == 0) a.lse[(size_t)b * kHq + qh] = (GM + __log2f(GL)) * kLn2;
}

}  // namespace

cudaError_t configure_decode() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<bool> configured[64] = {};
    if (dev < 0 || dev >= 64 || !configured[dev].load()) {
        e = cudaFuncSetAttribute(decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev].store(true);
    }
    return cudaSuccess;
}

cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &k_map, const CUtensorMap &v_map,
                          int num_sms, cudaStream_t stream) {
    (void)num_sms;
    if (a.batch == 0) return cudaSuccess;
    cudaError_t e = configure_decode();
    if (e != cudaSuccess) return e;
    // Programmatic dependent launch: the prologue may overlap the previous kernel on the
    // stream; the producer waits for it (griddepcontrol.wait) before reading the pools.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.batch * kHkv, a.nsplit);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.cluster_merge) {
        if (a.nsplit < 1 || a.nsplit > 8) return cudaErrorInvalidValue;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 1;
        attr[1].val.clusterDim.y = (unsigned)a.nsplit;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, decode_kernel<true>, k_map, v_map, a);
        if (e != cudaErrorLaunchOutOfResources && e != cudaErrorInvalidClusterSize && e != cudaErrorNotSupported &&
            e != cudaErrorCooperativeLaunchTooLarge)
            return e;
        // The cluster was refused (e.g. SMs partitioned or shared with other work): clear the
        // launch error and merge through the workspace and counters instead, which gives the
        // same bits (both merges run the same steps in the same order).
        cudaGetLastError();
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, decode_kernel<false>, k_map, v_map, a);
}

// ------------------------------------------------------------------ fixed scratch
// Scratch for paged_attn_decode_static, for callers that cannot allocate device memory
// themselves (no cudaMalloc allowed, no workspace handed to them): the split-K partial
// results, the merge counters and an error word live in this file-scope array instead
// of a caller workspace.  Every GPU that loads the library keeps these bytes reserved
// until the process exits, and all calls share them.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Unique ID of the context current on this thread (0 if none is current or the driver
// cannot say).  The driver entry points are looked up once through the runtime, so the
// library needs no link-time dependency on libcuda.
static unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

void *static_scratch_address(cudaError_t *status) {
    // In host code g_static_scratch names a host-side stand-in, not device memory: the
    // device address comes from cudaGetSymbolAddress, looked up while the device is
    // current.  The address belongs to the context the module was loaded into, so it is
    // cached per context (a context torn down and created again, e.g. after
    // cudaDeviceReset, gets a fresh lookup); where the context cannot be identified it is
    // looked up on every call (the lookup allocates nothing).
    static std::mutex mu;
    struct Entry {
        unsigned long long ctx;
        void *ptr;
    };
    static Entry cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        *status = e != cudaSuccess ? e : cudaErrorInvalidDevice;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    unsigned long long ctx = current_context_id();
    if (ctx != 0 && cache[dev].ctx == ctx && cache[dev].ptr) {
        *status = cudaSuccess;
        return cache[dev].ptr;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);   // also creates the context if needed
    if (e != cudaSuccess) {
        *status = e;
        return nullptr;
    }
    if (ctx == 0) ctx = current_context_id();
    cache[dev].ctx = ctx;
    cache[dev].ptr = ctx != 0 ? p : nullptr;
    *status = cudaSuccess;
    return p;
}

}  // namespace pa
