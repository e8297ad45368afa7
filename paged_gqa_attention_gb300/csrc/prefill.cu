// prefill.cu -- causal (chunked) prefill attention over the paged KV cache on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory, TMA-fed).
//
// Page "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎，C++/CUDA 实现性能追平 98%":
//   §4.4.1 flash_attn_prefill  tiled attention that never builds the N x N matrix and
//                              skips key tiles after the query tile (causal);
//   §4.4.2                     four query heads share one KV head.
// Page "从零搭建AI工程能力：手写KV Cache与动态批处理实战" §3.3: long prompts are cut into
// chunks that attend to the cached context before them (chunked prefill).
// Page "从零手搓AI推理引擎：避开调包陷阱的工程实践指南" §2.2: softmax(QK^T/sqrt(d))V,
// maximum subtracted first; a position sees itself and earlier positions.
//
// The pages' FlashAttention-2 loop renormalises nothing between key tiles; here the
// running max/sum of the online softmax does that (the plain definition is the target).
//
// Work tile: 32 query positions x the 4 query heads of one KV head = 128 MMA rows
// (row r = position (r / 4), head (r % 4)), so every K/V tile fetched serves 4 heads.
// Key/value tiles are 128 tokens (half a cache block) fetched by TMA straight from
// the paged pool: the block table lookup is the TMA coordinate.
//
// CTA = 6 warps, persistent (one per SM), tiles dealt in a snake order, latest query
// blocks (most keys) first:
//   warps 0-3  softmax + epilogue; thread r owns MMA row r (= TMEM lane r)
//   warp 4     TMA producer (Q double-buffered, K and V rings of 2 stages)
//   warp 5     TMEM allocator and the single-thread tcgen05.mma issuer
// Tensor memory (512 columns): S0, S1 (fp32 scores, 128 cols each), O (fp32, 128),
// P0, P1 (bf16 probabilities packed in pairs, 64 cols each).
// Per key tile:  S = Q K^T (SS-MMA)  ->  softmax reads S, writes P (bf16) into TMEM
// and, when its running max rose by more than 2^8, rescales O  ->  O += P V (TS-MMA,
// P from TMEM, V from shared memory, MN-major).  The MMA warp issues S for tile j+1
// before O += P V for tile j, so the tensor core works while the softmax runs.
// Every wait is bounded; on expiry the CTA records PA_ERR_TIMEOUT, unwinds, waits
// (bounded) for its own copies and MMAs, frees tensor memory and exits.
#include "common.cuh"
#include "launch.h"

namespace pa {
namespace {

constexpr int kRows = 128;                  // MMA M
constexpr int kKT = kPrefillKvTile;         // keys per tile (MMA N of S, K of PV)
constexpr int kQPos = kPrefillQPositions;   // query positions per tile
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128;   // score buffers
constexpr uint32_t kColO = 256;                // output accumulator
constexpr uint32_t kColP0 = 384, kColP1 = 448; // probability buffers
__device__ __forceinline__ uint32_t col_s(int st) { return st ? kColS1 : kColS0; }
__device__ __forceinline__ uint32_t col_p(int st) { return st ? kColP1 : kColP0; }
constexpr int kHalf = kRows * 128;          // 128 rows x 64 dims x 2 B = 16 KiB
constexpr uint32_t kTileBytes = 2 * kHalf;  // a full 128 x 128 bf16 tile
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O when the max grows > 2^8
constexpr float kLn2 = 0.693147180559945309f;
constexpr uint32_t kIdescQK = idesc_bf16(kRows, kKT, false);  // B = K tile, K-major
constexpr uint32_t kIdescPV = idesc_bf16(kRows, kD, true);    // B = V tile, MN-major

struct PrefillSmem {
    uint8_t q[2][2][kHalf];   // [buffer][dims 0-63 | 64-127]
    uint8_t k[2][2][kHalf];   // [stage][half]
    uint8_t v[2][2][kHalf];
    uint64_t q_full[2], q_empty[2];
    uint64_t k_full[2], k_empty[2];
    uint64_t v_full[2], v_empty[2];
    uint64_t s_full[2], s_free[2], p_full[2];
    uint64_t o_done;
    uint64_t mma_idle;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = sizeof(PrefillSmem) + 1024;

struct Tile {
    bool run;       // has work
    bool error;     // inconsistent lengths (recorded once, then skipped)
    int s, g;
    int tok0;       // row of q/out holding the tile's first query position
    int rows;       // real positions in this tile (1..32)
    int pos0;       // absolute position of the tile's first query
    int seq_len;    // context length (keys 0 .. seq_len-1 exist)
    int n_kt;       // key tiles to visit: 0 .. (last position) / 128
};

__device__ __forceinline__ Tile tile_at(const PrefillArgs &a, int idx, int qblocks) {
    Tile t;
    const int per_qb = a.num_seqs * kHkv;
    const int qb = qblocks - 1 - idx / per_qb;   // latest query block first
    const int rem = idx - (idx / per_qb) * per_qb;
    t.s = rem / kHkv;
    t.g = rem % kHkv;
    t.run = false;
    t.error = false;
    const int c0 = __ldg(a.cu_q_lens + t.s);
    const int c1 = __ldg(a.cu_q_lens + t.s + 1);
    const int q_len = c1 - c0;
    const int seq_len = __ldg(a.seq_lens + t.s);
    if (q_len < 0 || q_len > a.max_q_len || c0 < 0 || c1 > a.total_tokens ||
        (q_len > 0 && (seq_len < q_len || seq_len > a.max_blocks_per_seq * kBlock))) {
        t.error = true;
        return t;
    }
    if (qb * kQPos >= q_len) return t;
    t.run = true;
    t.tok0 = c0 + qb * kQPos;
    t.rows = min(kQPos, q_len - qb * kQPos);
    t.pos0 = seq_len - q_len + qb * kQPos;
    t.seq_len = seq_len;
    t.n_kt = (t.pos0 + t.rows - 1) / kKT + 1;
    return t;
}

// Index of this CTA's r-th tile in the snake order (or -1 past the end).
__device__ __forceinline__ int snake(int r, int total) {
    const int G = gridDim.x;
    const int idx = r * G + ((r & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
    return idx < total ? idx : -1;
}

// Bounded wait shared by all roles: gives up when another role has aborted or after
// the time limit (then raises the abort flag and records the timeout).
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              uint32_t *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            record_error(err, kErrTimeout);
            return false;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
               const __grid_constant__ CUtensorMap v_map, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    PrefillSmem &sm = *reinterpret_cast<PrefillSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    volatile int *abort_flag = &sm.abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int qblocks = (a.max_q_len + kQPos - 1) / kQPos;
    const int total = a.num_seqs * kHkv * qblocks;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sm.q_full[i]), 1);
            mbar_init(smem_u32(&sm.q_empty[i]), 1);
            mbar_init(smem_u32(&sm.k_full[i]), 1);
            mbar_init(smem_u32(&sm.k_empty[i]), 1);
            mbar_init(smem_u32(&sm.v_full[i]), 1);
            mbar_init(smem_u32(&sm.v_empty[i]), 1);
            mbar_init(smem_u32(&sm.s_full[i]), 1);
            mbar_init(smem_u32(&sm.s_free[i]), 4);   // one arrive per softmax warp
            mbar_init(smem_u32(&sm.p_full[i]), 4);
        }
        mbar_init(smem_u32(&sm.o_done), 1);
        mbar_init(smem_u32(&sm.mma_idle), 1);
        sm.abort = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            tma_prefetch_map(&q_map);
            tma_prefetch_map(&k_map);
            tma_prefetch_map(&v_map);
            int tcount = 0, it = 0;              // tiles / key tiles started
            int q_issued = 0, k_issued = 0, v_issued = 0;
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int idx = snake(r, total);
                if (idx < 0) break;
                const Tile t = tile_at(a, idx, qblocks);
                if (t.error) record_error(a.err, kErrDevice | kErrQLen);
                if (!t.run) continue;
                const int qbuf = tcount & 1;
                if (tcount >= 2 &&
                    !(ok = wait_or_abort(smem_u32(&sm.q_empty[qbuf]), ((tcount >> 1) - 1) & 1, abort_flag, a.err)))
                    break;
                const uint32_t qbar = smem_u32(&sm.q_full[qbuf]);
                mbar_arrive_expect_tx(qbar, kTileBytes);
                tma_load_3d(smem_u32(sm.q[qbuf][0]), &q_map, qbar, 0, t.g * kGroup, t.tok0);
                tma_load_3d(smem_u32(sm.q[qbuf][1]), &q_map, qbar, 64, t.g * kGroup, t.tok0);
                ++q_issued;
                const int32_t *bt = a.block_table + (size_t)t.s * a.max_blocks_per_seq;
                for (int j = 0; j < t.n_kt; ++j, ++it) {
                    const int st = it & 1;
                    int blk = __ldg(bt + (j >> 1));
                    if (blk < 0 || blk >= a.num_blocks) {
                        record_error(a.err, kErrDevice | kErrBadBlock);
                        blk = 0;   // stay inside the pool; the result is flagged as invalid
                    }
                    const int off = (j & 1) * kKT;
                    if (it >= 2 &&
                        !(ok = wait_or_abort(smem_u32(&sm.k_empty[st]), ((it >> 1) - 1) & 1, abort_flag, a.err)))
                        break;
                    const uint32_t kbar = smem_u32(&sm.k_full[st]);
                    mbar_arrive_expect_tx(kbar, kTileBytes);
                    tma_load_4d(smem_u32(sm.k[st][0]), &k_map, kbar, 0, t.g, off, blk);
                    tma_load_4d(smem_u32(sm.k[st][1]), &k_map, kbar, 64, t.g, off, blk);
                    ++k_issued;
                    if (it >= 2 &&
                        !(ok = wait_or_abort(smem_u32(&sm.v_empty[st]), ((it >> 1) - 1) & 1, abort_flag, a.err)))
                        break;
                    const uint32_t vbar = smem_u32(&sm.v_full[st]);
                    mbar_arrive_expect_tx(vbar, kTileBytes);
                    tma_load_4d(smem_u32(sm.v[st][0]), &v_map, vbar, 0, t.g, off, blk);
                    tma_load_4d(smem_u32(sm.v[st][1]), &v_map, vbar, 64, t.g, off, blk);
                    ++v_issued;
                }
                ++tcount;
            }
            // Drain: no TMA copy may still be landing when the CTA exits.  In the normal
            // path every load has been consumed and these waits return at once.
            for (int i = max(0, q_issued - 2); i < q_issued; ++i)
                mbar_wait(smem_u32(&sm.q_full[i & 1]), (i >> 1) & 1);
            for (int i = max(0, k_issued - 2); i < k_issued; ++i)
                mbar_wait(smem_u32(&sm.k_full[i & 1]), (i >> 1) & 1);
            for (int i = max(0, v_issued - 2); i < v_issued; ++i)
                mbar_wait(smem_u32(&sm.v_full[i & 1]), (i >> 1) & 1);
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int tcount = 0, it = 0;
            int pend_it = -1, pend_j = 0;   // O += P V still to issue for key tile pend_it
            bool ok = true;
            auto issue_pv = [&](int pit, int pj) -> bool {
                const int st = pit & 1;
                if (!wait_or_abort(smem_u32(&sm.v_full[st]), (pit >> 1) & 1, abort_flag, a.err)) return false;
                if (!wait_or_abort(smem_u32(&sm.p_full[st]), (pit >> 1) & 1, abort_flag, a.err)) return false;
                tc_fence_after();
                const uint32_t v0 = smem_u32(sm.v[st][0]);
#pragma unroll
                for (int kk = 0; kk < kKT / 16; ++kk) {
                    // V tile [128 keys][128 dims], dims contiguous (MN-major): 16 keys per step
                    // = two 8-row swizzle atoms (2 KiB); the dim halves are 16 KiB apart.
                    const uint64_t bdesc = sdesc_sw128(v0 + kk * 2048, (uint32_t)kHalf, 1024);
                    umma_ts(tmem + kColO, tmem + col_p(st) + kk * 8, bdesc, kIdescPV,
                            (pj > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(smem_u32(&sm.o_done));
                umma_commit(smem_u32(&sm.v_empty[st]));
                return true;
            };
            for (int r = 0; ok; ++r) {
                const int idx = snake(r, total);
                if (idx < 0) break;
                const Tile t = tile_at(a, idx, qblocks);
                if (!t.run) continue;
                const int qbuf = tcount & 1;
                if (!(ok = wait_or_abort(smem_u32(&sm.q_full[qbuf]), (tcount >> 1) & 1, abort_flag, a.err)))
                    break;
                for (int j = 0; j < t.n_kt; ++j, ++it) {
                    const int st = it & 1;
                    if (!(ok = wait_or_abort(smem_u32(&sm.k_full[st]), (it >> 1) & 1, abort_flag, a.err))) break;
                    if (it >= 2 &&
                        !(ok = wait_or_abort(smem_u32(&sm.s_free[st]), ((it >> 1) - 1) & 1, abort_flag, a.err)))
                        break;
                    tc_fence_after();
                    const uint32_t q0 = smem_u32(sm.q[qbuf][0]);
                    const uint32_t q1 = smem_u32(sm.q[qbuf][1]);
                    const uint32_t k0 = smem_u32(sm.k[st][0]);
                    const uint32_t k1 = smem_u32(sm.k[st][1]);
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        // K-major, 128-byte swizzle: 16 dims = 32 bytes along the row
                        const uint32_t off = (kk & 3) * 32;
                        const uint64_t adesc = sdesc_sw128((kk < 4 ? q0 : q1) + off, 16, 1024);
                        const uint64_t bdesc = sdesc_sw128((kk < 4 ? k0 : k1) + off, 16, 1024);
                        umma_ss(tmem + col_s(st), adesc, bdesc, kIdescQK, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(smem_u32(&sm.s_full[st]));
                    umma_commit(smem_u32(&sm.k_empty[st]));
                    if (j == t.n_kt - 1) umma_commit(smem_u32(&sm.q_empty[qbuf]));
                    if (pend_it >= 0 && !(ok = issue_pv(pend_it, pend_j))) break;
                    pend_it = it;
                    pend_j = j;
                }
                ++tcount;
            }
            if (ok && pend_it >= 0) issue_pv(pend_it, pend_j);
            // Every MMA issued must have finished before tensor memory is released.
            umma_commit(smem_u32(&sm.mma_idle));
            mbar_wait(smem_u32(&sm.mma_idle), 0);
        }
    } else {
        // ---------------------------------------------------------------- softmax warps
        const int row = warp * 32 + lane;          // MMA row == TMEM lane
        const int pl = row >> 2;                   // query position within the tile
        const int hl = row & 3;                    // query head within the group
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        int it = 0;
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int idx = snake(r, total);
            if (idx < 0) break;
            const Tile t = tile_at(a, idx, qblocks);
            if (!t.run) continue;
            const int pos = t.pos0 + pl;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < t.n_kt; ++j, ++it) {
                const int st = it & 1;
                ok = wait_or_abort(smem_u32(&sm.s_full[st]), (it >> 1) & 1, abort_flag, a.err);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t x[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + col_s(st) + c * 32, x[c]);
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_wait_ld(x[c]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sm.s_free[st]));

                // scaled scores (log2 units), causal mask on the tiles that reach past
                // this tile's first query position
                const bool need_mask = (j * kKT + kKT - 1) > t.pos0;
                float rmax = -INFINITY;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        float v = __uint_as_float(x[c][e]) * a.scale_log2;
                        if (need_mask && (j * kKT + c * 32 + e) > pos) v = -INFINITY;
                        x[c][e] = __float_as_uint(v);
                        rmax = fmaxf(rmax, v);
                    }
                }
                const float m_new = fmaxf(m, rmax);
                const bool rescale = m_new > m + kRescaleThreshold;   // also when m == -inf
                const float m_use = rescale ? m_new : m;
                const float alpha = rescale ? fast_exp2(m - m_new) : 1.f;
                float rsum = 0.f;
                uint32_t pk[2][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float p0 = fast_exp2(__uint_as_float(x[c][e]) - m_use);
                        const float p1 = fast_exp2(__uint_as_float(x[c][e + 1]) - m_use);
                        const uint32_t pp = pack_bf16x2(p0, p1);
                        // the row sum uses the same bf16-rounded weights the PV product uses,
                        // so the normalised weights sum to one exactly (up to fp32 rounding)
                        rsum += bf16_lo(pp) + bf16_hi(pp);
                        pk[c >> 1][(c & 1) * 16 + e / 2] = pp;
                    }
                }
                l = l * alpha + rsum;
                m = m_use;

                if (j > 0) {
                    // O must hold the previous tile's P V before it is rescaled, and the
                    // P buffer being overwritten must have been consumed.
                    ok = wait_or_abort(smem_u32(&sm.o_done), (it - 1) & 1, abort_flag, a.err);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint32_t o[32];
                            tmem_ld32(lane_base + kColO + c * 32, o);
                            tmem_wait_ld(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(lane_base + kColO + c * 32, o);
                        }
                    }
                }
                // V rows past the end of the context (the tail of the last block) may hold
                // anything, NaN included; P is 0 there but 0 * NaN is not, so zero them.
                const int kv_valid = t.seq_len - j * kKT;
                if (kv_valid < kKT) {
                    ok = wait_or_abort(smem_u32(&sm.v_full[st]), (it >> 1) & 1, abort_flag, a.err);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    if (row >= kv_valid) {
                        uint4 *r0 = reinterpret_cast<uint4 *>(sm.v[st][0] + row * 128);
                        uint4 *r1 = reinterpret_cast<uint4 *>(sm.v[st][1] + row * 128);
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            r0[v] = make_uint4(0u, 0u, 0u, 0u);
                            r1[v] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    fence_proxy_async_smem();   // generic writes -> visible to the MMA's reads
                }
                tmem_st32(lane_base + col_p(st), pk[0]);
                tmem_st32(lane_base + col_p(st) + 32, pk[1]);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sm.p_full[st]));
            }
            if (!ok) break;

            // ------------------------------------------------------------ epilogue
            ok = wait_or_abort(smem_u32(&sm.o_done), (it - 1) & 1, abort_flag, a.err);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const float inv_l = 1.f / l;
            const bool row_ok = pl < t.rows;
            __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) +
                                 ((size_t)(t.tok0 + pl) * kHq + t.g * kGroup + hl) * kD;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tmem_ld32(lane_base + kColO + c * 32, o);
                tmem_wait_ld(o);
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2)
                    w[e / 2] = pack_bf16x2(__uint_as_float(o[e]) * inv_l, __uint_as_float(o[e + 1]) * inv_l);
                if (row_ok) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v) d4[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
                }
            }
            if (row_ok && a.lse)
                a.lse[(size_t)(t.tok0 + pl) * kHq + t.g * kGroup + hl] = (m + __log2f(l)) * kLn2;
            tc_fence_before();
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// One CTA waiting on a barrier nothing completes: exercises the bounded-wait path.
__global__ void wait_selftest_kernel(uint32_t *err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0, limit_ns)) record_error(err, kErrTimeout);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, const CUtensorMap &q_map, const CUtensorMap &k_map,
                           const CUtensorMap &v_map, int num_sms, cudaStream_t stream) {
    if (a.num_seqs == 0 || a.max_q_len == 0 || a.total_tokens == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool configured[64] = {};
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    const long long tiles = (long long)a.num_seqs * kHkv * ((a.max_q_len + kQPos - 1) / kQPos);
    const int grid = (int)(tiles < num_sms ? tiles : num_sms);
    prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(q_map, k_map, v_map, a);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint32_t *err, uint64_t limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace pa
