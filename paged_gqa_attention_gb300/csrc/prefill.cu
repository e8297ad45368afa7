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
// CTA = 11 warps, persistent (one per SM), tiles dealt in a snake order, latest query
// blocks (most keys) first:
//   warps 0-7  softmax + epilogue in two warpgroups; warp w owns MMA rows (= TMEM
//              lanes) 32*(w%4) .. +31, columns 64*(w/4) .. +63 of each
//   warp 8     TMA producer of Q and K (ring of 2 stages)
//   warp 9     TMEM allocator and the single-thread tcgen05.mma issuer
//   warp 10    TMA producer of V (ring of 3 stages)
// Tensor memory (512 columns): S0, S1 (fp32 scores, 128 cols each), O (fp32, 128),
// L (fp32 row sums, 16).  P (bf16, packed in pairs) is written over the first 64
// columns of the S buffer it came from.
// Per key tile:  S = Q K^T (SS-MMA)  ->  softmax reads S, writes P (bf16) into TMEM
// and, when its running max rose by more than 2^8, rescales O and L  ->  O += P V
// (TS-MMA, P from TMEM, V from shared memory, MN-major) and L += P 1 (TS-MMA against a
// ones tile: the row sums of exactly the bf16 weights that multiply V).  The MMA warp
// issues S for tile j+1 before O += P V for tile j, so the tensor core works while the
// softmax runs; tcgen05.mma ops of one thread execute in issue order, so S for tile
// j+2 cannot overwrite P of tile j before O += P V of tile j has read it.
// Every wait is bounded; on expiry the CTA records PA_ERR_TIMEOUT, unwinds, waits
// (bounded) for its own copies and MMAs, frees tensor memory and exits.
#include "common.cuh"
#include "launch.h"

namespace pa {
namespace {

constexpr int kRows = 128;                  // MMA M
constexpr int kKT = kPrefillKvTile;         // keys per tile (MMA N of S, K of PV)
constexpr int kQPos = kPrefillQPositions;   // query positions per tile
constexpr int kSoftmaxWarps = 8;            // two warpgroups, one per half of each row
constexpr int kProducerWarp = 8;            // Q and K loads
constexpr int kMmaWarp = 9;
constexpr int kVProducerWarp = 10;          // V loads
constexpr int kThreads = (kSoftmaxWarps + 3) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128;   // score buffers; P (bf16 pairs) is written
                                               // over the first 64 columns of its own S
constexpr uint32_t kColO = 256;                // output accumulator
constexpr uint32_t kColL = 384;                // row sums of P (16 equal columns)
__device__ __forceinline__ uint32_t col_s(int st) { return st ? kColS1 : kColS0; }
constexpr int kHalf = kRows * 128;          // 128 rows x 64 dims x 2 B = 16 KiB
// Shared-memory rings (32 KiB per slot).  The V ring is the deepest: V of key tile j
// may only be requested once O += P V of tile j-3 has finished with its slot, and an
// L2-served 32 KiB load takes over a microsecond under this load.
constexpr int kQBufs = 1;
constexpr int kKStages = 2;
constexpr int kVStages = 3;
constexpr uint32_t kTileBytes = 2 * kHalf;  // a full 128 x 128 bf16 tile
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O when the max grows > 2^8
constexpr float kLn2 = 0.693147180559945309f;
constexpr uint32_t kIdescQK = idesc_bf16(kRows, kKT, false);  // B = K tile, K-major
constexpr uint32_t kIdescPV = idesc_bf16(kRows, kD, true);    // B = V tile, MN-major
constexpr uint32_t kIdescL = idesc_bf16(kRows, 16, false);    // B = ones [16 keys x 16]

struct PrefillSmem {
    uint8_t q[kQBufs][2][kHalf];    // [buffer][dims 0-63 | 64-127]
    uint8_t k[kKStages][2][kHalf];  // [stage][half]
    uint8_t v[kVStages][2][kHalf];
    uint64_t q_full[kQBufs], q_empty[kQBufs];
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2], s_free[2], p_full[2];
    uint64_t o_done;
    uint64_t mma_idle;
    uint64_t xbar[2];                  // softmax half-row exchange rounds
    float xchg[2][2][kRows];           // [round parity][half][row]
    alignas(128) uint16_t ones[512];   // bf16 1.0: B operand of the row-sum MMA
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
        for (int i = 0; i < kQBufs; ++i) {
            mbar_init(smem_u32(&sm.q_full[i]), 1);
            mbar_init(smem_u32(&sm.q_empty[i]), 1);
        }
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(smem_u32(&sm.k_full[i]), 1);
            mbar_init(smem_u32(&sm.k_empty[i]), 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(smem_u32(&sm.v_full[i]), 1);
            mbar_init(smem_u32(&sm.v_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sm.s_full[i]), 1);
            mbar_init(smem_u32(&sm.s_free[i]), kSoftmaxWarps);   // one arrive per softmax warp
            mbar_init(smem_u32(&sm.p_full[i]), kSoftmaxWarps);
            mbar_init(smem_u32(&sm.xbar[i]), kSoftmaxWarps);
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

    if (warp == kProducerWarp || warp == kVProducerWarp) {
        // ---------------------------------------------------------------- TMA producers
        // Two independent producers, so a K tile is requested as soon as its stage is
        // free, never behind a V tile waiting for its own stage: warp 8 loads Q and K,
        // warp 10 loads V.
        if (lane == 0) {
            const bool qk = (warp == kProducerWarp);
            if (qk) {
                tma_prefetch_map(&q_map);
                tma_prefetch_map(&k_map);
            } else {
                tma_prefetch_map(&v_map);
            }
            // The pools may be written by the kernel just before this one on the stream
            // (kv_append lets us launch early): wait for it before the first load.
            asm volatile("griddepcontrol.wait;" ::: "memory");
            uint64_t *full = qk ? sm.k_full : sm.v_full;
            uint64_t *empty = qk ? sm.k_empty : sm.v_empty;
            const int ns = qk ? kKStages : kVStages;
            const CUtensorMap *map = qk ? &k_map : &v_map;
            int tcount = 0, it = 0;              // tiles / key tiles started
            int q_issued = 0, kv_issued = 0;
            bool ok = true;
            for (int r = 0; ok; ++r) {
                const int idx = snake(r, total);
                if (idx < 0) break;
                const Tile t = tile_at(a, idx, qblocks);
                if (qk && t.error) record_error(a.err, kErrDevice | kErrQLen);
                if (!t.run) continue;
                if (qk) {
                    const int qbuf = tcount % kQBufs;
                    if (tcount >= kQBufs &&
                        !(ok = wait_or_abort(smem_u32(&sm.q_empty[qbuf]), ((tcount / kQBufs) - 1) & 1,
                                             abort_flag, a.err)))
                        break;
                    const uint32_t qbar = smem_u32(&sm.q_full[qbuf]);
                    mbar_arrive_expect_tx(qbar, kTileBytes);
                    tma_load_3d(smem_u32(sm.q[qbuf][0]), &q_map, qbar, 0, t.g * kGroup, t.tok0);
                    tma_load_3d(smem_u32(sm.q[qbuf][1]), &q_map, qbar, 64, t.g * kGroup, t.tok0);
                    ++q_issued;
                }
                const int32_t *bt = a.block_table + (size_t)t.s * a.max_blocks_per_seq;
                for (int j = 0; j < t.n_kt; ++j, ++it) {
                    const int st = it % ns;
                    int blk = __ldg(bt + (j >> 1));
                    if (blk < 0 || blk >= a.num_blocks) {
                        if (qk) record_error(a.err, kErrDevice | kErrBadBlock);
                        blk = 0;   // stay inside the pool; the result is flagged as invalid
                    }
                    const int off = (j & 1) * kKT;
                    if (it >= ns &&
                        !(ok = wait_or_abort(smem_u32(&empty[st]), ((it / ns) - 1) & 1, abort_flag, a.err)))
                        break;
                    const uint32_t bar = smem_u32(&full[st]);
                    uint8_t (*dst)[kHalf] = qk ? sm.k[st] : sm.v[st];
                    mbar_arrive_expect_tx(bar, kTileBytes);
                    tma_load_4d(smem_u32(dst[0]), map, bar, 0, t.g, off, blk);
                    tma_load_4d(smem_u32(dst[1]), map, bar, 64, t.g, off, blk);
                    ++kv_issued;
                }
                ++tcount;
            }
            // Drain: no TMA copy may still be landing when the CTA exits.  In the normal
            // path every load has been consumed and these waits return at once.
            for (int i = max(0, q_issued - kQBufs); i < q_issued; ++i)
                mbar_wait(smem_u32(&sm.q_full[i % kQBufs]), (i / kQBufs) & 1);
            for (int i = max(0, kv_issued - ns); i < kv_issued; ++i)
                mbar_wait(smem_u32(&full[i % ns]), (i / ns) & 1);
        }
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        // the ones tile of the row-sum MMA (written by the generic proxy, read by the MMA)
        for (int i = lane; i < 512; i += 32) sm.ones[i] = 0x3F80;   // bf16 1.0
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            int tcount = 0, it = 0;
            int pend_it = -1, pend_j = 0;   // O += P V still to issue for key tile pend_it
            // Matrix descriptors are built once; per MMA only a constant is added to the
            // start-address field (units of 16 bytes): +2 per 16 dims along a 128-byte row,
            // +1024 per 64-dim half (16 KiB), +2048 per ring slot (32 KiB), +128 per 16
            // keys of an MN-major V tile (2 KiB).
            const uint64_t ones_desc = sdesc_noswizzle(smem_u32(sm.ones), 128, 256);
            const uint64_t qd0 = sdesc_sw128(smem_u32(sm.q[0][0]), 16, 1024);
            const uint64_t kd0 = sdesc_sw128(smem_u32(sm.k[0][0]), 16, 1024);
            const uint64_t vd0 = sdesc_sw128(smem_u32(sm.v[0][0]), (uint32_t)kHalf, 1024);
            bool ok = true;
            auto issue_pv = [&](int pit, int pj) -> bool {
                const int vs = pit % kVStages;   // V slot
                const int st = pit & 1;          // S/P buffer
                if (!wait_or_abort(smem_u32(&sm.v_full[vs]), (pit / kVStages) & 1, abort_flag, a.err)) return false;
                if (!wait_or_abort(smem_u32(&sm.p_full[st]), (pit >> 1) & 1, abort_flag, a.err)) return false;
                tc_fence_after();
                // O += P V and L += P 1, 16 keys per step; V is [128 keys][128 dims] with dims
                // contiguous (MN-major), its two 64-dim halves 16 KiB apart.
                const uint64_t vb = vd0 + (uint64_t)(vs * 2048);
                const uint32_t pa = tmem + col_s(st);
                const uint32_t acc0 = pj > 0 ? 1u : 0u;
                umma_ts(tmem + kColO, pa, vb, kIdescPV, acc0);
                umma_ts(tmem + kColL, pa, ones_desc, kIdescL, acc0);
#pragma unroll
                for (int kk = 1; kk < kKT / 16; ++kk) {
                    umma_ts_c<true>(tmem + kColO, pa + kk * 8, vb + (uint64_t)(kk * 128), kIdescPV);
                    umma_ts_c<true>(tmem + kColL, pa + kk * 8, ones_desc, kIdescL);
                }
                umma_commit(smem_u32(&sm.o_done));
                umma_commit(smem_u32(&sm.v_empty[vs]));
                return true;
            };
            for (int r = 0; ok; ++r) {
                const int idx = snake(r, total);
                if (idx < 0) break;
                const Tile t = tile_at(a, idx, qblocks);
                if (!t.run) continue;
                const int qbuf = tcount % kQBufs;
                if (!(ok = wait_or_abort(smem_u32(&sm.q_full[qbuf]), (tcount / kQBufs) & 1, abort_flag, a.err)))
                    break;
                for (int j = 0; j < t.n_kt; ++j, ++it) {
                    const int st = it & 1;            // S/P buffer
                    const int ks = it % kKStages;     // K slot
                    if (!(ok = wait_or_abort(smem_u32(&sm.k_full[ks]), (it / kKStages) & 1, abort_flag, a.err)))
                        break;
                    if (it >= 2 &&
                        !(ok = wait_or_abort(smem_u32(&sm.s_free[st]), ((it >> 1) - 1) & 1, abort_flag, a.err)))
                        break;
                    tc_fence_after();
                    // S = Q K^T over 128 dims in 8 steps of 16 (K-major, 128-byte swizzle)
                    const uint64_t qa = qd0 + (uint64_t)(qbuf * 2048);
                    const uint64_t kb = kd0 + (uint64_t)(ks * 2048);
                    const uint32_t sd = tmem + col_s(st);
                    umma_ss_c<false>(sd, qa, kb, kIdescQK);
#pragma unroll
                    for (int kk = 1; kk < kD / 16; ++kk) {
                        const uint64_t off = (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2);
                        umma_ss_c<true>(sd, qa + off, kb + off, kIdescQK);
                    }
                    umma_commit(smem_u32(&sm.s_full[st]));
                    umma_commit(smem_u32(&sm.k_empty[ks]));
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
        // Two warpgroups share every score row: warpgroup ch (= warp / 4) owns columns
        // ch*64 .. ch*64+63 of S and O and keys ch*64 .. ch*64+63 of P for the row
        // (= TMEM lane) row.  The two halves of a row exchange their maxima through
        // shared memory, synchronised by an mbarrier per exchange round.
        const int ch = warp >> 2;                  // column half
        const int row = (warp & 3) * 32 + lane;    // MMA row == TMEM lane
        const int pl = row >> 2;                   // query position within the tile
        const int hl = row & 3;                    // query head within the group
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const float sl2 = a.scale_log2;
        int it = 0;
        int xc = 0;                                // exchange rounds so far
        bool ok = true;
        // Publish v for this row, wait for all 8 warps, return the other half's value.
        auto exchange = [&](float v, bool &good) -> float {
            const int buf = xc & 1;
            sm.xchg[buf][ch][row] = v;
            tc_fence_before();       // this warp's tcgen05.ld of S precede the other half's P stores
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.xbar[buf]));
            good = wait_or_abort(smem_u32(&sm.xbar[buf]), (xc >> 1) & 1, abort_flag, a.err);
            good = __all_sync(0xffffffffu, good);
            tc_fence_after();
            const float other = sm.xchg[buf][ch ^ 1][row];
            ++xc;
            return other;
        };
        for (int r = 0; ok; ++r) {
            const int idx = snake(r, total);
            if (idx < 0) break;
            const Tile t = tile_at(a, idx, qblocks);
            if (!t.run) continue;
            const int pos = t.pos0 + pl;
            float m = -INFINITY;                   // running max, log2 units (scaled)
            for (int j = 0; j < t.n_kt; ++j, ++it) {
                const int st = it & 1;
                ok = wait_or_abort(smem_u32(&sm.s_full[st]), (it >> 1) & 1, abort_flag, a.err);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t x[2][32];
                tmem_ld32(lane_base + col_s(st) + ch * 64, x[0]);
                tmem_ld32(lane_base + col_s(st) + ch * 64 + 32, x[1]);
                tmem_wait_ld(x[0]);
                tmem_wait_ld(x[1]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sm.s_free[st]));

                // causal mask (only on tiles reaching past the tile's first query position)
                // and the row maximum of the raw scores
                const int key0 = j * kKT + ch * 64;
                const bool need_mask = (j * kKT + kKT - 1) > t.pos0;
                if (need_mask) {
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if ((key0 + c * 32 + e) > pos) x[c][e] = __float_as_uint(-INFINITY);
                }
                float rmax = -INFINITY;
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        rmax = fmax3(rmax, __uint_as_float(x[c][e]), __uint_as_float(x[c][e + 1]));
                rmax = fmaxf(rmax, exchange(rmax, ok));
                if (!ok) break;
                const float m_new = fmaxf(m, rmax * sl2);
                const bool rescale = m_new > m + kRescaleThreshold;   // also when m == -inf
                const float m_use = rescale ? m_new : m;
                const float alpha = rescale ? fast_exp2(m - m_new) : 1.f;
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float p0 = fast_exp2(fmaf(__uint_as_float(x[c][e]), sl2, -m_use));
                        const float p1 = fast_exp2(fmaf(__uint_as_float(x[c][e + 1]), sl2, -m_use));
                        pk[c * 16 + e / 2] = pack_bf16x2(p0, p1);
                    }
                }
                m = m_use;

                if (j > 0) {
                    // O must hold the previous tile's P V before it is rescaled, and the
                    // P buffer being overwritten must have been consumed.
                    ok = wait_or_abort(smem_u32(&sm.o_done), (it - 1) & 1, abort_flag, a.err);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            uint32_t o[32];
                            tmem_ld32(lane_base + kColO + ch * 64 + c * 32, o);
                            tmem_wait_ld(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(lane_base + kColO + ch * 64 + c * 32, o);
                        }
                        if (ch == 0) {   // the row sum (its first column) scales with O
                            uint32_t lv = tmem_ld1(lane_base + kColL);
                            tmem_wait_ld1(lv);
                            tmem_st1(lane_base + kColL, __float_as_uint(__uint_as_float(lv) * alpha));
                        }
                    }
                }
                // V rows past the end of the context (the tail of the last block) may hold
                // anything, NaN included; P is 0 there but 0 * NaN is not, so zero them.
                const int kv_valid = t.seq_len - j * kKT;
                if (kv_valid < kKT) {
                    const int vs = it % kVStages;
                    ok = wait_or_abort(smem_u32(&sm.v_full[vs]), (it / kVStages) & 1, abort_flag, a.err);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    if (row >= kv_valid) {
                        uint4 *rv = reinterpret_cast<uint4 *>(sm.v[vs][ch] + row * 128);
#pragma unroll
                        for (int v = 0; v < 8; ++v) rv[v] = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();   // generic writes -> visible to the MMA's reads
                }
                tmem_st32(lane_base + col_s(st) + ch * 32, pk);
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
            uint32_t lbits = tmem_ld1(lane_base + kColL);
            tmem_wait_ld1(lbits);
            const float l_row = __uint_as_float(lbits);
            const float inv_l = 1.f / l_row;
            const bool row_ok = pl < t.rows;
            __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) +
                                 ((size_t)(t.tok0 + pl) * kHq + t.g * kGroup + hl) * kD + ch * 64;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t o[32];
                tmem_ld32(lane_base + kColO + ch * 64 + c * 32, o);
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
            if (row_ok && ch == 0 && a.lse)
                a.lse[(size_t)(t.tok0 + pl) * kHq + t.g * kGroup + hl] = (m + __log2f(l_row)) * kLn2;
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
    // Programmatic dependent launch (see decode): the producer waits before its loads.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_kernel, q_map, k_map, v_map, a);
}

cudaError_t launch_wait_selftest(uint32_t *err, uint64_t limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace pa
