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
// Work unit: 64 query positions x the 4 query heads of one KV head, split into two
// MMA tiles A and B of 128 rows (row r = position r / 4, head r % 4 within the tile).
// Key/value tiles are 128 tokens (half a cache block) fetched by TMA straight from the
// paged pool: the block-table lookup is the TMA coordinate.  Both query tiles consume
// every K/V tile the unit fetches, so a CTA moves 64 KiB of K/V from L2 per 256 x 128
// score block; at 128 rows per K/V tile the L2-to-SM delivery (not the tensor core) was
// the limit.
//
// CTA = 11 warps, persistent (one per SM), units dealt in a snake order, most key tiles
// first (one sequence: latest query blocks first; several: in the order a planning
// kernel sorts them into, longest processing time first):
//   warps 0-3   softmax + epilogue of tile A; thread = one row (= TMEM lane) of A
//   warps 4-7   softmax + epilogue of tile B
//   warp 8      TMA producer of Q and K (ring of 2 slots)
//   warp 9      TMEM allocator and the single-thread tcgen05.mma issuer
//   warp 10     TMA producer of V (ring of 2 slots)
// Tensor memory (512 columns): S_A, S_B (fp32 scores), O_A, O_B (fp32 output), 128
// columns each.  P (bf16, packed in pairs) is written over the first 64 columns of its
// own S buffer.  Per key tile j the MMA thread issues, in this order,
//     S_A(j) = Q_A K_j^T,  O_B += P_B(j-1) V_{j-1},  S_B(j) = Q_B K_j^T,  O_A += P_A(j) V_j
// so the tensor core computes one tile's products while the other tile's softmax runs.
// tcgen05.mma operations of one thread execute in issue order, hence S_X(j+1) cannot
// overwrite P_X(j) before O_X += P_X(j) V_j has read it.  The softmax keeps a running
// max and, only when it grows by more than 2^8, rescales O (lazy rescaling); the row
// sum accumulates the same bf16-rounded weights the PV product uses.
// Every wait is bounded; on expiry the CTA records PA_ERR_TIMEOUT, unwinds, waits
// (bounded) for its own copies and MMAs, frees tensor memory and exits.
#include "common.cuh"
#include "launch.h"

namespace pa {
namespace {

constexpr int kRows = 128;                    // MMA M (one query tile)
constexpr int kKT = kPrefillKvTile;           // keys per K/V tile (MMA N of S, K of PV)
constexpr int kTilePos = kPrefillQPositions;  // query positions per MMA tile (32)
constexpr int kUnitPos = 2 * kTilePos;        // query positions per work unit (64)
constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;              // Q and K loads
constexpr int kMmaWarp = 9;
constexpr int kVProducerWarp = 10;            // V loads
constexpr int kAppendWarp = 11;               // fused append only: new K/V rows into the pools
constexpr int kThreads = (kSoftmaxWarps + 3) * 32;
constexpr int kThreadsAppend = kThreads + 32;
constexpr uint32_t kTmemCols = 512;
constexpr int kHalf = kRows * 128;            // 128 rows x 64 dims x 2 B = 16 KiB
constexpr uint32_t kTileBytes = 2 * kHalf;    // a full 128 x 128 bf16 tile
constexpr int kKStages = 2;                   // (a third stage measured no faster)
constexpr int kVStages = 2;
constexpr uint32_t kParkNs = 20000;           // longest hardware park per wait attempt
constexpr float kRescaleThreshold = 8.0f;     // log2 units: rescale O when the max grows > 2^8
constexpr float kLn2 = 0.693147180559945309f;
constexpr uint32_t kIdescQK = idesc_bf16(kRows, kKT, false);  // B = K tile, K-major
constexpr uint32_t kIdescPV = idesc_bf16(kRows, kD, true);    // B = V tile, MN-major

// TMEM columns of query tile x (0 = A, 1 = B): S_A 0-127, S_B 128-255, O_A 256-383, O_B 384-511
__device__ __forceinline__ uint32_t col_s(int x) { return x ? 128u : 0u; }
__device__ __forceinline__ uint32_t col_o(int x) { return x ? 384u : 256u; }

struct PrefillSmem {
    uint8_t q[2][2][kHalf];          // [tile A|B][dims 0-63 | 64-127]
    uint8_t k[kKStages][2][kHalf];   // [slot][half]
    uint8_t v[kVStages][2][kHalf];
    uint64_t q_full, q_empty;
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2], p_half[2][2], o_done[2];   // per query tile (P in two key halves)
    uint64_t mma_idle;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t kSmemBytes = sizeof(PrefillSmem) + 1024;

struct Unit {
    bool run;       // has work
    bool error;     // inconsistent lengths (recorded once, then skipped)
    int s, g;
    int tok0;       // row of q/out holding the unit's first query position
    int positions;  // real positions in this unit (1..64)
    int pos0;       // absolute position of the unit's first query
    int seq_len;    // context length (keys 0 .. seq_len-1 exist)
    int kt0;        // first key tile visited (0 unless the keys are split)
    int n_kt;       // key tiles to visit: kt0 .. kt0 + n_kt - 1
    int ks;         // key split of the unit (shared-prefix mode)
    // Key tiles 0 .. n_old-1 hold positions 128j .. 128j+127 of the cache, only those below c0
    // being keys; with a fused append the tiles after them hold the new positions from c0 on,
    // 128 a tile (c0 + 128(j - n_old) + r), read from k_new rows tok_base + 128(j - n_old) + r.
    // Without one, c0 = seq_len and every tile is a cache tile.
    int c0;
    int n_old;
    int tok_base;
};

// Position of row 0 of key tile jg and the bound past which its rows are not keys.
__device__ __forceinline__ void key_tile_span(const Unit &t, int jg, int &base, int &limit) {
    const bool old_tile = jg < t.n_old;
    base = old_tile ? jg * kKT : t.c0 + (jg - t.n_old) * kKT;
    limit = old_tile ? t.c0 : t.seq_len;
}

template <bool kAppend>
__device__ __forceinline__ Unit unit_at(const PrefillArgs &a, int idx, int qblocks) {
    Unit t;
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
    if (qb * kUnitPos >= q_len) return t;
    t.run = true;
    t.tok0 = c0 + qb * kUnitPos;
    t.positions = min(kUnitPos, q_len - qb * kUnitPos);
    t.pos0 = seq_len - q_len + qb * kUnitPos;
    t.seq_len = seq_len;
    t.kt0 = 0;
    t.ks = 0;
    t.tok_base = c0;
    if constexpr (kAppend) {
        t.c0 = seq_len - q_len;
        t.n_old = (t.c0 + kKT - 1) / kKT;
        t.n_kt = t.n_old + (t.pos0 + t.positions - 1 - t.c0) / kKT + 1;
    } else {
        t.c0 = seq_len;
        t.n_kt = (t.pos0 + t.positions - 1) / kKT + 1;
        t.n_old = t.n_kt;
    }
    return t;
}

// Shared-prefix mode: unit idx = ((query block) x 8 + KV head) x n_kv_splits + key split;
// every query sees keys 0 .. prefix_len-1 of table row 0.
__device__ __forceinline__ Unit unit_at_prefix(const PrefillArgs &a, int idx, int qblocks) {
    Unit t;
    const int ks = idx % a.n_kv_splits;
    const int rest = idx / a.n_kv_splits;
    const int qb = qblocks - 1 - rest / kHkv;
    t.s = 0;
    t.g = rest % kHkv;
    t.error = false;
    t.run = qb * kUnitPos < a.total_tokens;
    t.tok0 = qb * kUnitPos;
    t.positions = min(kUnitPos, a.total_tokens - qb * kUnitPos);
    t.pos0 = 0;
    t.seq_len = a.prefix_len;
    t.kt0 = ks * a.kv_split_tiles;
    t.n_kt = min(a.kv_split_tiles, (a.prefix_len + kKT - 1) / kKT - t.kt0);
    t.ks = ks;
    t.c0 = t.seq_len;
    t.n_old = t.kt0 + t.n_kt;
    t.tok_base = 0;
    if (t.n_kt <= 0) t.run = false;
    return t;
}

template <bool kPrefix, bool kPlanned, bool kAppend>
__device__ __forceinline__ Unit unit_for(const PrefillArgs &a, int idx, int qblocks) {
    if constexpr (kPrefix) return unit_at_prefix(a, idx, qblocks);
    else if constexpr (kPlanned) return unit_at<kAppend>(a, __ldg(a.order + idx), qblocks);
    else return unit_at<kAppend>(a, idx, qblocks);
}

// Key tiles of unit idx (the unit_at rule; 0 for a unit without work, which sorts last).
template <bool kAppend>
__device__ __forceinline__ int plan_key(const PrefillArgs &a, int idx, int qblocks) {
    const Unit t = unit_at<kAppend>(a, idx, qblocks);
    return t.run ? t.n_kt : 0;
}

constexpr int kPlanThreads = 1024;
constexpr int kPlanMaxKeys = 12288;   // histogram buckets in shared memory (48 KiB)
// key buckets: a unit visits at most 2 * max_blocks_per_seq key tiles
inline int plan_keys(const PrefillArgs &a) { return 2 * a.max_blocks_per_seq + 2; }

// Planning kernel for several sequences: a counting sort of the units by key tiles, most
// first (longest processing time first), written as order[rank] = unit.  Units with equal
// keys take their ranks in whatever order the atomics resolve; every unit is computed by
// one CTA on its own, so the outputs do not depend on that order.  nk = key buckets.
template <bool kAppend>
__global__ void __launch_bounds__(kPlanThreads, 1) prefill_plan_kernel(const PrefillArgs a, int qblocks, int total,
                                                                       int nk) {
    __shared__ int hist[kPlanMaxKeys];
    __shared__ int warp_sum[kPlanThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int k = tid; k < nk; k += kPlanThreads) hist[k] = 0;
    __syncthreads();
    for (int idx = tid; idx < total; idx += kPlanThreads)
        atomicAdd(&hist[min(plan_key<kAppend>(a, idx, qblocks), nk - 1)], 1);
    __syncthreads();
    // hist[k] <- first rank of key k = number of units with more key tiles.  Thread t owns
    // the keys hi, hi - 1, ..., hi - per + 1 counted from the top.
    const int per = (nk + kPlanThreads - 1) / kPlanThreads;
    const int hi = nk - 1 - tid * per;
    int sum = 0;
    for (int i = 0; i < per; ++i)
        if (hi - i >= 0) sum += hist[hi - i];
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += n;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sum[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += n;
        }
        warp_sum[lane] = w;   // inclusive over warps
    }
    __syncthreads();
    int run = incl - sum + (warp > 0 ? warp_sum[warp - 1] : 0);
    for (int i = 0; i < per; ++i) {
        const int k = hi - i;
        if (k >= 0) {
            const int v = hist[k];
            hist[k] = run;
            run += v;
        }
    }
    __syncthreads();
    for (int idx = tid; idx < total; idx += kPlanThreads) {
        const int rank = atomicAdd(&hist[min(plan_key<kAppend>(a, idx, qblocks), nk - 1)], 1);
        a.order[rank] = idx;
    }
    // Complete only after the kernel before this one on the stream (kv_append lets its
    // dependents start early): the prefill launched after this kernel relies on it.
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Index of this CTA's r-th unit in the snake order (or -1 past the end).
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
        if (mbar_try_wait_parked(bar, parity, kParkNs)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            record_error(err, kErrTimeout);
            return false;
        }
    }
}

// The fused append's warp: this CTA's share of the new tokens' K and V rows (2 KiB each, all
// 8 KV heads) copied into their cache slots by the kv_append rule, two tokens at a time with
// 16-byte accesses.  Nothing in this kernel reads those slots (the attention takes the new
// rows from k_new / v_new), so the copies run beside the attention without any ordering; the
// kernel's completion publishes them.
__device__ __forceinline__ void append_share(const PrefillArgs &a, int lane) {
    const long long tt = a.total_tokens;
    const int t_lo = (int)(tt * blockIdx.x / gridDim.x), t_hi = (int)(tt * (blockIdx.x + 1) / gridDim.x);
    if (t_lo >= t_hi) return;
    int lo = 0, hi = a.num_seqs - 1;   // the sequence of the share's first token
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(a.cu_q_lens + mid) <= t_lo) lo = mid;
        else hi = mid - 1;
    }
    int s = lo, q0 = __ldg(a.cu_q_lens + s), q1 = __ldg(a.cu_q_lens + s + 1), seq_len = __ldg(a.seq_lens + s);
    int cached_j = -1, blk = -1;
    for (int t = t_lo; t < t_hi; t += 2) {
        uint4 r[2][8];
        long long dst[2] = {-1, -1};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int tu = t + u;
            if (tu >= t_hi) break;
            while (tu >= q1 && s + 1 < a.num_seqs) {   // next sequence (empty ones skipped)
                ++s;
                q0 = q1;
                q1 = __ldg(a.cu_q_lens + s + 1);
                seq_len = __ldg(a.seq_lens + s);
                cached_j = -1;
            }
            const uint4 *ks = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.k_new) + (size_t)tu * kTokenBytes);
            const uint4 *vs = reinterpret_cast<const uint4 *>(static_cast<const char *>(a.v_new) + (size_t)tu * kTokenBytes);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                r[u][k] = __ldg(ks + lane + 32 * k);
                r[u][4 + k] = __ldg(vs + lane + 32 * k);
            }
            const int q_len = q1 - q0, i = tu - q0;
            if (i < 0 || i >= q_len || seq_len < q_len || seq_len > a.max_blocks_per_seq * kBlock) {
                if (lane == 0) record_error(a.err, kErrDevice | kErrQLen);
                continue;
            }
            const int p = seq_len - q_len + i;
            if (p / kBlock != cached_j) {
                cached_j = p / kBlock;
                blk = __ldg(a.block_table + (size_t)s * a.max_blocks_per_seq + cached_j);
            }
            if (blk < 0 || blk >= a.num_blocks) {
                if (lane == 0) record_error(a.err, kErrDevice | kErrBadBlock);
                continue;
            }
            dst[u] = ((long long)blk * kBlock + p % kBlock) * kTokenBytes;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            if (dst[u] < 0) continue;
            uint4 *kd = reinterpret_cast<uint4 *>(static_cast<char *>(a.k_pool_w) + dst[u]);
            uint4 *vd = reinterpret_cast<uint4 *>(static_cast<char *>(a.v_pool_w) + dst[u]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                kd[lane + 32 * k] = r[u][k];
                vd[lane + 32 * k] = r[u][4 + k];
            }
        }
    }
}

template <bool kPrefix, bool kPlanned, bool kAppend>
__global__ void __launch_bounds__(kAppend ? kThreadsAppend : kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
               const __grid_constant__ CUtensorMap v_map, const __grid_constant__ CUtensorMap kn_map,
               const __grid_constant__ CUtensorMap vn_map, const PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    PrefillSmem &sm = *reinterpret_cast<PrefillSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    volatile int *abort_flag = &sm.abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int qblocks = (a.max_q_len + kUnitPos - 1) / kUnitPos;
    const int total = kPrefix ? kHkv * qblocks * a.n_kv_splits : a.num_seqs * kHkv * qblocks;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&sm.q_full), 1);
        mbar_init(smem_u32(&sm.q_empty), 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(smem_u32(&sm.k_full[i]), 1);
            mbar_init(smem_u32(&sm.k_empty[i]), 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(smem_u32(&sm.v_full[i]), 1);
            mbar_init(smem_u32(&sm.v_empty[i]), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(smem_u32(&sm.s_full[x]), 1);
            mbar_init(smem_u32(&sm.p_half[x][0]), 4);   // the 4 warps of the tile's softmax
            mbar_init(smem_u32(&sm.p_half[x][1]), 4);
            mbar_init(smem_u32(&sm.o_done[x]), 1);
        }
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
        // Two independent producers, so a K tile is requested as soon as its slot is
        // free, never behind a V tile waiting for its own slot.  As in the MMA warp, the
        // whole warp runs the loop and one elected lane issues the copies.
        const bool leader = elect_one();
        const bool qk = (warp == kProducerWarp);
        if (leader) {
            if (qk) {
                tma_prefetch_map(&q_map);
                tma_prefetch_map(&k_map);
                if constexpr (kAppend) tma_prefetch_map(&kn_map);
            } else {
                tma_prefetch_map(&v_map);
                if constexpr (kAppend) tma_prefetch_map(&vn_map);
            }
        }
        // The pools may be written by the kernel just before this one on the stream
        // (kv_append lets us launch early): wait for it before the first load.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        uint64_t *full = qk ? sm.k_full : sm.v_full;
        uint64_t *empty = qk ? sm.k_empty : sm.v_empty;
        const int ns = qk ? kKStages : kVStages;
        const CUtensorMap *map = qk ? &k_map : &v_map;
        const CUtensorMap *new_map = qk ? &kn_map : &vn_map;
        int tcount = 0, it = 0;              // units / key tiles started
        int q_issued = 0, kv_issued = 0;
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int idx = snake(r, total);
            if (idx < 0) break;
            const Unit t = unit_for<kPrefix, kPlanned, kAppend>(a, idx, qblocks);
            if (qk && leader && t.error) record_error(a.err, kErrDevice | kErrQLen);
            if (!t.run) continue;
            if (qk) {
                if (tcount >= 1 &&
                    !(ok = __all_sync(0xffffffffu, wait_or_abort(smem_u32(&sm.q_empty), (tcount - 1) & 1,
                                                                abort_flag, a.err))))
                    break;
                if (leader) {
                    const uint32_t qbar = smem_u32(&sm.q_full);
                    mbar_arrive_expect_tx(qbar, 2 * kTileBytes);
                    for (int x = 0; x < 2; ++x) {
                        tma_load_3d(smem_u32(sm.q[x][0]), &q_map, qbar, 0, t.g * kGroup, t.tok0 + x * kTilePos);
                        tma_load_3d(smem_u32(sm.q[x][1]), &q_map, qbar, 64, t.g * kGroup, t.tok0 + x * kTilePos);
                    }
                }
                __syncwarp();
                ++q_issued;
            }
            const int32_t *bt = a.block_table + (size_t)t.s * a.max_blocks_per_seq;
            for (int j = 0; j < t.n_kt; ++j, ++it) {
                const int st = it % ns;
                const int jg = t.kt0 + j;              // key tile within the context
                const bool cache_tile = !kAppend || jg < t.n_old;
                int blk = cache_tile ? __ldg(bt + (jg >> 1)) : 0;
                if (blk < 0 || blk >= a.num_blocks) {
                    if (qk && leader) record_error(a.err, kErrDevice | kErrBadBlock);
                    blk = 0;   // stay inside the pool; the result is flagged as invalid
                }
                const int off = (jg & 1) * kKT;
                if (it >= ns &&
                    !(ok = __all_sync(0xffffffffu, wait_or_abort(smem_u32(&empty[st]), ((it / ns) - 1) & 1,
                                                                abort_flag, a.err))))
                    break;
                if (leader) {
                    const uint32_t bar = smem_u32(&full[st]);
                    uint8_t (*dst)[kHalf] = qk ? sm.k[st] : sm.v[st];
                    mbar_arrive_expect_tx(bar, kTileBytes);
                    if (cache_tile) {
                        tma_load_4d(smem_u32(dst[0]), map, bar, 0, t.g, off, blk);
                        tma_load_4d(smem_u32(dst[1]), map, bar, 64, t.g, off, blk);
                    } else {
                        // 128 new rows of k_new / v_new (past the sequence's last one: rows of
                        // the next sequence, or zeros past the tensor's end; never keys here)
                        const int row = t.tok_base + (jg - t.n_old) * kKT;
                        tma_load_3d(smem_u32(dst[0]), new_map, bar, 0, t.g, row);
                        tma_load_3d(smem_u32(dst[1]), new_map, bar, 64, t.g, row);
                    }
                }
                __syncwarp();
                ++kv_issued;
            }
            ++tcount;
        }
        // Drain: no TMA copy may still be landing when the CTA exits.  In the normal
        // path every load has been consumed and these waits return at once.
        if (q_issued > 0) mbar_wait(smem_u32(&sm.q_full), (q_issued - 1) & 1);
        for (int i = max(0, kv_issued - ns); i < kv_issued; ++i)
            mbar_wait(smem_u32(&full[i % ns]), (i / ns) & 1);
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        // The whole warp runs the loop and the waits, so the descriptors and counters are
        // warp-uniform; one elected lane issues the MMAs and commits.  Confined to a
        // single-lane branch, the same stream competed for issue slots with the softmax
        // warps of its sub-partition and fed the tensor core at about half its rate.
        const bool leader = elect_one();
        // The unit order is written by the planning kernel just before this one.
        if constexpr (kPlanned) asm volatile("griddepcontrol.wait;" ::: "memory");
        // Matrix descriptors are built once; per MMA only a constant is added to the
        // start-address field (units of 16 bytes): +2 per 16 dims along a 128-byte row,
        // +1024 per 64-dim half (16 KiB), +2048 per tile or ring slot (32 KiB), +128 per
        // 16 keys of an MN-major V tile (2 KiB).
        const uint64_t qd0 = sdesc_sw128(smem_u32(sm.q[0][0]), 16, 1024);
        const uint64_t kd0 = sdesc_sw128(smem_u32(sm.k[0][0]), 16, 1024);
        const uint64_t vd0 = sdesc_sw128(smem_u32(sm.v[0][0]), (uint32_t)kHalf, 1024);
        int tcount = 0, it = 0;
        int pend_it = -1, pend_j = 0;   // O_B += P_B V still to issue for key tile pend_it
        bool ok = true;
        auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, wait_or_abort(smem_u32(bar), parity, abort_flag, a.err));
        };
        // S_x = Q_x K^T over 128 dims in 8 steps of 16 (K-major, 128-byte swizzle)
        auto issue_s = [&](int x, int ks) {
            const uint64_t qa = qd0 + (uint64_t)(x * 2048);
            const uint64_t kb = kd0 + (uint64_t)(ks * 2048);
            const uint32_t sd = tmem + col_s(x);
            if (leader) {
                umma_ss_c<false>(sd, qa, kb, kIdescQK);
#pragma unroll
                for (int kk = 1; kk < kD / 16; ++kk) {
                    const uint64_t off = (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2);
                    umma_ss_c<true>(sd, qa + off, kb + off, kIdescQK);
                }
                umma_commit(smem_u32(&sm.s_full[x]));
            }
            __syncwarp();
        };
        // O_x += P_x V over 128 keys in 8 steps of 16; V is [128 keys][128 dims] with dims
        // contiguous (MN-major), its two 64-dim halves 16 KiB apart.
        // Tile A (x = 0) takes keys 0-63 as soon as their P is stored and keys 64-127 when the
        // rest is.  Tile B's product is issued a key tile later, when its P is long complete:
        // it waits only for the second half (whose barrier completes after every softmax warp
        // has arrived on the first), and not for V, which tile A's product already waited for.
        // Every wait costs the issuing thread time in which the tensor core can run dry.
        auto issue_pv = [&](int x, int pit, int pj) -> bool {
            const int vs = pit % kVStages;
            if (x == 0 && !wait_all(&sm.v_full[vs], (pit / kVStages) & 1)) return false;
            const uint64_t vb = vd0 + (uint64_t)(vs * 2048);
            const uint32_t pa = tmem + col_s(x);
            if (!wait_all(&sm.p_half[x][x], pit & 1)) return false;
            tc_fence_after();
            if (leader) {
                umma_ts(tmem + col_o(x), pa, vb, kIdescPV, pj > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 1; kk < kKT / 32; ++kk)
                    umma_ts_c<true>(tmem + col_o(x), pa + kk * 8, vb + (uint64_t)(kk * 128), kIdescPV);
            }
            __syncwarp();
            if (x == 0) {
                if (!wait_all(&sm.p_half[x][1], pit & 1)) return false;
                tc_fence_after();
            }
            if (leader) {
#pragma unroll
                for (int kk = kKT / 32; kk < kKT / 16; ++kk)
                    umma_ts_c<true>(tmem + col_o(x), pa + kk * 8, vb + (uint64_t)(kk * 128), kIdescPV);
                umma_commit(smem_u32(&sm.o_done[x]));
                if (x == 1) umma_commit(smem_u32(&sm.v_empty[vs]));   // B is the V tile's last reader
            }
            __syncwarp();
            return true;
        };
        for (int r = 0; ok; ++r) {
            const int idx = snake(r, total);
            if (idx < 0) break;
            const Unit t = unit_for<kPrefix, kPlanned, kAppend>(a, idx, qblocks);
            if (!t.run) continue;
            if (!(ok = wait_all(&sm.q_full, tcount & 1))) break;
            for (int j = 0; j < t.n_kt; ++j, ++it) {
                const int ks = it % kKStages;
                if (!(ok = wait_all(&sm.k_full[ks], (it / kKStages) & 1))) break;
                tc_fence_after();
                issue_s(0, ks);                                        // S_A(j)
                if (pend_it >= 0 && !(ok = issue_pv(1, pend_it, pend_j))) break;   // O_B, tile j-1
                issue_s(1, ks);                                        // S_B(j)
                if (leader) {
                    umma_commit(smem_u32(&sm.k_empty[ks]));
                    if (j == t.n_kt - 1) umma_commit(smem_u32(&sm.q_empty));
                }
                __syncwarp();
                if (!(ok = issue_pv(0, it, j))) break;                 // O_A, tile j
                pend_it = it;
                pend_j = j;
            }
            // the unit's last O_B += P_B V now, not behind the next unit's Q and first S_A
            if (ok && pend_it >= 0) ok = issue_pv(1, pend_it, pend_j);
            pend_it = -1;
            ++tcount;
        }
        // Every MMA issued must have finished before tensor memory is released.
        if (leader) umma_commit(smem_u32(&sm.mma_idle));
        __syncwarp();
        mbar_wait(smem_u32(&sm.mma_idle), 0);
    } else if (kAppend && warp == kAppendWarp) {
        // ---------------------------------------------------------------- fused append
        // k_new / v_new and the pools may come from the kernel just before this one
        asm volatile("griddepcontrol.wait;" ::: "memory");
        // The copies are due only by the kernel's end: keep them off the start, where every
        // CTA's first Q, K and V tiles are on their way, by waiting for this CTA's first
        // O += P V product (if it has any unit to compute; bounded, then it copies anyway).
        bool has_unit = false;
        for (int r = 0; !has_unit; ++r) {
            const int idx = snake(r, total);
            if (idx < 0) break;
            has_unit = unit_for<kPrefix, kPlanned, kAppend>(a, idx, qblocks).run;
        }
        if (has_unit) mbar_wait(smem_u32(&sm.o_done[0]), 0, 200000ull);
        append_share(a, lane);
    } else {
        // ---------------------------------------------------------------- softmax warps
        // Warpgroup x (= warp / 4) owns query tile x; thread = one row = one TMEM lane.
        if constexpr (kPlanned) asm volatile("griddepcontrol.wait;" ::: "memory");
        const int x = warp >> 2;
        const int row = (warp & 3) * 32 + lane;    // MMA row == TMEM lane
        const int pl = row >> 2;                   // query position within the tile
        const int hl = row & 3;                    // query head within the group
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t s_col = col_s(x), o_col = col_o(x);
        const float sl2 = a.scale_log2;
        int it = 0;
        bool ok = true;
        for (int r = 0; ok; ++r) {
            const int idx = snake(r, total);
            if (idx < 0) break;
            const Unit t = unit_for<kPrefix, kPlanned, kAppend>(a, idx, qblocks);
            if (!t.run) continue;
            // the last key each row may see: its own position (causal), or the whole prefix
            const int pos_first = kPrefix ? t.seq_len - 1 : t.pos0 + x * kTilePos;
            const int pos = kPrefix ? t.seq_len - 1 : pos_first + pl;
            float m = -INFINITY;                   // running max, log2 units (scaled)
            float l = 0.f;                         // running sum of the bf16 weights
            for (int j = 0; j < t.n_kt; ++j, ++it) {
                ok = wait_or_abort(smem_u32(&sm.s_full[x]), it & 1, abort_flag, a.err);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                uint32_t s[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + s_col + c * 32, s[c]);
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_wait_ld(s[c]);

                // mask of the keys past each row's last visible key and of the tile's rows that
                // are no keys (past its span; only on tiles reaching past either) and the row
                // maximum of the raw scores
                const int jg = t.kt0 + j;                  // key tile within the context
                int base = jg * kKT, kv_valid = t.seq_len - jg * kKT;   // rows 0 .. kv_valid-1 are keys
                if constexpr (kAppend) {
                    int limit;
                    key_tile_span(t, jg, base, limit);
                    kv_valid = limit - base;
                }
                // (without the fused append a tile's rows past kv_valid lie past every query's
                // position, so the causal mask covers them)
                if (base + kKT - 1 > pos_first || (kAppend && kv_valid < kKT)) {
                    if constexpr (kAppend) {
                        // one bound per row, tile rows 0 .. lim-1 being keys this row may see
                        // (one compare per score instead of two: 2.8 % of the fused step)
                        const int lim = min(kv_valid, pos - base + 1);
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (c * 32 + e >= lim) s[c][e] = __float_as_uint(-INFINITY);
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                if (base + c * 32 + e > pos) s[c][e] = __float_as_uint(-INFINITY);
                    }
                }
                // independent partial maxima (one per 32-column chunk) keep the dependency
                // chain short: floating-point max/add are not reassociated by the compiler
                float cmax[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    // r0 over columns 0-15, r1 over columns 16-31
                    float r0 = fmaxf(__uint_as_float(s[c][0]), __uint_as_float(s[c][1]));
                    float r1 = fmaxf(__uint_as_float(s[c][16]), __uint_as_float(s[c][17]));
#pragma unroll
                    for (int e = 2; e < 16; e += 2) {
                        r0 = fmax3(r0, __uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1]));
                        r1 = fmax3(r1, __uint_as_float(s[c][e + 16]), __uint_as_float(s[c][e + 17]));
                    }
                    cmax[c] = fmaxf(r0, r1);
                }
                const float rmax = fmaxf(fmaxf(cmax[0], cmax[1]), fmaxf(cmax[2], cmax[3]));
                const float m_new = fmaxf(m, rmax * sl2);
                const bool rescale = m_new > m + kRescaleThreshold;   // also when m == -inf
                const float m_use = rescale ? m_new : m;
                const float alpha = rescale ? fast_exp2(m - m_new) : 1.f;
                // a row with every key so far masked keeps m = -inf; its weights are 0
                const float m_sub = m_use == -INFINITY ? 0.f : m_use;
                // The O rescale and the zeroing of V rows below both precede the release
                // of the first half of P.
                if (j > 0 && __any_sync(0xffffffffu, rescale)) {
                    // O must hold O += P V of the previous tile before it is rescaled (that
                    // product was issued before this tile's S, so it has completed).
                    ok = wait_or_abort(smem_u32(&sm.o_done[x]), (it - 1) & 1, abort_flag, a.err);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                    // 8 columns at a time: the scores of this tile are still live in registers
#pragma unroll 1
                    for (int c = 0; c < 16; ++c) {
                        uint32_t o[8];
                        tmem_ld8(lane_base + o_col + c * 8, o);
                        tmem_wait_ld8(o);
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st8(lane_base + o_col + c * 8, o);
                    }
                }
                // V rows that are no keys (past the end of the context, past the cached
                // positions, or rows of another sequence in k_new) may hold anything, NaN
                // included; P is 0 there but 0 * NaN is not, so tile A (the V tile's first
                // reader) zeroes them.
                if (x == 0 && kv_valid < kKT) {
                    const int vs = it % kVStages;
                    ok = wait_or_abort(smem_u32(&sm.v_full[vs]), (it / kVStages) & 1, abort_flag, a.err);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    if (row >= kv_valid) {
                        uint4 *r0 = reinterpret_cast<uint4 *>(sm.v[vs][0] + row * 128);
                        uint4 *r1 = reinterpret_cast<uint4 *>(sm.v[vs][1] + row * 128);
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            r0[v] = make_uint4(0u, 0u, 0u, 0u);
                            r1[v] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    fence_proxy_async_smem();   // generic writes -> visible to the MMA's reads
                }
                float part[4] = {0.f, 0.f, 0.f, 0.f};   // 4 partial row sums
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int c = 2 * h; c < 2 * h + 2; ++c) {
                        uint32_t pk[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float x0, x1;
                            ffma2(x0, x1, __uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1]), sl2, sl2,
                                  -m_sub, -m_sub);
                            const uint32_t pp = pack_bf16x2(fast_exp2(x0), fast_exp2(x1));
                            // the row sum uses the same bf16-rounded weights the PV product uses
                            const int k = (e >> 1) & 1;
                            part[2 * k] = add_bf16_lo(pp, part[2 * k]);
                            part[2 * k + 1] = add_bf16_hi(pp, part[2 * k + 1]);
                            pk[e / 2] = pp;
                        }
                        // P columns 16c..16c+15 go over S columns already read into registers
                        tmem_st16(lane_base + s_col + 16 * c, pk);
                    }
                    // P of keys 64h..64h+63 is in tensor memory: release that half of O += P V
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sm.p_half[x][h]));
                }
                const float rsum = (part[0] + part[1]) + (part[2] + part[3]);
                l = l * alpha + rsum;
                m = m_use;
            }
            if (!ok) break;

            // ------------------------------------------------------------ epilogue
            ok = wait_or_abort(smem_u32(&sm.o_done[x]), (it - 1) & 1, abort_flag, a.err);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const float inv_l = 1.f / l;
            const bool row_ok = x * kTilePos + pl < t.positions;
            // shared-prefix mode: fp32 partials of key split ks, [ks][token][32][128]
            const size_t orow = (size_t)t.ks * a.total_tokens * kHq +
                                (size_t)(t.tok0 + x * kTilePos + pl) * kHq + t.g * kGroup + hl;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tmem_ld32(lane_base + o_col + c * 32, o);
                tmem_wait_ld(o);
                if constexpr (kPrefix) {
                    if (row_ok) {
                        float4 *d4 = reinterpret_cast<float4 *>(static_cast<float *>(a.out) + orow * kD + c * 32);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            d4[v] = make_float4(__uint_as_float(o[4 * v]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                                __uint_as_float(o[4 * v + 2]) * inv_l,
                                                __uint_as_float(o[4 * v + 3]) * inv_l);
                    }
                } else {
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        w[e / 2] = pack_bf16x2(__uint_as_float(o[e]) * inv_l, __uint_as_float(o[e + 1]) * inv_l);
                    // 32-byte stores: each writes whole sectors (out is 32-byte aligned, rows
                    // are 256 bytes); 16-byte ones left every sector of a warp's store half written
                    if (row_ok) {
                        __nv_bfloat16 *d = static_cast<__nv_bfloat16 *>(a.out) + orow * kD + c * 32;
                        st_global_32b(d, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                        st_global_32b(d + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
                    }
                }
            }
            if (row_ok && a.lse) a.lse[orow] = (m + __log2f(l)) * kLn2;
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

template <bool kPrefix, bool kPlanned, bool kAppend>
cudaError_t launch_prefill_mode(const PrefillArgs &a, const CUtensorMap &q_map, const CUtensorMap &k_map,
                                const CUtensorMap &v_map, const CUtensorMap &kn_map, const CUtensorMap &vn_map,
                                int num_sms, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool configured[64] = {};
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(prefill_kernel<kPrefix, kPlanned, kAppend>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    const long long qblocks = (a.max_q_len + kUnitPos - 1) / kUnitPos;
    const long long units = kPrefix ? kHkv * qblocks * a.n_kv_splits : (long long)a.num_seqs * kHkv * qblocks;
    const int grid = (int)(units < num_sms ? units : num_sms);
    // Programmatic dependent launch: the producers wait (griddepcontrol.wait) before their
    // first load, so the launch and prologue may overlap the previous kernel on the stream.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (kPlanned) {
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(kPlanThreads);
        cfg.dynamicSmemBytes = 0;
        e = cudaLaunchKernelEx(&cfg, prefill_plan_kernel<kAppend>, a, (int)qblocks, (int)units, plan_keys(a));
        if (e != cudaSuccess) return e;
    }
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kAppend ? kThreadsAppend : kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    return cudaLaunchKernelEx(&cfg, prefill_kernel<kPrefix, kPlanned, kAppend>, q_map, k_map, v_map, kn_map, vn_map,
                              a);
}

}  // namespace

long long prefill_plan_units(const PrefillArgs &a) {
    if (a.num_seqs <= 1 || plan_keys(a) > kPlanMaxKeys) return 0;
    return (long long)a.num_seqs * kHkv * ((a.max_q_len + kUnitPos - 1) / kUnitPos);
}

cudaError_t launch_prefill(const PrefillArgs &a, const CUtensorMap &q_map, const CUtensorMap &k_map,
                           const CUtensorMap &v_map, int num_sms, cudaStream_t stream) {
    if (a.num_seqs == 0 || a.max_q_len == 0 || a.total_tokens == 0) return cudaSuccess;
    // (the maps of the new rows are unused without the fused append)
    if (a.order) return launch_prefill_mode<false, true, false>(a, q_map, k_map, v_map, k_map, v_map, num_sms, stream);
    return launch_prefill_mode<false, false, false>(a, q_map, k_map, v_map, k_map, v_map, num_sms, stream);
}

cudaError_t launch_prefill_append(const PrefillArgs &a, const CUtensorMap &q_map, const CUtensorMap &k_map,
                                  const CUtensorMap &v_map, const CUtensorMap &kn_map, const CUtensorMap &vn_map,
                                  int num_sms, cudaStream_t stream) {
    if (a.num_seqs == 0 || a.max_q_len == 0 || a.total_tokens == 0 || !a.k_new) return cudaSuccess;
    if (a.order) return launch_prefill_mode<false, true, true>(a, q_map, k_map, v_map, kn_map, vn_map, num_sms, stream);
    return launch_prefill_mode<false, false, true>(a, q_map, k_map, v_map, kn_map, vn_map, num_sms, stream);
}

cudaError_t launch_prefill_prefix(const PrefillArgs &a, const CUtensorMap &q_map, const CUtensorMap &k_map,
                                  const CUtensorMap &v_map, int num_sms, cudaStream_t stream) {
    if (a.num_seqs == 0 || a.max_q_len == 0 || a.total_tokens == 0) return cudaSuccess;
    return launch_prefill_mode<true, false, false>(a, q_map, k_map, v_map, k_map, v_map, num_sms, stream);
}

cudaError_t launch_wait_selftest(uint32_t *err, uint64_t limit_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace pa
