// qkv.cu -- the merged Q/K/V projection of a batch of new tokens, with K and V written
// straight into their slots of the paged cache.
//
// Page "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎，C++/CUDA 实现性能追平 98%":
//   §4.4.3 QKV fusion   the three projections are one matrix product with the weights
//                       stacked (w_qkv_merged), whose output is sliced into q, k, v;
//   §4.4.2 GQA          k and v have the 8 KV heads (1024 columns each), q the 32 heads;
//   §4.3.1              KV in 256-token blocks reached through a block table.
// Page "从零搭建AI工程能力：手写KV Cache与动态批处理实战" §3.2: the new tokens' K and V are
// appended to the cache.
//
// out[t][n] = sum_k x[t][k] * w[n][k]  (w stored [6144 out][hidden in], as a linear layer's
// weight), fp32 accumulation, one bf16 rounding.  Columns 0-4095 are q (head n / 128,
// dim n % 128) and go to q_out[t]; columns 4096-5119 are k of KV head (n - 4096) / 128 and
// 5120-6143 v, written to the cache slot of token t (position seq_len - q_len + i of its
// sequence, as kv_append places it), so K and V never make a round trip through memory
// before they reach the cache.
//
// Rotary position embedding (optional; the pages define no position encoding, so its
// definition is RoFormer's, Su et al. 2021, in the pairing Qwen3 uses): dims i and i + 64 of
// every q and k head are turned by the angle p * theta^(-i/64) at the token's absolute
// position p, in fp32 on the accumulator before the single bf16 rounding; v is not turned.
// So that one epilogue thread holds both dims of a pair, a tile's output columns are taken
// in 32-column runs reordered as [dims 0-31 | dims 64-95 | dims 32-63 | dims 96-127] of each
// head (the weight rows are loaded in that order); every 64 tile columns are then the two
// halves of 32 pairs of one head.  The angle is a float-float product p * (hi + lo) of the
// frequency, reduced by 2 pi in three parts (Cody and Waite's method) before the sine and
// cosine: about 1e-6 rad at any position below 2^24.  The optional per-head normalisation of
// q and k (QK-norm) needs whole heads, which the product tiles below do not hold: it runs as a
// second, memory-bound kernel (qk_norm_kernel, at the end of this file) over the rows the
// projection wrote without a rotation, and applies the rotation after it.
//
// GEMM on the 5th-generation tensor cores: with more than 256 tokens a pair of CTAs on two
// SMs computes 256 tokens x 192 output columns (tcgen05.mma.cta_group::2, see the pair kernel
// below); with fewer, one CTA computes 128 tokens x 64 columns (the weights dominate the
// bytes).  The hidden dimension goes in steps of 64 through a TMA ring; two accumulators in
// tensor memory, so the epilogue of one tile overlaps the products of the next.  With at most 32 tokens only 32
// rows of x are loaded per stage (BMA = 32): the ring then holds twice the weight bytes in
// flight.  The MMA still reads 128 rows; rows 32-127 come from the neighbouring shared
// memory, their results are discarded.  CTA = 6 warps, persistent (both kernels):
//   warps 0-3  epilogue: thread = one token row = TMEM lane
//   warp 4     TMA producer (x and w tiles, 128-byte swizzle)
//   warp 5     TMEM allocator and the tcgen05.mma issuer (in a pair: rank 0's)
// Every wait is bounded; on expiry the CTA records PA_ERR_TIMEOUT and unwinds.
#include "common.cuh"
#include "launch.h"

namespace pa {
namespace {

constexpr int kQCols = kHq * kD;               // 4096
constexpr int kKVCols = kHkv * kD;             // 1024
constexpr int kBM = 128;                       // tokens per tile (MMA M)
constexpr int kBK = 64;                        // hidden elements per sub-tile (one 128-byte row)
constexpr int kEpiWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr uint32_t kParkNs = 20000;
constexpr uint32_t kRingBytes = 192 * 1024;    // the TMA ring's share of shared memory
constexpr int kRunCols = 32;                   // weight rows per TMA box: one run of 32 columns

// Output column (weight row) where logical 32-column run r starts: runs 4h .. 4h+3 are dims
// 0-31, 64-95, 32-63 and 96-127 of head h (heads 0-31 q, 32-39 k, 40-47 v), so logical columns
// 64c .. 64c+63 are the two halves of pairs (32c' + e, 32c' + e + 64), c' = c % 2, of head c / 2.
__host__ __device__ __forceinline__ int run_row(int r) {
    return (r >> 2) * kD + (r & 1) * (kD / 2) + ((r >> 1) & 1) * kRunCols;
}

// 2 pi in three fp32 parts (hi + mid + lo, each the rounding of what remains) and 1 / (2 pi)
constexpr double kTwoPiD = 6.28318530717958647692528676655900577;
constexpr float kTwoPiHi = (float)kTwoPiD;
constexpr float kTwoPiMid = (float)(kTwoPiD - (double)kTwoPiHi);
constexpr float kTwoPiLo = (float)(kTwoPiD - (double)kTwoPiHi - (double)kTwoPiMid);
constexpr float kInvTwoPi = (float)(1.0 / kTwoPiD);

// BN output columns per tile, BMA rows of x loaded per stage (128, or 32 for <= 32 tokens).
// A stage covers kSub adjacent sub-tiles of 64 hidden elements: with few tokens the weights
// come from DRAM once, and 4 sub-tiles make each weight row's share of a stage 512
// contiguous bytes instead of 128 (one DRAM page opened per 128 bytes held reads of the
// weights at a third of the bandwidth).
template <int BN, int BMA>
struct QkvCfg {
    static constexpr int kSub = 4;
    static constexpr uint32_t kASub = BMA * kBK * 2;
    static constexpr uint32_t kBSub = BN * kBK * 2;
    static constexpr uint32_t kABytes = kSub * kASub;
    static constexpr uint32_t kBBytes = kSub * kBSub;
    static constexpr int kStages = (int)(kRingBytes / (kABytes + kBBytes));
    static constexpr uint32_t kTmemCols = 2 * BN;   // two accumulators
    static constexpr uint32_t kIdesc = idesc_bf16(kBM, BN, false);   // both operands K-major
};

// A work item: tile row mt (its tokens) x `width` output columns from col0; width 0 past
// the end.  Tiles are dealt round-robin over the g workers (CTAs, or CTA pairs).
struct QkvItem {
    int mt, col0, width;
};

template <int BN>
__device__ __forceinline__ QkvItem qkv_item_of(int k, int m_tiles, int g, int c) {
    constexpr int n_tiles = (kQCols + 2 * kKVCols) / BN;
    QkvItem w = {0, 0, 0};
    const int t = c + k * g;
    if (t >= m_tiles * n_tiles) return w;
    w.mt = t / n_tiles;
    w.col0 = (t - w.mt * n_tiles) * BN;
    w.width = BN;
    return w;
}

// The item sequence of this CTA (one CTA per tile).
template <int BN>
__device__ __forceinline__ QkvItem qkv_item(int k, int m_tiles) {
    return qkv_item_of<BN>(k, m_tiles, (int)gridDim.x, (int)blockIdx.x);
}

template <int BN, int BMA>
struct QkvSmem {
    // the A stages first: an MMA over a 32-row stage reads 96 more rows after it, which
    // stay inside this struct (the next stages, then the B ring)
    uint8_t a[QkvCfg<BN, BMA>::kStages][QkvCfg<BN, BMA>::kABytes];
    uint8_t b[QkvCfg<BN, BMA>::kStages][QkvCfg<BN, BMA>::kBBytes];
    uint64_t full[QkvCfg<BN, BMA>::kStages], empty[QkvCfg<BN, BMA>::kStages];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t mma_idle;
    uint32_t tmem_base;
    int abort;
};

template <int BN, int BMA>
constexpr size_t qkv_smem_bytes() { return sizeof(QkvSmem<BN, BMA>) + 1024; }
static_assert(qkv_smem_bytes<64, 128>() <= 232448 &&
              qkv_smem_bytes<64, 32>() <= 232448, "shared memory");
// the 128-row MMA reads of the last 32-row A stage end inside the B ring
static_assert(QkvCfg<64, 32>::kStages * QkvCfg<64, 32>::kABytes + QkvCfg<64, 32>::kBBytes * QkvCfg<64, 32>::kStages >=
              QkvCfg<64, 32>::kStages * QkvCfg<64, 32>::kABytes - QkvCfg<64, 32>::kASub + kBM * kBK * 2,
              "A over-read");

// 2-D tiled TMA load (col, row) completing its bytes on the mbarrier
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

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

// Cache slot and absolute position of token t (the kv_append rule).  Returns the element
// offset of (slot, KV head 0, dim 0) in a pool, or -1 when the token's sequence data are
// inconsistent or its block id is outside the pool (recorded in the error word); *pos gets
// p = seq_len - q_len + i, or -1 when the sequence data are inconsistent.
// Token t's sequence (*seq) and absolute position p = seq_len - q_len + i, or -1 when the
// sequence data are inconsistent (recorded in the error word).
__device__ __forceinline__ int token_position(const QkvArgs &a, int t, int *seq) {
    int lo = 0, hi = a.num_seqs - 1;   // the sequence s with cu_q_lens[s] <= t < cu_q_lens[s + 1]
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(a.cu_q_lens + mid) <= t) lo = mid;
        else hi = mid - 1;
    }
    const int s = lo;
    *seq = s;
    const int c0 = __ldg(a.cu_q_lens + s), c1 = __ldg(a.cu_q_lens + s + 1);
    const int seq_len = __ldg(a.seq_lens + s);
    const int q_len = c1 - c0;
    if (c0 > t || t >= c1 || q_len > seq_len || seq_len > a.max_blocks_per_seq * kBlock) {
        record_error(a.err, kErrDevice | kErrBadCuQ);
        return -1;
    }
    return seq_len - q_len + (t - c0);
}

__device__ __forceinline__ long long token_slot(const QkvArgs &a, int t, int *pos) {
    int s;
    const int p = token_position(a, t, &s);
    *pos = p;
    if (p < 0) return -1;
    const int blk = __ldg(a.block_table + (size_t)s * a.max_blocks_per_seq + p / kBlock);
    if (blk < 0 || blk >= a.num_blocks) {
        record_error(a.err, kErrDevice | kErrBadBlock);
        return -1;
    }
    return ((long long)blk * kBlock + p % kBlock) * kHkv * kD;
}

// cos and sin of the rotation angle at position pf (an integer below 2^24, exact in fp32) for
// the frequency fh + fl (pair i's: rope_cos_sin).  p * freq is formed as hi + lo (the product's rounding error recovered with an fma),
// the multiple of 2 pi nearest hi is taken off in three parts (Cody and Waite), lo is added
// back, and the reduced angle (|r| < 4) goes to the fast sine/cosine.
__device__ __forceinline__ void angle_cos_sin(float pf, float fh, float fl, float &c, float &s) {
    const float ah = __fmul_rn(pf, fh);
    const float al = fmaf(pf, fl, fmaf(pf, fh, -ah));
    const float k = rintf(__fmul_rn(ah, kInvTwoPi));
    float r = fmaf(-k, kTwoPiHi, ah);
    r = fmaf(-k, kTwoPiMid, r);
    r = fmaf(-k, kTwoPiLo, r);
    __sincosf(__fadd_rn(r, al), &s, &c);
}

__device__ __forceinline__ void rope_cos_sin(const QkvArgs &a, int i, float pf, float &c, float &s) {
    angle_cos_sin(pf, a.rope_freq_hi[i], a.rope_freq_lo[i], c, s);
}

// The epilogue of one tile for this thread's token row: logical columns col0 .. col0+width-1
// of the accumulator at tensor-memory address tcol, 64 at a time (the halves of 32 pairs of one
// head), rotated when they are q or k dims and the rotation is on, rounded once to bf16 and
// stored to q_out (q heads) or the token's cache slot (k, v heads; dst_row < 0: not written).
// A q or k row whose position is unknown (inconsistent sequence data) comes out NaN.
__device__ __forceinline__ void store_tile_row(const QkvArgs &a, uint32_t tcol, int col0, int width, int tok,
                                               bool live, long long dst_row, int pos) {
#pragma unroll 1
    for (int j = 0; j < width / 64; ++j) {
        const int cp = (col0 >> 6) + j;            // 64-column group over the 6144 outputs
        const int head = cp >> 1, half = cp & 1;   // dims half*32 .. +31 and 64 + half*32 .. +31
        uint32_t lo[32], hi[32];
        tmem_ld32(tcol + (uint32_t)(j * 64), lo);
        tmem_ld32(tcol + (uint32_t)(j * 64 + 32), hi);
        tmem_wait_ld(lo);
        tmem_wait_ld(hi);
        if (a.rope && head < kHq + kHkv) {
            const float pf = (float)pos;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                float c, sn;
                rope_cos_sin(a, half * 32 + e, pf, c, sn);
                if (pos < 0) c = sn = __int_as_float(0x7fc00000);
                const float x0 = __uint_as_float(lo[e]), x1 = __uint_as_float(hi[e]);
                lo[e] = __float_as_uint(fmaf(x0, c, -__fmul_rn(x1, sn)));
                hi[e] = __float_as_uint(fmaf(x1, c, __fmul_rn(x0, sn)));
            }
        }
        __nv_bfloat16 *dst = nullptr;
        if (head < kHq) {
            if (live) dst = static_cast<__nv_bfloat16 *>(a.q_out) + (size_t)tok * kQCols + head * kD;
        } else if (dst_row >= 0) {
            const bool is_k = head < kHq + kHkv;
            dst = static_cast<__nv_bfloat16 *>(is_k ? a.k_pool : a.v_pool) + dst_row +
                  (head - kHq - (is_k ? 0 : kHkv)) * kD;
        }
        if (dst) {
            uint4 *d_lo = reinterpret_cast<uint4 *>(dst + half * 32);
            uint4 *d_hi = reinterpret_cast<uint4 *>(dst + kD / 2 + half * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                d_lo[q] = make_uint4(pack_bf16x2(__uint_as_float(lo[8 * q]), __uint_as_float(lo[8 * q + 1])),
                                     pack_bf16x2(__uint_as_float(lo[8 * q + 2]), __uint_as_float(lo[8 * q + 3])),
                                     pack_bf16x2(__uint_as_float(lo[8 * q + 4]), __uint_as_float(lo[8 * q + 5])),
                                     pack_bf16x2(__uint_as_float(lo[8 * q + 6]), __uint_as_float(lo[8 * q + 7])));
                d_hi[q] = make_uint4(pack_bf16x2(__uint_as_float(hi[8 * q]), __uint_as_float(hi[8 * q + 1])),
                                     pack_bf16x2(__uint_as_float(hi[8 * q + 2]), __uint_as_float(hi[8 * q + 3])),
                                     pack_bf16x2(__uint_as_float(hi[8 * q + 4]), __uint_as_float(hi[8 * q + 5])),
                                     pack_bf16x2(__uint_as_float(hi[8 * q + 6]), __uint_as_float(hi[8 * q + 7])));
            }
        }
    }
}

template <int BN, int BMA>
__global__ void __launch_bounds__(kThreads, 1)
qkv_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap w_map,
           const __grid_constant__ QkvArgs a) {
    using Cfg = QkvCfg<BN, BMA>;
    constexpr int kStages = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    QkvSmem<BN, BMA> &sm = *reinterpret_cast<QkvSmem<BN, BMA> *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    volatile int *abort_flag = &sm.abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int m_tiles = (a.total_tokens + kBM - 1) / kBM;
    const int ksteps = a.hidden / (kBK * Cfg::kSub);   // stages per tile

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&sm.full[i]), 1);
            mbar_init(smem_u32(&sm.empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sm.acc_full[i]), 1);
            mbar_init(smem_u32(&sm.acc_empty[i]), kEpiWarps);
        }
        mbar_init(smem_u32(&sm.mma_idle), 1);
        sm.abort = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&sm.tmem_base), Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------------- TMA producer
        const bool leader = elect_one();
        if (leader) {
            tma_prefetch_map(&x_map);
            tma_prefetch_map(&w_map);
        }
        // x may be written by the kernel just before this one on the stream
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int it = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const QkvItem w = qkv_item<BN>(k, m_tiles);
            if (!w.width) break;
            const uint32_t b_bytes = Cfg::kBBytes;
            for (int kc = 0; kc < ksteps; ++kc, ++it) {
                const int s = it % kStages;
                if (it >= kStages &&
                    !(ok = __all_sync(0xffffffffu, wait_or_abort(smem_u32(&sm.empty[s]), ((it / kStages) - 1) & 1,
                                                                abort_flag, a.err))))
                    break;
                if (leader) {
                    const uint32_t bar = smem_u32(&sm.full[s]);
                    mbar_arrive_expect_tx(bar, Cfg::kABytes + b_bytes);
#pragma unroll
                    for (int j = 0; j < Cfg::kSub; ++j) {
                        const int k0 = (kc * Cfg::kSub + j) * kBK;
                        tma_load_2d(smem_u32(sm.a[s] + j * Cfg::kASub), &x_map, bar, k0, w.mt * kBM);
                        // the weight rows in runs of 32 (128 B each), stacked in logical order
                        for (int r = 0; r < w.width / kRunCols; ++r)
                            tma_load_2d(smem_u32(sm.b[s] + j * Cfg::kBSub + r * kRunCols * 128), &w_map, bar, k0,
                                        run_row(w.col0 / kRunCols + r));
                    }
                }
                __syncwarp();
            }
        }
        // no copy may still be landing when the CTA exits
        for (int i = max(0, it - kStages); i < it; ++i) mbar_wait(smem_u32(&sm.full[i % kStages]), (i / kStages) & 1);
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        const bool leader = elect_one();
        const uint64_t ad0 = sdesc_sw128(smem_u32(sm.a[0]), 16, 1024);
        const uint64_t bd0 = sdesc_sw128(smem_u32(sm.b[0]), 16, 1024);
        int it = 0, lt = 0;
        bool ok = true;
        for (int k = 0; ok; ++k, ++lt) {
            const QkvItem w = qkv_item<BN>(k, m_tiles);
            if (!w.width) break;
            const uint32_t idesc = Cfg::kIdesc;
            const int acc = lt & 1;
            if (lt >= 2 && !(ok = __all_sync(0xffffffffu, wait_or_abort(smem_u32(&sm.acc_empty[acc]),
                                                                         ((lt >> 1) - 1) & 1, abort_flag, a.err))))
                break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * BN);
            for (int kc = 0; kc < ksteps; ++kc, ++it) {
                const int s = it % kStages;
                if (!(ok = __all_sync(0xffffffffu, wait_or_abort(smem_u32(&sm.full[s]), (it / kStages) & 1,
                                                                abort_flag, a.err))))
                    break;
                tc_fence_after();
                // +2 per 16 elements along the 128-byte row; a stage is BMA / BN rows of 128 B
                const uint64_t ad = ad0 + (uint64_t)(s * (Cfg::kABytes >> 4));
                const uint64_t bd = bd0 + (uint64_t)(s * (Cfg::kBBytes >> 4));
                if (leader) {
#pragma unroll
                    for (int j = 0; j < Cfg::kSub; ++j) {
                        const uint64_t adj = ad + (uint64_t)(j * (Cfg::kASub >> 4));
                        const uint64_t bdj = bd + (uint64_t)(j * (Cfg::kBSub >> 4));
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            if (kc == 0 && j == 0 && kk == 0) umma_ss_c<false>(d, adj, bdj, idesc);
                            else umma_ss_c<true>(d, adj + (uint64_t)(kk * 2), bdj + (uint64_t)(kk * 2), idesc);
                        }
                    }
                    umma_commit(smem_u32(&sm.empty[s]));
                }
                __syncwarp();
            }
            if (!ok) break;
            if (leader) umma_commit(smem_u32(&sm.acc_full[acc]));
            __syncwarp();
        }
        // every MMA issued must have finished before tensor memory is released
        if (leader) umma_commit(smem_u32(&sm.mma_idle));
        __syncwarp();
        mbar_wait(smem_u32(&sm.mma_idle), 0);
    } else {
        // ---------------------------------------------------------------- epilogue warps
        // q_out and the pools may still be read by the kernel before this one on the stream
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int row = warp * 32 + lane;                       // token row = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        int lt = 0, cached_mt = -1, pos = -1;
        long long dst_row = -1;
        for (int k = 0;; ++k, ++lt) {
            const QkvItem w = qkv_item<BN>(k, m_tiles);
            if (!w.width) break;
            const int mt = w.mt;
            const int acc = lt & 1;
            const int tok = mt * kBM + row;
            const bool live = tok < a.total_tokens;
            // K/V columns need the token's cache slot, rotated q or k columns its position
            if ((w.col0 + w.width > kQCols || a.rope) && mt != cached_mt) {
                dst_row = live ? token_slot(a, tok, &pos) : -1;
                cached_mt = mt;
            }
            const bool ok = wait_or_abort(smem_u32(&sm.acc_full[acc]), (lt >> 1) & 1, abort_flag, a.err);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            store_tile_row(a, lane_base + (uint32_t)(acc * BN), w.col0, w.width, tok, live, dst_row, pos);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.acc_empty[acc]));
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}


// ------------------------------------------------------------------ CTA pairs (many tokens)
// With many tokens a 128 x 256 tile of one CTA needs ~190 GB/s of L2 -> SM traffic at the
// full tensor rate, more than one SM receives.  A pair of CTAs on two SMs (a 2-CTA cluster)
// computes a 256 x 192 tile with tcgen05.mma.cta_group::2 (M = 256): each SM holds its own
// 128 token rows and loads only half of the 192 weight rows, the MMA reading the other half
// from the peer's shared memory (~147 GB/s per SM at the full rate; 192 rather than 256
// columns deal 4096 tokens' 512 tiles over 76 pairs in 6.7 rounds instead of 5.05).  Rank 0's MMA warp issues for
// both; both halves of a stage complete on rank 0's barrier (pair-scoped TMA), rank 0's
// commits reach both CTAs (multicast), and both CTAs' epilogue warps hand an accumulator back
// on rank 0's barrier.  Each CTA's tensor memory holds its rows' two accumulators.
constexpr int kPairBM = 2 * kBM;                       // tokens per pair tile
constexpr int kPairBN = 192;                           // 4096 tokens: 512 tiles, 6.7 per pair
constexpr uint32_t kPairABytes = kBM * kBK * 2;        // this CTA's 128 rows x 64: 16 KiB
constexpr uint32_t kPairBBytes = (kPairBN / 2) * kBK * 2;   // this CTA's 96 weight rows: 12 KiB
constexpr int kPairStages = (int)(kRingBytes / (kPairABytes + kPairBBytes));
constexpr uint32_t kPairIdesc = idesc_bf16(kPairBM, kPairBN, false);

struct QkvPairSmem {
    uint8_t a[kPairStages][kPairABytes];
    uint8_t b[kPairStages][kPairBBytes];
    uint64_t full[kPairStages], empty[kPairStages];    // full: rank 0's counts both CTAs' copies
    uint64_t acc_full[2], acc_empty[2];                // acc_empty: rank 0's, both CTAs' epilogues
    uint64_t mma_idle;
    uint32_t tmem_base;
    int abort;
};
constexpr size_t kPairSmemBytes = sizeof(QkvPairSmem) + 1024;
static_assert(kPairSmemBytes <= 232448, "shared memory");

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// Arrive on a barrier of either CTA of the pair (release at CTA scope: what it announces is
// tensor memory this thread has finished reading).
__device__ __forceinline__ void arrive_remote(uint32_t cluster_bar) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Every thread of both CTAs.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 2-D TMA load into this CTA's shared memory completing on a barrier of either CTA
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t cluster_bar, int c0,
                                                 int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(cluster_bar)
        : "memory");
}

// D rows 0-127 in rank 0's tensor memory, 128-255 in rank 1's; A rows likewise from each
// CTA's shared memory at the same address; B columns 0 .. N/2-1 from rank 0, the rest from
// rank 1.
template <bool kAcc>
__device__ __forceinline__ void umma_ss_pair_c(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "n"(kAcc ? 1 : 0)
        : "memory");
}

// Arrive on the barrier at this offset in both CTAs once every prior pair MMA has completed.
__device__ __forceinline__ void umma_commit_both(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                 ::"r"(bar), "h"((uint16_t)3)
                 : "memory");
}

__device__ __forceinline__ void umma_commit_local(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
qkv_pair_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap w_map,
                const __grid_constant__ QkvArgs a) {
    extern __shared__ uint8_t smem_raw[];
    QkvPairSmem &sm = *reinterpret_cast<QkvPairSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    volatile int *abort_flag = &sm.abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool lead = rank == 0;
    const int m_tiles = (a.total_tokens + kPairBM - 1) / kPairBM;
    const int clusters = (int)gridDim.x >> 1, cid = (int)blockIdx.x >> 1;
    const int ksteps = a.hidden / kBK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kPairStages; ++i) {
            mbar_init(smem_u32(&sm.full[i]), 1);
            mbar_init(smem_u32(&sm.empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sm.acc_full[i]), 1);
            mbar_init(smem_u32(&sm.acc_empty[i]), 2 * kEpiWarps);
        }
        mbar_init(smem_u32(&sm.mma_idle), 1);
        sm.abort = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        // one warp of each CTA allocates the pair's tensor memory together
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&sm.tmem_base)),
                     "r"(512u)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    // both CTAs' barriers and tensor memory exist before either issues anything to the other
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == kProducerWarp) {
        // ---------------------------------------------------------------- TMA producer
        const bool leader = elect_one();
        if (leader) {
            tma_prefetch_map(&x_map);
            tma_prefetch_map(&w_map);
        }
        // x may be written by the kernel just before this one on the stream
        asm volatile("griddepcontrol.wait;" ::: "memory");
        int it = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const QkvItem w = qkv_item_of<kPairBN>(k, m_tiles, clusters, cid);
            if (!w.width) break;
            const int cols = w.width / 2;                  // weight rows this CTA loads
            for (int kc = 0; kc < ksteps; ++kc, ++it) {
                const int s = it % kPairStages;
                if (it >= kPairStages &&
                    !(ok = __all_sync(0xffffffffu, wait_or_abort(smem_u32(&sm.empty[s]),
                                                                ((it / kPairStages) - 1) & 1, abort_flag, a.err))))
                    break;
                if (leader) {
                    const uint32_t bar = smem_u32(&sm.full[s]);
                    if (lead) mbar_arrive_expect_tx(bar, 2 * (kPairABytes + (uint32_t)cols * 128));
                    const uint32_t bar0 = peer_addr(bar, 0);
                    const int k0 = kc * kBK;
                    tma_load_2d_pair(smem_u32(sm.a[s]), &x_map, bar0, k0, w.mt * kPairBM + (int)rank * kBM);
                    // this CTA's half of the tile's weight rows, in runs of 32 in logical order
                    for (int r = 0; r < cols / kRunCols; ++r)
                        tma_load_2d_pair(smem_u32(sm.b[s] + r * kRunCols * 128), &w_map, bar0, k0,
                                         run_row((w.col0 + (int)rank * cols) / kRunCols + r));
                }
                __syncwarp();
            }
        }
        // No copy may still be landing when the CTA exits: both CTAs' copies complete on rank
        // 0's barriers, which rank 0 waits on here (the MMA warp consumed them all in the
        // normal path); rank 1 stays until the cluster barrier below.
        if (lead)
            for (int i = max(0, it - kPairStages); i < it; ++i)
                mbar_wait(smem_u32(&sm.full[i % kPairStages]), (i / kPairStages) & 1);
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer (rank 0)
        if (lead) {
            const bool leader = elect_one();
            const uint64_t ad0 = sdesc_sw128(smem_u32(sm.a[0]), 16, 1024);
            const uint64_t bd0 = sdesc_sw128(smem_u32(sm.b[0]), 16, 1024);
            int it = 0, lt = 0;
            bool ok = true;
            for (int k = 0; ok; ++k, ++lt) {
                const QkvItem w = qkv_item_of<kPairBN>(k, m_tiles, clusters, cid);
                if (!w.width) break;
                const uint32_t idesc = kPairIdesc;
                const int acc = lt & 1;
                if (lt >= 2 && !(ok = __all_sync(0xffffffffu, wait_or_abort(smem_u32(&sm.acc_empty[acc]),
                                                                             ((lt >> 1) - 1) & 1, abort_flag, a.err))))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * kPairBN);
                for (int kc = 0; kc < ksteps; ++kc, ++it) {
                    const int s = it % kPairStages;
                    if (!(ok = __all_sync(0xffffffffu, wait_or_abort(smem_u32(&sm.full[s]), (it / kPairStages) & 1,
                                                                    abort_flag, a.err))))
                        break;
                    tc_fence_after();
                    // +2 per 16 elements along the 128-byte row; +stage size per stage
                    const uint64_t ad = ad0 + (uint64_t)(s * (kPairABytes >> 4));
                    const uint64_t bd = bd0 + (uint64_t)(s * (kPairBBytes >> 4));
                    if (leader) {
                        if (kc == 0) umma_ss_pair_c<false>(d, ad, bd, idesc);
                        else umma_ss_pair_c<true>(d, ad, bd, idesc);
#pragma unroll
                        for (int kk = 1; kk < kBK / 16; ++kk)
                            umma_ss_pair_c<true>(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc);
                        umma_commit_both(smem_u32(&sm.empty[s]));
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (leader) umma_commit_both(smem_u32(&sm.acc_full[acc]));
                __syncwarp();
            }
            // every MMA issued must have finished before tensor memory is released
            if (leader) umma_commit_local(smem_u32(&sm.mma_idle));
            __syncwarp();
            mbar_wait(smem_u32(&sm.mma_idle), 0);
        }
    } else {
        // ---------------------------------------------------------------- epilogue warps
        // q_out and the pools may still be read by the kernel before this one on the stream
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int row = warp * 32 + lane;                       // token row = TMEM lane
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const uint32_t acc_empty0 = peer_addr(smem_u32(&sm.acc_empty[0]), 0);   // + 8 per accumulator
        int lt = 0, cached_mt = -1, pos = -1;
        long long dst_row = -1;
        for (int k = 0;; ++k, ++lt) {
            const QkvItem w = qkv_item_of<kPairBN>(k, m_tiles, clusters, cid);
            if (!w.width) break;
            const int acc = lt & 1;
            const int tok = w.mt * kPairBM + (int)rank * kBM + row;
            const bool live = tok < a.total_tokens;
            // K/V columns need the token's cache slot, rotated q or k columns its position
            if ((w.col0 + w.width > kQCols || a.rope) && w.mt != cached_mt) {
                dst_row = live ? token_slot(a, tok, &pos) : -1;
                cached_mt = w.mt;
            }
            const bool ok = wait_or_abort(smem_u32(&sm.acc_full[acc]), (lt >> 1) & 1, abort_flag, a.err);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            store_tile_row(a, lane_base + (uint32_t)(acc * kPairBN), w.col0, w.width, tok, live, dst_row, pos);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_remote(acc_empty0 + (uint32_t)acc * 8u);
        }
    }

    // ---------------------------------------------------------------- teardown
    // Both CTAs meet before tensor memory is released or either exits: rank 0's MMAs read the
    // peer's shared memory and write its tensor memory until mma_idle.
    __syncthreads();
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    if (warp == kMmaWarp) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512u) : "memory");
    }
}

cudaError_t launch_qkv_pair(const QkvArgs &a, const CUtensorMap &x_map, const CUtensorMap &w_map, int num_sms,
                            cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static int max_clusters[64] = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kPairSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (max_clusters[dev] == 0) {
        e = cudaFuncSetAttribute(qkv_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPairSmemBytes);
        if (e != cudaSuccess) return e;
        int n = 0;
        cfg.gridDim = dim3(2 * (num_sms / 2));
        e = cudaOccupancyMaxActiveClusters(&n, qkv_pair_kernel, &cfg);
        if (e != cudaSuccess) return e;
        if (n < 1) return cudaErrorInvalidConfiguration;
        max_clusters[dev] = n;
    }
    const long long tiles = (long long)((a.total_tokens + kPairBM - 1) / kPairBM) * ((kQCols + 2 * kKVCols) / kPairBN);
    const int clusters = (int)(tiles < max_clusters[dev] ? tiles : max_clusters[dev]);
    cfg.gridDim = dim3(2 * clusters);
    return cudaLaunchKernelEx(&cfg, qkv_pair_kernel, x_map, w_map, a);
}

template <int BN, int BMA>
cudaError_t launch_qkv_bn(const QkvArgs &a, const CUtensorMap &x_map, const CUtensorMap &w_map, int num_sms,
                          cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool configured[64] = {};
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        e = cudaFuncSetAttribute(qkv_kernel<BN, BMA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)qkv_smem_bytes<BN, BMA>());
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    const long long tiles = (long long)((a.total_tokens + kBM - 1) / kBM) * ((kQCols + 2 * kKVCols) / BN);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles < num_sms ? tiles : num_sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = qkv_smem_bytes<BN, BMA>();
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qkv_kernel<BN, BMA>, x_map, w_map, a);
}

// ------------------------------------------------------------------ QK-norm (optional)
// Per-head RMS normalisation of the q and k heads.  The pages define none; Qwen3 normalises
// each q and k head before the rotary embedding with RMSNorm (Zhang and Sennrich 2019, §3):
// a head x of 128 values, as the projection wrote it (bf16, not rotated), becomes
//     y[d] = g[d] * x[d] / sqrt(mean(x^2) + eps)
// in fp32, g the q or the k gain; with the rotation on it is then turned by the token's
// angles (the rotation store_tile_row applies), and it is rounded to bf16 in place.
//
// A token's heads come in 5 groups of 8: groups 0-3 are q heads 8g .. 8g+7 (2 KiB contiguous
// in q_out), group 4 the token's 8 k heads (2 KiB contiguous at its cache slot).  A warp takes
// `groups_per_warp` consecutive groups of one token (all 5 when there are many tokens, so the
// token's lookup and angles are computed once; 1 when there are few, for parallelism).  Lane l
// holds dims 2l, 2l+1, 64+2l and 65+2l of each head -- both dims of two rotation pairs -- so
// only the sums of squares cross lanes, and every load and store of the warp is 128 contiguous
// bytes.  The rows it reads were just written by the projection and sit in L2; its instruction
// count mattered (a first form with 40 shuffles and an IEEE division and square root per head
// took twice as long), hence the packed fp32 arithmetic, rsqrtf and a reduce-scatter of the eight
// sums (17 shuffles instead of 40).
constexpr int kNormGroups = kHq / 8 + 1;       // 4 groups of q heads + the k heads
constexpr int kNormThreads = 256;
constexpr int kNormCtasPerSm = 4;              // 64 registers a thread

// The sums of v[0..7] over the warp, for every lane: reduce-scatter (after the steps over lane
// bits 16, 8 and 4 a lane holds a partial of head h(lane) = 4 b16 + 2 b8 + b4, the steps over
// bits 2 and 1 complete it; lanes that share h compute the same value since each addition
// commutes), then one shuffle per head from a lane that holds it.  f(total) is applied once per
// lane, before the gather.
template <typename F>
__device__ __forceinline__ void warp_sums8(float (&v)[8], int lane, F f) {
    const bool b16 = lane & 16, b8 = lane & 8, b4 = lane & 4;
    float u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float keep = b16 ? v[i + 4] : v[i], send = b16 ? v[i] : v[i + 4];
        u[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    float t[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float keep = b8 ? u[i + 2] : u[i], send = b8 ? u[i] : u[i + 2];
        t[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float r = (b4 ? t[1] : t[0]) + __shfl_xor_sync(0xffffffffu, b4 ? t[0] : t[1], 4);
    r += __shfl_xor_sync(0xffffffffu, r, 2);
    r += __shfl_xor_sync(0xffffffffu, r, 1);
    r = f(r);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __shfl_sync(0xffffffffu, r, ((j & 4) << 2) | ((j & 2) << 2) | ((j & 1) << 2));
}

__global__ void __launch_bounds__(kNormThreads, kNormCtasPerSm)
qk_norm_kernel(const __grid_constant__ QkvArgs a, int groups_per_warp) {
    // q_out and the cache rows are the projection's, launched just before on the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    // the rotation frequencies, copied once into shared memory: read from the argument space at
    // an index that differs between lanes, every read would be serialised
    __shared__ float2 freq[kRopePairs];            // (hi, lo) of pair i
    if (threadIdx.x < kRopePairs) freq[threadIdx.x] = make_float2(a.rope_freq_hi[threadIdx.x], a.rope_freq_lo[threadIdx.x]);
    __syncthreads();
    const int chunks = (kNormGroups + groups_per_warp - 1) / groups_per_warp;
    const long long work = (long long)a.total_tokens * chunks;
    const long long step = (long long)gridDim.x * (kNormThreads / 32);
    for (long long w = (long long)blockIdx.x * (kNormThreads / 32) + (threadIdx.x >> 5); w < work; w += step) {
        const int tok = (int)(w / chunks);
        const int g0 = (int)(w % chunks) * groups_per_warp;
        const int g1 = min(kNormGroups, g0 + groups_per_warp);
        int pos = -1;
        long long slot = -1;
        if (g1 == kNormGroups) {
            slot = token_slot(a, tok, &pos);
        } else if (a.rope) {
            int seq;
            pos = token_position(a, tok, &seq);
        }
        float c0 = 1.f, s0 = 0.f, c1 = 1.f, s1 = 0.f;   // pairs 2l and 2l+1
        if (a.rope) {
            const float pf = (float)pos;
            const float2 f0 = freq[2 * lane], f1 = freq[2 * lane + 1];
            angle_cos_sin(pf, f0.x, f0.y, c0, s0);
            angle_cos_sin(pf, f1.x, f1.y, c1, s1);
            if (pos < 0) c0 = s0 = c1 = s1 = __int_as_float(0x7fc00000);   // position unknown
        }
        for (int g = g0; g < g1; ++g) {
            const bool is_k = g == kNormGroups - 1;
            if (is_k && slot < 0) break;          // no k row was written for this token
            uint32_t *row = is_k ? reinterpret_cast<uint32_t *>(static_cast<__nv_bfloat16 *>(a.k_pool) + slot)
                                 : reinterpret_cast<uint32_t *>(static_cast<__nv_bfloat16 *>(a.q_out) +
                                                                ((size_t)tok * kHq + g * 8) * kD);
            uint32_t w_lo[8], w_hi[8];            // dims (2l, 2l+1) and (64+2l, 65+2l) of 8 heads
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                w_lo[h] = row[h * (kD / 2) + lane];
                w_hi[h] = row[h * (kD / 2) + 32 + lane];
            }
            // this lane's gains (dims 2l, 2l+1, 64+2l, 65+2l), from L1 after the first group, and the
            // coefficients of out[2l] = inv (x[2l] g c0 - x[64+2l] g' s0), out[64+2l] = inv (x[64+2l] g' c0
            // + x[2l] g s0) (the same for dims 2l+1, 65+2l with c1, s1), inv = 1 / the head's RMS
            const uint32_t *gw = static_cast<const uint32_t *>(is_k ? a.k_norm : a.q_norm);
            const uint32_t gl = __ldg(gw + lane), gh = __ldg(gw + 32 + lane);
            const float G0 = bf16_lo(gl), G1 = bf16_hi(gl);
            const float G2 = bf16_lo(gh), G3 = bf16_hi(gh);
            const float A0 = G0 * c0, A1 = G1 * c1, nB0 = -(G2 * s0), nB1 = -(G3 * s1);   // -> dims 2l, 2l+1
            const float A2 = G2 * c0, A3 = G3 * c1, B2 = G0 * s0, B3 = G1 * s1;           // -> dims 64+2l, 65+2l
            float ss[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const float x0 = bf16_lo(w_lo[h]), x1 = bf16_hi(w_lo[h]);
                const float x2 = bf16_lo(w_hi[h]), x3 = bf16_hi(w_hi[h]);
                float p, q;
                ffma2(p, q, x0, x1, x0, x1, 0.f, 0.f);
                ffma2(p, q, x2, x3, x2, x3, p, q);
                ss[h] = p + q;
            }
            const float eps = a.norm_eps;
            warp_sums8(ss, lane, [eps](float t) { return rsqrtf(fmaf(t, 1.0f / kD, eps)); });
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const float x0 = bf16_lo(w_lo[h]), x1 = bf16_hi(w_lo[h]);
                const float x2 = bf16_lo(w_hi[h]), x3 = bf16_hi(w_hi[h]);
                float o0, o1, o2, o3;
                ffma2(o0, o1, x0, x1, A0, A1, 0.f, 0.f);
                ffma2(o0, o1, x2, x3, nB0, nB1, o0, o1);
                ffma2(o0, o1, o0, o1, ss[h], ss[h], 0.f, 0.f);
                ffma2(o2, o3, x2, x3, A2, A3, 0.f, 0.f);
                ffma2(o2, o3, x0, x1, B2, B3, o2, o3);
                ffma2(o2, o3, o2, o3, ss[h], ss[h], 0.f, 0.f);
                row[h * (kD / 2) + lane] = pack_bf16x2(o0, o1);
                row[h * (kD / 2) + 32 + lane] = pack_bf16x2(o2, o3);
            }
        }
    }
}

}  // namespace

int qkv_tile_cols(int total_tokens) { return total_tokens <= 2 * kBM ? 64 : kPairBN; }
int qkv_weight_box_rows() { return kRunCols; }
int qkv_tile_rows_loaded(int total_tokens) { return total_tokens <= 32 ? 32 : kBM; }

cudaError_t launch_qkv(const QkvArgs &a, const CUtensorMap &x_map, const CUtensorMap &w_map, int num_sms,
                       cudaStream_t stream) {
    if (a.total_tokens == 0) return cudaSuccess;
    if (qkv_tile_rows_loaded(a.total_tokens) == 32) return launch_qkv_bn<64, 32>(a, x_map, w_map, num_sms, stream);
    if (a.total_tokens <= 2 * kBM) return launch_qkv_bn<64, 128>(a, x_map, w_map, num_sms, stream);
    return launch_qkv_pair(a, x_map, w_map, num_sms, stream);
}

cudaError_t launch_qk_norm(const QkvArgs &a, int num_sms, cudaStream_t stream) {
    if (a.total_tokens == 0) return cudaSuccess;
    const long long resident = (long long)num_sms * kNormCtasPerSm * (kNormThreads / 32);   // warps in one wave
    // many tokens: a warp per token (lookup and angles once); few: a warp per group of 8 heads
    const int groups_per_warp = (long long)a.total_tokens * kNormGroups > 2 * resident ? kNormGroups : 1;
    const long long work = (long long)a.total_tokens * ((kNormGroups + groups_per_warp - 1) / groups_per_warp);
    const long long need = (work + kNormThreads / 32 - 1) / (kNormThreads / 32);
    const long long ctas = (long long)num_sms * kNormCtasPerSm;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(need < ctas ? need : ctas));
    cfg.blockDim = dim3(kNormThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, qk_norm_kernel, a, groups_per_warp);
}

}  // namespace pa
