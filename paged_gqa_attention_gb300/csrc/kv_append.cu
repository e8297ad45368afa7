// kv_append.cu -- scatter of new K/V rows into their cache blocks.
//
// Page "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎，C++/CUDA 实现性能追平 98%" §4.3.1
// (KVBlockManager::append): tokens fill a sequence's last 256-token block in order,
// a new block is taken when it is full.  Here the host has already extended the
// block table; the bf16 kernel only moves bytes.  New token i of sequence s lands at
// absolute position p = seq_lens[s] - q_len + i, slot p % 256 of block
// block_table[s][p / 256].  In the pool layout [block][slot][kv_head][dim] one
// token's K (or V) for all 8 KV heads is 2 KiB contiguous, so each copy is one
// contiguous 2 KiB move: one warp per (token, K|V), 16-byte vector accesses.
//
// The 8-bit cache variant (k_scale set) quantises instead of copying: each (token, KV
// head) row of 128 values gets scale = amax / 448 (fp32, 1 for an all-zero row) and codes
// E4M3(x / scale) (fp32 division, round to nearest even, saturating at 448), one half-
// warp per row; the codes keep the pool layout (128 bytes per row) and the scale goes to
// [block][head][slot].  Page "从零搭建AI工程能力：手写KV Cache与动态批处理实战" §3.2: an 8-bit
// KV cache halves its memory.
//
// The kernel is a chain of dependent loads (which sequence owns the token, its
// length, its block id, then the data), so its time is latency: the owner is first
// guessed in proportion (exact for one token per sequence and for one sequence) and
// only on a miss found by a warp-wide 32-way search.  It lets the next kernel on the
// stream start its own prologue early (programmatic dependent launch); that kernel
// waits for this one to finish before it reads the pools.
#include "common.cuh"
#include "launch.h"

namespace pa {
namespace {

constexpr int kWarps = 8;  // 4 tokens x {K, V} per CTA

// Largest s in [0, n) with cu[s] <= t (cu non-decreasing, cu[0] <= t): each round the
// 32 lanes probe 32 evenly spaced entries, narrowing the range 32-fold.
__device__ __forceinline__ int warp_find_sequence(const int32_t *cu, int n, int t, int lane) {
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) / 32;
        const int idx = lo + lane * step;
        const bool le = idx < hi && __ldg(cu + idx) <= t;
        const unsigned m = __ballot_sync(0xffffffffu, le);
        const int last = m ? 31 - __clz(m) : 0;
        lo = lo + last * step;
        hi = min(hi, lo + step);
    }
    return lo;
}

template <bool kFp8>
__global__ void __launch_bounds__(kWarps * 32) kv_append_kernel(AppendArgs a) {
    // The pools are this kernel's only output: a dependent kernel may launch now and
    // run its prologue; it waits for our completion before touching the pools.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (kWarps / 2) + (warp >> 1);
    const bool is_v = warp & 1;
    if (t >= a.total_tokens) return;
    // The row's 2 KiB does not depend on where it goes: its loads are issued first, so they
    // overlap the chain that finds the destination.  2 KiB = 128 x 16 B: four 16-byte vectors
    // per lane.
    const uint4 *src = reinterpret_cast<const uint4 *>(
        static_cast<const char *>(is_v ? a.v_new : a.k_new) + (size_t)t * kTokenBytes);
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = __ldg(src + lane + 32 * k);

    if (blockIdx.x == 0 && threadIdx.x == 0) {
        // cu_q_lens must start at 0 and end at total_tokens
        if (__ldg(a.cu_q_lens) != 0 || __ldg(a.cu_q_lens + a.num_seqs) != a.total_tokens)
            record_error(a.err, kErrDevice | kErrBadCuQ);
    }
    int s = (int)((long long)t * a.num_seqs / a.total_tokens);
    int q0 = __ldg(a.cu_q_lens + s);
    int q1 = __ldg(a.cu_q_lens + s + 1);
    int seq_len = __ldg(a.seq_lens + s);
    if (!(q0 <= t && t < q1)) {
        s = warp_find_sequence(a.cu_q_lens, a.num_seqs, t, lane);
        q0 = __ldg(a.cu_q_lens + s);
        q1 = __ldg(a.cu_q_lens + s + 1);
        seq_len = __ldg(a.seq_lens + s);
    }
    const int q_len = q1 - q0;
    const int i = t - q0;
    if (i < 0 || i >= q_len) {
        if (lane == 0 && !is_v) record_error(a.err, kErrDevice | kErrBadCuQ);
        return;
    }
    if (seq_len < q_len || seq_len > a.max_blocks_per_seq * kBlock) {
        if (lane == 0 && !is_v) record_error(a.err, kErrDevice | kErrBadSeqLen);
        return;
    }
    const int p = seq_len - q_len + i;
    const int blk = __ldg(a.block_table + (size_t)s * a.max_blocks_per_seq + p / kBlock);
    if (blk < 0 || blk >= a.num_blocks) {
        if (lane == 0 && !is_v) record_error(a.err, kErrDevice | kErrBadBlock);
        return;
    }
    const int slot = p % kBlock;
    if constexpr (!kFp8) {
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<char *>(is_v ? a.v_pool : a.k_pool) +
                                               ((size_t)blk * kBlock + slot) * kTokenBytes);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[lane + 32 * k] = v[k];
    } else {
        // vector k of lane l: KV head 2k + l/16, dims 8 (l%16) .. 8 (l%16) + 7
        uint8_t *codes = static_cast<uint8_t *>(is_v ? a.v_pool : a.k_pool) +
                         ((size_t)blk * kBlock + slot) * (kHkv * kD);
        float *scales = is_v ? a.v_scale : a.k_scale;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
            float x[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[2 * e] = bf16_lo(w[e]);
                x[2 * e + 1] = bf16_hi(w[e]);
            }
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
            uint2 c;
            c.x = f32x2_to_e4m3x2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale)) |
                  f32x2_to_e4m3x2(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale)) << 16;
            c.y = f32x2_to_e4m3x2(__fdiv_rn(x[4], scale), __fdiv_rn(x[5], scale)) |
                  f32x2_to_e4m3x2(__fdiv_rn(x[6], scale), __fdiv_rn(x[7], scale)) << 16;
            const int head = 2 * k + (lane >> 4), chunk = lane & 15;
            *reinterpret_cast<uint2 *>(codes + head * kD + chunk * 8) = c;
            if (chunk == 0) scales[((size_t)blk * kHkv + head) * kBlock + slot] = scale;
        }
    }
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs &a, cudaStream_t stream) {
    if (a.total_tokens == 0) return cudaSuccess;
    const int tokens_per_cta = kWarps / 2;
    const int grid = (a.total_tokens + tokens_per_cta - 1) / tokens_per_cta;
    if (a.k_scale)
        kv_append_kernel<true><<<grid, kWarps * 32, 0, stream>>>(a);
    else
        kv_append_kernel<false><<<grid, kWarps * 32, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace pa
