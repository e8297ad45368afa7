// kv_append.cu -- scatter of new K/V rows into their cache blocks.
//
// Page "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎，C++/CUDA 实现性能追平 98%" §4.3.1
// (KVBlockManager::append): tokens fill a sequence's last 256-token block in order,
// a new block is taken when it is full.  Here the host has already extended the
// block table; the kernel only moves bytes.  New token i of sequence s lands at
// absolute position p = seq_lens[s] - q_len + i, slot p % 256 of block
// block_table[s][p / 256].  In the pool layout [block][slot][kv_head][dim] one
// token's K (or V) for all 8 KV heads is 2 KiB contiguous, so each copy is one
// contiguous 2 KiB move: one warp per (token, K|V), 16-byte vector accesses.
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

__global__ void __launch_bounds__(kWarps * 32) kv_append_kernel(AppendArgs a) {
    // The pools are this kernel's only output: a dependent kernel may launch now and
    // run its prologue; it waits for our completion before touching the pools.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (kWarps / 2) + (warp >> 1);
    const bool is_v = warp & 1;
    if (t >= a.total_tokens) return;

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
    const uint4 *src = reinterpret_cast<const uint4 *>(
        static_cast<const char *>(is_v ? a.v_new : a.k_new) + (size_t)t * kTokenBytes);
    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<char *>(is_v ? a.v_pool : a.k_pool) +
                                           ((size_t)blk * kBlock + (p % kBlock)) * kTokenBytes);
    // 2 KiB = 128 x 16 B: four 16-byte vectors per lane, all loads issued first
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = __ldg(src + lane + 32 * k);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[lane + 32 * k] = v[k];
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs &a, cudaStream_t stream) {
    if (a.total_tokens == 0) return cudaSuccess;
    const int tokens_per_cta = kWarps / 2;
    const int grid = (a.total_tokens + tokens_per_cta - 1) / tokens_per_cta;
    kv_append_kernel<<<grid, kWarps * 32, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace pa
