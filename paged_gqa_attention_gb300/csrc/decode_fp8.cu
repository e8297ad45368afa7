// decode_fp8.cu -- batched single-token GQA attention over the 8-bit KV cache.
//
// Page "从零搭建AI工程能力：手写KV Cache与动态批处理实战" §3.2: an 8-bit KV cache halves
// its memory.  Here a K or V row (one token, one KV head, 128 values) is 128 E4M3 codes
// plus one fp32 scale (the row means code * scale), so a decode step reads 264 bytes per
// token and KV head instead of 512.  The attention itself is that of decode.cu (page
// "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎，C++/CUDA 实现性能追平 98%" §4.4.2: the four query
// heads of a group share every KV read; split-K over the context with a log-sum-exp
// merge), with these differences:
//   * a stage is 128 tokens of K codes and V codes (16 KiB each, TMA, 128-byte swizzle)
//     and their 128 + 128 scales (512-byte bulk copies), consumed by 8 warps of 16 tokens;
//     three stages, two CTAs per SM.  A consumer warp's work per stage is one dependent
//     chain (S, softmax, PV) of about 0.8 us whatever the data type, so a stage of half-
//     size rows needs twice the tokens to move the bytes a bf16 stage moves;
//   * the tensor-core products run in f16 (the GPU converts E4M3 pairs to f16 pairs
//     exactly): ldmatrix on the code bytes gives each lane four consecutive codes of a
//     row, which become the A fragments of two k16 steps once Q is loaded in the
//     matching order of dimensions (dims 4t..4t+3 of a 16-dim step for lane column t);
//   * S is scaled per token by the K row's scale in fp32;
//   * for O^T += V^T P^T the transposed ldmatrix gives a lane the codes of two tokens for
//     two dimensions; one byte permute pairs them by dimension, so accumulator row r of
//     a 16-dim tile holds dimension 2r (r < 8) or 2(r-8)+1;
//   * fused append (k_new / v_new given): the warp whose 16 rows hold each sequence's new
//     token quantises the token's K and V rows of its KV head (kv_append_fp8's rule),
//     writes codes and scales to the cache and patches them into the landed stage;
//   * the V scale enters through P: each warp keeps a running reference sigma (the
//     largest V scale it has seen), accumulates P * (s_v / sigma) in f16 and rescales
//     its accumulator when sigma grows, as the online softmax does for its maximum; the
//     warp merge multiplies by sigma back.
#include <atomic>

#include "common.cuh"
#include "launch.h"

namespace pa {
namespace {

constexpr int kTile = kDecodeFp8TileTokens;   // 128 tokens per stage (half a cache block)
constexpr int kStages = 3;
constexpr int kCtasPerSm = 2;
constexpr int kConsumerWarps = kTile / 16;    // 8
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kCodeBytes = kTile * kD;        // 128 tokens x 128 codes = 16 KiB
constexpr int kScaleBytes = kTile * 4;        // 512 B
constexpr uint32_t kStageTx = 2 * kCodeBytes + 2 * kScaleBytes;
constexpr float kLn2 = 0.693147180559945309f;

struct MergeArrays {                          // the warps' partial results, after the stages
    float o[kConsumerWarps][kGroup][kD];
    float m[kConsumerWarps][kGroup];
    float l[kConsumerWarps][kGroup];
    float sigma[kConsumerWarps];
};

struct DecodeFp8Smem {
    union {
        uint8_t codes[kStages][2][kCodeBytes];  // [stage][K, V], each 1 KiB aligned
        MergeArrays mg;                         // reused once every stage is consumed
    };
    float scales[kStages][2][kTile];          // [stage][K, V]
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int last_cta;
    int poison;
};

constexpr size_t kSmemBytes = sizeof(DecodeFp8Smem) + 1024;

__device__ __forceinline__ void store_out4(__nv_bfloat16 *dst, const float (&v)[4], float inv) {
    uint2 w;
    w.x = pack_bf16x2(v[0] * inv, v[1] * inv);
    w.y = pack_bf16x2(v[2] * inv, v[3] * inv);
    *reinterpret_cast<uint2 *>(dst) = w;
}

// Transposed-ldmatrix register of V codes: bytes {tok 2t: dim 2g, 2g+1; tok 2t+1: dim 2g,
// 2g+1} -> f16 pairs by dimension: lo = dim 2g (tokens 2t, 2t+1), hi = dim 2g+1.
__device__ __forceinline__ void v_pairs(uint32_t r, uint32_t &lo, uint32_t &hi) {
    e4m3x4_to_f16x2x2(__byte_perm(r, 0u, 0x3120), lo, hi);
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
decode_fp8_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                  const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    DecodeFp8Smem &sm = *reinterpret_cast<DecodeFp8Smem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int pair = blockIdx.x;          // sequence * 8 + kv head
    const int b = pair / kHkv;
    const int g = pair % kHkv;
    // the highest splits start first (longest work first, as in decode.cu)
    const int split = (int)(gridDim.y - 1 - blockIdx.y);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int32_t *bt = a.block_table + (size_t)b * a.max_blocks_per_seq;
    int blk0 = 0;
    if (warp == kConsumerWarps && lane == 0) {
        tma_prefetch_map(&k_map);
        tma_prefetch_map(&v_map);
        blk0 = __ldg(bt + (split * a.split_tokens) / kBlock);   // < max_blocks_per_seq
    }
    const int seq_len = __ldg(a.seq_lens + b);
    if (seq_len < 1 || seq_len > a.max_blocks_per_seq * kBlock) {
        if (split == 0 && g == 0 && threadIdx.x == 0) record_error(a.err, kErrDevice | kErrBadSeqLen);
        return;
    }
    const int t_begin = split * a.split_tokens;
    if (t_begin >= seq_len) return;
    const int t_end = min(t_begin + a.split_tokens, seq_len);
    const int nsplit_b = (seq_len + a.split_tokens - 1) / a.split_tokens;
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
        if (lane == 0) {
            // the cache may be written by the kernel just before this one on the stream
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
                    record_error(a.err, kErrDevice | kErrBadBlock);
                    sm.poison = 1;
                    blk = 0;
                }
                const int off = tok % kBlock;
                const uint32_t bar = smem_u32(&sm.full[st]);
                const size_t srow = ((size_t)blk * kHkv + g) * kBlock + off;   // 64 scales, 256 B aligned
                mbar_arrive_expect_tx(bar, kStageTx);
                tma_load_4d(smem_u32(sm.codes[st][0]), &k_map, bar, 0, g, off, blk);
                tma_load_4d(smem_u32(sm.codes[st][1]), &v_map, bar, 0, g, off, blk);
                bulk_load(smem_u32(sm.scales[st][0]), a.k_scale + srow, kScaleBytes, bar);
                bulk_load(smem_u32(sm.scales[st][1]), a.v_scale + srow, kScaleBytes, bar);
                issued = i + 1;
            }
            for (int i = max(0, issued - kStages); i < issued; ++i)
                mbar_wait(smem_u32(&sm.full[i % kStages]), (i / kStages) & 1);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int w = warp;
    const int gq = lane >> 2;   // fragment row group
    const int tq = lane & 3;    // fragment column pair
    const int mi = lane >> 3;   // ldmatrix: which 8x8 matrix this lane addresses
    const int ri = lane & 7;    // ldmatrix: row within it

    // q may come from the kernel just before this one on the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // Q^T as the B operand of S^T = K Q^T, f16: k16 step s holds dims 16s+4tq .. 16s+4tq+3
    // of head gq (the order the code fragments arrive in); heads 4..7 are zero.
    uint32_t qb[8][2];
    {
        const uint2 *qrow = reinterpret_cast<const uint2 *>(
            static_cast<const __nv_bfloat16 *>(a.q) + ((size_t)b * kHq + g * kGroup + (gq & 3)) * kD);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint2 v = gq < kGroup ? __ldg(qrow + ks * 4 + tq) : make_uint2(0u, 0u);
            qb[ks][0] = bf16x2_to_f16x2(v.x);
            qb[ks][1] = bf16x2_to_f16x2(v.y);
        }
    }

    float m0 = -INFINITY, m1 = -INFINITY;   // running max (log2 units) of heads 2tq, 2tq+1
    float l0 = 0.f, l1 = 0.f;               // this thread's share of the running sums
    float sigma = 0.f;                      // reference V scale of the accumulator
    float inv_sigma = 0.f;                  // its reciprocal
    float acc[8][4];                        // O^T tiles, in units of sigma
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;

    const int row = w * 16 + ri + ((mi & 1) << 3);   // token row addressed by this lane

    // Fused append: the CTA whose range ends the context owns the new token at position
    // seq_len - 1; the warp whose rows hold it quantises the token's K (lanes 0-15) and V
    // (lanes 16-31) row of this KV head, 8 values a lane, stores codes and scale into the
    // cache and patches them over the stale row of the landed stage before using it.
    const int p_new = seq_len - 1;
    const int i_new = (a.k_new && t_end == seq_len) ? (p_new - t_begin) / kTile : -1;
    const int r_new = (p_new - t_begin) % kTile;        // row within that stage
    const bool new_here = i_new >= 0 && (r_new >> 4) == w;
    uint2 new_codes = make_uint2(0u, 0u);
    float new_scale = 0.f;
    if (new_here) {
        const int kv = lane >> 4, chunk = lane & 15;
        const uint4 src = __ldg(reinterpret_cast<const uint4 *>(
            static_cast<const char *>(kv ? a.v_new : a.k_new) + ((size_t)b * kHkv + g) * kRowBytes) + chunk);
        const uint32_t wv[4] = {src.x, src.y, src.z, src.w};
        float x[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[2 * e] = bf16_lo(wv[e]);
            x[2 * e + 1] = bf16_hi(wv[e]);
        }
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        new_scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
        new_codes.x = f32x2_to_e4m3x2(__fdiv_rn(x[0], new_scale), __fdiv_rn(x[1], new_scale)) |
                      f32x2_to_e4m3x2(__fdiv_rn(x[2], new_scale), __fdiv_rn(x[3], new_scale)) << 16;
        new_codes.y = f32x2_to_e4m3x2(__fdiv_rn(x[4], new_scale), __fdiv_rn(x[5], new_scale)) |
                      f32x2_to_e4m3x2(__fdiv_rn(x[6], new_scale), __fdiv_rn(x[7], new_scale)) << 16;
        const int blk = __ldg(bt + p_new / kBlock);
        if (blk >= 0 && blk < a.num_blocks) {
            const int slot = p_new % kBlock;
            uint8_t *dst = static_cast<uint8_t *>(kv ? a.v_pool_w : a.k_pool_w) +
                           (((size_t)blk * kBlock + slot) * kHkv + g) * kD + chunk * 8;
            *reinterpret_cast<uint2 *>(dst) = new_codes;
            if (chunk == 0)
                const_cast<float *>(kv ? a.v_scale : a.k_scale)[((size_t)blk * kHkv + g) * kBlock + slot] = new_scale;
        }   // a bad block id is reported by the producer and poisons the result
    }

    for (int i = 0; i < n_tiles; ++i) {
        const int st = i % kStages;
        if (!mbar_wait(smem_u32(&sm.full[st]), (i / kStages) & 1)) {
            if (lane == 0) record_error(a.err, kErrTimeout);
            break;
        }
        if (new_here && i == i_new) {
            // the new token's row: lane (kv, chunk) holds codes of dims 8 chunk .. 8 chunk + 7,
            // half (chunk % 2) of swizzled 16-byte chunk chunk / 2 of row r_new
            const int kv = lane >> 4, chunk = lane & 15;
            *reinterpret_cast<uint2 *>(sm.codes[st][kv] + sw128(r_new, chunk >> 1) + (chunk & 1) * 8) = new_codes;
            if (chunk == 0) sm.scales[st][kv][r_new] = new_scale;
            fence_proxy_async_smem();   // generic writes before the stage is refilled by TMA
            __syncwarp();
        }
        const int my_valid = min(max(t_end - (t_begin + i * kTile) - w * 16, 0), 16);
        if (my_valid > 0) {
            const uint32_t kc = smem_u32(sm.codes[st][0]);
            const uint32_t vc = smem_u32(sm.codes[st][1]);
            const float *ksc = sm.scales[st][0] + w * 16;
            const float *vsc = sm.scales[st][1] + w * 16;

            // S^T[16 tokens x 8 heads] = K[16 x 128] . Q^T, 32 dims per ldmatrix, as two
            // independent accumulations (even / odd k16 steps) to halve the dependent chain
            float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t r[4], af[4], bf[4];
                ldsm_x4(r, kc + sw128(row, 2 * j + (mi >> 1)));
                e4m3x4_to_f16x2x2(r[0], af[0], af[2]);   // token gq
                e4m3x4_to_f16x2x2(r[1], af[1], af[3]);   // token gq + 8
                mma_16816_f16(s, af, qb[2 * j][0], qb[2 * j][1]);
                e4m3x4_to_f16x2x2(r[2], bf[0], bf[2]);
                e4m3x4_to_f16x2x2(r[3], bf[1], bf[3]);
                mma_16816_f16(s2, bf, qb[2 * j + 1][0], qb[2 * j + 1][1]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) s[e] += s2[e];
            // s[0]: (token gq, head 2tq)   s[1]: (token gq, head 2tq+1)
            // s[2]: (token gq+8, head 2tq) s[3]: (token gq+8, head 2tq+1)
            const bool v_lo_ok = gq < my_valid;
            const bool v_hi_ok = gq + 8 < my_valid;
            float x0, x1, x2, x3;
            if (tq < 2) {
                const float k_lo = v_lo_ok ? ksc[gq] * a.scale_log2 : 0.f;
                const float k_hi = v_hi_ok ? ksc[gq + 8] * a.scale_log2 : 0.f;
                x0 = v_lo_ok ? s[0] * k_lo : -INFINITY;
                x1 = v_lo_ok ? s[1] * k_lo : -INFINITY;
                x2 = v_hi_ok ? s[2] * k_hi : -INFINITY;
                x3 = v_hi_ok ? s[3] * k_hi : -INFINITY;
            } else {  // padding heads 4..7: finite dummies, results discarded
                x0 = x1 = x2 = x3 = 0.f;
            }
            // lazy rescaling: the running max moves only when the tile's max exceeds it by
            // more than 2^8 (weights stay <= 2^8, far inside f16), so most tiles rescale
            // nothing; one vote finds those tiles, and only they reduce the maxima over the
            // warp (six dependent shuffles off the common path)
            float alpha0 = 1.f, alpha1 = 1.f;
            if (__any_sync(0xffffffffu, fmaxf(x0, x2) > m0 + 8.f || fmaxf(x1, x3) > m1 + 8.f)) {
                float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
                }
                const bool up0 = mx0 > m0 + 8.f, up1 = mx1 > m1 + 8.f;   // also when m == -inf
                const float mn0 = up0 ? mx0 : m0, mn1 = up1 ? mx1 : m1;
                alpha0 = up0 ? fast_exp2(m0 - mn0) : 1.f;
                alpha1 = up1 ? fast_exp2(m1 - mn1) : 1.f;
                m0 = mn0;
                m1 = mn1;
            }
            const float p0 = fast_exp2(x0 - m0), p1 = fast_exp2(x1 - m1);
            const float p2 = fast_exp2(x2 - m0), p3 = fast_exp2(x3 - m1);
            l0 = l0 * alpha0 + p0 + p2;
            l1 = l1 * alpha1 + p1 + p3;

            // V scales of this warp's tokens (0 past the context end: scale slots there
            // may hold anything) and their maximum
            const float sv_lo = v_lo_ok ? vsc[gq] : 0.f;
            const float sv_hi = v_hi_ok ? vsc[gq + 8] : 0.f;
            // the accumulator's reference V scale grows with the largest scale seen; its
            // reciprocal is recomputed only then (an approximate reciprocal: the factor it
            // introduces is undone exactly by the same values in grow and the final sigma)
            // (floored at 2^-100 so that the reciprocal stays finite: a V row whose scale is
            // below it contributes less than the output's bf16 resolution near zero)
            // (one vote finds the stages that raise it; only they reduce over the warp)
            float grow = 1.f;
            if (__any_sync(0xffffffffu, fmaxf(fmaxf(sv_lo, sv_hi), 0x1p-100f) > sigma)) {
                float svm = fmaxf(sv_lo, sv_hi);
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, o));
                const float svr = fmaxf(svm, 0x1p-100f);
                if (svr > sigma) {
                    inv_sigma = fast_rcp(svr);
                    grow = sigma * inv_sigma;              // 0 on the first tile (acc is 0)
                    sigma = svr;
                }
            }
            const float r_lo = sv_lo * inv_sigma, r_hi = sv_hi * inv_sigma;
            const uint32_t pp_lo = pack_f16x2(p0 * r_lo, p1 * r_lo);   // token gq:   heads 2tq, 2tq+1
            const uint32_t pp_hi = pack_f16x2(p2 * r_hi, p3 * r_hi);   // token gq+8: heads 2tq, 2tq+1
            const float f0 = alpha0 * grow, f1 = alpha1 * grow;
            if (__any_sync(0xffffffffu, f0 != 1.f || f1 != 1.f)) {
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    acc[mt][0] *= f0;
                    acc[mt][1] *= f1;
                    acc[mt][2] *= f0;
                    acc[mt][3] *= f1;
                }
            }
            // P^T as the B operand of O^T += V^T P^T: transpose the 8x8 16-bit blocks.
            const uint32_t pb0 = movmatrix_trans(pp_lo);
            const uint32_t pb1 = movmatrix_trans(pp_hi);
            // V codes of tokens past the context end are zeroed in the fragment.
            const uint32_t keep_lo = (2 * tq < my_valid ? 0x0000ffffu : 0u) |
                                     (2 * tq + 1 < my_valid ? 0xffff0000u : 0u);
            const uint32_t keep_hi = (2 * tq + 8 < my_valid ? 0x0000ffffu : 0u) |
                                     (2 * tq + 9 < my_valid ? 0xffff0000u : 0u);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // matrices: tokens 0-7 / 8-15 of the warp x dims 32j..32j+15 / 32j+16..32j+31
                uint32_t r[4], af[4], bf[4];
                ldsm_x4_trans(r, vc + sw128(row, 2 * j + (mi >> 1)));
                v_pairs(r[0], af[0], af[1]);   // rows gq (dim 2gq) and gq+8 (dim 2gq+1), tokens 2tq, 2tq+1
                v_pairs(r[1], af[2], af[3]);   // the same, tokens 2tq+8, 2tq+9
                af[0] &= keep_lo;
                af[1] &= keep_lo;
                af[2] &= keep_hi;
                af[3] &= keep_hi;
                mma_16816_f16(acc[2 * j], af, pb0, pb1);
                v_pairs(r[2], bf[0], bf[1]);
                v_pairs(r[3], bf[2], bf[3]);
                bf[0] &= keep_lo;
                bf[1] &= keep_lo;
                bf[2] &= keep_hi;
                bf[3] &= keep_hi;
                mma_16816_f16(acc[2 * j + 1], bf, pb0, pb1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.empty[st]));
    }

    // ------------------------------------------------------------ merge the warps
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    // the merge arrays overlay the stages: every consumer warp must be done with them
    named_barrier(1, kConsumerWarps * 32);
    if (tq < 2) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int d = mt * 16 + 2 * gq;      // accumulator rows gq, gq+8 = dims 2gq, 2gq+1
            sm.mg.o[w][2 * tq][d] = acc[mt][0];
            sm.mg.o[w][2 * tq + 1][d] = acc[mt][1];
            sm.mg.o[w][2 * tq][d + 1] = acc[mt][2];
            sm.mg.o[w][2 * tq + 1][d + 1] = acc[mt][3];
        }
        if (gq == 0) {
            sm.mg.m[w][2 * tq] = m0;
            sm.mg.m[w][2 * tq + 1] = m1;
            sm.mg.l[w][2 * tq] = l0;
            sm.mg.l[w][2 * tq + 1] = l1;
        }
    }
    if (lane == 0) sm.mg.sigma[w] = sigma;
    named_barrier(1, kConsumerWarps * 32);
    const bool bad = *reinterpret_cast<volatile int *>(&sm.poison) != 0;

    // the first 128 consumer threads merge (4 heads x 32 threads x 4 dims)
    const int c = threadIdx.x;
    if (c >= kGroup * 32) {
        // the others only take part in the partials' barriers below
        if (nsplit_b > 1) {
            named_barrier(2, kConsumerWarps * 32);
            named_barrier(2, kConsumerWarps * 32);
        }
        return;
    }
    const int h = c >> 5;               // query head within the group
    const int d0 = (c & 31) * 4;        // 4 dims per thread
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kConsumerWarps; ++ww) M = fmaxf(M, sm.mg.m[ww][h]);
    float L = 0.f, o4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ww = 0; ww < kConsumerWarps; ++ww) {
        const float e = fast_exp2(sm.mg.m[ww][h] - M);
        L += sm.mg.l[ww][h] * e;
        const float eo = e * sm.mg.sigma[ww];
#pragma unroll
        for (int k = 0; k < 4; ++k) o4[k] += sm.mg.o[ww][h][d0 + k] * eo;
    }
    if (bad) {
        M = L = __int_as_float(0x7fc00000);
#pragma unroll
        for (int k = 0; k < 4; ++k) o4[k] = __int_as_float(0x7fc00000);
    }
    const int qh = g * kGroup + h;      // query head
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + ((size_t)b * kHq + qh) * kD + d0;

    if (nsplit_b == 1) {
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
    __threadfence();
    named_barrier(2, kConsumerWarps * 32);
    if (c == 0) {
        const int prev = atomicAdd(a.counters + pair, 1);
        sm.last_cta = (prev == nsplit_b - 1);
    }
    named_barrier(2, kConsumerWarps * 32);
    if (!sm.last_cta) return;

    // The last CTA of this (sequence, KV head) merges every split by log-sum-exp.
    __threadfence();
    if (c == 0) a.counters[pair] = 0;   // ready for the next call
    const size_t e0 = (size_t)pair * a.nsplit;
    float GM = -INFINITY;
    for (int k = 0; k < nsplit_b; ++k) GM = fmaxf(GM, __ldcg(a.part_ml + ((e0 + k) * kGroup + h) * 2));
    float GL = 0.f, go[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < nsplit_b; ++k) {
        const float mk = __ldcg(a.part_ml + ((e0 + k) * kGroup + h) * 2);
        const float lk = __ldcg(a.part_ml + ((e0 + k) * kGroup + h) * 2 + 1);
        const float e = fast_exp2(mk - GM);
        const float4 ok = __ldcg(reinterpret_cast<const float4 *>(a.part_o + ((e0 + k) * kGroup + h) * kD + d0));
        GL += lk * e;
        go[0] += ok.x * e;
        go[1] += ok.y * e;
        go[2] += ok.z * e;
        go[3] += ok.w * e;
    }
    store_out4(out, go, 1.f / GL);
    if (a.lse && (c & 31) == 0) a.lse[(size_t)b * kHq + qh] = (GM + __log2f(GL)) * kLn2;
}

}  // namespace

cudaError_t launch_decode_fp8(const DecodeArgs &a, const CUtensorMap &k_map, const CUtensorMap &v_map,
                              cudaStream_t stream) {
    if (a.batch == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<bool> configured[64] = {};
    if (dev < 0 || dev >= 64 || !configured[dev].load()) {
        e = cudaFuncSetAttribute(decode_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev].store(true);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.batch * kHkv, a.nsplit);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_fp8_kernel, k_map, v_map, a);
}

}  // namespace pa
