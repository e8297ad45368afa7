"""The 8-bit KV cache on the GPU against the oracle: the append (codes and scales bit-exact)
and the decode over the cache (within the bf16 output tolerance)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (assert_close, assert_lse_close, gpu, lib_ready, oracle_appended_pools, to_cpu,
                         workspace_for)
from paged_gqa_attention_gb300 import ops
from paged_gqa_attention_gb300 import workloads as wl

pytestmark = gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def oracle_cache(batch: wl.Batch, drop_last: int = 0):
    """The 8-bit cache holding the batch's context, quantised by the oracle (host arrays):
    positions 0 .. seq_len - 1 - drop_last of every sequence."""
    kp, vp = oracle_appended_pools(batch)            # bf16 context incl. the new tokens
    k_rows, v_rows, cu, lens = wl.context_rows(batch, torch.from_numpy(kp.view(np.int16)).view(torch.bfloat16),
                                               torch.from_numpy(vp.view(np.int16)).view(torch.bfloat16),
                                               drop_last=drop_last)
    kc, vc, ks, vs = ops.fp8_cache(batch.num_blocks, device="cpu")
    return oracle.kv_append_fp8(kc.numpy(), vc.numpy(), ks.numpy(), vs.numpy(), k_rows, v_rows,
                                to_cpu(batch.block_table), cu, lens)


def upload(cache):
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in cache]


def same_bits(gpu_t, host):
    g = to_cpu(gpu_t).contiguous()
    if g.dtype == torch.float32:
        return np.array_equal(g.view(torch.int32).numpy(), np.ascontiguousarray(host).view(np.int32))
    return np.array_equal(g.numpy(), host)


def scaled_rows(n, seed, device="cuda"):
    """bf16 rows whose magnitudes span many binades (per row and within a row), a zero row
    and values that fall into E4M3's subnormal range after scaling."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(n, 8, 128, generator=g, device=device)
    x = x * torch.exp2(torch.randint(-12, 13, (n, 8, 1), generator=g, device=device).float())
    x[:, :, :8] *= 2.0 ** -9                     # small elements: subnormal codes
    x[0, 3] = 0.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("lens,q_lens", [([300, 40, 513], [5, 40, 1]), ([1, 256, 257, 1000], [1, 1, 1, 1])])
def test_kv_append_fp8_is_bit_exact(lens, q_lens):
    b = wl.build_batch("fp8_append", 51, lens, q_lens, num_blocks=sum((l + 255) // 256 for l in lens) + 2,
                       device="cuda")
    kn, vn = scaled_rows(b.total_tokens, 52), scaled_rows(b.total_tokens, 53)
    kc, vc, ks, vs = ops.fp8_cache(b.num_blocks)
    ref = oracle.kv_append_fp8(to_cpu(kc).numpy(), to_cpu(vc).numpy(), to_cpu(ks).numpy(), to_cpu(vs).numpy(),
                               to_cpu(kn), to_cpu(vn), to_cpu(b.block_table), to_cpu(b.cu_q_lens),
                               to_cpu(b.seq_lens))
    ws = workspace_for(b)
    ops.kv_append_fp8(kc, vc, ks, vs, kn, vn, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    ops.check_error(ws)
    for got, want, name in zip((kc, vc, ks, vs), ref, ("k_codes", "v_codes", "k_scale", "v_scale")):
        assert same_bits(got, want), f"{name} differs from the oracle"


@pytest.mark.parametrize("lens", [[1, 63, 64, 65, 255, 256, 257, 1000], [4096, 3000, 17]])
def test_decode_fp8_matches_oracle(lens):
    b = wl.build_batch("fp8_decode", 54 + len(lens), lens, [1] * len(lens),
                       num_blocks=sum((l + 255) // 256 for l in lens) + 3, device="cuda")
    cache = oracle_cache(b)
    kc, vc, ks, vs = upload(cache)
    ws = workspace_for(b)
    lse = torch.empty(b.num_seqs, ops.NUM_Q_HEADS, dtype=torch.float32, device="cuda")
    out = ops.paged_attn_decode_fp8(b.q, kc, vc, ks, vs, b.block_table, b.seq_lens, ws, lse=lse)
    ops.check_error(ws)
    ref, ref_lse = oracle.attention_fp8(to_cpu(b.q), *cache, to_cpu(b.block_table), to_cpu(b.cu_q_lens),
                                        to_cpu(b.seq_lens), scale=wl.SCALE)
    assert_close(out, ref, f"fp8 decode {lens}")
    assert_lse_close(lse, ref_lse, f"fp8 decode {lens}")


@pytest.mark.parametrize("split_tokens", [1024, 0])
def test_decode_fp8_late_score_spike(split_tokens):
    """A key late in the context whose score exceeds everything before it by far more than
    the rescale threshold (2^8).  With 1024-token splits each spike lies in a later stage of a
    warp that has already accumulated earlier stages, so that warp must take the warp-wide
    maximum path and rescale its accumulator (the library's own split, with this few
    sequences, gives each CTA one stage)."""
    lens = [3000, 700, 1800]
    b = wl.build_batch("fp8_spike", 61, lens, [1] * len(lens), num_blocks=sum((l + 255) // 256 for l in lens) + 3,
                       device="cuda")
    for s_, pos in ((0, 2500), (1, 650), (2, 1300)):
        blk = int(b.block_table[s_, pos // 256])
        for g in range(ops.NUM_KV_HEADS):
            # aligned with the group's first query head, 8 times its length: a score ~ 8 |q|^2 / sqrt(128)
            b.k_pool[blk, pos % 256, g] = (8.0 * b.q[s_, 4 * g].float()).to(torch.bfloat16)
    cache = oracle_cache(b)
    kc, vc, ks, vs = upload(cache)
    ws = workspace_for(b)
    lse = torch.empty(b.num_seqs, ops.NUM_Q_HEADS, dtype=torch.float32, device="cuda")
    out = ops.paged_attn_decode_fp8(b.q, kc, vc, ks, vs, b.block_table, b.seq_lens, ws, lse=lse,
                                    split_tokens=split_tokens)
    ops.check_error(ws)
    ref, ref_lse = oracle.attention_fp8(to_cpu(b.q), *cache, to_cpu(b.block_table), to_cpu(b.cu_q_lens),
                                        to_cpu(b.seq_lens), scale=wl.SCALE)
    assert_close(out, ref, f"fp8 decode, late score spike (split {split_tokens})")
    assert_lse_close(lse, ref_lse, f"fp8 decode, late score spike (split {split_tokens})")


def test_decode_fp8_after_gpu_append_of_the_new_tokens():
    """The decode step over the 8-bit cache: the context before the new tokens quantised by
    the oracle, the new tokens appended by the GPU, then the GPU decode."""
    lens = [700, 129, 2048, 5]
    b = wl.build_batch("fp8_step", 58, lens, [1] * len(lens), num_blocks=sum((l + 255) // 256 for l in lens) + 2,
                       device="cuda")
    before = oracle_cache(b, drop_last=1)
    full = oracle_cache(b)
    kc, vc, ks, vs = upload(before)
    ws = workspace_for(b)
    ops.kv_append_fp8(kc, vc, ks, vs, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    out = ops.paged_attn_decode_fp8(b.q, kc, vc, ks, vs, b.block_table, b.seq_lens, ws)
    ops.check_error(ws)
    for got, want in zip((kc, vc, ks, vs), full):
        assert same_bits(got, want)
    ref, _ = oracle.attention_fp8(to_cpu(b.q), *full, to_cpu(b.block_table), to_cpu(b.cu_q_lens),
                                  to_cpu(b.seq_lens), scale=wl.SCALE)
    assert_close(out, ref, "fp8 step")


def test_decode_fp8_single_key_returns_its_row():
    b = wl.build_batch("fp8_one", 59, [1, 1], [1, 1], num_blocks=4, device="cuda")
    cache = oracle_cache(b)
    kc, vc, ks, vs = upload(cache)
    ws = workspace_for(b)
    out = ops.paged_attn_decode_fp8(b.q, kc, vc, ks, vs, b.block_table, b.seq_lens, ws)
    ops.check_error(ws)
    ref, _ = oracle.attention_fp8(to_cpu(b.q), *cache, to_cpu(b.block_table), to_cpu(b.cu_q_lens),
                                  to_cpu(b.seq_lens), scale=wl.SCALE)
    # one key: the output is its V row (code * scale), rounded to bf16 after an fp32 product:
    # within one bf16 step of the exact value
    got = to_cpu(out).double().numpy()
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-30)


def test_decode_fp8_full_size_batched():
    """The benchmark's 8-bit workload (batch 32, contexts U{128..4096}): the plain decode over the
    oracle's cache, and the benchmark's fused step (each new token appended, then the decode) on
    the cache without the new tokens; all 32 x 32 rows and their lse against the oracle, the
    appended codes and scales bit-exact."""
    b = wl.batched_decode(device="cuda")
    full = oracle_cache(b)
    ws = workspace_for(b)
    lse = torch.empty(b.num_seqs, ops.NUM_Q_HEADS, dtype=torch.float32, device="cuda")
    out = ops.paged_attn_decode_fp8(b.q, *upload(full), b.block_table, b.seq_lens, ws, lse=lse)
    ops.check_error(ws)
    ref, ref_lse = oracle.attention_fp8(to_cpu(b.q), *full, to_cpu(b.block_table), to_cpu(b.cu_q_lens),
                                        to_cpu(b.seq_lens), scale=wl.SCALE)
    assert_close(out, ref, "fp8 batched decode, full size")
    assert_lse_close(lse, ref_lse, "fp8 batched decode, full size")
    c1 = upload(oracle_cache(b, drop_last=1))
    lse_f = torch.empty_like(lse)
    out_f = ops.paged_attn_decode_append_fp8(b.q, b.k_new, b.v_new, *c1, b.block_table, b.seq_lens, ws, lse=lse_f)
    ops.check_error(ws)
    for got, want in zip(c1, full):
        assert same_bits(got, want)
    assert_close(out_f, ref, "fp8 fused append + decode, full size")
    assert_lse_close(lse_f, ref_lse, "fp8 fused append + decode, full size")


def test_decode_fp8_bad_block_is_reported():
    b = wl.build_batch("fp8_bad", 60, [600, 300], [1, 1], num_blocks=6, device="cuda")
    cache = oracle_cache(b)
    kc, vc, ks, vs = upload(cache)
    ws = workspace_for(b)
    ref, _ = oracle.attention_fp8(to_cpu(b.q), *cache, to_cpu(b.block_table), to_cpu(b.cu_q_lens),
                                  to_cpu(b.seq_lens), scale=wl.SCALE)
    bt = b.block_table.clone()
    bt[0, 1] = b.num_blocks + 5
    out = ops.paged_attn_decode_fp8(b.q, kc, vc, ks, vs, bt, b.seq_lens, ws)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.check_error(ws)
    assert e.value.status == 4
    assert torch.isnan(out[0].float()).any()
    assert_close(out[1], ref[1], "unaffected sequence")


@pytest.mark.parametrize("lens", [[700, 129, 2048, 5, 1, 128, 256, 257], [4096, 3000, 17]])
def test_fused_append_fp8_equals_the_two_calls(lens):
    b = wl.build_batch("fp8_fused", 61 + len(lens), lens, [1] * len(lens),
                       num_blocks=sum((l + 255) // 256 for l in lens) + 2, device="cuda")
    before = oracle_cache(b, drop_last=1)
    full = oracle_cache(b)
    ws = workspace_for(b)
    c2 = upload(before)
    ops.kv_append_fp8(*c2, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    lse2 = torch.empty(b.num_seqs, ops.NUM_Q_HEADS, dtype=torch.float32, device="cuda")
    out2 = ops.paged_attn_decode_fp8(b.q, *c2, b.block_table, b.seq_lens, ws, lse=lse2)
    c1 = upload(before)
    lse1 = torch.empty_like(lse2)
    out1 = ops.paged_attn_decode_append_fp8(b.q, b.k_new, b.v_new, *c1, b.block_table, b.seq_lens, ws, lse=lse1)
    ops.check_error(ws)
    for got, want in zip(c1, full):
        assert same_bits(got, want)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1.view(torch.int32), lse2.view(torch.int32))
    ref, ref_lse = oracle.attention_fp8(to_cpu(b.q), *full, to_cpu(b.block_table), to_cpu(b.cu_q_lens),
                                        to_cpu(b.seq_lens), scale=wl.SCALE)
    assert_close(out1, ref, f"fused fp8 step {lens}")
    assert_lse_close(lse1, ref_lse, f"fused fp8 step {lens}")
