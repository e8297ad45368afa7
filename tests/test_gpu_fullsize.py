"""Whole-tensor parity at full size on the three large workloads: every output element and
every lse of the GPU path, in the launch configuration the benchmark times, against the fp64
oracle on the same seeded inputs.

  causal_prefill        4096-token prompt: kv_append, then paged_attn_prefill, and the fused
                        paged_attn_prefill_append (131 072 rows each)
  mixed_batch           one append for 120 decode tokens + 8 chunks of 512, then the decode
                        of the 120 sequences and the prefill of the 8 chunks; and the two
                        fused calls (decode with append, prefill with append) (all rows)
  prefix_shared_decode  batch 128 x 32 768 with a 64-block shared prefix: the fused append +
                        decode step, the plain decode and the cascade decode (all rows of each)

The oracle appends on its own host copy of the pools, taken before the GPU's append, and
attends over that copy; nothing it consumes comes from the CUDA path.  The bars are those of
every other parity test: over the whole output tensor max-abs <= 1e-2 and relative RMS
<= 5e-3, lse within 2.5e-3.
"""
import numpy as np
import torch

from gpu_helpers import (assert_close, assert_lse_close, gpu, lib_ready, oracle_appended_pools,
                         oracle_attention, workspace_for)
from paged_gqa_attention_gb300 import ops
from paged_gqa_attention_gb300 import workloads as wl

pytestmark = gpu


def setup_module(module):
    lib_ready()


def _lse(n):
    return torch.full((n, 32), float("nan"), dtype=torch.float32, device="cuda")


def _pool_rows_equal(pool, ref, blocks):
    """The listed blocks of a device pool equal the oracle's (uint16 bit patterns)."""
    idx = torch.as_tensor(blocks, dtype=torch.long, device=pool.device)
    got = pool.index_select(0, idx).view(torch.int16).cpu().numpy().view(np.uint16)
    return np.array_equal(got, ref[np.asarray(blocks)])


def test_causal_prefill_whole_tensor():
    """kv_append then paged_attn_prefill, and the fused paged_attn_prefill_append (the step the
    benchmark times) on a copy of the same pools: all rows of both against one oracle result."""
    b = wl.causal_prefill(device="cuda")
    kp, vp = oracle_appended_pools(b)
    k0, v0 = b.k_pool.clone(), b.v_pool.clone()
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    lse = _lse(b.total_tokens)
    out = ops.paged_attn_prefill(b.q, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens,
                                 b.max_q_len, ws, lse=lse)
    ops.check_error(ws)
    blocks = b.block_table[0, :16].cpu().tolist()
    assert _pool_rows_equal(b.k_pool, kp, blocks) and _pool_rows_equal(b.v_pool, vp, blocks)
    ref, ref_lse = oracle_attention(b, kp, vp)
    assert_close(out, ref, "causal_prefill, all 4096 x 32 rows")
    assert_lse_close(lse, ref_lse, "causal_prefill, all 4096 x 32 rows")
    lse_f = _lse(b.total_tokens)
    out_f = ops.paged_attn_prefill_append(b.q, b.k_new, b.v_new, k0, v0, b.block_table, b.cu_q_lens, b.seq_lens,
                                          b.max_q_len, ws, lse=lse_f)
    ops.check_error(ws)
    assert _pool_rows_equal(k0, kp, blocks) and _pool_rows_equal(v0, vp, blocks)
    assert_close(out_f, ref, "causal_prefill fused append, all 4096 x 32 rows")
    assert_lse_close(lse_f, ref_lse, "causal_prefill fused append, all 4096 x 32 rows")
    # from position 0 both paths cut the keys into the same tiles: the same bits
    assert torch.equal(out.view(torch.int16), out_f.view(torch.int16))


def test_mixed_batch_whole_tensor():
    """The three calls (one append for all, decode, prefill) and the two fused calls (decode
    with its append, prefill with its append) on a copy of the same pools."""
    b = wl.mixed_batch(device="cuda")
    kp, vp = oracle_appended_pools(b)
    k0, v0 = b.k_pool.clone(), b.v_pool.clone()
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    n_dec = b.info["n_decode"]
    dec = b.select(slice(0, n_dec))
    pre = b.select(slice(n_dec, b.num_seqs))
    lse_d, lse_p = _lse(dec.total_tokens), _lse(pre.total_tokens)
    out_d = ops.paged_attn_decode(dec.q, dec.k_pool, dec.v_pool, dec.block_table, dec.seq_lens, ws, lse=lse_d)
    out_p = ops.paged_attn_prefill(pre.q, pre.k_pool, pre.v_pool, pre.block_table, pre.cu_q_lens,
                                   pre.seq_lens, pre.max_q_len, ws, lse=lse_p)
    ops.check_error(ws)
    ref_d, ref_lse_d = oracle_attention(dec, kp, vp)
    assert_close(out_d, ref_d, "mixed_batch decode part, all 120 x 32 rows")
    assert_lse_close(lse_d, ref_lse_d, "mixed_batch decode part, all 120 x 32 rows")
    ref_p, ref_lse_p = oracle_attention(pre, kp, vp)
    assert_close(out_p, ref_p, "mixed_batch prefill part, all 4096 x 32 rows")
    assert_lse_close(lse_p, ref_lse_p, "mixed_batch prefill part, all 4096 x 32 rows")
    lse_fd, lse_fp = _lse(dec.total_tokens), _lse(pre.total_tokens)
    out_fd = ops.paged_attn_decode_append(dec.q, dec.k_new, dec.v_new, k0, v0, dec.block_table, dec.seq_lens, ws,
                                          lse=lse_fd)
    out_fp = ops.paged_attn_prefill_append(pre.q, pre.k_new, pre.v_new, k0, v0, pre.block_table, pre.cu_q_lens,
                                           pre.seq_lens, pre.max_q_len, ws, lse=lse_fp)
    ops.check_error(ws)
    assert torch.equal(k0.view(torch.int16), b.k_pool.view(torch.int16))
    assert torch.equal(v0.view(torch.int16), b.v_pool.view(torch.int16))
    assert_close(out_fd, ref_d, "mixed_batch fused decode part, all 120 x 32 rows")
    assert_lse_close(lse_fd, ref_lse_d, "mixed_batch fused decode part, all 120 x 32 rows")
    assert_close(out_fp, ref_p, "mixed_batch fused prefill part, all 4096 x 32 rows")
    assert_lse_close(lse_fp, ref_lse_p, "mixed_batch fused prefill part, all 4096 x 32 rows")


def test_prefix_shared_decode_whole_tensor():
    """The fused decode step (append + decode, one kernel), then the plain decode and the
    cascade over the appended cache: all 128 x 32 rows of each against one oracle result."""
    b = wl.prefix_shared_decode(device="cuda")
    kp, vp = oracle_appended_pools(b)
    ref, ref_lse = oracle_attention(b, kp, vp)
    ws = workspace_for(b)
    lse_f = _lse(b.num_seqs)
    out_f = ops.paged_attn_decode_append(b.q, b.k_new, b.v_new, b.k_pool, b.v_pool, b.block_table,
                                         b.seq_lens, ws, lse=lse_f)
    ops.check_error(ws)
    # the new token of every sequence sits in the last slot of its last (private) block
    last = b.block_table[:, 127].cpu().tolist()
    assert _pool_rows_equal(b.k_pool, kp, last) and _pool_rows_equal(b.v_pool, vp, last)
    assert_close(out_f, ref, "prefix_shared fused append + decode, all 128 x 32 rows")
    assert_lse_close(lse_f, ref_lse, "prefix_shared fused append + decode, all 128 x 32 rows")

    lse_p = _lse(b.num_seqs)
    out_p = ops.paged_attn_decode(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, ws, lse=lse_p)
    ops.check_error(ws)
    assert_close(out_p, ref, "prefix_shared plain decode, all 128 x 32 rows")
    assert_lse_close(lse_p, ref_lse, "prefix_shared plain decode, all 128 x 32 rows")

    shared = b.info["shared_blocks"]
    cws = ops.make_cascade_workspace(b.num_seqs, b.max_blocks_per_seq, shared)
    lse_c = _lse(b.num_seqs)
    out_c = ops.paged_attn_decode_cascade(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, shared, cws,
                                          lse=lse_c)
    ops.check_error(cws)
    assert_close(out_c, ref, "prefix_shared cascade decode, all 128 x 32 rows")
    assert_lse_close(lse_c, ref_lse, "prefix_shared cascade decode, all 128 x 32 rows")
