"""Decode parity: paged_attn_decode (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

from gpu_helpers import (assert_close, assert_lse_close, gpu, lib_ready, oracle_appended_pools,
                         oracle_attention, workspace_for)
from paged_gqa_attention_gb300 import ops
from paged_gqa_attention_gb300 import workloads as wl

pytestmark = gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def run_decode(batch, ws=None, split_tokens=0, with_lse=True):
    ws = workspace_for(batch) if ws is None else ws
    lse = torch.empty(batch.num_seqs, 32, dtype=torch.float32, device="cuda") if with_lse else None
    out = ops.paged_attn_decode(batch.q, batch.k_pool, batch.v_pool, batch.block_table,
                                batch.seq_lens, ws, lse=lse, split_tokens=split_tokens)
    ops.check_error(ws)
    return out, lse


def decode_batch(lens, seed=0, num_blocks=None, maxb=None):
    """Pre-filled context (every position present) and one query per sequence."""
    need = sum((l + 255) // 256 for l in lens)
    b = wl.build_batch("decode_case", seed, lens, [0] * len(lens), num_blocks=num_blocks or need + 3,
                       device="cuda", max_blocks_per_seq=maxb)
    return _with_queries(b, seed)


def _with_queries(b, seed):
    """Give a q_len-0 batch one query per sequence (its context already holds every key)."""
    g = torch.Generator(device="cuda").manual_seed(seed + 77)
    n = b.num_seqs
    b.q = torch.randn(n, 32, 128, generator=g, device="cuda").to(torch.bfloat16)
    b.cu_q_lens = torch.arange(n + 1, dtype=torch.int32, device="cuda")
    b.q_lens_host = [1] * n
    b.max_q_len = 1
    return b


def test_single_sequence_512():
    b = wl.single_decode(device="cuda")
    kp, vp = oracle_appended_pools(b)
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    out, lse = run_decode(b, ws)
    ref, ref_lse = oracle_attention(b, kp, vp)
    assert_close(out, ref, "single_decode")
    assert_lse_close(lse, ref_lse, "single_decode")


def test_batched_decode_full_size():
    b = wl.batched_decode(device="cuda")
    kp, vp = oracle_appended_pools(b)
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    out, lse = run_decode(b, ws)
    ref, ref_lse = oracle_attention(b, kp, vp)
    assert_close(out, ref, "batched_decode")
    assert_lse_close(lse, ref_lse, "batched_decode")


@pytest.mark.parametrize("seed", [0, 2])
def test_batched_decode_other_seeds(seed):
    b = wl.batched_decode(device="cuda", seed=seed)
    kp, vp = oracle_appended_pools(b)
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    out, _ = run_decode(b, ws)
    ref, _ = oracle_attention(b, kp, vp)
    assert_close(out, ref, f"batched_decode seed {seed}")


BOUNDARY_LENS = [1, 2, 63, 64, 65, 127, 128, 255, 256, 257, 511, 512, 513, 1000, 4096]


def test_ragged_boundary_lengths():
    b = decode_batch(BOUNDARY_LENS, seed=5)
    out, lse = run_decode(b)
    ref, ref_lse = oracle_attention(b)
    assert_close(out, ref, "boundary lengths")
    assert_lse_close(lse, ref_lse, "boundary lengths")


@pytest.mark.parametrize("split", [64, 128, 256, 448, 1024, 4096])
def test_split_length_does_not_change_the_result(split):
    b = decode_batch([3000, 1, 700, 4096, 129], seed=6, maxb=16)
    ref, ref_lse = oracle_attention(b)
    out, lse = run_decode(b, split_tokens=split)
    assert_close(out, ref, f"split {split}")
    assert_lse_close(lse, ref_lse, f"split {split}")


def test_block_placement_is_bit_exact():
    b = decode_batch([900, 33, 2048], seed=7, num_blocks=40)
    out1, lse1 = run_decode(b)
    # move every block to another physical slot and rewrite the tables accordingly
    perm = torch.randperm(b.num_blocks, generator=torch.Generator().manual_seed(1)).to("cuda")
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(b.num_blocks, device="cuda")
    k2 = torch.empty_like(b.k_pool)
    v2 = torch.empty_like(b.v_pool)
    k2[perm] = b.k_pool
    v2[perm] = b.v_pool
    bt = b.block_table.clone()
    valid = bt >= 0
    bt[valid] = perm[bt[valid].long()].to(torch.int32)
    b.k_pool, b.v_pool, b.block_table = k2, v2, bt
    out2, lse2 = run_decode(b)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)


def test_single_key_returns_v_bit_exactly():
    b = decode_batch([1, 1, 1], seed=8)
    out, _ = run_decode(b)
    bt = b.block_table.cpu()
    for s in range(3):
        v = b.v_pool[int(bt[s, 0]), 0]                      # [8, 128]
        expect = v.repeat_interleave(4, dim=0)              # q-head h reads kv-head h // 4
        assert torch.equal(out[s].view(torch.int16), expect.view(torch.int16))


def test_identical_keys_give_mean_of_v():
    b = decode_batch([777], seed=9)
    bt = b.block_table.cpu()
    k0 = b.k_pool[int(bt[0, 0]), 0].clone()
    for j in range(4):
        blk = int(bt[0, j])
        n = min(256, 777 - 256 * j)
        b.k_pool[blk, :n] = k0
    out, _ = run_decode(b)
    vs = torch.cat([b.v_pool[int(bt[0, j]), :min(256, 777 - 256 * j)] for j in range(4)])
    mean = vs.double().mean(0).repeat_interleave(4, dim=0).cpu().numpy()
    assert_close(out[0], mean, "identical keys")


def test_append_then_decode_step_matches_oracle():
    b = wl.batched_decode(device="cuda", seed=11, batch=8, hi=1500, num_blocks=64)
    kp, vp = oracle_appended_pools(b)
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    out, _ = run_decode(b, ws)
    ref, _ = oracle_attention(b, kp, vp)
    assert_close(out, ref, "append + decode")


def test_repeated_calls_reuse_the_workspace():
    """The merge counters reset themselves: ten calls on one workspace agree bit for bit."""
    b = decode_batch([3000, 2500, 100], seed=12, maxb=16)
    ws = workspace_for(b)
    first, _ = run_decode(b, ws)
    for _ in range(9):
        again, _ = run_decode(b, ws)
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))


def test_empty_batch_is_a_no_op():
    b = decode_batch([10], seed=13)
    ws = workspace_for(b)
    out = ops.paged_attn_decode(b.q[:0], b.k_pool, b.v_pool, b.block_table[:0], b.seq_lens[:0], ws)
    ops.check_error(ws)
    assert out.shape[0] == 0


@pytest.mark.parametrize("seed", [1, 3])
def test_fused_append_decode_equals_the_two_calls(seed):
    """paged_attn_decode_append == kv_append followed by paged_attn_decode: identical pools
    (bit for bit) and identical outputs; and both match the oracle."""
    b = wl.batched_decode(device="cuda", seed=seed)
    kp, vp = oracle_appended_pools(b)
    k2, v2 = b.k_pool.clone(), b.v_pool.clone()
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    lse1 = torch.empty(b.num_seqs, 32, dtype=torch.float32, device="cuda")
    out1 = ops.paged_attn_decode(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, ws, lse=lse1)
    ops.check_error(ws)
    lse2 = torch.empty_like(lse1)
    out2 = ops.paged_attn_decode_append(b.q, b.k_new, b.v_new, k2, v2, b.block_table, b.seq_lens, ws,
                                        lse=lse2)
    ops.check_error(ws)
    assert torch.equal(k2.view(torch.int16), b.k_pool.view(torch.int16))
    assert torch.equal(v2.view(torch.int16), b.v_pool.view(torch.int16))
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1, lse2)
    ref, ref_lse = oracle_attention(b, kp, vp)
    assert_close(out2, ref, "fused append + decode")
    assert_lse_close(lse2, ref_lse, "fused append + decode")


def test_fused_append_decode_boundary_lengths_and_splits():
    lens = [1, 2, 64, 65, 256, 257, 1000]
    b = wl.build_batch("fused_edges", 31, lens, [1] * len(lens), num_blocks=16, device="cuda")
    kp, vp = oracle_appended_pools(b)
    ws = workspace_for(b)
    ref, _ = oracle_attention(b, kp, vp)
    for split in (0, 64, 128):
        k2, v2 = b.k_pool.clone(), b.v_pool.clone()
        if split:
            ops.kv_append(k2, v2, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
            out = ops.paged_attn_decode(b.q, k2, v2, b.block_table, b.seq_lens, ws, split_tokens=split)
        else:
            out = ops.paged_attn_decode_append(b.q, b.k_new, b.v_new, k2, v2, b.block_table, b.seq_lens, ws)
        ops.check_error(ws)
        assert np.array_equal(k2.view(torch.int16).cpu().numpy().view(np.uint16), kp)
        assert np.array_equal(v2.view(torch.int16).cpu().numpy().view(np.uint16), vp)
        assert_close(out, ref, f"fused edges split {split}")


@pytest.mark.parametrize("pinned", [True, False])
def test_decode_step_from_host_buffers(pinned):
    """pa_decode_step_host: host inputs in, one fused decode step, host output back.  Pinned
    buffers are read and written in place by the kernel; pageable ones go through the
    staging copies."""
    b = wl.batched_decode(device="cuda", seed=5, batch=16, hi=2000, num_blocks=160)
    kp, vp = oracle_appended_pools(b)
    ws = workspace_for(b)
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    host = {k: pin(getattr(b, k).cpu()) for k in ("q", "k_new", "v_new", "block_table", "seq_lens")}
    out_host = pin(torch.empty(b.q.shape, dtype=torch.bfloat16))
    lse_host = pin(torch.empty(b.num_seqs, 32, dtype=torch.float32))
    staging = ops.decode_step_host_staging(b.num_seqs, b.max_blocks_per_seq)
    for _ in range(2):   # the second step re-appends the same token: results must not change
        ops.decode_step_host(out_host, host["q"], host["k_new"], host["v_new"], host["block_table"],
                             host["seq_lens"], b.k_pool, b.v_pool, staging, ws, lse_host=lse_host)
        torch.cuda.synchronize()
        ops.check_error(ws)
        ref, ref_lse = oracle_attention(b, kp, vp)
        assert_close(out_host, ref, "decode step from host buffers")
        assert_lse_close(lse_host, ref_lse, "decode step from host buffers")
    assert np.array_equal(b.k_pool.view(torch.int16).cpu().numpy().view(np.uint16), kp)


def test_cluster_merge_with_an_invalid_length():
    """A sequence whose length is invalid on the cluster-merge path (short contexts, one wave):
    the error is reported, its output is left alone, the other sequence is still right."""
    b = decode_batch([300, 200], seed=31, maxb=2)
    ref, _ = oracle_attention(b)
    sl = b.seq_lens.clone()
    sl[0] = 0                                   # invalid: no context at all
    ws = workspace_for(b)
    out = torch.full_like(b.q, 7.0)
    ops.paged_attn_decode(b.q, b.k_pool, b.v_pool, b.block_table, sl, ws, out=out)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.check_error(ws)
    assert e.value.status == 4
    assert torch.all(out[0] == 7.0)
    assert_close(out[1:], ref[1:], "the valid sequence")


@pytest.mark.parametrize("lens", [[512, 100, 1, 300], [65, 512, 257, 2]])
def test_fused_append_decode_on_the_cluster_merge_path(lens):
    """Short contexts of mixed lengths (tables 2 blocks wide, at most 4 sequences): the grid
    fits in one wave with 8 splits of 64 tokens a pair, so the splits merge as a cluster;
    sequences shorter than 512 leave splits idle (they only meet the others at the cluster
    barriers).  The fused append + decode must match the oracle, leave the pools bit-identical
    to kv_append's, and give the same bits as kv_append followed by paged_attn_decode."""
    b = wl.build_batch("cluster_fused", 41 + len(lens), lens, [1] * len(lens), num_blocks=12,
                       device="cuda", max_blocks_per_seq=2)
    kp, vp = oracle_appended_pools(b)
    ref, ref_lse = oracle_attention(b, kp, vp)
    ws = workspace_for(b)
    k2, v2 = b.k_pool.clone(), b.v_pool.clone()
    lse = torch.empty(b.num_seqs, 32, dtype=torch.float32, device="cuda")
    out = ops.paged_attn_decode_append(b.q, b.k_new, b.v_new, k2, v2, b.block_table, b.seq_lens, ws, lse=lse)
    ops.check_error(ws)
    assert np.array_equal(k2.view(torch.int16).cpu().numpy().view(np.uint16), kp)
    assert np.array_equal(v2.view(torch.int16).cpu().numpy().view(np.uint16), vp)
    assert_close(out, ref, f"fused cluster path {lens}")
    assert_lse_close(lse, ref_lse, f"fused cluster path {lens}")
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    lse2 = torch.empty_like(lse)
    out2 = ops.paged_attn_decode(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, ws, lse=lse2)
    ops.check_error(ws)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse, lse2)


@pytest.mark.parametrize("batch,hi,seed", [(70, 3000, 51), (200, 2500, 52), (512, 700, 53), (513, 700, 54)])
def test_decode_many_sequences(batch, hi, seed):
    """Batches of 70 to 513 sequences whose splits take several waves of CTAs: the result must
    match the oracle and repeat bit for bit (the merge counters put themselves back)."""
    lens = wl.randint_lens(seed, batch, 1, hi)
    b = decode_batch(lens, seed=seed, maxb=(hi + 255) // 256)
    ref, ref_lse = oracle_attention(b)
    ws = workspace_for(b)
    out, lse = run_decode(b, ws)
    assert_close(out, ref, f"decode, batch {batch}")
    assert_lse_close(lse, ref_lse, f"decode, batch {batch}")
    for _ in range(2):
        again, lse2 = run_decode(b, ws)
        assert torch.equal(out.view(torch.int16), again.view(torch.int16))
        assert torch.equal(lse, lse2)
