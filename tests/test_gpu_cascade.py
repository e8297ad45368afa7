"""Cascade decode over a shared prefix (paged_attn_decode_cascade) against the oracle and
against the plain decode: the same attention, computed as the shared prefix for every query
at once plus each sequence's private suffix."""
import pytest
import torch

import oracle
from gpu_helpers import (assert_close, assert_lse_close, gpu, lib_ready, oracle_appended_pools, oracle_attention,
                         to_cpu, workspace_for)
from paged_gqa_attention_gb300 import ops
from paged_gqa_attention_gb300 import workloads as wl

pytestmark = gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def shared_case(lens, shared, seed, extra=3):
    nblk = sum(max(0, (l + 255) // 256 - shared) for l in lens) + shared + extra
    return wl.build_batch("cascade", seed, lens, [1] * len(lens), num_blocks=nblk, device="cuda",
                          shared_prefix_blocks=shared)


def run_cascade(b, shared):
    ws = ops.make_cascade_workspace(b.num_seqs, b.max_blocks_per_seq, shared)
    lse = torch.empty(b.num_seqs, ops.NUM_Q_HEADS, dtype=torch.float32, device="cuda")
    out = ops.paged_attn_decode_cascade(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, shared, ws, lse=lse)
    return out, lse, ws


@pytest.mark.parametrize("lens,shared", [
    ([513, 700, 1000, 515, 2048], 2),       # suffixes from 1 token to several blocks
    ([300] * 9, 1),                         # equal lengths
    ([4096, 769, 1025], 3),
    ([600 + 37 * i for i in range(70)], 2),  # 70 queries: a ragged second query block
])
def test_cascade_matches_oracle_and_plain_decode(lens, shared):
    b = shared_case(lens, shared, seed=71 + len(lens))
    kp, vp = oracle_appended_pools(b)
    ref, ref_lse = oracle_attention(b, kp, vp)
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    out, lse, cws = run_cascade(b, shared)
    ops.check_error(cws)
    assert_close(out, ref, f"cascade {lens[:4]}")
    assert_lse_close(lse, ref_lse, f"cascade {lens[:4]}")
    plain = ops.paged_attn_decode(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, ws)
    ops.check_error(ws)
    assert (out.float() - plain.float()).abs().max().item() <= 1e-2


def test_cascade_repeated_calls_on_one_workspace():
    b = shared_case([700, 513, 1300], 2, seed=75)
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    cws = ops.make_cascade_workspace(b.num_seqs, b.max_blocks_per_seq, 2)
    outs = [ops.paged_attn_decode_cascade(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, 2, cws)
            for _ in range(3)]
    ops.check_error(cws)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_cascade_rejects_a_table_that_does_not_share_the_prefix():
    b = shared_case([700, 900, 1100], 2, seed=76)
    kp, vp = oracle_appended_pools(b)
    ref, _ = oracle_attention(b, kp, vp)
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    bt = b.block_table.clone()
    bt[1, 1] = bt[1, 2]                      # sequence 1's second entry is no longer the shared block
    cws = ops.make_cascade_workspace(b.num_seqs, b.max_blocks_per_seq, 2)
    out = ops.paged_attn_decode_cascade(b.q, b.k_pool, b.v_pool, bt, b.seq_lens, 2, cws)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.check_error(cws)
    assert e.value.status == 4
    assert torch.isnan(out[1].float()).all()
    assert_close(out[0], ref[0], "unaffected sequence 0")
    assert_close(out[2], ref[2], "unaffected sequence 2")


def test_cascade_context_must_extend_past_the_prefix():
    b = shared_case([600, 512], 2, seed=77)     # sequence 1 ends exactly at the prefix
    cws = ops.make_cascade_workspace(b.num_seqs, b.max_blocks_per_seq, 2)
    ops.paged_attn_decode_cascade(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, 2, cws)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.check_error(cws)
    assert e.value.status == 4
    with pytest.raises(ops.PagedAttnError):
        ops.paged_attn_decode_cascade(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, 0, cws)
