"""kv_append: bit-exact against the oracle's append; untouched slots stay untouched."""
import numpy as np
import pytest
import torch

from gpu_helpers import gpu, lib_ready, oracle_appended_pools, workspace_for
from paged_gqa_attention_gb300 import ops
from paged_gqa_attention_gb300 import workloads as wl

pytestmark = gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("name", ["single_decode", "batched_decode", "causal_prefill", "mixed_batch"])
def test_append_is_bit_exact(name):
    b = wl.WORKLOADS[name](device="cuda")
    kp, vp = oracle_appended_pools(b)
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    ops.check_error(ws)
    # the whole pool, NaN sentinels included, equals the oracle's pool bit for bit
    assert np.array_equal(bits(b.k_pool), kp)
    assert np.array_equal(bits(b.v_pool), vp)


def test_append_crossing_block_edges_and_empty_sequences():
    seq_lens = [300, 5, 700, 256]
    q_lens = [100, 0, 450, 1]
    b = wl.build_batch("append_edges", 31, seq_lens, q_lens, num_blocks=12, device="cuda")
    kp, vp = oracle_appended_pools(b)
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    ops.check_error(ws)
    assert np.array_equal(bits(b.k_pool), kp)
    assert np.array_equal(bits(b.v_pool), vp)


def _batch_with_table(seq_lens, q_lens, rows, num_blocks, seed):
    """A batch whose block table is given (rows of physical block ids, -1 padding)."""
    b = wl.build_batch("append_table", seed, seq_lens, q_lens, num_blocks=num_blocks, device="cuda")
    width = max(len(r) for r in rows)
    bt = torch.full((len(rows), width), -1, dtype=torch.int32)
    for i, r in enumerate(rows):
        bt[i, :len(r)] = torch.tensor(r, dtype=torch.int32)
    b.block_table = bt.cuda()
    return b


@pytest.mark.parametrize("case", ["many_empty", "adjacent_blocks", "one_token_each", "scattered"])
def test_append_runs_of_tokens(case):
    """The append moves runs of consecutive new tokens at once: runs that span more than 32
    sequences (empty ones between), runs that continue into a physically adjacent block,
    one token per sequence, and tokens scattered over blocks in no order."""
    if case == "many_empty":
        q_lens = [3] + [0] * 40 + [5] + [0] * 3 + [20] + [0] * 50 + [7]
        seq_lens = [q + 10 * (i % 3) if q else 4 for i, q in enumerate(q_lens)]
        b = wl.build_batch("append_runs", 51, seq_lens, q_lens, num_blocks=len(q_lens) + 4, device="cuda")
    elif case == "adjacent_blocks":
        # sequence 0's positions 200..300 run from block 5 into block 6, sequence 1 from 7 into 2
        b = _batch_with_table([301, 400], [101, 300], [[5, 6], [7, 2]], num_blocks=9, seed=52)
    elif case == "one_token_each":
        lens = [17 + 37 * i for i in range(70)]
        b = wl.build_batch("append_runs", 53, lens, [1] * 70, num_blocks=sum((n + 255) // 256 for n in lens) + 8,
                           device="cuda")
    else:
        b = wl.build_batch("append_runs", 54, [1000, 33, 513], [999, 20, 513], num_blocks=12, device="cuda")
    kp, vp = oracle_appended_pools(b)
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    ops.check_error(ws)
    assert np.array_equal(bits(b.k_pool), kp)
    assert np.array_equal(bits(b.v_pool), vp)
