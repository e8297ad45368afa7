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
