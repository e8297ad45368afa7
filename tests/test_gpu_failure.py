"""Failure paths on the GPU, without faulting it: device-side argument checks and bounded
waits report through the workspace error word, and the context stays usable."""
import pytest
import torch

from gpu_helpers import assert_close, gpu, lib_ready, oracle_appended_pools, oracle_attention, workspace_for
from paged_gqa_attention_gb300 import ops
from paged_gqa_attention_gb300 import workloads as wl

pytestmark = gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def decode_case(lens, seed):
    need = sum((l + 255) // 256 for l in lens)
    b = wl.build_batch("fail_case", seed, lens, [1] * len(lens), num_blocks=need + 2, device="cuda")
    return b


def test_bounded_wait_times_out_and_context_survives():
    b = decode_case([300, 40], seed=41)
    kp, vp = oracle_appended_pools(b)           # the oracle's own append, on the host
    ws = workspace_for(b)
    ops.selftest_wait_timeout(ws, timeout_us=20000)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.check_error(ws)
    assert e.value.status == 5          # PA_ERR_TIMEOUT
    # the error word was cleared and the GPU still computes correctly
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    out = ops.paged_attn_decode(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, ws)
    ops.check_error(ws)
    ref, _ = oracle_attention(b, kp, vp)
    assert_close(out, ref, "after timeout")


def test_decode_bad_block_id_is_reported_and_poisons_only_its_sequence():
    b = decode_case([600, 300], seed=42)
    kp, vp = oracle_appended_pools(b)           # the oracle's own append, on the host
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    ops.check_error(ws)
    ref, _ = oracle_attention(b, kp, vp)
    bt = b.block_table.clone()
    bt[0, 1] = b.num_blocks + 5                     # out of range
    out = ops.paged_attn_decode(b.q, b.k_pool, b.v_pool, bt, b.seq_lens, ws)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.check_error(ws)
    assert e.value.status == 4                      # PA_ERR_DEVICE
    assert torch.isnan(out[0].float()).any()
    assert_close(out[1], ref[1], "unaffected sequence")
    # and the next call on the same workspace is clean
    out = ops.paged_attn_decode(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, ws)
    ops.check_error(ws)
    assert_close(out, ref, "after device error")


def test_decode_bad_context_length_is_reported():
    b = decode_case([100], seed=43)
    ws = workspace_for(b)
    sl = torch.tensor([0], dtype=torch.int32, device="cuda")
    ops.paged_attn_decode(b.q, b.k_pool, b.v_pool, b.block_table, sl, ws)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.check_error(ws)
    assert e.value.status == 4


def test_append_bad_block_id_writes_nothing_out_of_place():
    b = decode_case([10, 20], seed=44)
    ws = workspace_for(b)
    bt = b.block_table.clone()
    bt[1, 0] = -3
    before_k = b.k_pool.clone()
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, bt, b.cu_q_lens, b.seq_lens, ws)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.check_error(ws)
    assert e.value.status == 4
    # sequence 0 was appended, sequence 1 was not written anywhere
    blk0 = int(b.block_table[0, 0])
    changed = (b.k_pool.view(torch.int16) != before_k.view(torch.int16)).flatten(1).any(1)
    assert changed.nonzero().flatten().tolist() == [blk0]


def test_prefill_inconsistent_lengths_are_reported():
    b = wl.build_batch("fail_prefill", 45, [100], [100], num_blocks=3, device="cuda")
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    ops.check_error(ws)
    # max_q_len smaller than the real q_len
    ops.paged_attn_prefill(b.q, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, 64, ws)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.check_error(ws)
    assert e.value.status == 4


def test_host_rejects_bad_arguments():
    b = decode_case([50], seed=46)
    ws = workspace_for(b)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.paged_attn_decode(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, ws[:64])
    assert e.value.status == 1
    with pytest.raises(TypeError):
        ops.paged_attn_decode(b.q.float(), b.k_pool, b.v_pool, b.block_table, b.seq_lens, ws)
