"""paged_attn_decode_static: batched decode that allocates nothing.

Some callers cannot allocate device memory: code running where cudaMalloc is not
allowed or not available, which is handed only its input and output buffers and no
scratch workspace.  For them the library keeps the decode's split-K scratch in a fixed
device array of its own.  This test calls that entry point through the C ABI and checks
it against paged_attn_decode (caller workspace) on two calls in a row; it creates all
its own data, so it passes alone in a fresh process as well as after the other tests.
"""
import ctypes

import pytest
import torch

from gpu_helpers import LSE_ABS, assert_close, gpu, lib_ready, workspace_for
from paged_gqa_attention_gb300 import ops
from paged_gqa_attention_gb300 import workloads as wl

pytestmark = gpu


def static_entry():
    lib = lib_ready()
    fn = lib.paged_attn_decode_static
    vp = ctypes.c_void_p
    fn.argtypes = [ops.pa_shape, vp, vp, vp, vp, vp, vp, ctypes.c_int32, ctypes.c_int32, vp,
                   ctypes.c_int32, ctypes.c_float, vp, vp]
    fn.restype = ctypes.c_int
    return fn


def test_static_scratch_decode_matches_workspace_decode_twice():
    fn = static_entry()
    b = wl.batched_decode(device="cuda", seed=21, batch=24, hi=3000, num_blocks=400)
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    ref_lse = torch.empty(b.num_seqs, 32, dtype=torch.float32, device="cuda")
    ref = ops.paged_attn_decode(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, ws, lse=ref_lse)
    ops.check_error(ws)
    ref_np = ref.float().cpu().double().numpy()
    err_word = torch.zeros(1, dtype=torch.int32, device="cuda")   # caller-owned error word
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full_like(b.q, float("nan"))
        lse = torch.full((b.num_seqs, 32), float("nan"), dtype=torch.float32, device="cuda")
        st = fn(ops.SHAPE, out.data_ptr(), lse.data_ptr(), b.q.data_ptr(), b.k_pool.data_ptr(),
                b.v_pool.data_ptr(), b.block_table.data_ptr(), b.block_table.shape[1],
                b.k_pool.shape[0], b.seq_lens.data_ptr(), b.num_seqs, wl.SCALE,
                err_word.data_ptr(), stream)
        assert st == 0, ops.STATUS.get(st, st)
        ops.check_error(err_word)          # the word reads like a workspace's first word
        assert_close(out, ref_np, f"static decode, call {call + 1}")
        assert float((lse - ref_lse).abs().max()) <= LSE_ABS


def test_static_scratch_decode_rejects_batches_beyond_its_limit():
    fn = static_entry()
    # 257 sequences exceed the fixed scratch: rejected before anything is launched
    st = fn(ops.SHAPE, None, None, None, None, None, None, 16, 1, None, 257, wl.SCALE, None, None)
    assert st == 6   # PA_ERR_WORKSPACE


def _static_decode(fn, b):
    out = torch.full_like(b.q, float("nan"))
    lse = torch.full((b.num_seqs, 32), float("nan"), dtype=torch.float32, device="cuda")
    err_word = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = fn(ops.SHAPE, out.data_ptr(), lse.data_ptr(), b.q.data_ptr(), b.k_pool.data_ptr(), b.v_pool.data_ptr(),
            b.block_table.data_ptr(), b.block_table.shape[1], b.k_pool.shape[0], b.seq_lens.data_ptr(),
            b.num_seqs, wl.SCALE, err_word.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, ops.STATUS.get(st, st)
    ops.check_error(err_word)
    return out, lse


@pytest.mark.parametrize("lens", [[512], [512, 300], [128, 64, 512, 1]])
def test_cluster_merge_equals_workspace_merge_bit_for_bit(lens):
    """Short contexts: paged_attn_decode's splits merge as a thread-block cluster (through
    shared memory); the static entry point merges the same splits through its scratch and a
    counter.  Same splits, same merge order and arithmetic: identical bits."""
    fn = static_entry()
    b = wl.build_batch("cluster_case", 23, lens, [1] * len(lens), num_blocks=8, device="cuda",
                       max_blocks_per_seq=2)
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    lse = torch.empty(b.num_seqs, 32, dtype=torch.float32, device="cuda")
    out = ops.paged_attn_decode(b.q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, ws, lse=lse)
    ops.check_error(ws)
    out_s, lse_s = _static_decode(fn, b)
    assert torch.equal(out.view(torch.int16), out_s.view(torch.int16))
    assert torch.equal(lse, lse_s)
