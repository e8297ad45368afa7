"""The multi-layer decode step captured as a CUDA graph (pa_decode_graph_*): every layer's
append and attention against the oracle, bit-identical to the same calls made one by one,
and replays that follow in-place updates of the inputs."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, assert_lse_close, gpu, lib_ready, to_cpu
from paged_gqa_attention_gb300 import ops
from paged_gqa_attention_gb300 import workloads as wl

pytestmark = gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def bits(t):
    return to_cpu(t).contiguous().view(torch.int16).numpy().view(np.uint16)


def oracle_step(b: wl.Batch, kp, vp):
    """The oracle's append of b's new tokens into pools (kp, vp), then its attention."""
    kp2, vp2 = oracle.kv_append(kp, vp, to_cpu(b.k_new), to_cpu(b.v_new), to_cpu(b.block_table),
                                to_cpu(b.cu_q_lens), to_cpu(b.seq_lens))
    out, lse = oracle.attention(to_cpu(b.q), kp2, vp2, to_cpu(b.block_table), to_cpu(b.cu_q_lens),
                                to_cpu(b.seq_lens), scale=wl.SCALE)
    return kp2, vp2, out, lse


def decode_case(lens, seed, layers, spare_tokens=0):
    need = sum((l + spare_tokens + 255) // 256 for l in lens)
    b = wl.build_batch("graph_case", seed, lens, [1] * len(lens), num_blocks=need + 3, device="cuda")
    return wl.layered(b, layers, seed + 1000)


def test_graph_step_matches_oracle_and_one_by_one_calls():
    L = decode_case([1, 255, 256, 257, 700, 1024], seed=61, layers=4)
    b0 = L.base
    ws = ops.make_workspace(b0.num_seqs, b0.max_blocks_per_seq)
    # one call per layer, on copies of the pools
    kp_e, vp_e = L.k_pool.clone(), L.v_pool.clone()
    out_e = torch.empty_like(L.q)
    for l in range(L.layers):
        ops.paged_attn_decode_append(L.q[l], L.k_new[l], L.v_new[l], kp_e[l], vp_e[l], b0.block_table,
                                     b0.seq_lens, ws, out=out_e[l])
    ops.check_error(ws)
    # the captured graph, on the layered tensors themselves
    refs = [oracle_step(L.layer(l), bits(L.k_pool[l]), bits(L.v_pool[l])) for l in range(L.layers)]
    out_g = torch.empty_like(L.q)
    lse_g = torch.empty(L.layers, b0.num_seqs, ops.NUM_Q_HEADS, dtype=torch.float32, device="cuda")
    g = ops.decode_graph(L.q, L.k_new, L.v_new, L.k_pool, L.v_pool, b0.block_table, b0.seq_lens, ws,
                         out=out_g, lse=lse_g)
    g.launch()
    ops.check_error(ws)
    assert torch.equal(out_g.view(torch.int16), out_e.view(torch.int16)), "graph differs from one-by-one calls"
    for l, (kp, vp, ref, ref_lse) in enumerate(refs):
        assert (bits(L.k_pool[l]) == kp).all() and (bits(L.v_pool[l]) == vp).all(), f"layer {l} pools"
        assert_close(out_g[l], ref, f"layer {l}")
        assert_lse_close(lse_g[l], ref_lse, f"layer {l}")
    g.close()


def test_graph_replays_follow_in_place_updates():
    # lengths that stay inside their last block for three more tokens
    L = decode_case([5, 100, 300, 610], seed=62, layers=3, spare_tokens=3)
    b0 = L.base
    ws = ops.make_workspace(b0.num_seqs, b0.max_blocks_per_seq)
    kps = [bits(L.k_pool[l]) for l in range(L.layers)]
    vps = [bits(L.v_pool[l]) for l in range(L.layers)]
    out = torch.empty_like(L.q)
    g = ops.decode_graph(L.q, L.k_new, L.v_new, L.k_pool, L.v_pool, b0.block_table, b0.seq_lens, ws,
                         out=out)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(63)
    for step in range(3):
        if step:
            # the next decode step: new queries and new K/V rows, one more token per context
            for t in (L.q, L.k_new, L.v_new):
                t.copy_(torch.randn(t.shape, generator=gen, device="cuda").to(torch.bfloat16))
            b0.seq_lens.add_(1)
        g.launch()
        ops.check_error(ws)
        for l in range(L.layers):
            kps[l], vps[l], ref, _ = oracle_step(L.layer(l), kps[l], vps[l])
            assert (bits(L.k_pool[l]) == kps[l]).all() and (bits(L.v_pool[l]) == vps[l]).all()
            assert_close(out[l], ref, f"step {step} layer {l}")
    g.close()


def test_graph_rejects_bad_arguments():
    L = decode_case([40], seed=64, layers=2)
    b0 = L.base
    ws = ops.make_workspace(b0.num_seqs, b0.max_blocks_per_seq)
    out = torch.empty_like(L.q)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.decode_graph(L.q, L.k_new, L.v_new, L.k_pool, L.v_pool, b0.block_table, b0.seq_lens, ws[:64],
                         out=out)
    assert e.value.status == 1          # workspace below the fixed header: invalid
    # a closed handle cannot be launched; closing twice is harmless
    g = ops.decode_graph(L.q, L.k_new, L.v_new, L.k_pool, L.v_pool, b0.block_table, b0.seq_lens, ws, out=out)
    g.close()
    g.close()
    with pytest.raises(RuntimeError):
        g.launch()
