"""The attention block of a Qwen3-8B layer through the library, end to end, against the same
pipeline in the oracle: the merged Q/K/V projection of a chunk of new tokens (QK-norm, rotary
embedding, k and v into their cache slots), the causal prefill over the cache, then one decode
step whose new token goes through the projection as well.  Only the hidden states x and the
weights are shared inputs; every intermediate (q, the appended cache rows) is each side's own."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, assert_lse_close, gpu, lib_ready, to_cpu, workspace_for
from paged_gqa_attention_gb300 import ops
from paged_gqa_attention_gb300 import workloads as wl

pytestmark = gpu

HIDDEN = 4096


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def _randn(shape, seed, scale=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(*shape, generator=g, device="cuda") * scale).to(torch.bfloat16)


def _bf16(q_exact):
    """The oracle's fp64 q rounded to bf16 (its own encoder), as the attention's input."""
    bits = oracle.bf16_round(q_exact)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


def _pools(k_bits, v_bits):
    return (torch.from_numpy(k_bits.view(np.int16)).view(torch.bfloat16),
            torch.from_numpy(v_bits.view(np.int16)).view(torch.bfloat16))


@pytest.mark.parametrize("qknorm", [False, True])
def test_projection_prefill_and_decode_step(qknorm):
    # a 200-token chunk after 300 cached tokens, and a fresh 130-token prompt; one more token each
    # for the decode step fits in the blocks already placed
    b = wl.build_batch("pipeline", 70, [500, 130], [200, 130], num_blocks=6, device="cuda")
    # weights ~N(0, 1/(4 hidden)): projected values ~N(0, 1/4), so outputs stay below 2, where one bf16
    # step of the inputs (each side rounds its own projection) moves an output well under the bar
    w = (torch.randn(ops.QKV_COLS, HIDDEN, generator=torch.Generator(device="cuda").manual_seed(71),
                     device="cuda") / (2 * np.sqrt(HIDDEN))).to(torch.bfloat16)
    x = _randn((b.total_tokens, HIDDEN), 72)
    gq, gk = (_randn((128,), 73, 0.5).float().add(1.0).to(torch.bfloat16),
              _randn((128,), 74, 0.5).float().add(1.0).to(torch.bfloat16)) if qknorm else (None, None)
    norm = dict(q_norm_weight=gq, k_norm_weight=gk) if qknorm else {}
    onorm = dict(q_norm=gq.cpu(), k_norm=gk.cpu()) if qknorm else {}
    theta = ops.QWEN3_ROPE_THETA
    kp0, vp0 = to_cpu(b.k_pool), to_cpu(b.v_pool)
    ws = workspace_for(b)

    # prefill: projection into the cache, then causal attention of the chunk
    q = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, ws,
                             rope_theta=theta, **norm)
    lse = torch.empty(b.total_tokens, 32, dtype=torch.float32, device="cuda")
    out = ops.paged_attn_prefill(q, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, b.max_q_len, ws,
                                 lse=lse)
    ops.check_error(ws)
    q_ref, kp, vp = oracle.qkv_append(x.cpu(), w.cpu(), kp0, vp0, to_cpu(b.block_table), to_cpu(b.cu_q_lens),
                                      to_cpu(b.seq_lens), rope_theta=theta, **onorm)
    kp_t, vp_t = _pools(kp, vp)
    ref, ref_lse = oracle.attention(_bf16(q_ref), kp_t, vp_t, to_cpu(b.block_table), to_cpu(b.cu_q_lens),
                                    to_cpu(b.seq_lens), scale=wl.SCALE)
    assert_close(out, ref, f"projection + prefill (qknorm={qknorm})")
    assert_lse_close(lse, ref_lse, f"projection + prefill (qknorm={qknorm})")

    # decode step: one new token per sequence through the projection, then the decode
    x1 = _randn((2, HIDDEN), 75)
    cu1 = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    sl1 = b.seq_lens + 1
    q1 = ops.paged_qkv_append(x1, w, b.k_pool, b.v_pool, b.block_table, cu1, sl1, ws, rope_theta=theta, **norm)
    lse1 = torch.empty(2, 32, dtype=torch.float32, device="cuda")
    out1 = ops.paged_attn_decode(q1, b.k_pool, b.v_pool, b.block_table, sl1, ws, lse=lse1)
    ops.check_error(ws)
    q1_ref, kp1, vp1 = oracle.qkv_append(x1.cpu(), w.cpu(), kp_t, vp_t, to_cpu(b.block_table), cu1.cpu(),
                                         sl1.cpu(), rope_theta=theta, **onorm)
    kp1_t, vp1_t = _pools(kp1, vp1)
    ref1, ref1_lse = oracle.attention(_bf16(q1_ref), kp1_t, vp1_t, to_cpu(b.block_table), cu1.cpu(), sl1.cpu(),
                                      scale=wl.SCALE)
    assert_close(out1, ref1, f"projection + decode step (qknorm={qknorm})")
    assert_lse_close(lse1, ref1_lse, f"projection + decode step (qknorm={qknorm})")
