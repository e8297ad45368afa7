"""Prefill parity: paged_attn_prefill (tcgen05 kernel, through the C ABI) against the oracle."""
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


def append_and_prefill(b, ws=None, with_lse=True):
    ws = workspace_for(b) if ws is None else ws
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    lse = torch.empty(b.total_tokens, 32, dtype=torch.float32, device="cuda") if with_lse else None
    out = ops.paged_attn_prefill(b.q, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens,
                                 b.max_q_len, ws, lse=lse)
    ops.check_error(ws)
    return out, lse


def small_batch(ctx_and_q, seed, extra_blocks=3):
    seq_lens = [c + q for c, q in ctx_and_q]
    q_lens = [q for _, q in ctx_and_q]
    need = sum((s + 255) // 256 for s in seq_lens)
    return wl.build_batch("prefill_case", seed, seq_lens, q_lens, num_blocks=need + extra_blocks,
                          device="cuda")


@pytest.mark.parametrize("ctx_and_q", [
    [(0, 1)],
    [(0, 32)],
    [(0, 128)],
    [(0, 300)],                       # several query tiles, ragged tail
    [(0, 777)],                       # crosses block edges, ragged key tile
    [(200, 100)],                     # chunk after a context ending mid-block
    [(511, 1), (1, 1), (0, 1)],       # decode-like rows through the prefill path
    [(0, 64), (37, 1), (255, 130), (1000, 77), (128, 128)],   # mixed batch
])
def test_prefill_matches_oracle(ctx_and_q):
    b = small_batch(ctx_and_q, seed=len(ctx_and_q) * 100 + ctx_and_q[0][1])
    kp, vp = oracle_appended_pools(b)
    out, lse = append_and_prefill(b)
    ref, ref_lse = oracle_attention(b, kp, vp)
    assert_close(out, ref, f"prefill {ctx_and_q}")
    assert_lse_close(lse, ref_lse, f"prefill {ctx_and_q}")


def plant_score_spikes(b, spikes):
    """Make the new key at token `key_tok` (a row of k_new) 8 times the first query head of
    each KV group at token `q_tok`: that row's score jumps by ~130 (log2 units) and about a
    quarter of the other rows' by more than 8, far past the running maximum of the key tiles
    before it."""
    for key_tok, q_tok in spikes:
        for g in range(ops.NUM_KV_HEADS):
            b.k_new[key_tok, g] = (8.0 * b.q[q_tok, 4 * g].float()).to(torch.bfloat16)


@pytest.mark.parametrize("fused", [False, True])
def test_prefill_late_score_spikes(fused):
    """Scores that exceed the running maximum by far more than the rescale threshold (2^8) in
    a key tile after the first: the rows must rescale their O accumulator mid-way (the
    threshold-crossing path), in the plain and the fused-append prefill alike."""
    b = small_batch([(0, 1000), (300, 700)], seed=23)
    plant_score_spikes(b, [(700, 900), (450, 999), (1000 + 500, 1000 + 650)])
    kp, vp = oracle_appended_pools(b)
    ws = workspace_for(b)
    lse = torch.empty(b.total_tokens, 32, dtype=torch.float32, device="cuda")
    if fused:
        out = ops.paged_attn_prefill_append(b.q, b.k_new, b.v_new, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens,
                                            b.seq_lens, b.max_q_len, ws, lse=lse)
    else:
        ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
        out = ops.paged_attn_prefill(b.q, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens,
                                     b.max_q_len, ws, lse=lse)
    ops.check_error(ws)
    ref, ref_lse = oracle_attention(b, kp, vp)
    assert_close(out, ref, f"prefill with late score spikes (fused={fused})")
    assert_lse_close(lse, ref_lse, f"prefill with late score spikes (fused={fused})")


def test_decode_equals_last_prefill_row():
    b = small_batch([(0, 700)], seed=21)
    out, _ = append_and_prefill(b)
    ws = workspace_for(b)
    for p in (0, 255, 256, 699):
        q = b.q[p:p + 1].contiguous()
        sl = torch.tensor([p + 1], dtype=torch.int32, device="cuda")
        d = ops.paged_attn_decode(q, b.k_pool, b.v_pool, b.block_table, sl, ws)
        ops.check_error(ws)
        diff = (d[0].float() - out[p].float()).abs().max().item()
        assert diff <= 1e-2, f"position {p}: decode vs prefill row differ by {diff}"


def test_chunked_equals_unchunked():
    b = small_batch([(0, 600)], seed=22)
    whole, _ = append_and_prefill(b)
    ws = workspace_for(b)
    parts = []
    for lo, hi in ((0, 129), (129, 300), (300, 600)):
        cu = torch.tensor([0, hi - lo], dtype=torch.int32, device="cuda")
        sl = torch.tensor([hi], dtype=torch.int32, device="cuda")
        parts.append(ops.paged_attn_prefill(b.q[lo:hi].contiguous(), b.k_pool, b.v_pool,
                                            b.block_table, cu, sl, hi - lo, ws))
    ops.check_error(ws)
    chunked = torch.cat(parts)
    diff = (chunked.float() - whole.float()).abs().max().item()
    assert diff <= 1e-2


def test_prefill_block_placement_is_bit_exact():
    b = small_batch([(100, 400), (0, 50)], seed=23, extra_blocks=10)
    out1, _ = append_and_prefill(b)
    perm = torch.randperm(b.num_blocks, generator=torch.Generator().manual_seed(3)).to("cuda")
    k2 = torch.empty_like(b.k_pool)
    v2 = torch.empty_like(b.v_pool)
    k2[perm] = b.k_pool
    v2[perm] = b.v_pool
    bt = b.block_table.clone()
    valid = bt >= 0
    bt[valid] = perm[bt[valid].long()].to(torch.int32)
    ws = workspace_for(b)
    out2 = ops.paged_attn_prefill(b.q, k2, v2, bt, b.cu_q_lens, b.seq_lens, b.max_q_len, ws)
    ops.check_error(ws)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_empty_sequences_are_skipped():
    b = small_batch([(10, 0), (0, 40), (300, 0)], seed=24)
    kp, vp = oracle_appended_pools(b)
    out, _ = append_and_prefill(b)
    ref, _ = oracle_attention(b, kp, vp)
    assert_close(out, ref, "empty sequences")


def test_work_plan_leaves_results_unchanged():
    """Several sequences: the units are first sorted by work (a planning kernel writing into
    the workspace).  A workspace holding only the error word leaves no room for that order,
    so the units go in their natural order; both runs must agree bit for bit (each unit is
    computed by one CTA on its own), and with the oracle."""
    ctx_and_q = [(0, 300), (700, 64), (33, 1), (2000, 129), (0, 5), (511, 200)]
    b = small_batch(ctx_and_q, seed=91)
    kp, vp = oracle_appended_pools(b)
    ws = workspace_for(b)
    ops.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    ops.check_error(ws)
    runs = []
    for w in (ws, torch.zeros(256, dtype=torch.uint8, device="cuda")):
        lse = torch.empty(b.total_tokens, 32, dtype=torch.float32, device="cuda")
        out = ops.paged_attn_prefill(b.q, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens,
                                     b.max_q_len, w, lse=lse)
        ops.check_error(w)
        runs.append((out, lse))
    (o1, l1), (o2, l2) = runs
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32))
    ref, ref_lse = oracle_attention(b, kp, vp)
    assert_close(o1, ref, "planned prefill")
    assert_lse_close(l1, ref_lse, "planned prefill")


def fused_prefill(b, ws=None):
    ws = workspace_for(b) if ws is None else ws
    lse = torch.empty(b.total_tokens, 32, dtype=torch.float32, device="cuda")
    out = ops.paged_attn_prefill_append(b.q, b.k_new, b.v_new, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens,
                                        b.seq_lens, b.max_q_len, ws, lse=lse)
    ops.check_error(ws)
    return out, lse


def pool_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("ctx_and_q", [
    [(0, 1)],
    [(0, 300)],                       # from position 0: the same key tiles as the two calls
    [(0, 777)],
    [(200, 100)],                     # a chunk after a context ending mid-tile
    [(100, 28)],                      # a chunk inside one key tile of the context
    [(511, 1), (1, 1), (0, 1)],
    [(0, 64), (37, 1), (255, 130), (1000, 77), (128, 128)],   # several sequences (planned order)
    [(10, 0), (300, 513), (40, 3)],   # an empty sequence
])
def test_prefill_append_matches_oracle(ctx_and_q):
    """paged_attn_prefill_append: the pools equal the oracle's append bit for bit (sentinels
    included) and the outputs and lse match the oracle."""
    b = small_batch(ctx_and_q, seed=len(ctx_and_q) * 100 + ctx_and_q[0][1] + 7)
    kp, vp = oracle_appended_pools(b)
    out, lse = fused_prefill(b)
    assert np.array_equal(pool_bits(b.k_pool), kp)
    assert np.array_equal(pool_bits(b.v_pool), vp)
    ref, ref_lse = oracle_attention(b, kp, vp)
    assert_close(out, ref, f"fused prefill {ctx_and_q}")
    assert_lse_close(lse, ref_lse, f"fused prefill {ctx_and_q}")


@pytest.mark.parametrize("ctx_and_q", [[(0, 300)], [(256, 100)], [(128, 77), (0, 5), (384, 260)]])
def test_prefill_append_equals_the_two_calls_on_aligned_contexts(ctx_and_q):
    """Where every earlier context is a multiple of 128 tokens both paths cut the keys into the
    same tiles: the fused call gives the bits of kv_append followed by paged_attn_prefill."""
    b = small_batch(ctx_and_q, seed=61 + len(ctx_and_q))
    k0, v0 = b.k_pool.clone(), b.v_pool.clone()
    out1, lse1 = append_and_prefill(b)
    b.k_pool, b.v_pool = k0, v0
    out2, lse2 = fused_prefill(b)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1.view(torch.int32), lse2.view(torch.int32))


def test_prefill_append_bad_block_is_reported_and_writes_nothing_stray():
    b = small_batch([(0, 300), (100, 20)], seed=66, extra_blocks=6)
    bt = b.block_table.clone()
    bt[1, 0] = b.num_blocks + 3                 # sequence 1's only block is outside the pool
    kp0 = pool_bits(b.k_pool).copy()
    kp, vp = oracle_appended_pools(b)           # (the oracle appends with the valid table)
    ws = workspace_for(b)
    ops.paged_attn_prefill_append(b.q, b.k_new, b.v_new, b.k_pool, b.v_pool, bt, b.cu_q_lens, b.seq_lens,
                                  b.max_q_len, ws)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.check_error(ws)
    assert e.value.status == 4
    # sequence 0's rows are appended as the oracle does; no byte of sequence 1's goes anywhere
    got = pool_bits(b.k_pool)
    seq0_blocks = [int(x) for x in b.block_table[0, :2].cpu()]
    assert np.array_equal(got[seq0_blocks], kp[seq0_blocks])
    others = np.ones(b.num_blocks, dtype=bool)
    others[seq0_blocks] = False
    assert np.array_equal(got[others], kp0[others])
