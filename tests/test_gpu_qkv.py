"""paged_qkv_append (merged Q/K/V projection with K and V written into the cache) against the
oracle.

Tolerance: each output is one bf16 rounding of a dot product accumulated in fp32 by the
tensor cores, so every element of q and of the appended K/V rows must lie within one bf16
step of the exact fp64 value (2^-8 relative) plus the accumulation error, which scales with
the sum of the absolute products rather than with the (possibly cancelled) result: we allow
2^-16 * sum_k |x_k w_k| (about 256 fp32 roundings of that sum).  The whole q must also be
within rel-RMS 5e-3.  Every pool byte outside the new tokens' slots must be unchanged
(bit-exact).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import REPORT, gpu, lib_ready, workspace_for
from paged_gqa_attention_gb300 import ops
from paged_gqa_attention_gb300 import workloads as wl

pytestmark = gpu

HIDDEN = 4096


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_ready()


def weights(seed, hidden=HIDDEN):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(ops.QKV_COLS, hidden, generator=g, device="cuda") / np.sqrt(hidden)).to(torch.bfloat16)


def inputs(seed, tokens, hidden=HIDDEN):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(tokens, hidden, generator=g, device="cuda").to(torch.bfloat16)


def batch_for(ctx_and_q, seed):
    seq_lens = [c + q for c, q in ctx_and_q]
    q_lens = [q for _, q in ctx_and_q]
    return wl.build_batch("qkv_case", seed, seq_lens, q_lens, num_blocks=sum((s + 255) // 256 for s in seq_lens) + 3,
                          device="cuda")


def abs_sums(x, w, rows=None):
    """sum_k |x[t][k] w[n][k]| for the listed token rows (the scale of the accumulation error)."""
    xa = x.cpu().double().abs().numpy()
    if rows is not None:
        xa = xa[rows]
    return xa @ w.cpu().double().abs().numpy().T


def within_tol(got, exact, abs_sum, what):
    got = np.asarray(got, dtype=np.float64)
    tol = np.abs(exact) * 2.0 ** -8 + abs_sum * 2.0 ** -16
    err = np.abs(got - exact)
    with np.errstate(divide="ignore", invalid="ignore"):      # zero rows: 0 / 0 in the report only
        ratio = np.where(tol > 0, err / tol, np.where(err > 0, np.inf, 0.0))
    i = np.unravel_index(np.nanargmax(ratio), err.shape)
    REPORT.append({"what": what, "kind": "bound", "max_ratio": float(ratio[i]), "elements": int(err.size)})
    assert (err <= tol).all(), (f"{what}: worst element {i}: got {got[i]!r} exact {exact[i]!r} "
                                f"tolerance {tol[i]!r} ({(err > tol).sum()} elements beyond it)")


def new_slots(b):
    """(block, slot) of every new token, in token order."""
    bt, cu, sl = b.block_table.cpu(), b.cu_q_lens.cpu(), b.seq_lens.cpu()
    out = []
    for s in range(b.num_seqs):
        q_len = int(cu[s + 1] - cu[s])
        for i in range(q_len):
            p = int(sl[s]) - q_len + i
            out.append((int(bt[s, p // 256]), p % 256))
    return out


def exact_and_bound(x, w, cu_q_lens, seq_lens, rope_theta, rows=None, projected=None):
    """The oracle's exact outputs (q and k heads rotated when rope_theta > 0) and the
    accumulation part of the bound: a rotated dim mixes the two columns of its pair, so it
    carries both their accumulation errors, and the fp32 angle (about 1e-6 rad) adds
    1e-5 x the pair's size.  projected: (y, sum|x w|) of the listed rows, if already at hand."""
    y, a = projected if projected is not None else (oracle.qkv_project(x.cpu(), w.cpu(), rows=rows),
                                                    abs_sums(x, w, rows))
    if rope_theta:
        pos = oracle.token_positions(cu_q_lens.cpu(), seq_lens.cpu())
        if rows is not None:
            pos = pos[np.asarray(rows)]
        rot = oracle.rope(y, pos, rope_theta, first_col=0, n_heads=32)
        rot = oracle.rope(rot, pos, rope_theta, first_col=4096, n_heads=8)
        cols = np.arange(5120)
        partner = cols ^ 64                       # the other dim of the pair in the same head
        a = a.copy()
        a[:, :5120] = a[:, cols] + a[:, partner] + 1e-5 * 2.0 ** 16 * (np.abs(y[:, cols]) + np.abs(y[:, partner]))
        y = rot
    return y, a


def check_case(b, x, w, rope_theta=0.0):
    kp0 = b.k_pool.view(torch.int16).cpu().numpy().view(np.uint16).copy()
    vp0 = b.v_pool.view(torch.int16).cpu().numpy().view(np.uint16).copy()
    ws = workspace_for(b)
    q = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, ws,
                             rope_theta=rope_theta)
    ops.check_error(ws)
    y, a = exact_and_bound(x, w, b.cu_q_lens, b.seq_lens, rope_theta)
    qg = q.float().cpu().numpy().astype(np.float64).reshape(x.shape[0], -1)
    within_tol(qg, y[:, :4096], a[:, :4096], "q")
    rel = np.sqrt(((qg - y[:, :4096]) ** 2).sum() / (y[:, :4096] ** 2).sum())
    assert rel <= 5e-3, rel
    kp = b.k_pool.view(torch.int16).cpu().numpy().view(np.uint16)
    vp = b.v_pool.view(torch.int16).cpu().numpy().view(np.uint16)
    touched = np.zeros(kp.shape[:2], dtype=bool)
    for t, (blk, slot) in enumerate(new_slots(b)):
        touched[blk, slot] = True
        kf = torch.from_numpy(kp[blk, slot].copy()).view(torch.bfloat16).double().numpy().reshape(-1)
        vf = torch.from_numpy(vp[blk, slot].copy()).view(torch.bfloat16).double().numpy().reshape(-1)
        within_tol(kf, y[t, 4096:5120], a[t, 4096:5120], f"k row of token {t}")
        within_tol(vf, y[t, 5120:], a[t, 5120:], f"v row of token {t}")
    assert np.array_equal(kp[~touched], kp0[~touched]), "k pool written outside the new slots"
    assert np.array_equal(vp[~touched], vp0[~touched]), "v pool written outside the new slots"


@pytest.mark.parametrize("ctx_and_q", [
    [(0, 1)],
    [(0, 37)],                                  # few tokens: 64-column tiles
    [(200, 100), (0, 64), (511, 1)],            # chunks after context, a decode-like row
    [(0, 300)],                                 # many tokens: 256-column tiles, a ragged last tile
    [(37, 130), (1000, 0), (255, 200)],         # a sequence with no new token
    [(100, 900)],                               # 192 tiles on 152 CTAs: the last round in halves
])
def test_qkv_append_matches_oracle(ctx_and_q):
    b = batch_for(ctx_and_q, seed=60 + len(ctx_and_q))
    x = inputs(61, b.total_tokens)
    w = weights(62)
    check_case(b, x, w)


@pytest.mark.parametrize("ctx_and_q", [
    [(0, 1)],
    [(0, 37)],                                  # 64-column tiles, 32 rows of x loaded
    [(200, 100), (0, 64), (511, 1)],            # 64-column tiles, 128 rows
    [(0, 300)],                                 # CTA pairs, a ragged last tile
    [(37, 130), (1000, 0), (255, 200)],
    [(131000, 40), (70000, 300)],               # large positions: angles of 10^5 rad
])
def test_qkv_append_with_rotary_embedding(ctx_and_q):
    """Qwen3's rotary embedding (theta 1e6) on q and k before the rounding, against the
    oracle's rotation of its exact projection at each token's absolute position."""
    b = batch_for(ctx_and_q, seed=160 + len(ctx_and_q))
    check_case(b, inputs(161, b.total_tokens), weights(162), rope_theta=ops.QWEN3_ROPE_THETA)


def test_rotary_embedding_near_the_largest_position():
    """Positions just below 2^24 (tables 65536 blocks wide, the widest a rotation accepts):
    every table entry but the last two points at block 0, the new tokens go to blocks 1, 2."""
    n = 40
    seq_len = (1 << 24) - 3
    width = 1 << 16
    bt = torch.zeros(1, width, dtype=torch.int32)
    p0 = seq_len - n
    bt[0, p0 // 256] = 1
    bt[0, (seq_len - 1) // 256] = 2
    g = torch.Generator(device="cuda").manual_seed(170)
    pools = [torch.randn(3, 256, 8, 128, generator=g, device="cuda").to(torch.bfloat16) for _ in range(2)]
    b = wl.Batch(name="far", q=torch.empty(n, 32, 128, dtype=torch.bfloat16, device="cuda"),
                 k_new=torch.empty(n, 8, 128, dtype=torch.bfloat16, device="cuda"),
                 v_new=torch.empty(n, 8, 128, dtype=torch.bfloat16, device="cuda"),
                 k_pool=pools[0], v_pool=pools[1], block_table=bt.cuda(),
                 seq_lens=torch.tensor([seq_len], dtype=torch.int32, device="cuda"),
                 cu_q_lens=torch.tensor([0, n], dtype=torch.int32, device="cuda"), max_q_len=n,
                 seq_lens_host=[seq_len], q_lens_host=[n])
    check_case(b, inputs(171, n), weights(172), rope_theta=ops.QWEN3_ROPE_THETA)
    # one block wider and the positions could reach 2^24: refused before any launch
    wide = torch.zeros(1, width + 1, dtype=torch.int32, device="cuda")
    ws = workspace_for(b)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.paged_qkv_append(inputs(171, n), weights(172), b.k_pool, b.v_pool, wide, b.cu_q_lens, b.seq_lens, ws,
                             rope_theta=ops.QWEN3_ROPE_THETA)
    assert e.value.status == 1


@pytest.mark.parametrize("hidden", [256, 1280])
@pytest.mark.parametrize("ctx_and_q", [[(10, 40)], [(0, 300)]])   # one CTA per tile; CTA pairs
def test_other_hidden_sizes(hidden, ctx_and_q):
    """hidden is any multiple of 256: 1 and 5 ring stages per tile (one CTA), 4 and 20 (pairs)."""
    b = batch_for(ctx_and_q, seed=80 + hidden % 7)
    x = inputs(81, b.total_tokens, hidden)
    w = weights(82, hidden)
    ws = workspace_for(b)
    q = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, ws)
    ops.check_error(ws)
    y = oracle.qkv_project(x.cpu(), w.cpu())
    a = abs_sums(x, w)
    qg = q.float().cpu().numpy().astype(np.float64).reshape(x.shape[0], -1)
    within_tol(qg, y[:, :4096], a[:, :4096], "q")
    for t, (blk, slot) in enumerate(new_slots(b)):
        kf = b.k_pool[blk, slot].double().cpu().numpy().reshape(-1)
        vf = b.v_pool[blk, slot].double().cpu().numpy().reshape(-1)
        within_tol(kf, y[t, 4096:5120], a[t, 4096:5120], f"k row of token {t}")
        within_tol(vf, y[t, 5120:], a[t, 5120:], f"v row of token {t}")


def test_decode_batch_one_token_per_sequence():
    b = wl.batched_decode(device="cuda", seed=63, batch=32, hi=2000, num_blocks=300)
    check_case(b, inputs(64, b.total_tokens), weights(65))


@pytest.mark.parametrize("rope_theta", [0.0, ops.QWEN3_ROPE_THETA])
def test_full_prefill_chunk_sampled_rows(rope_theta):
    """4096 new tokens (the causal prefill workload's prompt), in the configuration the
    benchmark times: sampled rows of q and of the cache against the oracle, every other
    cache row untouched is not re-checked here."""
    b = wl.causal_prefill(device="cuda")
    x = inputs(66, b.total_tokens)
    w = weights(67)
    ws = workspace_for(b)
    q = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, ws,
                             rope_theta=rope_theta)
    ops.check_error(ws)
    rows = [0, 1, 127, 128, 2047, 2048, 4000, 4095]
    y, a = exact_and_bound(x, w, b.cu_q_lens, b.seq_lens, rope_theta, rows=rows)
    slots = new_slots(b)
    qg = q.float().cpu().numpy().astype(np.float64).reshape(b.total_tokens, -1)
    for r, t in enumerate(rows):
        within_tol(qg[t], y[r, :4096], a[r, :4096], f"q row {t}")
        blk, slot = slots[t]
        kf = b.k_pool[blk, slot].double().cpu().numpy().reshape(-1)
        vf = b.v_pool[blk, slot].double().cpu().numpy().reshape(-1)
        within_tol(kf, y[r, 4096:5120], a[r, 4096:5120], f"k row {t}")
        within_tol(vf, y[r, 5120:], a[r, 5120:], f"v row {t}")


@pytest.mark.parametrize("ctx_and_q", [
    [(0, 40), (100, 20)],                       # one CTA per tile
    [(0, 300), (100, 20)],                      # CTA pairs
])
def test_bad_block_writes_no_kv_but_keeps_q(ctx_and_q):
    b = batch_for(ctx_and_q, seed=68)
    n0 = ctx_and_q[0][1]                        # sequence 0's new tokens
    x = inputs(69, b.total_tokens)
    w = weights(70)
    bt = b.block_table.clone()
    bt[1, 0] = b.num_blocks + 7                 # sequence 1's only block is outside the pool
    kp0 = b.k_pool.clone()
    ws = workspace_for(b)
    q = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, bt, b.cu_q_lens, b.seq_lens, ws)
    with pytest.raises(ops.PagedAttnError) as e:
        ops.check_error(ws)
    assert e.value.status == 4
    y = oracle.qkv_project(x.cpu(), w.cpu())
    qg = q.float().cpu().numpy().astype(np.float64).reshape(b.total_tokens, -1)
    within_tol(qg, y[:, :4096], abs_sums(x, w)[:, :4096], "q")
    # sequence 0's rows are appended, nothing of sequence 1 is written anywhere
    touched = np.zeros((b.num_blocks, 256), dtype=bool)
    for t, (blk, slot) in enumerate(new_slots(b)[:n0]):
        touched[blk, slot] = True
    a = b.k_pool.view(torch.int16).cpu().numpy()
    o = kp0.view(torch.int16).cpu().numpy()
    assert np.array_equal(a[~touched], o[~touched])


@pytest.mark.parametrize("rope_theta", [0.0, ops.QWEN3_ROPE_THETA])
def test_fused_append_feeds_the_decode(rope_theta):
    """The fused projection + append (with or without the rotary embedding) followed by the
    decode equals the decode over the oracle's appended cache (within the attention
    tolerance)."""
    from gpu_helpers import assert_close
    b = wl.batched_decode(device="cuda", seed=71, batch=8, hi=1500, num_blocks=64)
    x = inputs(72, b.total_tokens)
    w = weights(73)
    q_ref, kp, vp = oracle.qkv_append(x.cpu(), w.cpu(), b.k_pool.cpu(), b.v_pool.cpu(), b.block_table.cpu(),
                                      b.cu_q_lens.cpu(), b.seq_lens.cpu(), rope_theta=rope_theta)
    ws = workspace_for(b)
    q = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, ws,
                             rope_theta=rope_theta)
    out = ops.paged_attn_decode(q, b.k_pool, b.v_pool, b.block_table, b.seq_lens, ws)
    ops.check_error(ws)
    # the oracle attends with the GPU's q (its own q is exact fp64, the GPU's is bf16)
    ref, _ = oracle.attention(q.cpu(), kp, vp, b.block_table.cpu(), b.cu_q_lens.cpu(), b.seq_lens.cpu(),
                              scale=wl.SCALE)
    assert_close(out, ref, "decode after the fused projection")


@pytest.mark.parametrize("rope_theta", [0.0, ops.QWEN3_ROPE_THETA])
@pytest.mark.parametrize("ctx_and_q", [[(0, 300)], [(0, 4096)]])
def test_repeated_calls_are_bit_identical(ctx_and_q, rope_theta):
    """The CTA-pair path is deterministic: q and the appended cache rows repeat bit for bit."""
    b = batch_for(ctx_and_q, seed=90)
    x = inputs(91, b.total_tokens)
    w = weights(92)
    ws = workspace_for(b)
    q1 = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, ws,
                              rope_theta=rope_theta).clone()
    k1, v1 = b.k_pool.clone(), b.v_pool.clone()
    for _ in range(3):
        q2 = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, ws,
                                  rope_theta=rope_theta)
        ops.check_error(ws)
        assert torch.equal(q1.view(torch.int16), q2.view(torch.int16))
        assert torch.equal(k1.view(torch.int16), b.k_pool.view(torch.int16))
        assert torch.equal(v1.view(torch.int16), b.v_pool.view(torch.int16))


# ------------------------------------------------------------------ QK-norm (paged_qkv_append_qknorm)

def norm_gains(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    q = (1.0 + 0.5 * torch.randn(128, generator=g, device="cuda")).to(torch.bfloat16)
    k = (1.0 + 0.5 * torch.randn(128, generator=g, device="cuda")).to(torch.bfloat16)
    return q, k


def qknorm_exact_and_bound(x, w, cu_q_lens, seq_lens, rope_theta, gq, gk, eps, rows=None, projected=None):
    """The oracle's q and k after the norm and the rotation (exact, before the last rounding),
    and per element the part of the bound that the projection's own error carries through
    the norm.  The GPU normalises its bf16 projection p', the oracle the rounded exact one p:
    |p' - p| <= d = 2^-7 |y| + 2^-16 sum|x w| (the projection's bound plus the oracle's half
    step).  To first order that moves n = g p / r (r the head's RMS with eps) by
    |g| d / r + |g p| (sum_j |p_j| d_j) / (128 r^3); a rotated dim mixes the two dims of its
    pair, and the fp32 arithmetic and angle add 1e-5 of the pair's size.  Returned scaled by
    2^16, in the units ``within_tol`` takes for its second term."""
    y, a = projected if projected is not None else (oracle.qkv_project(x.cpu(), w.cpu(), rows=rows),
                                                    abs_sums(x, w, rows))
    p = (oracle.bf16_round(y[:, :5120]).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    d = 2.0 ** -7 * np.abs(y[:, :5120]) + 2.0 ** -16 * a[:, :5120]
    n = np.concatenate([oracle.rms_norm_heads(p[:, :4096], gq.cpu(), eps, n_heads=32),
                        oracle.rms_norm_heads(p[:, 4096:], gk.cpu(), eps, n_heads=8)], axis=1)
    g = np.concatenate([np.tile(gq.double().cpu().numpy(), 32), np.tile(gk.double().cpu().numpy(), 8)])
    ph, dh = p.reshape(len(p), 40, 128), d.reshape(len(p), 40, 128)
    r = np.sqrt((ph ** 2).mean(axis=2) + eps)[:, :, None]
    cross = (np.abs(ph) * dh).sum(axis=2)[:, :, None]
    dn = (np.abs(g).reshape(1, 40, 128) * (dh / r + np.abs(ph) * cross / (128 * r ** 3))).reshape(len(p), 5120)
    if rope_theta:
        pos = oracle.token_positions(cu_q_lens.cpu(), seq_lens.cpu())
        if rows is not None:
            pos = pos[np.asarray(rows)]
        e = oracle.rope(n, pos, rope_theta, first_col=0, n_heads=32)
        e = oracle.rope(e, pos, rope_theta, first_col=4096, n_heads=8)
        cols = np.arange(5120)
        partner = cols ^ 64
        bound = dn[:, cols] + dn[:, partner] + 1e-5 * (np.abs(n[:, cols]) + np.abs(n[:, partner]))
    else:
        e = n
        bound = dn + 1e-6 * np.abs(n)
    return e, bound * 2.0 ** 16, y, a


def check_qknorm_case(b, x, w, rope_theta, eps=ops.QWEN3_NORM_EPS, seed=90):
    gq, gk = norm_gains(seed)
    kp0 = b.k_pool.view(torch.int16).cpu().numpy().copy()
    vp0 = b.v_pool.view(torch.int16).cpu().numpy().copy()
    ws = workspace_for(b)
    q = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, ws,
                             rope_theta=rope_theta, q_norm_weight=gq, k_norm_weight=gk, norm_eps=eps)
    ops.check_error(ws)
    e, bound, y, a = qknorm_exact_and_bound(x, w, b.cu_q_lens, b.seq_lens, rope_theta, gq, gk, eps)
    qg = q.float().cpu().numpy().astype(np.float64).reshape(x.shape[0], -1)
    within_tol(qg, e[:, :4096], bound[:, :4096], "normalised q")
    rel = np.sqrt(((qg - e[:, :4096]) ** 2).sum() / (e[:, :4096] ** 2).sum())
    assert rel <= 5e-3, rel
    kp = b.k_pool.view(torch.int16).cpu().numpy()
    vp = b.v_pool.view(torch.int16).cpu().numpy()
    touched = np.zeros(kp.shape[:2], dtype=bool)
    for t, (blk, slot) in enumerate(new_slots(b)):
        touched[blk, slot] = True
        kf = b.k_pool[blk, slot].double().cpu().numpy().reshape(-1)
        vf = b.v_pool[blk, slot].double().cpu().numpy().reshape(-1)
        within_tol(kf, e[t, 4096:], bound[t, 4096:], f"normalised k row of token {t}")
        within_tol(vf, y[t, 5120:], a[t, 5120:], f"v row of token {t}")
    assert np.array_equal(kp[~touched], kp0[~touched]), "k pool written outside the new slots"
    assert np.array_equal(vp[~touched], vp0[~touched]), "v pool written outside the new slots"
    return q


@pytest.mark.parametrize("rope_theta", [0.0, ops.QWEN3_ROPE_THETA])
@pytest.mark.parametrize("ctx_and_q", [
    [(0, 1)],
    [(0, 37)],                                  # 64-column tiles, 32 rows of x loaded
    [(200, 100), (0, 64), (511, 1)],            # chunks after context, a decode-like row
    [(0, 300)],                                 # CTA pairs, a ragged last tile
    [(37, 130), (1000, 0), (255, 200)],         # a sequence with no new token
    [(131000, 40), (70000, 300)],               # large positions
])
def test_qkv_append_qknorm_matches_oracle(ctx_and_q, rope_theta):
    """Qwen3's QK-norm (RMSNorm of every q and k head with its own gain, eps 1e-6) on the bf16
    projection, then the rotation, against the oracle's norm and rotation."""
    b = batch_for(ctx_and_q, seed=180 + len(ctx_and_q))
    check_qknorm_case(b, inputs(181, b.total_tokens), weights(182), rope_theta)


def test_qknorm_large_eps_and_a_zero_row():
    """eps large against the heads' mean square (0.5 of it) weighs in the result; a zero input
    row gives zero q and k heads (0 / sqrt(eps))."""
    b = batch_for([(10, 50)], seed=183)
    x = inputs(184, b.total_tokens)
    x[7] = 0
    w = weights(185)
    q = check_qknorm_case(b, x, w, ops.QWEN3_ROPE_THETA, eps=0.5)
    assert torch.count_nonzero(q[7]).item() == 0


def test_qknorm_full_prefill_chunk_sampled_rows():
    """4096 new tokens: sampled rows of q and of the cache against the oracle."""
    b = wl.causal_prefill(device="cuda")
    x = inputs(186, b.total_tokens)
    w = weights(187)
    gq, gk = norm_gains(188)
    ws = workspace_for(b)
    q = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, ws,
                             rope_theta=ops.QWEN3_ROPE_THETA, q_norm_weight=gq, k_norm_weight=gk)
    ops.check_error(ws)
    rows = [0, 1, 127, 128, 2047, 2048, 4000, 4095]
    e, bound, y, a = qknorm_exact_and_bound(x, w, b.cu_q_lens, b.seq_lens, ops.QWEN3_ROPE_THETA, gq, gk,
                                            ops.QWEN3_NORM_EPS, rows=rows)
    slots = new_slots(b)
    qg = q.float().cpu().numpy().astype(np.float64).reshape(b.total_tokens, -1)
    for r, t in enumerate(rows):
        within_tol(qg[t], e[r, :4096], bound[r, :4096], f"q row {t}")
        blk, slot = slots[t]
        kf = b.k_pool[blk, slot].double().cpu().numpy().reshape(-1)
        vf = b.v_pool[blk, slot].double().cpu().numpy().reshape(-1)
        within_tol(kf, e[r, 4096:], bound[r, 4096:], f"k row {t}")
        within_tol(vf, y[r, 5120:], a[r, 5120:], f"v row {t}")


def test_qknorm_bad_block_writes_no_kv_but_keeps_q():
    """A token whose block is outside the pool: no k or v row anywhere, its q still
    normalised and rotated, PA_ERR_DEVICE recorded."""
    b = batch_for([(0, 40), (100, 20)], seed=189)
    x = inputs(190, b.total_tokens)
    w = weights(191)
    gq, gk = norm_gains(192)
    bt = b.block_table.clone()
    bt[1, 0] = b.num_blocks + 7
    kp0, vp0 = b.k_pool.clone(), b.v_pool.clone()
    ws = workspace_for(b)
    q = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, bt, b.cu_q_lens, b.seq_lens, ws,
                             rope_theta=ops.QWEN3_ROPE_THETA, q_norm_weight=gq, k_norm_weight=gk)
    with pytest.raises(ops.PagedAttnError) as err:
        ops.check_error(ws)
    assert err.value.status == 4
    e, bound, _, _ = qknorm_exact_and_bound(x, w, b.cu_q_lens, b.seq_lens, ops.QWEN3_ROPE_THETA, gq, gk,
                                            ops.QWEN3_NORM_EPS)
    qg = q.float().cpu().numpy().astype(np.float64).reshape(b.total_tokens, -1)
    within_tol(qg, e[:, :4096], bound[:, :4096], "q")
    touched = np.zeros((b.num_blocks, 256), dtype=bool)
    for blk, slot in new_slots(b)[:40]:
        touched[blk, slot] = True
    for pool, pool0 in ((b.k_pool, kp0), (b.v_pool, vp0)):
        a = pool.view(torch.int16).cpu().numpy()
        o = pool0.view(torch.int16).cpu().numpy()
        assert np.array_equal(a[~touched], o[~touched])


def test_qknorm_rejects_bad_gains():
    b = batch_for([(0, 8)], seed=193)
    x, w = inputs(194, 8), weights(195)
    gq, gk = norm_gains(196)
    ws = workspace_for(b)
    for kw in (dict(norm_eps=-1.0), dict(norm_eps=float("nan")), dict(norm_eps=float("inf"))):
        with pytest.raises(ops.PagedAttnError) as err:
            ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, ws,
                                 q_norm_weight=gq, k_norm_weight=gk, **kw)
        assert err.value.status == 1
    with pytest.raises(ValueError):
        ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, ws, q_norm_weight=gq)


@pytest.mark.parametrize("qknorm", [False, True])
def test_inconsistent_sequence_gets_nan_q_and_no_kv(qknorm):
    """A sequence whose new tokens outnumber its length (q_len 20 > seq_len 5): its tokens get no
    K/V row anywhere and, with the rotation, NaN q rows (their positions are unknown); the other
    sequence is computed as usual; PA_ERR_DEVICE is recorded."""
    b = batch_for([(10, 30), (0, 20)], seed=197)
    x, w = inputs(198, b.total_tokens), weights(199)
    bad_lens = b.seq_lens.clone()
    bad_lens[1] = 5
    gq, gk = norm_gains(200) if qknorm else (None, None)
    kp0, vp0 = b.k_pool.clone(), b.v_pool.clone()
    ws = workspace_for(b)
    q = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, bad_lens, ws,
                             rope_theta=ops.QWEN3_ROPE_THETA, q_norm_weight=gq, k_norm_weight=gk)
    with pytest.raises(ops.PagedAttnError) as err:
        ops.check_error(ws)
    assert err.value.status == 4
    assert torch.isnan(q[30:].float()).all()
    rows = list(range(30))
    if qknorm:
        e, bound, _, _ = qknorm_exact_and_bound(x, w, b.cu_q_lens, b.seq_lens, ops.QWEN3_ROPE_THETA, gq, gk,
                                                ops.QWEN3_NORM_EPS, rows=rows)
    else:
        e, bound = exact_and_bound(x, w, b.cu_q_lens, b.seq_lens, ops.QWEN3_ROPE_THETA, rows=rows)
    qg = q[:30].float().cpu().numpy().astype(np.float64).reshape(30, -1)
    within_tol(qg, e[:, :4096], bound[:, :4096], "q of the consistent sequence")
    touched = np.zeros((b.num_blocks, 256), dtype=bool)
    for blk, slot in new_slots(b)[:30]:
        touched[blk, slot] = True
    for pool, pool0 in ((b.k_pool, kp0), (b.v_pool, vp0)):
        a = pool.view(torch.int16).cpu().numpy()
        o = pool0.view(torch.int16).cpu().numpy()
        assert np.array_equal(a[~touched], o[~touched])


# ------------------------------------------------------------------ whole tensors at full size

@pytest.fixture(scope="module")
def full_chunk():
    """The 4096-token prompt of the causal prefill workload (the benchmark's projection): inputs
    and the oracle's exact projection of every row, computed once for the tests below."""
    b = wl.causal_prefill(device="cuda")
    x, w = inputs(66, b.total_tokens), weights(67)
    return b, x, w, (oracle.qkv_project(x.cpu(), w.cpu()), abs_sums(x, w))


def cache_rows(b, pool):
    """The new tokens' rows of a pool, [tokens, 8 * 128] float64, in token order."""
    blk, slot = (torch.tensor(v, device=pool.device) for v in zip(*new_slots(b)))
    return pool[blk, slot].double().cpu().numpy().reshape(len(blk), -1)


@pytest.mark.parametrize("qknorm", [False, True])
def test_full_prefill_chunk_whole_tensors(full_chunk, qknorm):
    """Every element of q and of the appended k and v rows for all 4096 new tokens, with Qwen3's
    rotary embedding (and, in the second case, its QK-norm), against the oracle."""
    b0, x, w, projected = full_chunk
    b = wl.causal_prefill(device="cuda")          # fresh pools for each case
    ws = workspace_for(b)
    if qknorm:
        gq, gk = norm_gains(201)
        q = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, ws,
                                 rope_theta=ops.QWEN3_ROPE_THETA, q_norm_weight=gq, k_norm_weight=gk)
        e, bound, y, a = qknorm_exact_and_bound(x, w, b.cu_q_lens, b.seq_lens, ops.QWEN3_ROPE_THETA, gq, gk,
                                                ops.QWEN3_NORM_EPS, projected=projected)
        k_exact, k_bound = e[:, 4096:], bound[:, 4096:]
    else:
        q = ops.paged_qkv_append(x, w, b.k_pool, b.v_pool, b.block_table, b.cu_q_lens, b.seq_lens, ws,
                                 rope_theta=ops.QWEN3_ROPE_THETA)
        e, bound = exact_and_bound(x, w, b.cu_q_lens, b.seq_lens, ops.QWEN3_ROPE_THETA, projected=projected)
        y, a = projected
        k_exact, k_bound = e[:, 4096:5120], bound[:, 4096:5120]
    ops.check_error(ws)
    qg = q.float().cpu().numpy().astype(np.float64).reshape(b.total_tokens, -1)
    within_tol(qg, e[:, :4096], bound[:, :4096], "q")
    rel = np.sqrt(((qg - e[:, :4096]) ** 2).sum() / (e[:, :4096] ** 2).sum())
    assert rel <= 5e-3, rel
    within_tol(cache_rows(b, b.k_pool), k_exact, k_bound, "k rows in the cache")
    within_tol(cache_rows(b, b.v_pool), y[:, 5120:], a[:, 5120:], "v rows in the cache")

