"""Pins of the oracle's per-head RMS normalisation of q and k (QK-norm) and of its place in
the projection.

The pages do not define it; the definition taken is Qwen3's QK-norm: RMSNorm (Zhang and
Sennrich, 2019, §3) of every 128-dim q and k head, y = g * x / sqrt(mean(x^2) + eps), with a
learned gain g per dim (one for q heads, one for k heads) and eps = 1e-6 (Qwen3's
configuration), applied to the projection's bf16 output before the rotary embedding.  The
pins check it against torch's own ``rms_norm`` and against what the definition fixes without
retracing the oracle's loop: a unit gain leaves a mean square of ms / (ms + eps); without eps
the result does not depend on the head's scale; a constant head maps to a / sqrt(a^2 + eps);
the gain acts per dim; heads do not mix.  In the projection: at position 0 q and k are the
normalised bf16 projection, elsewhere turning them back by the token's angle recovers it
(normalised first, rotated second), and v is untouched.
"""
import numpy as np
import torch

import oracle

D = 128


def heads(seed, n, h=1, scale_spread=0.0):
    g = np.random.default_rng(seed)
    y = g.standard_normal((n, h * D))
    if scale_spread:
        y *= np.exp2(g.uniform(-scale_spread, scale_spread, (n, h)).repeat(D, axis=1))
    return y


def gain(seed, d=D):
    g = torch.Generator().manual_seed(seed)
    return (1.0 + 0.5 * torch.randn(d, generator=g)).to(torch.bfloat16)


def unit_gain(d=D):
    return torch.ones(d, dtype=torch.bfloat16)


def test_matches_torch_rms_norm():
    for eps in (0.0, 1e-6, 0.25):
        y = heads(1, 9, h=3, scale_spread=20.0)
        g = gain(2)
        got = oracle.rms_norm_heads(y, g, eps, n_heads=3)
        ref = torch.nn.functional.rms_norm(torch.from_numpy(y).view(9, 3, D), (D,), weight=g.double(),
                                           eps=eps).reshape(9, 3 * D).numpy()
        assert np.allclose(got, ref, rtol=1e-13, atol=0), eps


def test_worked_example():
    # x = (3, 4), unit gain, no eps: the root mean square is sqrt(12.5)
    got = oracle.rms_norm_heads(np.array([[3.0, 4.0]]), unit_gain(2), 0.0, head_dim=2)
    assert np.allclose(got, [[0.848528137423857, 1.131370849898476]], rtol=1e-14, atol=0)


def test_unit_gain_leaves_mean_square_ms_over_ms_plus_eps():
    y = heads(3, 6, h=2, scale_spread=4.0)
    eps = 1e-2
    got = oracle.rms_norm_heads(y, unit_gain(), eps, n_heads=2)
    for h in range(2):
        ms = (y[:, h * D:(h + 1) * D] ** 2).mean(axis=1)
        out_ms = (got[:, h * D:(h + 1) * D] ** 2).mean(axis=1)
        assert np.allclose(out_ms, ms / (ms + eps), rtol=1e-13, atol=0)


def test_without_eps_the_scale_of_a_head_does_not_matter():
    y = heads(4, 5)
    g = gain(5)
    base = oracle.rms_norm_heads(y, g, 0.0)
    for c in (2.0 ** -40, 3.0, 1e30):
        assert np.allclose(oracle.rms_norm_heads(c * y, g, 0.0), base, rtol=1e-13, atol=0)
    assert np.allclose(oracle.rms_norm_heads(-y, g, 0.0), -base, rtol=1e-13, atol=0)


def test_constant_head_and_zero_head():
    eps = 1e-6
    for a in (1e-4, 0.5, -7.0):
        got = oracle.rms_norm_heads(np.full((1, D), a), unit_gain(), eps)
        assert np.allclose(got, a / np.sqrt(a * a + eps), rtol=1e-14, atol=0)
    assert np.array_equal(oracle.rms_norm_heads(np.zeros((2, D)), gain(6), eps), np.zeros((2, D)))


def test_gain_acts_per_dim():
    y = heads(7, 3)
    rms = np.sqrt((y ** 2).mean(axis=1) + 1e-6)
    for d in (0, 1, 63, 64, 127):
        g = torch.zeros(D, dtype=torch.bfloat16)
        g[d] = 2.5
        got = oracle.rms_norm_heads(y, g, 1e-6)
        expect = np.zeros_like(y)
        expect[:, d] = 2.5 * y[:, d] / rms
        assert np.allclose(got, expect, rtol=1e-14, atol=0), d


def test_heads_are_normalised_each_on_its_own():
    y = heads(8, 4, h=2)
    wide = np.concatenate([np.full((4, 5), 9.0), y, np.full((4, 3), -2.0)], axis=1)
    g = gain(9)
    got = oracle.rms_norm_heads(wide, g, 1e-6, first_col=5, n_heads=2)
    assert np.array_equal(got[:, :5], wide[:, :5]) and np.array_equal(got[:, -3:], wide[:, -3:])
    alone = oracle.rms_norm_heads(y[:, D:], g, 1e-6)
    assert np.array_equal(got[:, 5 + D:5 + 2 * D], alone)
    y2 = y.copy()
    y2[:, D:] *= 1000.0                       # the second head's size leaves the first head alone
    got2 = oracle.rms_norm_heads(y2, g, 1e-6, n_heads=2)
    assert np.array_equal(got2[:, :D], got[:, 5:5 + D])


def test_input_checks():
    y = heads(10, 2)
    for bad in (dict(first_col=1), dict(n_heads=2)):
        try:
            oracle.rms_norm_heads(y, unit_gain(), 1e-6, **bad)
        except ValueError:
            continue
        raise AssertionError(bad)


# ------------------------------------------------------------------ inside the projection

def projection_case(seed, ctx_and_q, hidden=256):
    g = torch.Generator().manual_seed(seed)
    seq_lens = [c + q for c, q in ctx_and_q]
    q_lens = [q for _, q in ctx_and_q]
    t = sum(q_lens)
    x = torch.randn(t, hidden, generator=g).to(torch.bfloat16)
    w = (torch.randn(6144, hidden, generator=g) / 16.0).to(torch.bfloat16)
    nblk = [(s + 255) // 256 for s in seq_lens]
    perm = torch.randperm(sum(nblk) + 2, generator=g).to(torch.int32)
    bt = torch.full((len(seq_lens), max(nblk)), -1, dtype=torch.int32)
    o = 0
    for s, n in enumerate(nblk):
        bt[s, :n] = perm[o:o + n]
        o += n
    pools = [torch.randn(sum(nblk) + 2, 256, 8, D, generator=g).to(torch.bfloat16) for _ in range(2)]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(q_lens)]), dtype=torch.int32)
    return x, w, pools, bt, cu, torch.tensor(seq_lens, dtype=torch.int32)


def bf16_projection(x, w):
    y = oracle.qkv_project(x, w)
    return torch.from_numpy(y).to(torch.bfloat16).double().numpy()      # round to nearest even


def cache_rows(pool, bt, cu, sl):
    bt, cu, sl = bt.numpy(), cu.numpy(), sl.numpy()
    out = []
    for s in range(len(sl)):
        q_len = cu[s + 1] - cu[s]
        for i in range(q_len):
            p = sl[s] - q_len + i
            out.append(pool[bt[s, p // 256], p % 256].double().numpy().reshape(-1))
    return np.array(out)


def torch_norm(v, g, n_heads, eps=1e-6):
    t = torch.from_numpy(v).view(v.shape[0], n_heads, D)
    return torch.nn.functional.rms_norm(t, (D,), weight=g.double(), eps=eps).reshape(v.shape[0], -1).numpy()


def test_projection_normalises_q_and_k_at_position_zero():
    x, w, (kp, vp), bt, cu, sl = projection_case(11, [(0, 1), (0, 1), (0, 1)])
    gq, gk = gain(12), gain(13)
    q, kp2, vp2 = oracle.qkv_append(x, w, kp, vp, bt, cu, sl, rope_theta=1e6, q_norm=gq, k_norm=gk)
    y = bf16_projection(x, w)
    assert np.allclose(q.reshape(3, -1), torch_norm(y[:, :4096], gq, 32), rtol=1e-13, atol=0)
    k_rows = cache_rows(torch.from_numpy(kp2).view(torch.bfloat16), bt, cu, sl)
    k_ref = torch.from_numpy(torch_norm(y[:, 4096:5120], gk, 8)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(k_rows, k_ref)
    v_rows = cache_rows(torch.from_numpy(vp2).view(torch.bfloat16), bt, cu, sl)
    assert np.array_equal(v_rows, y[:, 5120:])


def test_projection_normalises_before_it_rotates():
    x, w, (kp, vp), bt, cu, sl = projection_case(14, [(300, 5), (0, 4)])
    gq, gk = gain(15), gain(16)
    q, _, _ = oracle.qkv_append(x, w, kp, vp, bt, cu, sl, rope_theta=1e6, q_norm=gq, k_norm=gk)
    pos = oracle.token_positions(cu, sl)
    back = oracle.rope(q.reshape(len(pos), -1), -pos, 1e6, n_heads=32)       # turn back by each angle
    y = bf16_projection(x, w)
    assert np.allclose(back, torch_norm(y[:, :4096], gq, 32), rtol=0, atol=1e-12)
    # the other order gives another result (the gains differ between the dims of a pair)
    other = oracle.rope(y[:, :4096], pos, 1e6, n_heads=32)
    other = torch_norm(other, gq, 32)
    assert not np.allclose(q.reshape(len(pos), -1), other, rtol=0, atol=1e-6)


def test_projection_without_norm_is_unchanged():
    x, w, (kp, vp), bt, cu, sl = projection_case(17, [(10, 3)])
    q0, k0, v0 = oracle.qkv_append(x, w, kp, vp, bt, cu, sl, rope_theta=1e6)
    y = oracle.qkv_project(x, w)
    pos = oracle.token_positions(cu, sl)
    assert np.array_equal(q0.reshape(3, -1), oracle.rope(y[:, :4096], pos, 1e6, n_heads=32))
