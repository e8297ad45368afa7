"""Pins of the oracle's rotary position embedding and of the token positions it uses.

The pages do not define a position encoding; the definition taken is RoFormer's (Su et al.,
2021) in the rotate-half pairing of Qwen3 and the Llama family: dims i and i + 64 of a
128-dim head form a pair, turned by p * theta^(-i/64) at position p (Qwen3: theta = 1e6).
The pins check what that definition fixes without retracing the oracle's loop: position 0
is the identity; every pair keeps its length; q.k after rotation depends only on the
difference of the positions; rotations compose; the angle of pair i read back with atan2
is the pair's own frequency times p (so the pairing, the sign and the exponent are fixed);
and each pair equals complex multiplication by e^{i p w} (numpy's complex exponential).
"""
import numpy as np
import torch

import oracle

THETA = 1.0e6
D = 128


def rows(seed, n, heads=1):
    return np.random.default_rng(seed).standard_normal((n, heads * D))


def test_position_zero_is_the_identity():
    y = rows(1, 5, heads=3)
    r = oracle.rope(y, [0] * 5, THETA, n_heads=3)
    assert np.array_equal(r, y)


def test_every_pair_keeps_its_length():
    y = rows(2, 7, heads=2)
    pos = [1, 17, 255, 256, 4095, 32767, 1000003]
    r = oracle.rope(y, pos, THETA, n_heads=2)
    for h in range(2):
        a, b = y[:, h * D:h * D + 64], y[:, h * D + 64:(h + 1) * D]
        ra, rb = r[:, h * D:h * D + 64], r[:, h * D + 64:(h + 1) * D]
        assert np.allclose(ra ** 2 + rb ** 2, a ** 2 + b ** 2, rtol=1e-12, atol=0)


def test_dot_products_depend_only_on_the_position_difference():
    q, k = rows(3, 1), rows(4, 1)
    base = None
    for m, n in ((10, 3), (107, 100), (5007, 5000), (70007, 70000)):
        rq = oracle.rope(q, [m], THETA)
        rk = oracle.rope(k, [n], THETA)
        d = float(rq[0] @ rk[0])
        base = d if base is None else base
        assert abs(d - base) <= 1e-10 * abs(base)
    # and it does change with the difference
    assert abs(float(oracle.rope(q, [11], THETA)[0] @ oracle.rope(k, [3], THETA)[0]) - base) > 1e-6


def test_rotations_compose():
    y = rows(5, 4)
    a, b = [3, 90, 4000, 12345], [5, 1, 60000, 7]
    twice = oracle.rope(oracle.rope(y, a, THETA), b, THETA)
    once = oracle.rope(y, [x + z for x, z in zip(a, b)], THETA)
    assert np.allclose(twice, once, rtol=0, atol=1e-10)


def test_pair_i_turns_by_its_own_frequency():
    """A unit vector in dim i at position 1 moves within the pair (i, i + 64) only, by the
    angle theta^(-i/64) (counter-clockwise: dim i + 64 gains +sin)."""
    for i in (0, 1, 31, 32, 63):
        y = np.zeros((1, D))
        y[0, i] = 1.0
        r = oracle.rope(y, [1], THETA)[0]
        others = np.delete(r, [i, i + 64])
        assert np.all(others == 0.0)
        ang = np.arctan2(r[i + 64], r[i])
        assert abs(ang - THETA ** (-i / 64)) <= 1e-15
    # pair 32 at position 1000: 1e6^(-1/2) * 1000 = 1 radian exactly
    y = np.zeros((1, D))
    y[0, 32] = 1.0
    r = oracle.rope(y, [1000], THETA)[0]
    assert abs(np.arctan2(r[96], r[32]) - 1.0) <= 1e-12


def test_equals_complex_multiplication():
    y = rows(6, 6, heads=2)
    pos = np.array([0, 1, 2, 511, 4096, 32769])
    r = oracle.rope(y, pos, THETA, n_heads=2)
    w = THETA ** (-np.arange(64) / 64.0)
    # numpy's vectorised power may differ from libm's in the last bit of a frequency; the
    # position multiplies that into the angle, so the bound grows with p
    tol = 1e-14 * (1.0 + pos[:, None])
    for h in range(2):
        z = y[:, h * D:h * D + 64] + 1j * y[:, h * D + 64:(h + 1) * D]
        zr = z * np.exp(1j * pos[:, None] * w[None, :])
        assert np.all(np.abs(r[:, h * D:h * D + 64] - zr.real) <= tol)
        assert np.all(np.abs(r[:, h * D + 64:(h + 1) * D] - zr.imag) <= tol)


def test_columns_outside_the_rotated_heads_are_untouched():
    y = rows(7, 3, heads=4)
    r = oracle.rope(y, [9, 99, 999], THETA, first_col=D, n_heads=2)
    assert np.array_equal(r[:, :D], y[:, :D]) and np.array_equal(r[:, 3 * D:], y[:, 3 * D:])
    assert not np.array_equal(r[:, D:3 * D], y[:, D:3 * D])


def test_token_positions_are_absolute():
    # decode rows, a chunk after a context of 700, a prompt from position 0, an empty sequence
    cu = [0, 1, 2, 6, 9, 9]
    sl = [1, 513, 704, 3, 40]
    assert oracle.token_positions(cu, sl).tolist() == [0, 512, 700, 701, 702, 703, 0, 1, 2]


def test_qkv_append_rotates_q_and_k_at_the_token_positions_and_leaves_v():
    """qkv_append = the projection (pinned on its own), then the rotation of the q and k heads
    at each token's absolute position, k and v rounded once into their cache slots."""
    hidden, tokens = 256, 5
    g = torch.Generator().manual_seed(8)
    x = torch.randn(tokens, hidden, generator=g).to(torch.bfloat16)
    w = (torch.randn(6144, hidden, generator=g) / 16).to(torch.bfloat16)
    nb, bs = 6, 256
    kp = torch.zeros(nb, bs, 8, D, dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    bt = torch.tensor([[4, 1], [0, -1]], dtype=torch.int32)
    cu = torch.tensor([0, 3, 5], dtype=torch.int32)
    sl = torch.tensor([300, 2], dtype=torch.int32)          # positions 297, 298, 299 | 0, 1
    y = oracle.qkv_project(x, w)
    pos = [297, 298, 299, 0, 1]
    q, kc, vc = oracle.qkv_append(x, w, kp, vp, bt, cu, sl, rope_theta=THETA)
    q0, _, _ = oracle.qkv_append(x, w, kp, vp, bt, cu, sl)
    exp_q = oracle.rope(y[:, :4096], pos, THETA, n_heads=32).reshape(tokens, 32, D)
    assert np.array_equal(q, exp_q)
    assert np.array_equal(q0, y[:, :4096].reshape(tokens, 32, D))
    exp_k = oracle.bf16_round(oracle.rope(y[:, 4096:5120], pos, THETA, n_heads=8)).reshape(tokens, 8, D)
    exp_v = oracle.bf16_round(y[:, 5120:]).reshape(tokens, 8, D)
    slots = [(1, 41), (1, 42), (1, 43), (0, 0), (0, 1)]   # table entry p // 256, slot p % 256
    for t, (b, s) in enumerate(slots):
        assert np.array_equal(kc[b, s], exp_k[t]) and np.array_equal(vc[b, s], exp_v[t])
