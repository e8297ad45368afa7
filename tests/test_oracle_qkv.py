"""Pins of the oracle's merged Q/K/V projection (page "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎，
C++/CUDA 实现性能追平 98%" §4.4.3 QKV fusion) and of its append into the cache.

The projection is checked against integer arithmetic (exact), an independent fp64 matrix
product, selection weights that copy chosen input columns (which fixes the slicing into q,
k and v and the placement of k and v in the cache), and the bf16 rounding against torch
and a brute-force nearest-even search.
"""
import numpy as np
import torch

import oracle
from oracle_cases import bf16_is_nearest_even, bf16_probe_values, qkv_integer_case

N_OUT = 32 * 128 + 2 * 8 * 128


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_integer_inputs_give_the_exact_product():
    x, w = qkv_integer_case(seed=41, tokens=9, hidden=128, n_out=70)
    y = oracle.qkv_project(x, w)
    exact = x.double().numpy().astype(np.int64) @ w.double().numpy().astype(np.int64).T
    assert np.array_equal(y, exact.astype(np.float64))


def test_matches_an_independent_fp64_product():
    g = torch.Generator().manual_seed(42)
    x = torch.randn(11, 256, generator=g).to(torch.bfloat16)
    w = (torch.randn(96, 256, generator=g) / 16).to(torch.bfloat16)
    y = oracle.qkv_project(x, w)
    ref = x.double().numpy() @ w.double().numpy().T
    assert np.allclose(y, ref, rtol=1e-14, atol=1e-13)


def test_row_subset():
    x, w = qkv_integer_case(seed=43, tokens=12)
    full = oracle.qkv_project(x, w)
    assert np.array_equal(oracle.qkv_project(x, w, rows=[11, 3, 3, 0]), full[[11, 3, 3, 0]])


def test_bf16_rounding_matches_torch_and_is_nearest_even():
    v = bf16_probe_values()
    ref = bits(torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16))
    got = oracle.bf16_round(v)
    assert np.array_equal(got, ref)
    assert bf16_is_nearest_even(v, got)
    # doubles that are not fp32 values (a double rounding through fp32 could differ)
    g = np.random.default_rng(44)
    d = g.standard_normal(5000) * np.exp2(g.uniform(-130, 126, 5000))
    assert bf16_is_nearest_even(d, oracle.bf16_round(d))
    assert oracle.bf16_round(np.array([np.nan]))[0] & 0x7FFF > 0x7F80            # NaN stays NaN
    assert list(oracle.bf16_round(np.array([1e39, -1e39]))) == [0x7F80, 0xFF80]   # overflow to inf


def selection_weights(hidden, seed):
    """w whose row n is the unit vector of input column sel[n]: y[t][n] = x[t][sel[n]] exactly."""
    sel = np.random.default_rng(seed).integers(0, hidden, N_OUT)
    w = np.zeros((N_OUT, hidden), dtype=np.float32)
    w[np.arange(N_OUT), sel] = 1.0
    return torch.from_numpy(w).to(torch.bfloat16), sel


def test_append_slices_q_k_v_and_places_them_by_position():
    hidden, bs, nb = 64, 256, 6
    g = torch.Generator().manual_seed(45)
    x = torch.randn(7, hidden, generator=g).to(torch.bfloat16)
    w, sel = selection_weights(hidden, 46)
    kpool = torch.randn(nb, bs, 8, 128, generator=g).to(torch.bfloat16)
    vpool = torch.randn(nb, bs, 8, 128, generator=g).to(torch.bfloat16)
    bt = torch.tensor([[4, 1, 0], [2, 5, -1]], dtype=torch.int32)
    cu = torch.tensor([0, 5, 7], dtype=torch.int32)
    sl = torch.tensor([258, 300], dtype=torch.int32)      # sequence 0 crosses a block edge
    q, kp, vp = oracle.qkv_append(x, w, kpool, vpool, bt, cu, sl)
    xb = x.double().numpy()
    assert np.array_equal(q.reshape(7, -1), xb[:, sel[:4096]])
    ek, ev = bits(kpool).copy(), bits(vpool).copy()
    xbits = bits(x)
    for t in range(7):
        s = 0 if t < 5 else 1
        i = t - int(cu[s])
        p = int(sl[s]) - (int(cu[s + 1]) - int(cu[s])) + i
        blk, slot = int(bt[s, p // bs]), p % bs
        ek[blk, slot] = xbits[t, sel[4096:5120]].reshape(8, 128)
        ev[blk, slot] = xbits[t, sel[5120:]].reshape(8, 128)
    assert np.array_equal(kp, ek)
    assert np.array_equal(vp, ev)


def test_append_rounds_k_and_v_once_to_bf16():
    g = torch.Generator().manual_seed(47)
    x = torch.randn(3, 128, generator=g).to(torch.bfloat16)
    w = (torch.randn(N_OUT, 128, generator=g) / 11).to(torch.bfloat16)
    kpool = torch.zeros(2, 256, 8, 128, dtype=torch.bfloat16)
    vpool = torch.zeros_like(kpool)
    bt = torch.tensor([[1]], dtype=torch.int32)
    q, kp, vp = oracle.qkv_append(x, w, kpool, vpool, bt, torch.tensor([0, 3], dtype=torch.int32),
                                  torch.tensor([3], dtype=torch.int32))
    y = x.double().numpy() @ w.double().numpy().T
    assert np.allclose(q.reshape(3, -1), y[:, :4096], rtol=1e-14, atol=1e-13)
    for t in range(3):
        assert bf16_is_nearest_even(y[t, 4096:5120], kp[1, t].reshape(-1))
        assert bf16_is_nearest_even(y[t, 5120:], vp[1, t].reshape(-1))
    assert not kp[0].any() and not kp[1, 3:].any()       # nothing else written
