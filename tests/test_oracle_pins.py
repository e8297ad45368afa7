"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics, not by the oracle.

Each pin is chosen so that a plausible slip in the oracle fails at least one of them:
  * closed forms: one key returns its V row exactly; identical keys return the mean
    of V; adding one vector to every key leaves the output unchanged; linearity in V;
  * a library routine: torch's scaled_dot_product_attention in float64 on tiny cases
    (causal, chunked with a bottom-right mask, several sequences, real head shapes),
    fed contiguous K/V that the test scatters into the paged pool itself;
  * invariants: GQA equals MHA with every KV head repeated; paged equals contiguous;
    block placement does not matter; decode equals the matching prefill row; a chunked
    prefill equals the unchunked one;
  * a 60-digit brute force on a tiny input;
  * the sizing example printed in §2.3 of the page
    "从零手搓AI推理引擎：避开调包陷阱的工程实践指南" (golden fixture).
``test_oracle_mutants.py`` plants mistakes in copies of the oracle and checks these pins
catch them.
"""
import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle
from oracle_cases import make_case, run_oracle, sdpa_lse, sdpa_reference
from paged_gqa_attention_gb300 import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


# ----------------------------------------------------------------- closed forms

def test_single_key_returns_v_exactly():
    c = make_case([1], [1], seed=1)
    out, lse = run_oracle(c, 0.25)
    v = c["v"][0].double().numpy()                   # [1, Hkv, D]
    rep = c["hq"] // c["hkv"]
    for h in range(c["hq"]):
        assert np.array_equal(out[0, h], v[0, h // rep])
    # lse of a single score is the score itself
    q = c["q"][0].double().numpy()
    k = c["k"][0].double().numpy()[0]
    for h in range(c["hq"]):
        assert lse[0, h] == pytest.approx(0.25 * float(q[h] @ k[h // rep]), rel=1e-14, abs=1e-14)


def test_identical_keys_give_mean_of_v():
    c = make_case([7], [1], seed=2)
    k0 = c["k"][0][0].clone()                       # [Hkv, D]
    for j in range(c["bt"].shape[1]):
        b = int(c["bt"][0, j])
        if b >= 0:
            c["k_pool"][b, :min(c["bs"], 7 - j * c["bs"])] = k0
    scale = 1.0 / math.sqrt(c["d"])
    out, lse = run_oracle(c, scale)
    v = c["v"][0].double().numpy()
    rep = c["hq"] // c["hkv"]
    for h in range(c["hq"]):
        np.testing.assert_allclose(out[0, h], v[:, h // rep].mean(0), rtol=0, atol=1e-14)
        score = float(c["q"][0, h].double() @ k0[h // rep].double()) * scale
        assert lse[0, h] == pytest.approx(score + math.log(7), rel=1e-13)


def test_key_shift_invariance():
    """Adding one vector c to every key adds q.c to every score of a row: the output of
    the row is unchanged and its lse moves by scale * q.c."""
    g = torch.Generator().manual_seed(3)
    bs, hkv, hq, d, sl = 4, 1, 2, 8, 9
    # small integers / 8 keep every bf16 sum exact
    k = (torch.randint(-8, 8, (sl, hkv, d), generator=g).float() / 8).to(torch.bfloat16)
    shift = (torch.randint(-8, 8, (1, hkv, d), generator=g).float() / 8).to(torch.bfloat16)
    v = torch.randn(sl, hkv, d, generator=g).to(torch.bfloat16)
    q = (torch.randint(-4, 4, (1, hq, d), generator=g).float() / 4).to(torch.bfloat16)
    bt = torch.tensor([[2, 0, 1]], dtype=torch.int32)

    def pool(x):
        p = torch.zeros(3, bs, hkv, d, dtype=torch.bfloat16)
        for j in range(sl):
            p[bt[0, j // bs], j % bs] = x[j]
        return p

    ks = (k.float() + shift.float()).to(torch.bfloat16)
    assert torch.equal(ks.float(), k.float() + shift.float())
    args = (torch.tensor([0, 1], dtype=torch.int32), torch.tensor([sl], dtype=torch.int32))
    o1, l1 = oracle.attention(q, pool(k), pool(v), bt, *args, scale=0.5)
    o2, l2 = oracle.attention(q, pool(ks), pool(v), bt, *args, scale=0.5)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    for h in range(hq):
        qc = float(q[0, h].double() @ shift[0, 0].double())
        assert l2[0, h] - l1[0, h] == pytest.approx(0.5 * qc, abs=1e-12)


def test_linearity_in_v():
    c = make_case([11, 5], [3, 1], seed=4)
    scale = 0.3
    out1, _ = run_oracle(c, scale)
    g = torch.Generator().manual_seed(5)
    v2 = (torch.randint(-4, 4, c["v_pool"].shape, generator=g).float() / 4).to(torch.bfloat16)
    v1 = (torch.randint(-4, 4, c["v_pool"].shape, generator=g).float() / 4).to(torch.bfloat16)
    combo = (2 * v1.float() - 3 * v2.float()).to(torch.bfloat16)   # exact in bf16
    assert torch.equal(combo.float(), 2 * v1.float() - 3 * v2.float())
    a = oracle.attention(c["q"], c["k_pool"], v1, c["bt"], c["cu"], c["seq_lens"], scale=scale)[0]
    b = oracle.attention(c["q"], c["k_pool"], v2, c["bt"], c["cu"], c["seq_lens"], scale=scale)[0]
    ab = oracle.attention(c["q"], c["k_pool"], combo, c["bt"], c["cu"], c["seq_lens"],
                          scale=scale)[0]
    np.testing.assert_allclose(ab, 2 * a - 3 * b, rtol=0, atol=1e-12)


# ----------------------------------------------------------------- library routine

@pytest.mark.parametrize("seq_lens,q_lens", [
    ([1], [1]),                 # decode with a single key
    ([13], [1]),                # decode
    ([9, 1, 17], [1, 1, 1]),    # batched decode, ragged
    ([16], [16]),               # unchunked causal prefill
    ([21], [6]),                # chunk after a context of 15
    ([10, 7, 19], [10, 3, 5]),  # several sequences: prefill + chunks
])
def test_matches_torch_sdpa_tiny(seq_lens, q_lens):
    c = make_case(seq_lens, q_lens, seed=sum(seq_lens) + len(q_lens))
    scale = 1.0 / math.sqrt(c["d"])
    out, lse = run_oracle(c, scale)
    np.testing.assert_allclose(out, sdpa_reference(c, scale), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, sdpa_lse(c, scale), rtol=1e-13, atol=1e-12)


@pytest.mark.parametrize("seq_len,q_len", [(255, 1), (256, 1), (257, 1), (511, 4), (512, 1),
                                           (513, 3)])
def test_matches_torch_sdpa_real_heads_block_edges(seq_len, q_len):
    """Real head shape (32 q / 8 kv heads, dim 128, 256-token blocks) at block-edge lengths."""
    c = make_case([seq_len], [q_len], hq=32, hkv=8, d=128, bs=256, extra_blocks=2,
                  seed=seq_len)
    scale = 1.0 / math.sqrt(128)
    out, lse = run_oracle(c, scale)
    np.testing.assert_allclose(out, sdpa_reference(c, scale), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, sdpa_lse(c, scale), rtol=1e-13, atol=1e-12)


# ----------------------------------------------------------------- invariants

def test_gqa_equals_mha_with_repeated_kv():
    c = make_case([12, 6], [4, 1], hq=8, hkv=2, seed=6)
    scale = 0.2
    out, lse = run_oracle(c, scale)
    rep = c["hq"] // c["hkv"]
    kp = c["k_pool"].repeat_interleave(rep, dim=2).contiguous()
    vp = c["v_pool"].repeat_interleave(rep, dim=2).contiguous()
    out2, lse2 = oracle.attention(c["q"], kp, vp, c["bt"], c["cu"], c["seq_lens"], scale=scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_paged_equals_contiguous_and_placement_free():
    c = make_case([14, 9], [5, 1], seed=7)
    scale = 0.25
    out, lse = run_oracle(c, scale)
    # contiguous layout: the identity table over per-sequence block runs
    bs = c["bs"]
    rows, blocks_k, blocks_v = [], [], []
    for s, sl in enumerate([14, 9]):
        n = (sl + bs - 1) // bs
        row = list(range(len(blocks_k), len(blocks_k) + n))
        rows.append(row + [-1] * (c["bt"].shape[1] - n))
        kk = torch.zeros(n * bs, c["hkv"], c["d"], dtype=torch.bfloat16)
        vv = torch.zeros_like(kk)
        kk[:sl] = c["k"][s]
        vv[:sl] = c["v"][s]
        blocks_k += list(kk.view(n, bs, c["hkv"], c["d"]))
        blocks_v += list(vv.view(n, bs, c["hkv"], c["d"]))
    kp = torch.stack(blocks_k)
    vp = torch.stack(blocks_v)
    bt = torch.tensor(rows, dtype=torch.int32)
    out2, lse2 = oracle.attention(c["q"], kp, vp, bt, c["cu"], c["seq_lens"], scale=scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_decode_equals_matching_prefill_row():
    c = make_case([20], [20], seed=8)
    scale = 0.25
    out, lse = run_oracle(c, scale)
    for p in (0, 7, 19):
        o, l = oracle.attention(c["q"][p:p + 1], c["k_pool"], c["v_pool"], c["bt"],
                                torch.tensor([0, 1], dtype=torch.int32),
                                torch.tensor([p + 1], dtype=torch.int32), scale=scale)
        assert np.array_equal(o[0], out[p]) and np.array_equal(l[0], lse[p])


def test_chunked_equals_unchunked():
    c = make_case([24], [24], seed=9)
    scale = 0.25
    out, lse = run_oracle(c, scale)
    pieces = []
    for lo, hi in ((0, 8), (8, 13), (13, 24)):
        o, l = oracle.attention(c["q"][lo:hi], c["k_pool"], c["v_pool"], c["bt"],
                                torch.tensor([0, hi - lo], dtype=torch.int32),
                                torch.tensor([hi], dtype=torch.int32), scale=scale)
        pieces.append(o)
    assert np.array_equal(np.concatenate(pieces), out)


def test_rows_api_matches_full():
    c = make_case([10, 6], [4, 1], seed=10)
    out, lse = run_oracle(c, 0.3)
    toks = [0, 3, 4, 2]
    heads = [1, 3, 0, 2]
    o, l = oracle.attention(c["q"], c["k_pool"], c["v_pool"], c["bt"], c["cu"], c["seq_lens"],
                            scale=0.3, rows=(toks, heads))
    for r, (t, h) in enumerate(zip(toks, heads)):
        assert np.array_equal(o[r], out[t, h]) and l[r] == lse[t, h]


# ----------------------------------------------------------------- brute force

def test_brute_force_60_digits():
    """softmax(q.k * scale) V evaluated term by term with 60-digit decimals."""
    getcontext().prec = 60
    c = make_case([3, 2], [2, 1], hq=2, hkv=1, d=4, bs=2, seed=11)
    scale = 0.7
    out, lse = run_oracle(c, scale)
    t = 0
    for s, (sl, ql) in enumerate(zip([3, 2], [2, 1])):
        for i in range(ql):
            p = sl - ql + i
            for h in range(2):
                q = [Decimal(float(x)) for x in c["q"][t, h].float()]
                xs = []
                for j in range(p + 1):
                    k = [Decimal(float(x)) for x in c["k"][s][j, 0].float()]
                    xs.append(Decimal(scale) * sum(a * b for a, b in zip(q, k)))
                m = max(xs)
                ws = [(x - m).exp() for x in xs]
                z = sum(ws)
                for dd in range(4):
                    num = sum(w * Decimal(float(c["v"][s][j, 0, dd])) for j, w in enumerate(ws))
                    assert abs(float(num / z) - out[t, h, dd]) <= 1e-14
                assert abs(float(m + z.ln()) - lse[t, h]) <= 1e-14
            t += 1


# ----------------------------------------------------------------- kv append

def test_kv_append_places_rows_and_leaves_the_rest():
    bs, hkv, d = 4, 2, 8
    g = torch.Generator().manual_seed(12)
    num_blocks = 6
    k_pool = torch.randn(num_blocks, bs, hkv, d, generator=g).to(torch.bfloat16)
    v_pool = torch.randn(num_blocks, bs, hkv, d, generator=g).to(torch.bfloat16)
    # seq 0: context 3 then 6 new tokens (crosses two block edges); seq 1: 1 new token at 4
    seq_lens = [9, 5]
    q_lens = [6, 1]
    bt = torch.tensor([[5, 2, 0], [3, 1, -1]], dtype=torch.int32)
    k_new = torch.randn(7, hkv, d, generator=g).to(torch.bfloat16)
    v_new = torch.randn(7, hkv, d, generator=g).to(torch.bfloat16)
    cu = torch.tensor([0, 6, 7], dtype=torch.int32)
    kp, vp = oracle.kv_append(k_pool, v_pool, k_new, v_new, bt, cu,
                              torch.tensor(seq_lens, dtype=torch.int32), block_size=bs)
    exp_k = k_pool.view(torch.int16).numpy().view(np.uint16).copy()
    exp_v = v_pool.view(torch.int16).numpy().view(np.uint16).copy()
    kn = k_new.view(torch.int16).numpy().view(np.uint16)
    vn = v_new.view(torch.int16).numpy().view(np.uint16)
    # positions 3..8 of seq 0 -> (block, slot): 3->(5,3) 4->(2,0) .. 7->(2,3) 8->(0,0)
    where = [(5, 3), (2, 0), (2, 1), (2, 2), (2, 3), (0, 0), (1, 0)]
    for t, (b, sl) in enumerate(where):
        exp_k[b, sl] = kn[t]
        exp_v[b, sl] = vn[t]
    assert np.array_equal(kp, exp_k) and np.array_equal(vp, exp_v)


def test_oracle_rejects_bad_input():
    c = make_case([5], [1], seed=13)
    bt = c["bt"].clone()
    bt[0, 0] = c["k_pool"].shape[0]        # out of range
    with pytest.raises(ValueError):
        oracle.attention(c["q"], c["k_pool"], c["v_pool"], bt, c["cu"], c["seq_lens"], scale=1.0)
    with pytest.raises(ValueError):        # q_len > seq_len
        oracle.attention(c["q"], c["k_pool"], c["v_pool"], c["bt"], c["cu"],
                         torch.tensor([0], dtype=torch.int32), scale=1.0)


# ----------------------------------------------------------------- printed example

def test_kv_sizing_matches_printed_example():
    with open(os.path.join(HERE, "golden", "kv_cache_sizing.json")) as f:
        gold = json.load(f)
    got = workloads.kv_cache_bytes(**gold["inputs"])
    assert got == gold["exact_bytes"] == 8 * 2 ** 30
    # "about 8 GB" as printed: within 8 +- 0.6 decimal GB
    assert abs(got / 1e9 - 8) < 0.6
