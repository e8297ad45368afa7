"""Shared tiny cases and library-routine references for the oracle pins (test side only)."""
import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle


def make_case(seq_lens, q_lens, hq=4, hkv=2, d=16, bs=4, extra_blocks=3, seed=0, lib=None):
    """Tiny paged case built from contiguous per-sequence K/V.

    Returns dict with contiguous K/V (for the library reference) and the paged pool,
    block table and cu_q_lens the oracle consumes.
    """
    g = torch.Generator().manual_seed(seed)
    nblk = [(sl + bs - 1) // bs for sl in seq_lens]
    num_blocks = sum(nblk) + extra_blocks
    perm = torch.randperm(num_blocks, generator=g).tolist()
    width = max(nblk) + 1
    bt = torch.full((len(seq_lens), width), -1, dtype=torch.int32)
    k_pool = torch.full((num_blocks, bs, hkv, d), float("nan")).to(torch.bfloat16)
    v_pool = k_pool.clone()
    ks, vs = [], []
    cur = 0
    for s, sl in enumerate(seq_lens):
        k = torch.randn(sl, hkv, d, generator=g).to(torch.bfloat16)
        v = torch.randn(sl, hkv, d, generator=g).to(torch.bfloat16)
        ks.append(k)
        vs.append(v)
        for j in range(nblk[s]):
            b = perm[cur]
            cur += 1
            bt[s, j] = b
            n = min(bs, sl - j * bs)
            k_pool[b, :n] = k[j * bs:j * bs + n]
            v_pool[b, :n] = v[j * bs:j * bs + n]
    q = torch.randn(sum(q_lens), hq, d, generator=g).to(torch.bfloat16)
    cu = torch.tensor([0] + list(np.cumsum(q_lens)), dtype=torch.int32)
    return dict(q=q, k=ks, v=vs, k_pool=k_pool, v_pool=v_pool, bt=bt, cu=cu,
                seq_lens=torch.tensor(seq_lens, dtype=torch.int32), q_lens=list(q_lens),
                hq=hq, hkv=hkv, d=d, bs=bs)


def run_oracle(c, scale, lib=None):
    return oracle.attention(c["q"], c["k_pool"], c["v_pool"], c["bt"], c["cu"], c["seq_lens"],
                            scale=scale, lib=lib)


def sdpa_reference(c, scale):
    """torch SDPA (float64, CPU) per sequence on contiguous K/V, bottom-right causal mask."""
    outs = []
    t0 = 0
    for s, ql in enumerate(c["q_lens"]):
        sl = int(c["seq_lens"][s])
        q = c["q"][t0:t0 + ql].double().permute(1, 0, 2).unsqueeze(0)   # [1,Hq,ql,D]
        rep = c["hq"] // c["hkv"]
        k = c["k"][s].double().permute(1, 0, 2).repeat_interleave(rep, 0).unsqueeze(0)
        v = c["v"][s].double().permute(1, 0, 2).repeat_interleave(rep, 0).unsqueeze(0)
        i = torch.arange(ql).unsqueeze(1)
        j = torch.arange(sl).unsqueeze(0)
        mask = j <= (sl - ql + i)
        o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
        outs.append(o[0].permute(1, 0, 2))
        t0 += ql
    return torch.cat(outs).numpy()


def sdpa_lse(c, scale):
    """log-sum-exp of the masked scores, from torch.logsumexp."""
    res = []
    t0 = 0
    for s, ql in enumerate(c["q_lens"]):
        sl = int(c["seq_lens"][s])
        q = c["q"][t0:t0 + ql].double()                                  # [ql,Hq,D]
        rep = c["hq"] // c["hkv"]
        k = c["k"][s].double().repeat_interleave(rep, 1)                 # [sl,Hq,D]
        sc = torch.einsum("ihd,jhd->hij", q, k) * scale
        i = torch.arange(ql).unsqueeze(1)
        j = torch.arange(sl).unsqueeze(0)
        sc = sc.masked_fill(~(j <= (sl - ql + i)), float("-inf"))
        res.append(torch.logsumexp(sc, dim=-1).permute(1, 0))
        t0 += ql
    return torch.cat(res).numpy()


def pin_battery(lib):
    """Run a compact set of pins against an oracle library; return the names that fail."""
    failed = []

    def check(name, fn):
        try:
            ok = fn()
        except Exception:
            ok = False
        if not ok:
            failed.append(name)

    for seq_lens, q_lens in (([13], [1]), ([9, 1, 17], [1, 1, 1]), ([16], [16]), ([21], [6]),
                             ([10, 7, 19], [10, 3, 5])):
        c = make_case(seq_lens, q_lens, seed=sum(seq_lens) + len(q_lens))
        scale = 1.0 / math.sqrt(c["d"])

        def sdpa_out(c=c, scale=scale):
            out, _ = run_oracle(c, scale, lib=lib)
            return np.allclose(out, sdpa_reference(c, scale), rtol=0, atol=1e-12)

        def sdpa_l(c=c, scale=scale):
            _, lse = run_oracle(c, scale, lib=lib)
            return np.allclose(lse, sdpa_lse(c, scale), rtol=1e-13, atol=1e-12)

        check(f"sdpa_out{seq_lens}{q_lens}", sdpa_out)
        check(f"sdpa_lse{seq_lens}{q_lens}", sdpa_l)

    def gqa():
        c = make_case([12, 6], [4, 1], hq=8, hkv=2, seed=6)
        out, lse = run_oracle(c, 0.2, lib=lib)
        kp = c["k_pool"].repeat_interleave(4, dim=2).contiguous()
        vp = c["v_pool"].repeat_interleave(4, dim=2).contiguous()
        out2, lse2 = oracle.attention(c["q"], kp, vp, c["bt"], c["cu"], c["seq_lens"],
                                      scale=0.2, lib=lib)
        return np.array_equal(out, out2) and np.array_equal(lse, lse2)

    check("gqa_equals_mha", gqa)

    def append():
        bs, hkv, d = 4, 2, 8
        g = torch.Generator().manual_seed(12)
        kpool = torch.randn(6, bs, hkv, d, generator=g).to(torch.bfloat16)
        vpool = torch.randn(6, bs, hkv, d, generator=g).to(torch.bfloat16)
        bt = torch.tensor([[5, 2, 0], [3, 1, -1]], dtype=torch.int32)
        kn = torch.randn(7, hkv, d, generator=g).to(torch.bfloat16)
        vn = torch.randn(7, hkv, d, generator=g).to(torch.bfloat16)
        kp, vp = oracle.kv_append(kpool, vpool, kn, vn, bt,
                                  torch.tensor([0, 6, 7], dtype=torch.int32),
                                  torch.tensor([9, 5], dtype=torch.int32), block_size=bs, lib=lib)
        ek = kpool.view(torch.int16).numpy().view(np.uint16).copy()
        ev = vpool.view(torch.int16).numpy().view(np.uint16).copy()
        knb = kn.view(torch.int16).numpy().view(np.uint16)
        vnb = vn.view(torch.int16).numpy().view(np.uint16)
        for t, (b, sl) in enumerate([(5, 3), (2, 0), (2, 1), (2, 2), (2, 3), (0, 0), (1, 0)]):
            ek[b, sl] = knb[t]
            ev[b, sl] = vnb[t]
        return np.array_equal(kp, ek) and np.array_equal(vp, ev)

    check("kv_append_placement", append)
    return failed
