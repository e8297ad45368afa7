"""Seeded synthetic workloads for paged GQA attention.

This module only draws inputs: random bf16 tensors, context lengths, block
placements and block tables.  It contains none of the attention arithmetic, so
both the CUDA path and the fp64 oracle can consume what it produces.

Shapes follow a Qwen3-8B-style attention layer: 32 query heads, 8 KV heads,
head_dim 128, KV stored in 256-token blocks ("BLOCK_SIZE 256" in §4.3.1 of the
page "扔掉 vLLM！从零构建 Qwen3-8B 推理引擎，C++/CUDA 实现性能追平 98%").
Values are ~N(0,1) drawn in fp32 and rounded to bf16.  Pool slots that no
sequence owns, slots past a sequence's length and block-table padding are filled
with sentinels (NaN bf16 / -1) so that a stray read shows up in the output.

Config names:
  single_decode        1 sequence, context 512 (2 blocks) in an 8-block pool
  batched_decode       batch 32, context ~U{128..4096}, 1024-block pool
  causal_prefill       1 sequence, 4096-token prompt appended into 16 blocks
  mixed_batch          120 decode sequences (context ~U{256..8192}) + 8 prefill
                       chunks of 512 tokens after contexts ~U{0..4096}, 4096 blocks
  prefix_shared_decode batch 128, context 32768, first 64 blocks shared by all
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 128
BLOCK_SIZE = 256
SCALE = 1.0 / math.sqrt(HEAD_DIM)

BF16_NAN_BITS = 0x7FC0
KV_BYTES_PER_TOKEN = 2 * NUM_KV_HEADS * HEAD_DIM * 2  # K and V, bf16


def kv_cache_bytes(num_layers: int, num_heads: int, head_dim: int, seq_len: int, batch: int,
                   bytes_per_elem: int) -> int:
    """Bytes of a dense KV cache: 2 (K and V) x layers x heads x head_dim x seq x batch x bytes.

    The sizing rule of §2.3 of the page "从零手搓AI推理引擎：避开调包陷阱的工程实践指南".
    """
    return 2 * num_layers * num_heads * head_dim * seq_len * batch * bytes_per_elem


def pool_bytes(num_blocks: int, block_size: int = BLOCK_SIZE, num_kv_heads: int = NUM_KV_HEADS,
               head_dim: int = HEAD_DIM, bytes_per_elem: int = 2) -> int:
    """Bytes of one paged pool (K or V): [num_blocks, block_size, Hkv, D]."""
    return num_blocks * block_size * num_kv_heads * head_dim * bytes_per_elem


@dataclass
class Batch:
    """One batch of paged-attention work.  All tensors live on ``device``.

    q          [T, Hq, D] bf16   queries of the T new tokens (grouped by sequence)
    k_new/v_new[T, Hkv, D] bf16  K/V of the new tokens, to be appended before attending
    k_pool/v_pool [N, 256, Hkv, D] bf16
    block_table [S, max_blocks] int32 (padding = -1)
    seq_lens   [S] int32         context length including the new tokens
    cu_q_lens  [S+1] int32       offsets of each sequence's new tokens in q/k_new/v_new
    """

    name: str
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    cu_q_lens: torch.Tensor
    max_q_len: int
    seq_lens_host: list = field(default_factory=list)
    q_lens_host: list = field(default_factory=list)
    info: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens_host)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.q_lens_host))

    @property
    def num_blocks(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    def select(self, seqs: slice) -> "Batch":
        """Sub-batch of a contiguous range of sequences sharing this batch's pools."""
        lo, hi, _ = seqs.indices(self.num_seqs)
        t0 = int(sum(self.q_lens_host[:lo]))
        t1 = int(sum(self.q_lens_host[:hi]))
        cu = self.cu_q_lens[lo:hi + 1] - self.cu_q_lens[lo]
        ql = self.q_lens_host[lo:hi]
        return Batch(name=f"{self.name}[{lo}:{hi}]", q=self.q[t0:t1], k_new=self.k_new[t0:t1],
                     v_new=self.v_new[t0:t1], k_pool=self.k_pool, v_pool=self.v_pool,
                     block_table=self.block_table[lo:hi], seq_lens=self.seq_lens[lo:hi],
                     cu_q_lens=cu.contiguous(), max_q_len=max(ql) if ql else 0,
                     seq_lens_host=self.seq_lens_host[lo:hi], q_lens_host=ql, info=dict(self.info))

    def kv_bytes(self) -> int:
        """Distinct K+V bytes a decode over this batch must read (valid tokens only)."""
        return int(sum(self.seq_lens_host)) * KV_BYTES_PER_TOKEN

    def causal_pairs(self) -> int:
        """Number of unmasked (query, key) pairs per query head."""
        n = 0
        for sl, ql in zip(self.seq_lens_host, self.q_lens_host):
            c0 = sl - ql
            # query i (0-based) at position c0 + i sees c0 + i + 1 keys
            n += ql * c0 + ql * (ql + 1) // 2
        return n

    def attention_flops(self) -> int:
        """4 * Hq * D flops per unmasked (query, key) pair (QK^T and PV, 2 flops per MAC)."""
        return 4 * NUM_Q_HEADS * HEAD_DIM * self.causal_pairs()


def _gen(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, gen: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def nan_bf16(shape, device) -> torch.Tensor:
    return torch.full(shape, BF16_NAN_BITS, dtype=torch.int16, device=device).view(torch.bfloat16)


def place_blocks(seq_lens, num_blocks: int, gen_cpu: torch.Generator, *,
                 shared_prefix_blocks: int = 0, max_blocks_per_seq: int | None = None,
                 block_size: int = BLOCK_SIZE) -> torch.Tensor:
    """Block tables for the given context lengths, blocks drawn from a random permutation.

    Physical blocks are taken in order from randperm(num_blocks): first the shared-prefix
    blocks (identical ids in every table), then each sequence's private blocks in turn.
    Table padding is -1.
    """
    need = [(sl + block_size - 1) // block_size for sl in seq_lens]
    width = max_blocks_per_seq or max(need + [1])
    perm = torch.randperm(num_blocks, generator=gen_cpu).tolist()
    shared = perm[:shared_prefix_blocks]
    cursor = shared_prefix_blocks
    rows = []
    for n in need:
        assert n <= width, "context does not fit the table width"
        own = max(0, n - shared_prefix_blocks)
        row = (shared[:min(n, shared_prefix_blocks)] + perm[cursor:cursor + own])
        cursor += own
        assert cursor <= num_blocks, "pool too small for the batch"
        rows.append(row + [-1] * (width - len(row)))
    return torch.tensor(rows, dtype=torch.int32).reshape(len(seq_lens), width)


def build_batch(name: str, seed: int, seq_lens, q_lens, num_blocks: int, device="cpu", *,
                shared_prefix_blocks: int = 0, max_blocks_per_seq: int | None = None,
                sentinel: bool = True, info: dict | None = None) -> Batch:
    """Draw a batch: pool contents for positions before each sequence's new tokens,
    plus q/k_new/v_new for the new tokens.  Block placement uses a CPU generator so it
    is identical on every device; tensor values use a generator on ``device``."""
    seq_lens = [int(x) for x in seq_lens]
    q_lens = [int(x) for x in q_lens]
    assert len(seq_lens) == len(q_lens) and all(0 <= ql <= sl for sl, ql in zip(seq_lens, q_lens))
    g_cpu = _gen(seed, "cpu")
    bt = place_blocks(seq_lens, num_blocks, g_cpu, shared_prefix_blocks=shared_prefix_blocks,
                      max_blocks_per_seq=max_blocks_per_seq)
    g = _gen(seed + 1000, device)
    shape = (num_blocks, BLOCK_SIZE, NUM_KV_HEADS, HEAD_DIM)
    k_pool = _randn_bf16(shape, g, device)
    v_pool = _randn_bf16(shape, g, device)
    if sentinel:
        # Every slot not holding a context token of some sequence becomes NaN.
        valid = torch.zeros(num_blocks * BLOCK_SIZE, dtype=torch.bool)
        for s, sl in enumerate(seq_lens):
            ctx = sl - q_lens[s]
            row = bt[s]
            for j in range((sl + BLOCK_SIZE - 1) // BLOCK_SIZE):
                lo = j * BLOCK_SIZE
                n = max(0, min(ctx - lo, BLOCK_SIZE))
                if n:
                    b = int(row[j])
                    valid[b * BLOCK_SIZE:b * BLOCK_SIZE + n] = True
        invalid = (~valid).nonzero().flatten().to(device)
        if invalid.numel():
            kv = k_pool.view(-1, NUM_KV_HEADS, HEAD_DIM)
            vv = v_pool.view(-1, NUM_KV_HEADS, HEAD_DIM)
            nan = nan_bf16((1, NUM_KV_HEADS, HEAD_DIM), device)
            kv.index_copy_(0, invalid, nan.expand(invalid.numel(), -1, -1).contiguous())
            vv.index_copy_(0, invalid, nan.expand(invalid.numel(), -1, -1).contiguous())
    t = sum(q_lens)
    q = _randn_bf16((t, NUM_Q_HEADS, HEAD_DIM), g, device)
    k_new = _randn_bf16((t, NUM_KV_HEADS, HEAD_DIM), g, device)
    v_new = _randn_bf16((t, NUM_KV_HEADS, HEAD_DIM), g, device)
    cu = [0]
    for ql in q_lens:
        cu.append(cu[-1] + ql)
    return Batch(name=name, q=q, k_new=k_new, v_new=v_new, k_pool=k_pool, v_pool=v_pool,
                 block_table=bt.to(device), seq_lens=torch.tensor(seq_lens, dtype=torch.int32,
                                                                 device=device),
                 cu_q_lens=torch.tensor(cu, dtype=torch.int32, device=device),
                 max_q_len=max(q_lens) if q_lens else 0, seq_lens_host=seq_lens,
                 q_lens_host=q_lens, info=dict(info or {}))


def randint_lens(seed: int, n: int, lo: int, hi: int) -> list:
    """n integers ~ U{lo..hi} (both ends inclusive) from a CPU generator."""
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


# ---------------------------------------------------------------- the five workloads

def single_decode(device="cpu", seed: int = 0) -> Batch:
    """1 sequence, context 512 = 2 blocks at shuffled slots of an 8-block pool."""
    return build_batch("single_decode", seed, [512], [1], num_blocks=8, device=device,
                       info={"batch": 1, "context": 512, "pool_blocks": 8})


def batched_decode(device="cpu", seed: int = 1, batch: int = 32, lo: int = 128,
                   hi: int = 4096, num_blocks: int = 1024) -> Batch:
    """batch 32, context ~U{128..4096}, blocks randomly permuted in a 1024-block pool."""
    lens = randint_lens(seed, batch, lo, hi)
    maxb = (hi + BLOCK_SIZE - 1) // BLOCK_SIZE
    return build_batch("batched_decode", seed, lens, [1] * batch, num_blocks=num_blocks,
                       device=device, max_blocks_per_seq=maxb,
                       info={"batch": batch, "context": f"U{{{lo}..{hi}}}",
                             "pool_blocks": num_blocks})


def causal_prefill(device="cpu", seed: int = 2, q_len: int = 4096,
                   num_blocks: int = 1024) -> Batch:
    """1 sequence, prompt of q_len tokens appended into randomly placed blocks."""
    return build_batch("causal_prefill", seed, [q_len], [q_len], num_blocks=num_blocks,
                       device=device, info={"batch": 1, "prompt": q_len,
                                            "pool_blocks": num_blocks})


def mixed_batch(device="cpu", seed: int = 3, n_decode: int = 120, n_chunks: int = 8,
                chunk: int = 512, dec_lo: int = 256, dec_hi: int = 8192, ctx_hi: int = 4096,
                num_blocks: int = 4096) -> Batch:
    """Continuous batch: n_decode decode sequences followed by n_chunks prefill chunks.

    Sequences [0, n_decode) have one new token each; the rest have `chunk` new tokens
    after an existing context ~U{0..ctx_hi}.  One block table covers all of them, so a
    single append call writes every new token; decode and prefill then run on the two
    contiguous sub-batches (Batch.select).
    """
    dec = randint_lens(seed, n_decode, dec_lo, dec_hi)
    ctx = randint_lens(seed + 500, n_chunks, 0, ctx_hi)
    seq_lens = dec + [c + chunk for c in ctx]
    q_lens = [1] * n_decode + [chunk] * n_chunks
    maxb = (max(dec_hi, ctx_hi + chunk) + BLOCK_SIZE - 1) // BLOCK_SIZE
    return build_batch("mixed_batch", seed, seq_lens, q_lens, num_blocks=num_blocks,
                       device=device, max_blocks_per_seq=maxb,
                       info={"n_decode": n_decode, "n_chunks": n_chunks, "chunk": chunk,
                             "pool_blocks": num_blocks})


def prefix_shared_decode(device="cpu", seed: int = 4, batch: int = 128, context: int = 32768,
                         shared_blocks: int = 64, slack_blocks: int = 64) -> Batch:
    """batch 128, context 32768; the first 64 blocks are the same physical blocks in
    every table (a shared prefix), the remaining 64 blocks of each sequence are private."""
    nblk = context // BLOCK_SIZE
    num_blocks = shared_blocks + batch * (nblk - shared_blocks) + slack_blocks
    return build_batch("prefix_shared_decode", seed, [context] * batch, [1] * batch,
                       num_blocks=num_blocks, device=device, shared_prefix_blocks=shared_blocks,
                       info={"batch": batch, "context": context, "shared_blocks": shared_blocks,
                             "pool_blocks": num_blocks})


def context_rows(batch: Batch, k_pool=None, v_pool=None, drop_last: int = 0):
    """Every context token's K/V rows gathered through the block table, as an append request
    that rebuilds the whole context: (k_rows, v_rows [T, Hkv, D], cu [S+1], lens [S]) with
    positions 0 .. seq_len - 1 - drop_last of each sequence (drop_last = 1 leaves out each
    sequence's newest token).  Pure data movement; the pools default to the batch's own."""
    kp = batch.k_pool if k_pool is None else k_pool
    vp = batch.v_pool if v_pool is None else v_pool
    bt = batch.block_table.cpu()
    blks, slots, lens = [], [], []
    for s, sl in enumerate(batch.seq_lens_host):
        n = sl - drop_last
        pos = torch.arange(n)
        blks.append(bt[s, pos // BLOCK_SIZE].long())
        slots.append(pos % BLOCK_SIZE)
        lens.append(n)
    blk = torch.cat(blks).to(kp.device)
    slot = torch.cat(slots).to(kp.device)
    cu = torch.tensor([0] + list(torch.tensor(lens).cumsum(0).tolist()), dtype=torch.int32, device=kp.device)
    return (kp[blk, slot].contiguous(), vp[blk, slot].contiguous(), cu,
            torch.tensor(lens, dtype=torch.int32, device=kp.device))


@dataclass
class Layers:
    """A decode batch repeated over L layers, layer-major: q [L, B, Hq, D], k_new / v_new
    [L, B, Hkv, D], k_pool / v_pool [L, N, 256, Hkv, D]; block_table and seq_lens are
    shared by every layer (the batch's own).  Layer 0 holds the batch's values; the other
    layers hold fresh values in the same pool slots (unowned slots stay sentinels)."""

    base: Batch
    q: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor

    @property
    def layers(self) -> int:
        return int(self.q.shape[0])

    def layer(self, l: int) -> Batch:
        """Layer l as a Batch (views into the layer-major tensors)."""
        return replace(self.base, name=f"{self.base.name}[{l}]", q=self.q[l], k_new=self.k_new[l],
                       v_new=self.v_new[l], k_pool=self.k_pool[l], v_pool=self.v_pool[l])

    def kv_bytes(self) -> int:
        return self.layers * self.base.kv_bytes()


def layered(batch: Batch, layers: int, seed: int) -> Layers:
    """Stack `layers` copies of a decode batch (one new token per sequence) with fresh
    seeded values per layer, for the multi-layer decode step."""
    assert all(ql == 1 for ql in batch.q_lens_host), "a decode batch (one new token per sequence)"
    dev = batch.q.device
    gen = _gen(seed, dev)
    qs, kns, vns, kps, vps = [batch.q], [batch.k_new], [batch.v_new], [batch.k_pool], [batch.v_pool]
    owned = ~torch.isnan(batch.k_pool.float())
    for _ in range(1, layers):
        qs.append(_randn_bf16(tuple(batch.q.shape), gen, dev))
        kns.append(_randn_bf16(tuple(batch.k_new.shape), gen, dev))
        vns.append(_randn_bf16(tuple(batch.v_new.shape), gen, dev))
        kps.append(torch.where(owned, _randn_bf16(tuple(batch.k_pool.shape), gen, dev), batch.k_pool))
        vps.append(torch.where(owned, _randn_bf16(tuple(batch.v_pool.shape), gen, dev), batch.v_pool))
    return Layers(batch, torch.stack(qs), torch.stack(kns), torch.stack(vns), torch.stack(kps),
                  torch.stack(vps))


def layered_decode(device="cpu", seed: int = 5, layers: int = 36) -> Layers:
    """The single-sequence decode (context 512, 8-block pool) over the 36 layers of the
    model: the launch-bound case the multi-layer CUDA graph serves."""
    return layered(single_decode(device=device), layers, seed)


WORKLOADS = {
    "single_decode": single_decode,
    "batched_decode": batched_decode,
    "causal_prefill": causal_prefill,
    "mixed_batch": mixed_batch,
    "prefix_shared_decode": prefix_shared_decode,
}


def unique_kv_bytes(batch: Batch) -> int:
    """Distinct K+V bytes behind the valid tokens (a shared block counted once)."""
    seen = {}
    bt = batch.block_table.cpu()
    for s, sl in enumerate(batch.seq_lens_host):
        for j in range((sl + BLOCK_SIZE - 1) // BLOCK_SIZE):
            b = int(bt[s, j])
            n = min(BLOCK_SIZE, sl - j * BLOCK_SIZE)
            seen[b] = max(seen.get(b, 0), n)
    return sum(seen.values()) * KV_BYTES_PER_TOKEN
