"""Seeded synthetic inputs for paged-KV varlen attention.

This module only draws inputs: sequence lengths, page pools, block tables and
the q / k / v values.  It holds none of the attention arithmetic, and both the
CUDA path's tests and the oracle's tests take their inputs from it, so that
the two sides read the same bytes.

Layouts follow the candle pages ("flash-attn-varlen paged expects k/v tensors
of rank 4", What it means; "flash-attn-varlen expects input tensors of rank
3", Source): q is (total_q, num_heads, head_dim); the paged caches are
(num_blocks, page_block_size, num_heads_k, head_dim) with the last dimension
contiguous; the block table holds one row of physical block ids per sequence.

Recipe (all draws seeded):
  * lengths: ``numpy.random.default_rng(seed)``, integer uniforms inclusive;
  * pages: each sequence needs ceil(sk / P) pages; the pool holds the needed
    pages plus ``spare`` extra blocks; a seeded permutation of the pool assigns
    physical blocks to pages in sequence order; unused table slots hold -1;
  * values: N(0, std^2) drawn in fp32 by ``torch.Generator`` (on the device the
    tensors live on) and rounded to the dtype;
  * ``nan_fill``: every cache slot no sequence owns (the tail of a last page
    and every spare block) is set to NaN so that a stray read shows.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional

import numpy as np


@dataclass
class Layout:
    """Lengths, pool size and block table of one synthetic batch (host numpy)."""

    name: str
    dtype: str
    num_heads: int
    num_heads_k: int
    head_dim: int
    page_block_size: int
    seqlens_q: List[int]
    seqlens_k: List[int]
    num_blocks: int
    block_table: np.ndarray  # int32 [batch, max_pages], -1 past each sequence's pages
    window_left: int = -1
    window_right: int = 0
    std: float = 1.0
    softmax_scale: float = 0.0
    seed: int = 0
    nan_fill: bool = True
    paged: bool = True

    @property
    def batch(self) -> int:
        return len(self.seqlens_q)

    @property
    def total_q(self) -> int:
        return int(sum(self.seqlens_q))

    @property
    def total_k(self) -> int:
        return int(sum(self.seqlens_k))

    @property
    def max_seqlen_q(self) -> int:
        return int(max(self.seqlens_q, default=0))

    @property
    def max_seqlen_k(self) -> int:
        return int(max(self.seqlens_k, default=0))

    def cu_seqlens(self):
        cq = np.zeros(self.batch + 1, dtype=np.int32)
        ck = np.zeros(self.batch + 1, dtype=np.int32)
        cq[1:] = np.cumsum(self.seqlens_q)
        ck[1:] = np.cumsum(self.seqlens_k)
        return cq, ck


def make_layout(name, dtype, seqlens_q, seqlens_k, *, num_heads, num_heads_k, head_dim,
                page_block_size, seed, spare=0.0, extra_blocks=0, window_left=-1,
                window_right=0, std=1.0, softmax_scale=None, nan_fill=True,
                extra_table_cols=0) -> Layout:
    """Assign physical blocks to each sequence's pages from a seeded permutation.

    ``spare`` is a fraction of the needed pages added to the pool (0.1 = 10 %),
    ``extra_blocks`` an absolute count on top of it.
    """
    P = int(page_block_size)
    sq = [int(x) for x in seqlens_q]
    sk = [int(x) for x in seqlens_k]
    pages = [(s + P - 1) // P for s in sk]
    needed = int(sum(pages))
    num_blocks = needed + int(math.ceil(needed * spare)) + int(extra_blocks)
    num_blocks = max(num_blocks, 1)
    rng = np.random.default_rng(seed + 7919)
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_pages = max(max(pages, default=0), 1) + int(extra_table_cols)
    bt = np.full((len(sk), max_pages), -1, dtype=np.int32)
    cursor = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[cursor:cursor + n]
        cursor += n
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(head_dim)
    return Layout(name=name, dtype=dtype, num_heads=num_heads, num_heads_k=num_heads_k,
                  head_dim=head_dim, page_block_size=P, seqlens_q=sq, seqlens_k=sk,
                  num_blocks=num_blocks, block_table=bt, window_left=window_left,
                  window_right=window_right, std=std, softmax_scale=float(softmax_scale),
                  seed=seed, nan_fill=nan_fill)


# --- the five serving-shaped workloads -------------------------------------------------

def tiny_fp16() -> Layout:
    """2 sequences, sq=[3,5], sk=[40,70]; H=4, Hkv=2, D=64, P=32; 8-block pool, causal, fp16."""
    return make_layout("tiny_fp16", "f16", [3, 5], [40, 70], num_heads=4, num_heads_k=2,
                       head_dim=64, page_block_size=32, seed=1, extra_blocks=3)


def decode_bf16(batch=64, lo=512, hi=4096, seed=2) -> Layout:
    """64 decode sequences (q_len 1), sk ~ U[512, 4096]; H=32, Hkv=8, D=128, P=32; pool +10 %."""
    rng = np.random.default_rng(seed)
    sk = rng.integers(lo, hi, size=batch, endpoint=True)
    return make_layout("decode_bf16", "bf16", [1] * batch, sk, num_heads=32, num_heads_k=8,
                       head_dim=128, page_block_size=32, seed=seed, spare=0.1)


def prefill_bf16(batch=8, lo=1024, hi=8192, seed=3) -> Layout:
    """8 causal prefill sequences, sq = sk ~ U[1024, 8192]; H=32, Hkv=8, D=128, P=64; exact pool."""
    rng = np.random.default_rng(seed)
    s = rng.integers(lo, hi, size=batch, endpoint=True)
    return make_layout("prefill_bf16", "bf16", s, s, num_heads=32, num_heads_k=8,
                       head_dim=128, page_block_size=64, seed=seed)


def prefill_d256_bf16(batch=8, lo=1024, hi=8192, seed=3) -> Layout:
    """The causal prefill batch at head_dim 256: 8 sequences, sq = sk ~ U[1024, 8192];
    H=16, Hkv=4, D=256, P=64; exact pool."""
    rng = np.random.default_rng(seed)
    s = rng.integers(lo, hi, size=batch, endpoint=True)
    return make_layout("prefill_d256_bf16", "bf16", s, s, num_heads=16, num_heads_k=4,
                       head_dim=256, page_block_size=64, seed=seed)


def mixed_bf16(n_chunks=4, chunk=512, ctx_lo=2048, ctx_hi=16384, n_decode=120, dec_lo=256,
               dec_hi=32768, seed=4) -> Layout:
    """4 chunked-prefill sequences (512 queries over 2048-16384 cached keys) then 120
    decode sequences (sk ~ U[256, 32768]); H=64, Hkv=8, D=128, P=128; window (4096, 0)."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_lo, ctx_hi, size=n_chunks, endpoint=True)
    dec = rng.integers(dec_lo, dec_hi, size=n_decode, endpoint=True)
    sq = [chunk] * n_chunks + [1] * n_decode
    sk = [int(c) + chunk for c in ctx] + [int(d) for d in dec]
    return make_layout("mixed_bf16", "bf16", sq, sk, num_heads=64, num_heads_k=8,
                       head_dim=128, page_block_size=128, seed=seed, spare=0.1,
                       window_left=4096, window_right=0)


def long_bf16(seed=5) -> Layout:
    """4 sequences, 4 queries each over sk=131072; H=16, Hkv=2, D=256, P=256; N(0, 0.5^2)."""
    return make_layout("long_bf16", "bf16", [4] * 4, [131072] * 4, num_heads=16, num_heads_k=2,
                       head_dim=256, page_block_size=256, seed=seed, spare=0.1, std=0.5)


def long_d512_bf16(seed=6) -> Layout:
    """2 sequences, 4 queries each over sk=16384; H=16, Hkv=2, D=512, P=32; N(0, 0.5^2)."""
    return make_layout("long_d512_bf16", "bf16", [4] * 2, [16384] * 2, num_heads=16,
                       num_heads_k=2, head_dim=512, page_block_size=32, seed=seed, spare=0.1,
                       std=0.5)


def skewed_decode_bf16(batch=64, lo=512, hi=4096, long_k=131072, seed=7) -> Layout:
    """The decode batch with one sequence far longer than the rest: 63 sequences with
    sk ~ U[512, 4096] and one (at a seeded position) with 131,072 keys; H=32, Hkv=8, D=128,
    P=32, q_len 1, pool +10 %."""
    rng = np.random.default_rng(seed)
    sk = rng.integers(lo, hi, size=batch, endpoint=True)
    sk[int(rng.integers(0, batch))] = long_k
    return make_layout("skewed_decode_bf16", "bf16", [1] * batch, sk, num_heads=32, num_heads_k=8,
                       head_dim=128, page_block_size=32, seed=seed, spare=0.1)


CONFIGS = {
    "tiny_fp16": tiny_fp16,
    "decode_bf16": decode_bf16,
    "prefill_bf16": prefill_bf16,
    "prefill_d256_bf16": prefill_d256_bf16,
    "mixed_bf16": mixed_bf16,
    "long_bf16": long_bf16,
    "long_d512_bf16": long_d512_bf16,
    "skewed_decode_bf16": skewed_decode_bf16,
}


# --- reduced variants the oracle finishes in seconds (several tiles, ragged tails) ---

def small(name: str) -> Layout:
    if name == "decode":
        rng = np.random.default_rng(12)
        sk = list(rng.integers(1, 700, size=11, endpoint=True)) + [1]
        return make_layout("decode_small", "bf16", [1] * len(sk), sk, num_heads=8, num_heads_k=2,
                           head_dim=128, page_block_size=32, seed=12, spare=0.1)
    if name == "prefill":
        rng = np.random.default_rng(13)
        s = rng.integers(60, 333, size=3, endpoint=True)
        return make_layout("prefill_small", "bf16", s, s, num_heads=4, num_heads_k=2,
                           head_dim=128, page_block_size=64, seed=13)
    if name == "mixed":
        rng = np.random.default_rng(14)
        ctx = rng.integers(100, 600, size=2, endpoint=True)
        dec = rng.integers(30, 900, size=6, endpoint=True)
        sq = [77, 150] + [1] * 6
        sk = [int(ctx[0]) + 77, int(ctx[1]) + 150] + [int(d) for d in dec]
        return make_layout("mixed_small", "bf16", sq, sk, num_heads=8, num_heads_k=2,
                           head_dim=128, page_block_size=128, seed=14, spare=0.1,
                           window_left=200, window_right=0)
    if name == "long":
        return make_layout("long_small", "bf16", [4, 4], [3000, 2345], num_heads=16,
                           num_heads_k=2, head_dim=256, page_block_size=256, seed=15,
                           spare=0.1, std=0.5)
    if name == "d512":
        return make_layout("d512_small", "bf16", [4, 3], [700, 333], num_heads=16,
                           num_heads_k=2, head_dim=512, page_block_size=32, seed=16,
                           spare=0.1, std=0.5)
    raise KeyError(name)


# --- materialisation --------------------------------------------------------------------

def _torch_dtype(dtype: str):
    import torch
    return {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]


@dataclass
class Inputs:
    layout: Layout
    q: "object"
    k_cache: "object"
    v_cache: "object"
    cu_seqlens_q: "object"
    cu_seqlens_k: "object"
    block_table: "object"

    def to(self, device):
        return Inputs(self.layout, *(None if t is None else t.to(device) for t in (
            self.q, self.k_cache, self.v_cache, self.cu_seqlens_q, self.cu_seqlens_k,
            self.block_table)))


def _randn(shape, std, dtype, gen, device, chunk_rows=1 << 14):
    """N(0, std^2) in fp32, rounded to ``dtype``; drawn in slabs to bound temporaries."""
    import torch
    out = torch.empty(shape, dtype=dtype, device=device)
    if out.numel() == 0:
        return out
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        x = torch.randn((r1 - r0, flat.shape[1]), generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[r0:r1].copy_(x)
    return out


def materialize(layout: Layout, device="cpu", seed: Optional[int] = None) -> Inputs:
    """Draw q / k_cache / v_cache for ``layout`` on ``device`` (torch tensors)."""
    import torch
    seed = layout.seed if seed is None else seed
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    dt = _torch_dtype(layout.dtype)
    H, Hkv, D, P = layout.num_heads, layout.num_heads_k, layout.head_dim, layout.page_block_size
    q = _randn((max(layout.total_q, 0), H, D), layout.std, dt, gen, device)
    if layout.paged:
        kv_shape = (layout.num_blocks, P, Hkv, D)
    else:
        kv_shape = (layout.total_k, Hkv, D)
    k = _randn(kv_shape, layout.std, dt, gen, device, chunk_rows=max(1, (1 << 22) // (kv_shape[1] * Hkv * D) if layout.paged else 1 << 14))
    v = _randn(kv_shape, layout.std, dt, gen, device, chunk_rows=max(1, (1 << 22) // (kv_shape[1] * Hkv * D) if layout.paged else 1 << 14))
    cq, ck = layout.cu_seqlens()
    if layout.paged and layout.nan_fill:
        owned = np.zeros((layout.num_blocks, P), dtype=bool)
        for b, s in enumerate(layout.seqlens_k):
            n = (s + P - 1) // P
            for p in range(n):
                blk = layout.block_table[b, p]
                owned[blk, : min(P, s - p * P)] = True
        free = torch.from_numpy(~owned).to(device)
        k[free] = float("nan")
        v[free] = float("nan")
    return Inputs(
        layout, q, k, v,
        torch.from_numpy(cq).to(device), torch.from_numpy(ck).to(device),
        torch.from_numpy(layout.block_table.copy()).to(device) if layout.paged else None,
    )


def with_block_permutation(inputs: Inputs, seed: int) -> Inputs:
    """Same logical cache under a random physical placement: blocks are permuted and the
    block table is rewritten to match (unused table slots stay -1)."""
    import torch
    lay = inputs.layout
    rng = np.random.default_rng(seed)
    perm = rng.permutation(lay.num_blocks)  # new position of old block b is perm[b]
    dev = inputs.k_cache.device
    inv = np.empty_like(perm)
    inv[perm] = np.arange(lay.num_blocks)
    idx = torch.from_numpy(inv).to(dev)
    k2 = inputs.k_cache.index_select(0, idx)
    v2 = inputs.v_cache.index_select(0, idx)
    bt = lay.block_table.copy()
    mask = bt >= 0
    bt[mask] = perm[bt[mask]]
    lay2 = replace(lay, block_table=bt)
    return Inputs(lay2, inputs.q, k2, v2, inputs.cu_seqlens_q, inputs.cu_seqlens_k,
                  torch.from_numpy(bt).to(dev))
