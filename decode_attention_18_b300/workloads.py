"""Seeded synthetic inputs for the decode-attention workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic. Both the CUDA path (tests, bench) and the fp64 checker
consume what it returns, so it is the one module they share.

Recipe (every tensor is drawn in float32 from a seeded ``torch.Generator`` on
the requested device, scaled by its standard deviation and rounded to bf16):

* sequence lengths: ``torch.randint`` from a generator seeded ``seed + 1000``
  (drawn first, because they fix the cache shapes);
* tensors, in this order, from a generator seeded ``seed``: queries
  (q, or q_nope then q_pe), keys (K, or Z), values (V, or K_pe), then the
  weights W_uk and W_uv for MLA;
* the physical page order of a paged cache: ``torch.randperm`` from a
  generator seeded ``seed + 2000``.

Cache slots past a sequence's length are filled with random values too (a
kernel that reads past the end therefore changes its result). Unused
block-table entries are -1.

The shapes follow the pages' model geometries: DeepSeek-V3-like MLA (h=128,
d=128, k=512, p=64, t=4096), a 64-query / 8-KV head GQA layer with head dim
128, and a 24-query-head, head-dim-256 layer with 24 / 4 / 1 KV heads over
long ragged contexts in 64-token pages.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

PAGE_SIZE = 64


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, g: torch.Generator, device, std: float = 1.0) -> torch.Tensor:
    """N(0, std^2) rounded to bf16. Large tensors are drawn in slabs along
    dim 0 to bound the float32 temporary."""
    shape = tuple(int(x) for x in shape)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if out.numel() == 0:
        return out
    per_row = max(1, out.numel() // max(1, shape[0]))
    rows = max(1, (1 << 27) // per_row)
    for r0 in range(0, shape[0], rows):
        r1 = min(shape[0], r0 + rows)
        tmp = torch.randn((r1 - r0,) + shape[1:], generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        out[r0:r1].copy_(tmp)
    return out


def ragged_seqlens(b: int, lo: int, hi: int, seed: int) -> list[int]:
    """Integer lengths uniform in [lo, hi] (inclusive)."""
    g = _gen(seed + 1000, "cpu")
    return [int(x) for x in torch.randint(lo, hi + 1, (b,), generator=g)]


def page_layout(seqlens, seed: int, page_size: int = PAGE_SIZE):
    """Random physical page order: returns (block_table [b, max_pages] int32
    with -1 padding, num_pages)."""
    n_pages = [(L + page_size - 1) // page_size for L in seqlens]
    total = sum(n_pages)
    max_pages = max(1, max(n_pages) if n_pages else 1)
    perm = torch.randperm(total, generator=_gen(seed + 2000, "cpu")).to(torch.int32) if total else \
        torch.zeros(0, dtype=torch.int32)
    table = torch.full((len(seqlens), max_pages), -1, dtype=torch.int32)
    pos = 0
    for i, n in enumerate(n_pages):
        table[i, :n] = perm[pos:pos + n]
        pos += n
    return table, total


@dataclass
class KVCache:
    """Keys/values of a grouped-head layer, contiguous or paged.

    contiguous: k, v are [b, capacity, Hkv, d]; paged: [num_pages, 64, Hkv, d]
    with block_table [b, max_pages]."""
    k: torch.Tensor
    v: torch.Tensor
    seqlens: list
    paged: bool
    capacity: int = 0
    block_table: torch.Tensor | None = None
    page_size: int = PAGE_SIZE

    def seq_rows(self, i: int, which: str) -> torch.Tensor:
        """Rows [L_i, Hkv, d] of sequence i in logical order (a gather of the
        stored tensor; used to hand the checker its inputs)."""
        t = self.k if which == "k" else self.v
        L = self.seqlens[i]
        if not self.paged:
            return t[i, :L]
        n = (L + self.page_size - 1) // self.page_size
        idx = self.block_table[i, :n].to(torch.long).to(t.device)
        return t.index_select(0, idx).reshape(-1, *t.shape[2:])[:L]


def make_gqa(b, hq, hkv, d, s, seqlens, *, paged=False, capacity=None, seed=0,
             device="cpu", q_std=1.0):
    """Query [b, Hq, s, d] and a K/V cache for grouped-head decode."""
    seqlens = [int(x) for x in seqlens]
    g = _gen(seed, device)
    q = randn_bf16((b, hq, s, d), g, device, q_std)
    if paged:
        table, total = page_layout(seqlens, seed)
        k = randn_bf16((max(total, 1), PAGE_SIZE, hkv, d), g, device)
        v = randn_bf16((max(total, 1), PAGE_SIZE, hkv, d), g, device)
        cache = KVCache(k, v, seqlens, True, 0, table.to(device))
    else:
        cap = int(capacity if capacity is not None else max(max(seqlens), 1))
        k = randn_bf16((b, cap, hkv, d), g, device)
        v = randn_bf16((b, cap, hkv, d), g, device)
        cache = KVCache(k, v, seqlens, False, cap)
    return q, cache


def make_gqa_fp8(b, hq, hkv, d, s, seqlens, *, paged=False, capacity=None, seed=0, device="cpu"):
    """Query [b, Hq, s, d] bf16 and an FP8 (OCP E4M3) K/V cache: values drawn
    N(0, 1) in fp32, stored as E4M3 bytes of value / scale with one scale per
    tensor (its largest magnitude maps to 448, the largest E4M3 value). Returns
    (q, cache with uint8 k / v, k_scale, v_scale)."""
    seqlens = [int(x) for x in seqlens]
    g = _gen(seed, device)
    q = randn_bf16((b, hq, s, d), g, device)

    def quantised(shape):
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        scale = float(x.abs().max()) / 448.0
        return (x / scale).to(torch.float8_e4m3fn).view(torch.uint8), scale

    if paged:
        table, total = page_layout(seqlens, seed)
        k, ks = quantised((max(total, 1), PAGE_SIZE, hkv, d))
        v, vs = quantised((max(total, 1), PAGE_SIZE, hkv, d))
        cache = KVCache(k, v, seqlens, True, 0, table.to(device))
    else:
        cap = int(capacity if capacity is not None else max(max(seqlens), 1))
        k, ks = quantised((b, cap, hkv, d))
        v, vs = quantised((b, cap, hkv, d))
        cache = KVCache(k, v, seqlens, False, cap)
    return q, cache, ks, vs


@dataclass
class MLAInputs:
    q_nope: torch.Tensor      # [b, h, s, d]
    q_pe: torch.Tensor        # [b, h, s, p]
    z: torch.Tensor           # [b, cap, k] or [pages, 64, k]
    k_pe: torch.Tensor        # [b, cap, p] or [pages, 64, p]
    w_uk: torch.Tensor        # [h, d, k]
    w_uv: torch.Tensor        # [h, k, d]
    seqlens: list
    paged: bool
    capacity: int = 0
    block_table: torch.Tensor | None = None
    scale: float = 0.0
    page_size: int = PAGE_SIZE

    def seq_rows(self, i: int, which: str) -> torch.Tensor:
        t = self.z if which == "z" else self.k_pe
        L = self.seqlens[i]
        if not self.paged:
            return t[i, :L]
        n = (L + self.page_size - 1) // self.page_size
        idx = self.block_table[i, :n].to(torch.long).to(t.device)
        return t.index_select(0, idx).reshape(-1, t.shape[-1])[:L]


def make_mla(b, h, d, k, p, s, seqlens, *, paged=False, capacity=None, seed=0,
             device="cpu", q_std=1.0):
    """Absorbed-MLA inputs: queries and cache ~N(0,1), weights ~N(0, 1/k),
    softmax scale 1/sqrt(d + p)."""
    seqlens = [int(x) for x in seqlens]
    g = _gen(seed, device)
    q_nope = randn_bf16((b, h, s, d), g, device, q_std)
    q_pe = randn_bf16((b, h, s, p), g, device, q_std)
    wstd = 1.0 / math.sqrt(k)
    if paged:
        table, total = page_layout(seqlens, seed)
        z = randn_bf16((max(total, 1), PAGE_SIZE, k), g, device)
        kpe = randn_bf16((max(total, 1), PAGE_SIZE, p), g, device)
        cap = 0
        table = table.to(device)
    else:
        cap = int(capacity if capacity is not None else max(max(seqlens), 1))
        z = randn_bf16((b, cap, k), g, device)
        kpe = randn_bf16((b, cap, p), g, device)
        table = None
    w_uk = randn_bf16((h, d, k), g, device, wstd)
    w_uv = randn_bf16((h, k, d), g, device, wstd)
    return MLAInputs(q_nope, q_pe, z, kpe, w_uk, w_uv, seqlens, paged, cap, table,
                     1.0 / math.sqrt(d + p))


# --- the five workloads -----------------------------------------------------

@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "gqa" or "mla"
    b: int
    heads: int                # Hq (gqa) or h (mla)
    d: int
    s: int = 1
    t: int = 4096
    hkv: int = 0              # gqa only
    k: int = 0                # mla only
    p: int = 0                # mla only
    paged: bool = False
    ragged: tuple = ()        # (lo, hi) for uniform ragged lengths
    seed: int = 0

    def seqlens(self):
        if self.ragged:
            return ragged_seqlens(self.b, self.ragged[0], self.ragged[1], self.seed)
        # context t prior tokens plus the s new ones when s > 1 (MTP); for s = 1
        # the new token's key is already among the t cached ones
        L = self.t + (self.s if self.s > 1 else 0)
        return [L] * self.b


WORKLOADS = {
    "mla_tiny": Workload("mla_tiny b2 h16 d32 k64 p16 t256 s1", "mla", 2, 16, 32, 1, 256, k=64, p=16),
    "gqa_64_8": Workload("gqa b32 hq64 hkv8 d128 t4096 s1", "gqa", 32, 64, 128, 1, 4096, hkv=8),
    "mla_dsv3": Workload("mla b32 h128 d128 k512 p64 t4096 s1", "mla", 32, 128, 128, 1, 4096, k=512, p=64),
    **{f"mla_mtp_s{s}": Workload(f"mla b32 h128 d128 k512 p64 t4096+{s} s{s} causal", "mla", 32, 128, 128, s,
                                 4096, k=512, p=64) for s in (2, 4, 8, 16, 32, 64, 128)},
    **{f"gqa_paged_hkv{hk}": Workload(f"gqa paged b8 hq24 hkv{hk} d256 L~U[16384,32768] s1", "gqa", 8, 24, 256,
                                      1, 0, hkv=hk, paged=True, ragged=(16384, 32768))
       for hk in (24, 4, 1)},
}
