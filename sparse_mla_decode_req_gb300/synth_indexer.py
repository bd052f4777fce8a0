"""Seeded synthetic inputs of the indexer step (the step that picks each decode token's
top-k positions) over an fp8 paged key cache.

Like ``synth``, this module makes inputs and nothing else: no logits, no selection, no
gather.  The one arithmetic here is the cache writer's quantisation rule, which fixes
the bytes a cache holds (a reading: the pages print the gather of this cache, not its
writer):

* a position's key is ``head_dim`` values drawn from N(0,1), stored as fp8 e4m3 bytes
  ``float8_e4m3fn(x / scale)`` (torch's round-to-nearest-even cast) with one float32
  scale per position, ``scale = amax / 448`` (amax > 0 for Gaussian rows);
* page layout 0: a page of ``P`` positions holds their ``P * head_dim`` key bytes, then
  their ``P`` little-endian float32 scales; layout 1 interleaves each position's bytes
  and scale;
* the query is fp8 e4m3 bytes of N(0,1) values (no scale of its own), the per-head
  weights are N(0,1) / sqrt(heads) in float32.

Requests own disjoint page ranges, each block-table row a random permutation of them
(the decode workloads' recipe); one query token per request.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

from .synth import SEED_BASE, _gen

FP8_MAX = 448.0


@dataclass(frozen=True)
class IndexerWorkload:
    name: str
    num_tokens: int
    topk: int
    ctx_lo: int
    ctx_hi: int
    num_heads: int = 64
    head_dim: int = 128
    block_size: int = 64
    extra_pages: int = 0
    description: str = ""


@dataclass
class IndexerInputs:
    workload: IndexerWorkload
    q: torch.Tensor            # uint8 e4m3 [T, H, D]
    weights: torch.Tensor      # float32 [T, H]
    cache: torch.Tensor        # uint8 [num_pages, P * (D + 4)]
    block_table: torch.Tensor  # int32 [T, max_blocks]
    req_id: torch.Tensor       # int32 [T]
    ctx_lens: torch.Tensor     # int32 [T]
    layout: int = 0
    ctx: list = field(default_factory=list)

    @property
    def num_pages(self) -> int:
        return int(self.cache.shape[0])

    @property
    def max_len(self) -> int:
        return max(self.ctx) if self.ctx else 0


INDEXER_WORKLOADS = [
    IndexerWorkload("indexer_midbatch_b32_h64_d128_k2048", 32, 2048, 4096, 32768,
                    description="the mid-batch decode's top-k source: 32 requests, context "
                                "U[4096, 32768], 64 indexer heads of 128, top-k 2048"),
    IndexerWorkload("indexer_largebatch_b256_h64_d128_k512", 256, 512, 8192, 8192,
                    description="the large-batch decode's top-k source: 256 requests of 8192 "
                                "positions, 64 indexer heads of 128, top-k 512"),
]


def small_indexer_workload(name="small_indexer", num_tokens=3, topk=40, ctx_lo=100, ctx_hi=300,
                           num_heads=64, head_dim=128, block_size=64, extra_pages=1) -> IndexerWorkload:
    return IndexerWorkload(name, num_tokens, topk, ctx_lo, ctx_hi, num_heads, head_dim, block_size, extra_pages)


def quantize_keys(x: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """float32 [n, D] -> (e4m3 bytes [n, D], float32 scales [n]) by the writer rule."""
    amax = x.abs().amax(dim=1).clamp_min(torch.finfo(torch.float32).tiny)
    scale = (amax / FP8_MAX).to(torch.float32)
    codes = (x / scale[:, None]).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale


def make_indexer_cache(num_pages: int, P: int, D: int, seed: int, device, layout: int = 0,
                       chunk_pages: int = 1024) -> torch.Tensor:
    cache = torch.empty(num_pages, P * (D + 4), dtype=torch.uint8, device=device)
    g = _gen(seed, device)
    for p0 in range(0, num_pages, chunk_pages):
        p1 = min(num_pages, p0 + chunk_pages)
        n = (p1 - p0) * P
        x = torch.randn(n, D, generator=g, device=device, dtype=torch.float32)
        codes, scale = quantize_keys(x)
        sb = scale.view(torch.uint8).reshape(n, 4)
        pages = cache[p0:p1]
        if layout == 0:
            pages[:, : P * D] = codes.reshape(p1 - p0, P * D)
            pages[:, P * D:] = sb.reshape(p1 - p0, P * 4)
        else:
            rows = torch.cat([codes, sb], dim=1)  # [n, D + 4]
            pages[:] = rows.reshape(p1 - p0, P * (D + 4))
    return cache


def make_indexer_inputs(w: IndexerWorkload, seed: int | None = None, device="cpu", layout: int = 0) -> IndexerInputs:
    if seed is None:
        seed = SEED_BASE + 100 + (INDEXER_WORKLOADS.index(w) if w in INDEXER_WORKLOADS else 0)
    T, H, D, P = w.num_tokens, w.num_heads, w.head_dim, w.block_size
    g_idx = _gen(seed * 4 + 1, device)
    g_q = _gen(seed * 4 + 2, device)
    g_w = _gen(seed * 4 + 3, device)
    if w.ctx_lo == w.ctx_hi:
        ctx = [w.ctx_lo] * T
    else:
        ctx = torch.randint(w.ctx_lo, w.ctx_hi + 1, (T,), generator=g_idx, device=device).tolist()
    nblk = [math.ceil(c / P) for c in ctx]
    max_blocks = max(nblk) if nblk else 1
    num_pages = sum(nblk) + w.extra_pages
    block_table = torch.full((T, max_blocks), -1, dtype=torch.int32, device=device)
    base = 0
    for r in range(T):
        perm = torch.randperm(nblk[r], generator=g_idx, device=device) + base
        block_table[r, : nblk[r]] = perm.to(torch.int32)
        base += nblk[r]
    q = torch.randn(T, H, D, generator=g_q, device=device).to(torch.float8_e4m3fn).view(torch.uint8)
    weights = (torch.randn(T, H, generator=g_w, device=device) / math.sqrt(H)).to(torch.float32)
    cache = make_indexer_cache(num_pages, P, D, seed * 4, device, layout)
    req_id = torch.arange(T, dtype=torch.int32, device=device)
    ctx_lens = torch.tensor(ctx, dtype=torch.int32, device=device)
    return IndexerInputs(w, q, weights, cache, block_table, req_id, ctx_lens, layout, ctx)
