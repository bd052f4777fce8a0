"""Seeded synthetic decode workloads in the ``fp8_ds_mla`` paged latent-cache format
(and plain bf16 latent caches).

This module is the one piece shared by the CUDA path's tests/benchmark and by the
float64 oracle: it makes inputs and nothing else.  It contains none of the decode
arithmetic (no index conversion, no dequantisation, no attention).  The only
arithmetic here is the cache *writer's* quantisation rule, which defines what bytes a
cache holds:

* NoPE values (448 per row) are quantised per group of 64 with a UE8M0 scale code
  ``clamp(ceil(log2(amax / 448)) + 127, 0, 254)`` (amax = 0 gives code 0); code 255
  is never written (vLLM PR #52212 report, "实现拆解" item 3 and the
  ``fused_compress_quant_cache.py`` snippet: scale-code cap lowered to 254).  The
  fp8 byte is ``float8_e4m3fn(x / 2**(code-127))`` with round-to-nearest-even,
  delegated to torch's cast.
* RoPE values (64 per row) are stored as raw little-endian bf16.

Row and page layout (SGLang PR #26208 report, "关键源码片段",
``triton_mla_kernels_decode_dsv4.py`` constants and ``_gather_dequant_dsv4_kernel``):
a row is 576 data bytes (448 fp8 NoPE then 64 bf16 RoPE) plus 8 scale bytes (7 codes
and one zero pad byte).  A page of ``P`` slots stores its ``P`` data rows first
(``P * 576`` bytes) and then its ``P`` scale rows (``P * 8`` bytes).

Workloads follow the five decode shapes the benchmark is quoted on: tiny (1 token,
16 heads), single request (64 heads, 8k context, top-k 512 + window 128), mid batch
(32 x 128 heads, context U[4096, 32768], top-k 2048), large batch (256 x 64 heads,
top-k 512 + window 128) and long context (4 x 128 heads, 128k context, top-k 2048 +
window 128, 10 % of entries -1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

D_LATENT = 512
D_NOPE = 448
D_ROPE = 64
QUANT_GROUP = 64
N_SCALES = D_NOPE // QUANT_GROUP          # 7
ROW_DATA_BYTES = D_NOPE + 2 * D_ROPE      # 576
ROW_SCALE_BYTES = 8                       # 7 codes + 1 pad
ROW_BYTES = ROW_DATA_BYTES + ROW_SCALE_BYTES  # 584
FP8_MAX = 448.0
SEED_BASE = 20261202


@dataclass(frozen=True)
class Workload:
    """One synthetic decode step: ``num_tokens`` tokens, one per request."""

    name: str
    num_tokens: int
    num_heads: int
    topk: int
    swa: int
    ctx_lo: int
    ctx_hi: int
    block_size: int = 64
    n_invalid: int = 0          # entries per token (over both scopes) forced to -1
    max_splits: int = 0         # 0 = selector's own cap (32)
    extra_pages: int = 0        # unreferenced pages appended to the cache
    description: str = ""

    @property
    def n_entries(self) -> int:
        return self.topk + self.swa


WORKLOADS = [
    Workload("tiny_b1_h16_k64", 1, 16, 64, 0, 1024, 1024, n_invalid=8,
             description="batch 1, 16 heads, 1024-slot cache in 16 pages, top-k 64 with 8 entries -1"),
    Workload("single_b1_h64_k512_w128", 1, 64, 512, 128, 8192, 8192, max_splits=8,
             description="batch 1, 64 heads, context 8192, top-k 512 + window 128, up to 8 splits"),
    Workload("midbatch_b32_h128_k2048", 32, 128, 2048, 0, 4096, 32768,
             description="batch 32, 128 heads, context U[4096,32768], top-k 2048"),
    Workload("largebatch_b256_h64_k512_w128", 256, 64, 512, 128, 8192, 8192, max_splits=1,
             description="batch 256, 64 heads, context 8192, top-k 512 + window 128, no split"),
    Workload("longctx_b4_h128_k2048_w128", 4, 128, 2048, 128, 131072, 131072, n_invalid=217,
             max_splits=32,
             description="batch 4, 128 heads, context 131072, top-k 2048 + window 128, 217 of 2176 entries -1"),
]


@dataclass
class DecodeInputs:
    """Everything one decode step reads, plus bookkeeping counts from construction."""

    workload: Workload
    q: torch.Tensor               # bf16 [T, H, 512]
    kv_cache: torch.Tensor        # uint8 [num_pages, P*584]
    block_table: torch.Tensor     # int32 [R, max_blocks]
    req_id: torch.Tensor          # int32 [T]
    topk_idx: torch.Tensor        # int32 [T, K]
    swa_idx: torch.Tensor         # int32 [T, W]
    sink: torch.Tensor            # float32 [H]
    scale: float
    ctx_lens: list = field(default_factory=list)
    n_set_invalid: int = 0        # entries the generator wrote as -1 (padding + forced)

    @property
    def num_pages(self) -> int:
        return int(self.kv_cache.shape[0])

    @property
    def block_size(self) -> int:
        return self.workload.block_size

    @property
    def n_valid(self) -> int:
        """Entries that address a real slot, counted from how they were built."""
        w = self.workload
        return w.num_tokens * w.n_entries - self.n_set_invalid


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def ue8m0_codes(amax: torch.Tensor) -> torch.Tensor:
    """Writer rule: smallest k with 448 * 2**k >= amax, code = clamp(k + 127, 0, 254).

    ``amax`` is float32; the search is done in float64, where 448 * 2**k is exact, so
    the result is the exact ceiling of log2(amax / 448).  amax == 0 gives code 0.
    """
    a = amax.to(torch.float64)
    ratio = a / FP8_MAX
    safe = torch.where(a > 0, ratio, torch.ones_like(ratio))
    _, e = torch.frexp(safe)
    k = e.to(torch.int64)  # safe = m * 2**e, m in [0.5, 1) -> ceil(log2) in {e-1, e}
    two = torch.full_like(a, 2.0)
    lower = FP8_MAX * torch.pow(two, (k - 1).to(torch.float64))
    k = torch.where(lower >= a, k - 1, k)
    upper = FP8_MAX * torch.pow(two, k.to(torch.float64))
    k = torch.where(upper < a, k + 1, k)
    code = torch.clamp(k + 127, 0, 254)
    code = torch.where(a > 0, code, torch.zeros_like(code))
    return code.to(torch.uint8)


def quantize_rows(nope: torch.Tensor, rope: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """Encode float32 NoPE [n,448] and bf16 RoPE [n,64] into (data u8 [n,576], scale u8 [n,8])."""
    n = nope.shape[0]
    groups = nope.reshape(n, N_SCALES, QUANT_GROUP)
    codes = ue8m0_codes(groups.abs().amax(dim=-1))                       # [n,7]
    inv = torch.pow(torch.full_like(codes, 2.0, dtype=torch.float64),
                    127.0 - codes.to(torch.float64))                     # 2**(127-code)
    y = (groups.to(torch.float64) * inv.unsqueeze(-1)).to(torch.float32)  # exact: power-of-2 scale
    fp8 = y.reshape(n, D_NOPE).to(torch.float8_e4m3fn).view(torch.uint8)
    rope_bytes = rope.to(torch.bfloat16).contiguous().view(torch.uint8).reshape(n, 2 * D_ROPE)
    data = torch.cat([fp8, rope_bytes], dim=1)
    scale = torch.zeros(n, ROW_SCALE_BYTES, dtype=torch.uint8, device=nope.device)
    scale[:, :N_SCALES] = codes
    return data, scale


def make_cache(num_pages: int, block_size: int, seed: int, device, chunk_pages: int = 2048
               ) -> torch.Tensor:
    """A cache of ``num_pages`` pages whose every slot holds a row quantised from N(0,1)."""
    P = block_size
    cache = torch.empty(num_pages, P * ROW_BYTES, dtype=torch.uint8, device=device)
    g = _gen(seed, device)
    chunk_pages = max(1, min(chunk_pages, max(1, (1 << 21) // P)))
    for p0 in range(0, num_pages, chunk_pages):
        p1 = min(num_pages, p0 + chunk_pages)
        n = (p1 - p0) * P
        nope = torch.randn(n, D_NOPE, generator=g, device=device, dtype=torch.float32)
        rope = torch.randn(n, D_ROPE, generator=g, device=device, dtype=torch.float32)
        data, scale = quantize_rows(nope, rope)
        pages = cache[p0:p1]
        pages[:, : P * ROW_DATA_BYTES] = data.reshape(p1 - p0, P * ROW_DATA_BYTES)
        pages[:, P * ROW_DATA_BYTES:] = scale.reshape(p1 - p0, P * ROW_SCALE_BYTES)
    return cache


ROW_BYTES_BF16 = 2 * D_LATENT  # a bf16 cache row: 512 little-endian bf16 values


def make_cache_bf16(num_pages: int, block_size: int, seed: int, device) -> torch.Tensor:
    """A bf16 latent cache u8 [num_pages, P * 1024]: every slot holds 512 N(0,1) values
    rounded to bf16 (NoPE then RoPE), one row after another."""
    g = _gen(seed, device)
    vals = torch.randn(num_pages * block_size, D_LATENT, generator=g, device=device).to(torch.bfloat16)
    return vals.view(torch.uint8).reshape(num_pages, block_size * ROW_BYTES_BF16)


def make_inputs(w: Workload, seed: int | None = None, device="cpu") -> DecodeInputs:
    """Build one decode step for workload ``w`` (seeded; separate streams per tensor)."""
    if seed is None:
        seed = SEED_BASE + WORKLOADS.index(w) if w in WORKLOADS else SEED_BASE
    P = w.block_size
    T, H, K, W = w.num_tokens, w.num_heads, w.topk, w.swa
    g_idx = _gen(seed * 4 + 1, device)
    g_q = _gen(seed * 4 + 2, device)
    g_sink = _gen(seed * 4 + 3, device)

    # context lengths (one request per token) and disjoint page ranges per request
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

    topk = torch.full((T, K), -1, dtype=torch.int32, device=device)
    swa = torch.full((T, W), -1, dtype=torch.int32, device=device)
    n_set_invalid = 0
    for t in range(T):
        c = ctx[t]
        kk = min(K, c)
        if kk:
            topk[t, :kk] = torch.randperm(c, generator=g_idx, device=device)[:kk].to(torch.int32)
        n_set_invalid += K - kk
        ww = min(W, c)
        if ww:
            swa[t, :ww] = torch.arange(c - ww, c, dtype=torch.int32, device=device)
        n_set_invalid += W - ww
    if w.n_invalid:
        both = torch.cat([topk, swa], dim=1)
        for t in range(T):
            valid_pos = (both[t] >= 0).nonzero().flatten()
            pick = valid_pos[torch.randperm(valid_pos.numel(), generator=g_idx,
                                            device=device)[: w.n_invalid]]
            both[t, pick] = -1
            n_set_invalid += int(pick.numel())
        topk = both[:, :K].contiguous()
        swa = both[:, K:].contiguous()

    q = torch.randn(T, H, D_LATENT, generator=g_q, device=device).to(torch.bfloat16)
    sink = torch.randn(H, generator=g_sink, device=device, dtype=torch.float32)
    cache = make_cache(num_pages, P, seed * 4 + 0, device)
    req_id = torch.arange(T, dtype=torch.int32, device=device)
    return DecodeInputs(w, q, cache, block_table, req_id, topk, swa, sink,
                        1.0 / math.sqrt(D_LATENT), ctx, n_set_invalid)


def small_workload(name="small", num_tokens=3, num_heads=16, topk=96, swa=32, ctx=300,
                   block_size=64, n_invalid=5, extra_pages=1) -> Workload:
    """A parametrised small shape for parity sweeps."""
    return Workload(name, num_tokens, num_heads, topk, swa, ctx, ctx, block_size=block_size,
                    n_invalid=n_invalid, extra_pages=extra_pages)
