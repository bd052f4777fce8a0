"""Float64 CPU oracle for sparse MLA decode over an ``fp8_ds_mla`` paged latent cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this module: only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference legs
use it.  It shares no code with the CUDA path (no kernels, headers, helpers, tables or
constants are common); its inputs are plain NumPy arrays.

Every function is the plain definition of one step, written out in float64:

* ``convert_req_index`` -- request-local index -> global slot through the block table
  (vLLM PR #41217 report, "关键源码片段", ``_convert_req_index_to_global_index_kernel``;
  the physical-page range check follows vLLM PR #52212 report, "关键源码片段",
  ``_cp_gather_indexer_quant_cache_gfx950_kernel``).  Invalid entries become -1.
* ``decode_e4m3`` / ``decode_ue8m0`` / ``decode_bf16`` / ``dequant_rows`` -- the cache
  row format (SGLang PR #26208 report, "关键源码片段", ``triton_mla_kernels_decode_dsv4.py``
  constants and ``_gather_dequant_dsv4_kernel`` offsets), with the decode-side scrub of
  non-finite values (vLLM PR #52212 report, "实现拆解" item 3 and the ``rocm.py``
  snippet: element-wise scrub unless the cache is trusted NaN-free).
* ``attend`` -- one 512-wide QK dot for all heads, softmax with a per-head sink logit
  in the denominator, PV over the same 512-wide latent (vLLM PR #52212 report, "实现拆解"
  item 1; SGLang PR #26208 report, ``_unified_sparse_decode_kernel`` interface
  ``Q, KV, Mask, AttnSink, Output, LSE, sm_scale``), with the -inf guard of the same
  report's "评论区精华".
* ``lse_combine`` -- log-sum-exp merge of split partials (vLLM PR #52212 report,
  "实现拆解" item 2 and the test symbol ``_launch_sparse_decode_reduce``).

Readings where the pages are silent:
invalid conversion output is -1 (not 0 + ragged lengths); out-of-range request ids
invalidate the whole token; the sink is an unscaled logit that enters only the
denominator; ``lse`` is the natural log of the full denominator including the sink;
duplicated entries count once per occurrence; a latent element that is non-finite
once held as bf16 (NaN byte, scale code 255, non-finite RoPE, or a product beyond
bf16's finite range) is zeroed.
"""
from __future__ import annotations

import numpy as np

# Format facts, restated from the pages (not shared with any other module).
NOPE_DIMS = 448
ROPE_DIMS = 64
LATENT_DIMS = NOPE_DIMS + ROPE_DIMS        # 512: K = V latent
GROUP = 64                                  # one UE8M0 scale per 64 NoPE values
N_GROUPS = NOPE_DIMS // GROUP               # 7
DATA_BYTES = NOPE_DIMS + 2 * ROPE_DIMS      # 576
SCALE_BYTES = 8                             # 7 codes + 1 pad
# Smallest magnitude that bf16 round-to-nearest-even turns into infinity:
# halfway between the largest finite bf16 (0x1.fep127) and 2**128.
BF16_OVERFLOW = float.fromhex("0x1.ffp127")


# --------------------------------------------------------------------------- format
def decode_e4m3(b) -> np.ndarray:
    """fp8 e4m3 (the 'fn' variant: no infinities) byte -> float64.

    1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is
    subnormal (m * 2**-9); S.1111.111 is NaN; the largest finite value is 448.
    """
    b = np.asarray(b).astype(np.int64)
    sign = np.where((b >> 7) & 1, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    normal = (1.0 + m / 8.0) * np.ldexp(1.0, (e - 7).astype(np.int32))
    sub = m * 2.0 ** -9
    val = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & (m == 7), np.nan, val)


def decode_ue8m0(c) -> np.ndarray:
    """UE8M0 scale code -> 2**(code-127); code 255 is NaN."""
    c = np.asarray(c).astype(np.int64)
    return np.where(c == 255, np.nan, np.ldexp(1.0, (c - 127).astype(np.int32)))


def decode_bf16(u16) -> np.ndarray:
    """bf16 bit pattern (uint16) -> float64 (bf16 is the top half of a float32)."""
    u = np.asarray(u16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


def row_offsets(slots: np.ndarray, block_size: int) -> tuple[np.ndarray, np.ndarray]:
    """Byte offsets of (data row, scale row) of each global slot in the flat cache.

    A page of P slots holds P data rows of 576 bytes, then P scale rows of 8 bytes.
    """
    P = int(block_size)
    slots = np.asarray(slots).astype(np.int64)
    page = slots // P
    off = slots % P
    page_bytes = P * (DATA_BYTES + SCALE_BYTES)
    return page * page_bytes + off * DATA_BYTES, page * page_bytes + P * DATA_BYTES + off * SCALE_BYTES


def dequant_rows(cache: np.ndarray, slots, block_size: int) -> np.ndarray:
    """Decode cache rows at global ``slots`` into float64 latent vectors [n, 512].

    k[d] = e4m3(byte d) * 2**(code[d // 64] - 127) for d < 448, k[448 + r] = rope[r];
    an element that is NaN/inf, or whose magnitude overflows bf16, is set to 0.
    """
    flat = np.ascontiguousarray(cache).reshape(-1)
    slots = np.asarray(slots).astype(np.int64).reshape(-1)
    d_off, s_off = row_offsets(slots, block_size)
    data = flat[d_off[:, None] + np.arange(DATA_BYTES)]
    codes = flat[s_off[:, None] + np.arange(N_GROUPS)]
    nope = decode_e4m3(data[:, :NOPE_DIMS]) * np.repeat(decode_ue8m0(codes), GROUP, axis=1)
    rope_bits = data[:, NOPE_DIMS:].astype(np.uint16)
    rope = decode_bf16(rope_bits[:, 0::2] | (rope_bits[:, 1::2] << np.uint16(8)))  # little-endian
    k = np.concatenate([nope, rope], axis=1)
    with np.errstate(invalid="ignore"):
        bad = ~np.isfinite(k) | (np.abs(k) >= BF16_OVERFLOW)
    k[bad] = 0.0
    return k


# ------------------------------------------------------------------ index conversion
def convert_req_index(req_id, block_table, topk_idx, swa_idx, block_size: int,
                      num_pages: int) -> np.ndarray:
    """Request-local indices -> global cache slots, int64 [T, K+W] (-1 = invalid).

    Top-k entries come first and the sliding-window entries follow at offset K.  For
    token t and index i: i < 0 -> invalid; block b = i // P and offset o = i % P;
    b outside [0, max_blocks) -> invalid; page = block_table[req_id[t], b]; page
    outside [0, num_pages) -> invalid; otherwise the slot is page * P + o.
    """
    P = int(block_size)
    bt = np.asarray(block_table).astype(np.int64)
    R, max_blocks = bt.shape
    req = np.asarray(req_id).astype(np.int64).reshape(-1)
    T = req.shape[0]
    parts = [np.asarray(a).astype(np.int64).reshape(T, -1) for a in (topk_idx, swa_idx)
             if a is not None]
    idx = np.concatenate(parts, axis=1) if parts else np.zeros((T, 0), np.int64)
    out = np.full(idx.shape, -1, dtype=np.int64)
    for t in range(T):
        r = req[t]
        if r < 0 or r >= R:
            continue
        for j in range(idx.shape[1]):
            i = idx[t, j]
            if i < 0:
                continue
            b, o = i // P, i % P
            if b >= max_blocks:
                continue
            page = bt[r, b]
            if page < 0 or page >= num_pages:
                continue
            out[t, j] = page * P + o
    return out


# ------------------------------------------------------------------------- attention
def attend(q: np.ndarray, k: np.ndarray, sink, scale: float) -> tuple[np.ndarray, np.ndarray]:
    """Sink-augmented softmax attention of H query heads over n latent rows (K = V).

    s[h, e] = scale * q[h] . k[e];  den[h] = sum_e exp(s[h, e]) + exp(sink[h]);
    out[h] = sum_e exp(s[h, e]) k[e] / den[h];  lse[h] = ln den[h].
    Evaluated max-shifted.  With no rows and no sink: out = 0 and lse = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64).reshape(-1, q.shape[-1])
    H = q.shape[0]
    sink = np.full(H, -np.inf) if sink is None else np.asarray(sink, dtype=np.float64)
    s = scale * (q @ k.T)                                   # [H, n]
    m = np.maximum(s.max(axis=1) if k.shape[0] else np.full(H, -np.inf), sink)
    out = np.zeros((H, q.shape[-1]))
    lse = np.full(H, -np.inf)
    live = np.isfinite(m)                                   # -inf guard
    if live.any():
        ml = m[live]
        w = np.exp(s[live] - ml[:, None])
        den = w.sum(axis=1) + np.exp(sink[live] - ml)
        out[live] = (w @ k) / den[:, None]
        lse[live] = ml + np.log(den)
    return out, lse


def lse_combine(o_parts, lse_parts, sink) -> tuple[np.ndarray, np.ndarray]:
    """Merge split partials (each normalised over its own rows, no sink) with the sink.

    M = max(max_s lse_s, sink); w_s = exp(lse_s - M); den = sum_s w_s + exp(sink - M);
    out = sum_s w_s o_s / den; lse = M + ln den.  o_parts [S, ..., D], lse_parts [S, ...].
    """
    o = np.asarray(o_parts, dtype=np.float64)
    l = np.asarray(lse_parts, dtype=np.float64)
    sk = np.full(l.shape[1:], -np.inf) if sink is None else np.broadcast_to(
        np.asarray(sink, dtype=np.float64), l.shape[1:])
    M = np.maximum(l.max(axis=0) if l.shape[0] else np.full(l.shape[1:], -np.inf), sk)
    out = np.zeros(o.shape[1:])
    lse = np.full(l.shape[1:], -np.inf)
    live = np.isfinite(M)
    if live.any():
        w = np.where(np.isfinite(l), np.exp(l - np.where(live, M, 0.0)), 0.0)
        w = np.where(live, w, 0.0)
        den = w.sum(axis=0) + np.where(live, np.exp(sk - np.where(live, M, 0.0)), 0.0)
        num = (w[..., None] * o).sum(axis=0)
        out[live] = num[live] / den[live][..., None]
        lse[live] = M[live] + np.log(den[live])
    return out, lse


# ----------------------------------------------------------------------- whole step
def sparse_mla_decode(q, kv_cache, block_table, req_id, topk_idx, swa_idx, sink, scale,
                      block_size: int, tokens=None) -> tuple[np.ndarray, np.ndarray]:
    """The decode step: convert, gather + dequantise the valid rows, attend per token.

    ``q`` is float64 [T, H, 512] (already decoded from bf16); returns float64 out
    [T', H, 512] and lse [T', H] for the tokens in ``tokens`` (default: all).
    """
    q = np.asarray(q, dtype=np.float64)
    T, H, _ = q.shape
    num_pages = np.asarray(kv_cache).shape[0]
    toks = range(T) if tokens is None else list(tokens)
    out = np.zeros((len(toks), H, LATENT_DIMS))
    lse = np.zeros((len(toks), H))
    bt = np.asarray(block_table)
    rid = np.asarray(req_id).reshape(-1)
    for n, t in enumerate(toks):
        g = convert_req_index(rid[t:t + 1], bt,
                              None if topk_idx is None else np.asarray(topk_idx)[t:t + 1],
                              None if swa_idx is None else np.asarray(swa_idx)[t:t + 1],
                              block_size, num_pages)[0]
        rows = g[g >= 0]
        k = dequant_rows(kv_cache, rows, block_size)
        out[n], lse[n] = attend(q[t], k, sink, scale)
    return out, lse
