"""Decode over a bf16 latent cache (CPU oracle; the next step after the fp8 path).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/`` may use it, and it
shares no code with the CUDA path.

vLLM PR #41217 report lists a bf16-KV decode path (key symbol ``_forward_bf16_kv``) beside
the fp8 one but prints no layout.  The plainest reading: the same paged addressing with
one row of 512 bf16 latent values (1024 bytes, little-endian, NoPE then RoPE) per slot
and no scale rows; the attention is the fp8 path's with the rows read as they are, and
a non-finite element is zeroed as the fp8 path's scrub does.
"""
from __future__ import annotations

import numpy as np

from .sparse_mla import attend, convert_req_index, decode_bf16

ROW_BYTES = 1024


def dequant_rows_bf16(cache: np.ndarray, slots, block_size: int) -> np.ndarray:
    """Rows at global ``slots`` of a bf16 cache u8 [num_pages, block_size * 1024] as float64 [n, 512]."""
    flat = np.ascontiguousarray(cache).reshape(-1)
    slots = np.asarray(slots).astype(np.int64).reshape(-1)
    P = int(block_size)
    base = (slots // P) * (P * ROW_BYTES) + (slots % P) * ROW_BYTES
    b = flat[base[:, None] + np.arange(ROW_BYTES)].astype(np.uint16)
    k = decode_bf16(b[:, 0::2] | (b[:, 1::2] << np.uint16(8)))
    k[~np.isfinite(k)] = 0.0
    return k


def sparse_mla_decode_bf16(q, kv_cache, block_table, req_id, topk_idx, swa_idx, sink, scale,
                           block_size: int) -> tuple[np.ndarray, np.ndarray]:
    """out float64 [T, H, 512] and lse [T, H] over a bf16 latent cache."""
    q = np.asarray(q, dtype=np.float64)
    T, H, D = q.shape
    num_pages = np.asarray(kv_cache).shape[0]
    rid = np.asarray(req_id).reshape(-1)
    out = np.zeros((T, H, D))
    lse = np.zeros((T, H))
    for t in range(T):
        g = convert_req_index(rid[t:t + 1], block_table,
                              None if topk_idx is None else np.asarray(topk_idx)[t:t + 1],
                              None if swa_idx is None else np.asarray(swa_idx)[t:t + 1],
                              block_size, num_pages)[0]
        out[t], lse[t] = attend(q[t], dequant_rows_bf16(kv_cache, g[g >= 0], block_size), sink, scale)
    return out, lse
