"""Ragged and length-limited index forms (CPU oracle; the next step after the dense path).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/`` may use it, and it
shares no code with the CUDA path.  Plain NumPy, integer arithmetic, one loop per rule.

* ``apply_topk_length`` -- the per-sequence top-k length cut of SGLang PR #26208 report,
  "关键源码片段", ``_gather_dequant_dsv4_kernel`` (its ``HAS_TOPK_LENGTH`` branch): the
  entry in column k of token t is invalid when k >= TopkLength[t // s_q], where s_q is
  the number of query tokens per sequence.
* ``convert_req_index_ragged`` -- the ragged form of the index conversion in vLLM PR
  #41217 report, "关键源码片段", ``_convert_req_index_to_global_index_kernel``: token t
  owns output positions [cu_seqlens[t], cu_seqlens[t + 1]) and fills position
  cu_seqlens[t] + j from column j of its request-local indices; an index that is
  negative or whose block lies outside [0, max_blocks) is written as 0 (the pages' fill,
  which a real slot 0 shares -- the reason the dense form here uses -1 instead).  That
  kernel checks neither the request id nor the physical page, and neither does this.
* ``compact`` -- the valid entries of a dense [T, N] slot array (-1 = invalid), in
  order, as (cu_seqlens, slots): the rows the gather has to fetch once the invalid ones
  are skipped (vLLM PR #41217 report, "实现拆解" item 2, sparse sequence lengths built
  ahead of the decode; the pages print no body for that builder, so the lengths are
  read as the count of valid entries per token).
"""
from __future__ import annotations

import numpy as np


def apply_topk_length(topk_idx, topk_length, queries_per_seq: int = 1) -> np.ndarray:
    """Copy of ``topk_idx`` [T, K] with column k of token t set to -1 when
    k >= topk_length[t // queries_per_seq]."""
    idx = np.array(topk_idx, dtype=np.int64, copy=True)
    lengths = np.asarray(topk_length, dtype=np.int64).reshape(-1)
    s_q = int(queries_per_seq)
    T, K = idx.shape
    for t in range(T):
        limit = lengths[t // s_q]
        for k in range(K):
            if k >= limit:
                idx[t, k] = -1
    return idx


def convert_req_index_ragged(req_id, block_table, token_indices, cu_seqlens,
                             block_size: int) -> np.ndarray:
    """Ragged conversion with 0 for invalid entries: int64 [cu_seqlens[-1]]."""
    P = int(block_size)
    bt = np.asarray(block_table, dtype=np.int64)
    max_blocks = bt.shape[1]
    req = np.asarray(req_id, dtype=np.int64).reshape(-1)
    ti = np.asarray(token_indices, dtype=np.int64)
    cu = np.asarray(cu_seqlens, dtype=np.int64).reshape(-1)
    out = np.zeros(int(cu[-1]), dtype=np.int64)
    for t in range(req.shape[0]):
        start, end = int(cu[t]), int(cu[t + 1])
        for j in range(end - start):
            tok = ti[t, j]
            block, off = tok // P, tok % P
            if tok < 0 or block < 0 or block >= max_blocks:
                out[start + j] = 0
            else:
                out[start + j] = bt[req[t], block] * P + off
    return out


def compact(slots) -> tuple[np.ndarray, np.ndarray]:
    """(cu_seqlens int64 [T + 1], valid slots int64 [cu_seqlens[-1]]) of a dense [T, N]
    slot array, keeping each token's valid entries in their original order."""
    g = np.asarray(slots, dtype=np.int64)
    T = g.shape[0]
    cu = np.zeros(T + 1, dtype=np.int64)
    kept = []
    for t in range(T):
        for s in g[t]:
            if s >= 0:
                kept.append(int(s))
        cu[t + 1] = len(kept)
    return cu, np.asarray(kept, dtype=np.int64)
