"""Indexer side of the sparse decode: the step that chooses each token's top-k positions
(CPU oracle).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may use it, and it shares no code
with the CUDA path.  Plain NumPy, float64 arithmetic, one loop per rule.

What the pages fix, and where:

* ``cp_gather_indexer_k`` -- vLLM PR #52212 report, "关键源码片段",
  ``_cp_gather_indexer_quant_cache_gfx950_kernel`` and "实现拆解" item 4: one program per
  token ``tid`` of a ragged batch; its sequence is ``token_to_seq[tid]``, valid when in
  ``[0, num_batches)``; the token must lie in ``[cu_seqlen[b], cu_seqlen[b + 1])``, else
  nothing is written; its position in the sequence, ``tid - cu_seqlen[b]``, selects a
  block-table entry whose page must lie in ``[0, NUM_BLOCKS)``; the token's fp8 key row
  (``HEAD_DIM`` bytes) is copied to ``k_fp8[tid]`` only from a valid page, and its scale
  is written to ``k_scale[tid]`` (0 for an invalid page).
* ``mqa_logits`` -- vLLM PR #41217 report, "实现拆解" item 6 (the fp8 paged MQA logits:
  per query token and cached position, one kernel in place of per-head scores followed
  by a sum over heads) and "关键源码片段", ``SparseAttnIndexer.forward`` (one projection
  gives the indexer key -- ``head_dim`` values per position -- and a weight per head; the
  query has ``n_head`` heads of ``head_dim``).
* ``topk_positions`` -- the indexer's output is the request-local top-k index list the
  sparse decode reads (``topk_idx`` of ``sparse_mla_decode``).

Readings where the pages are silent:

* Cache layout.  The gather kernel takes a LAYOUT switch it does not print.  Layout 0
  (the one the logits use) stores a page of ``P`` positions as ``P * D`` fp8 bytes then
  ``P`` little-endian float32 scales -- the same values-then-scales split as the
  ``fp8_ds_mla`` page; layout 1 interleaves each position's ``D`` bytes and its scale.
* Key value: ``k[d] = e4m3(byte[d]) * scale`` (one float32 scale per position).
* Logit: ``logit[t, s] = sum_h w[t, h] * max(0, sum_d e4m3(q[t, h, d]) * k_s[d])``.  The
  pages name per-head scores summed with per-head weights; a score linear in q would let
  the heads fold into one vector before the dot, so the per-head stage implies a
  per-head non-linearity, read here as the rectifier.  The query carries no scale of its
  own (the weights absorb it).
* Positions at or past the token's context, and positions whose page is outside the
  cache or whose block is outside the table, get ``-inf``.
* Top-k: the ``K`` positions with the largest finite logits, in descending order of
  logit and ascending position among equal logits; ``-1`` pads a token with fewer than
  ``K`` finite logits.  Any other order of the same positions selects the same rows.
"""
from __future__ import annotations

import numpy as np

from .sparse_mla import decode_e4m3


def page_offsets(pos_in_page: int, P: int, D: int, layout: int) -> tuple[int, int]:
    """Byte offsets, within a page, of a position's D key bytes and of its float32 scale."""
    if layout == 0:
        return pos_in_page * D, P * D + 4 * pos_in_page
    if layout == 1:
        return pos_in_page * (D + 4), pos_in_page * (D + 4) + D
    raise ValueError("layout is 0 (values then scales) or 1 (interleaved)")


def _scale_at(page_bytes: np.ndarray, off: int) -> float:
    return float(np.frombuffer(page_bytes[off:off + 4].tobytes(), dtype="<f4")[0])


def cp_gather_indexer_k(cache, block_table, cu_seqlen, token_to_seq, num_batches: int, P: int, D: int,
                        layout: int = 0, k_init=None, s_init=None):
    """Gather each ragged token's key bytes and scale (see the module notes).

    cache u8 [num_blocks, page_bytes]; block_table int [B, W]; cu_seqlen int [B + 1];
    token_to_seq int [n].  Returns (k u8 [n, D], k_scale f32 [n]) starting from copies of
    ``k_init`` / ``s_init`` (the untouched contents; zeros if not given), so that entries
    the rule does not write keep their old value."""
    cache = np.asarray(cache, dtype=np.uint8)
    bt = np.asarray(block_table)
    cu = np.asarray(cu_seqlen)
    tts = np.asarray(token_to_seq)
    n = tts.shape[0]
    num_blocks = cache.shape[0]
    k = np.zeros((n, D), np.uint8) if k_init is None else np.array(k_init, dtype=np.uint8, copy=True)
    s = np.zeros(n, np.float32) if s_init is None else np.array(s_init, dtype=np.float32, copy=True)
    for tid in range(n):
        b = int(tts[tid])
        if not (0 <= b < num_batches):
            continue
        start, end = int(cu[b]), int(cu[b + 1])
        if not (start <= tid < end):
            continue
        pos = tid - start
        blk, off = divmod(pos, P)
        page = int(bt[b, blk]) if blk < bt.shape[1] else -1
        if not (0 <= page < num_blocks):
            s[tid] = 0.0
            continue
        vo, so = page_offsets(off, P, D, layout)
        k[tid] = cache[page, vo:vo + D]
        s[tid] = _scale_at(cache[page], so)
    return k, s


def key_rows(cache, pages_offsets, P: int, D: int, layout: int = 0) -> np.ndarray:
    """float64 keys [n, D] of the (page, in-page position) pairs: e4m3 bytes times scale."""
    cache = np.asarray(cache, dtype=np.uint8)
    out = np.empty((len(pages_offsets), D))
    for i, (page, off) in enumerate(pages_offsets):
        vo, so = page_offsets(off, P, D, layout)
        out[i] = decode_e4m3(cache[page, vo:vo + D]) * _scale_at(cache[page], so)
    return out


def mqa_logits(q_codes, weights, cache, block_table, req_id, ctx_lens, P: int, D: int, layout: int = 0,
               max_len: int | None = None) -> np.ndarray:
    """float64 logits [T, L] (L = max_len or the largest context) of every query token
    against every position of its request's context (see the module notes)."""
    q = decode_e4m3(np.asarray(q_codes, dtype=np.uint8))          # [T, H, D]
    w = np.asarray(weights, dtype=np.float64)                       # [T, H]
    cache = np.asarray(cache, dtype=np.uint8)
    bt = np.asarray(block_table)
    ctx = np.asarray(ctx_lens)
    T = q.shape[0]
    L = int(max_len if max_len is not None else (ctx.max() if T else 0))
    out = np.full((T, L), -np.inf)
    num_blocks = cache.shape[0]
    for t in range(T):
        r = int(req_id[t])
        n = min(int(ctx[t]), L)
        if not (0 <= r < bt.shape[0]) or n <= 0:
            continue
        pos = np.arange(n)
        blk, off = pos // P, pos % P
        ok = blk < bt.shape[1]
        page = np.full(n, -1)
        page[ok] = bt[r, blk[ok]]
        ok &= (page >= 0) & (page < num_blocks)
        idx = np.nonzero(ok)[0]
        if idx.size == 0:
            continue
        k = key_rows(cache, list(zip(page[idx].tolist(), off[idx].tolist())), P, D, layout)  # [m, D]
        scores = q[t] @ k.T                                       # [H, m]
        out[t, idx] = (w[t][:, None] * np.maximum(scores, 0.0)).sum(axis=0)
    return out


def topk_positions(logits, K: int) -> np.ndarray:
    """int32 [T, K]: per row the K positions of the largest finite logits, descending by
    logit, ascending by position among equal logits; -1 pads rows with fewer."""
    lg = np.asarray(logits)
    T = lg.shape[0]
    out = np.full((T, K), -1, dtype=np.int32)
    for t in range(T):
        fin = np.nonzero(np.isfinite(lg[t]))[0]
        order = sorted(fin.tolist(), key=lambda s: (-lg[t, s], s))
        take = order[:K]
        out[t, :len(take)] = take
    return out
