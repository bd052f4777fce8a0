"""Two-cache decode: top-k entries over one paged cache, window entries over another.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/`` may use it, and it
shares no code with the CUDA path.

The DeepSeek-V4 decode the pages describe attends over two scopes in one softmax: the
main (top-k) entries of the compressed cache and the sliding-window entries of the window
cache (vLLM PR #52212 report, "实现拆解" item 1: main and SWA work handled by one partial
kernel, with the sink and the invalid-index semantics kept; item 3: the compressed
"extra" cache beside the window cache; SGLang PR #26208 report, "功能与动机" item 3: the
fused dual-scope attention).  Both caches use the ``fp8_ds_mla`` row format; each has its
own block table and page size.  The plainest reading: each scope's request-local indices
go through its own block table and page range exactly as in ``convert_req_index``, the
valid rows of both scopes (top-k first, then the window) form one list, and ``attend``
runs once over it.
"""
from __future__ import annotations

import numpy as np

from .sparse_mla import attend, convert_req_index, dequant_rows


def sparse_mla_decode_dual(q, req_id, sink, scale,
                           main_cache, main_block_table, main_block_size, topk_idx,
                           swa_cache, swa_block_table, swa_block_size, swa_idx,
                           tokens=None) -> tuple[np.ndarray, np.ndarray]:
    """out float64 [T', H, 512] and lse [T', H] over both scopes (``q`` float64 [T, H, 512])."""
    q = np.asarray(q, dtype=np.float64)
    T, H, D = q.shape
    rid = np.asarray(req_id).reshape(-1)
    toks = range(T) if tokens is None else list(tokens)
    out = np.zeros((len(toks), H, D))
    lse = np.zeros((len(toks), H))
    main_pages = np.asarray(main_cache).shape[0]
    swa_pages = np.asarray(swa_cache).shape[0]
    for n, t in enumerate(toks):
        rows = []
        if topk_idx is not None:
            g = convert_req_index(rid[t:t + 1], main_block_table, np.asarray(topk_idx)[t:t + 1], None,
                                  main_block_size, main_pages)[0]
            rows.append(dequant_rows(main_cache, g[g >= 0], main_block_size))
        if swa_idx is not None:
            g = convert_req_index(rid[t:t + 1], swa_block_table, None, np.asarray(swa_idx)[t:t + 1],
                                  swa_block_size, swa_pages)[0]
            rows.append(dequant_rows(swa_cache, g[g >= 0], swa_block_size))
        k = np.concatenate(rows, axis=0) if rows else np.zeros((0, D))
        out[n], lse[n] = attend(q[t], k, sink, scale)
    return out, lse
