"""Float64 CPU oracle for sparse MLA decode (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package; the product path never does.
"""
from .sparse_mla import (  # noqa: F401
    attend, convert_req_index, decode_bf16, decode_e4m3, decode_ue8m0, dequant_rows,
    lse_combine, row_offsets, sparse_mla_decode,
)
from .indexer import cp_gather_indexer_k, mqa_logits, topk_positions  # noqa: F401,E402
