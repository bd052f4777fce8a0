"""Thin ctypes binding of libsmd (``include/smd.h``), with the same names.

Argument marshalling only: shapes, strides and device pointers are read from torch
tensors and passed to the C ABI; every step of the decode runs in the library's CUDA
kernels.  There is no CPU fallback: if ``libsmd.so`` is missing or fails to load, the
first call raises.  Build it with ``python -m sparse_mla_decode_req_gb300.build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsmd.so")

SMD_OK = 0
SMD_ERR_INVALID_ARG = -1
SMD_ERR_UNSUPPORTED = -2
SMD_ERR_WORKSPACE = -3
SMD_ERR_CUDA = -4
SMD_ERR_TIMEOUT = -5
SMD_ERR_DEVICE_CHECK = -6
LATENT_DIM = 512
ROW_BYTES = 584
ROW_BYTES_BF16 = 1024
MAX_SPLITS = 32
CACHE_FP8_DS_MLA = 0
CACHE_BF16 = 1


class SmdError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libsmd status {status}: {message}")
        self.status = status


class Dims(ctypes.Structure):
    """``smd_dims`` (include/smd.h)."""

    _fields_ = [
        ("num_tokens", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("num_requests", ctypes.c_int32),
        ("max_blocks_per_req", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
        ("block_size", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("swa", ctypes.c_int32),
        ("cache_format", ctypes.c_int32),
        ("bt_stride", ctypes.c_int64),
        ("topk_stride", ctypes.c_int64),
        ("swa_stride", ctypes.c_int64),
    ]


class IndexerDims(ctypes.Structure):
    """``smd_indexer_dims`` (include/smd.h)."""

    _fields_ = [
        ("num_tokens", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("num_requests", ctypes.c_int32),
        ("max_blocks_per_req", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
        ("bt_stride", ctypes.c_int64),
        ("max_len", ctypes.c_int32),
        ("layout", ctypes.c_int32),
    ]


class DecodeOpts(ctypes.Structure):
    """``smd_decode_opts`` (include/smd.h)."""

    _fields_ = [
        ("swa_kv_cache", ctypes.c_void_p),
        ("swa_block_table", ctypes.c_void_p),
        ("swa_num_pages", ctypes.c_int64),
        ("swa_bt_stride", ctypes.c_int64),
        ("swa_block_size", ctypes.c_int32),
        ("swa_max_blocks_per_req", ctypes.c_int32),
        ("topk_length", ctypes.c_void_p),
        ("compact", ctypes.c_int32),
        ("reserved_", ctypes.c_int32),
    ]


_lib = None

# name -> (restype, argtypes), mirroring include/smd.h
_P = ctypes.c_void_p
_SIGS = {
    "smd_select_num_splits": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_int]),
    "smd_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(Dims), ctypes.c_int, ctypes.c_int]),
    "smd_sparse_mla_decode": (ctypes.c_int, [ctypes.POINTER(Dims), _P, _P, _P, _P, _P, _P, _P, ctypes.c_float,
                                             _P, _P, ctypes.c_int, _P, ctypes.c_size_t, _P]),
    "smd_sparse_mla_decode_ex": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.POINTER(DecodeOpts), _P, _P, _P, _P,
                                                _P, _P, _P, ctypes.c_float, _P, _P, ctypes.c_int, _P,
                                                ctypes.c_size_t, _P]),
    "smd_sparse_mla_attention": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.POINTER(DecodeOpts), _P, _P, _P, _P,
                                                _P, ctypes.c_float, ctypes.c_int, _P, _P, _P, _P, _P, _P]),
    "smd_set_wait_limit_ns": (ctypes.c_uint64, [ctypes.c_uint64]),
    "smd_convert_req_index": (ctypes.c_int, [ctypes.POINTER(Dims), _P, _P, _P, _P, _P, _P]),
    "smd_convert_req_index_ex": (ctypes.c_int, [ctypes.POINTER(Dims), ctypes.POINTER(DecodeOpts), _P, _P, _P, _P,
                                                _P, _P, _P]),
    "smd_convert_req_index_ragged": (ctypes.c_int, [ctypes.POINTER(Dims), _P, _P, _P, ctypes.c_int32,
                                                    ctypes.c_int64, _P, _P, _P]),
    "smd_gather_dequant": (ctypes.c_int, [ctypes.POINTER(Dims), _P, _P, ctypes.c_int64, _P, _P]),
    "smd_lse_combine": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P, _P, _P, _P, _P, _P]),
    "smd_sparse_mla_decode_static_scratch": (ctypes.c_int, [ctypes.POINTER(Dims), _P, _P, _P, _P, _P, _P, _P,
                                                            ctypes.c_float, _P, _P, ctypes.c_int, _P]),
    "smd_read_status": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
    "smd_read_static_scratch_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32), _P]),
    "smd_indexer_gather_k": (ctypes.c_int, [_P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, _P, _P, ctypes.c_int32,
                                            _P, _P, _P]),
    "smd_indexer_mqa_logits": (ctypes.c_int, [ctypes.POINTER(IndexerDims), _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "smd_indexer_topk": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, _P, ctypes.c_int32,
                                        _P, _P]),
    "smd_last_error": (ctypes.c_char_p, []),
    "smd_version": (ctypes.c_int, []),
}


def lib_path() -> str:
    return _LIB_PATH


_LIB_DEBUG_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsmd_debug.so")
_handles: dict[str, ctypes.CDLL] = {}
_active = _LIB_PATH


def _open(path: str) -> ctypes.CDLL:
    if path not in _handles:
        if not os.path.exists(path):
            raise ImportError(f"{path} is not built; run python -m sparse_mla_decode_req_gb300.build")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _handles[path] = lib
    return _handles[path]


def load() -> ctypes.CDLL:
    """The active library (libsmd.so unless use_debug_library(True)); raise if it is not built."""
    global _lib
    _lib = _open(_active)
    return _lib


def use_debug_library(on: bool) -> None:
    """Route every call of this module to libsmd_debug.so (the SMD_DEBUG range-checking
    build) or back to libsmd.so."""
    global _active, _lib
    _active = _LIB_DEBUG_PATH if on else _LIB_PATH
    _lib = None
    load()


def last_error() -> str:
    return load().smd_last_error().decode()


def _check(status: int) -> int:
    if status < 0:
        raise SmdError(status, last_error())
    return status


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _row_stride(t, n_cols):
    if t is None or n_cols == 0:
        return max(n_cols, 0)
    st = t.stride()
    assert t.dtype is torch.int32 and len(st) == 2 and st[1] == 1, \
        "index tensors: int32 [rows, cols], unit column stride"
    return st[0]


def make_dims(q, kv_cache, block_table, req_id, topk_idx, swa_idx, block_size: int = 64,
              cache_format: int = CACHE_FP8_DS_MLA) -> Dims:
    """smd_dims from tensor shapes (q [T,H,512], kv_cache [pages, P*row bytes], block_table [R, B])."""
    T = req_id.shape[0]
    H = q.shape[1] if q is not None else 1
    K = 0 if topk_idx is None else topk_idx.shape[1]
    W = 0 if swa_idx is None else swa_idx.shape[1]
    R, B = block_table.shape
    # positional, in smd_dims field order (cheaper than keywords on every call)
    return Dims(T, H, R, B, kv_cache.shape[0], int(block_size), K, W, int(cache_format),
                _row_stride(block_table, B), _row_stride(topk_idx, K), _row_stride(swa_idx, W))


def make_opts(swa_kv_cache=None, swa_block_table=None, swa_block_size: int = 64, topk_length=None,
              compact: bool = False):
    """smd_decode_opts, or None when every option is off."""
    if swa_kv_cache is None and swa_block_table is None and topk_length is None and not compact:
        return None
    o = DecodeOpts()
    if swa_kv_cache is not None:
        assert swa_block_table is not None, "swa_kv_cache needs swa_block_table"
        B = int(swa_block_table.shape[1])
        o.swa_kv_cache = swa_kv_cache.data_ptr()
        o.swa_block_table = swa_block_table.data_ptr()
        o.swa_num_pages = int(swa_kv_cache.shape[0])
        o.swa_bt_stride = _row_stride(swa_block_table, B)
        o.swa_block_size = int(swa_block_size)
        o.swa_max_blocks_per_req = B
    if topk_length is not None:
        assert topk_length.dtype == torch.int32 and topk_length.is_contiguous()
        o.topk_length = topk_length.data_ptr()
    o.compact = int(bool(compact))
    return o


def _opts_ref(o):
    return None if o is None else ctypes.byref(o)


def select_num_splits(dims: Dims, num_splits: int = 0, num_sms: int = 0) -> int:
    return _check(load().smd_select_num_splits(ctypes.byref(dims), int(num_splits), int(num_sms)))


def workspace_size(dims: Dims, num_splits: int = 0, num_sms: int = 0) -> int:
    n = load().smd_workspace_size(ctypes.byref(dims), int(num_splits), int(num_sms))
    if n == 0:
        raise SmdError(SMD_ERR_INVALID_ARG, last_error())
    return int(n)


def sparse_mla_decode(q, kv_cache, block_table, req_id, topk_idx, swa_idx, sink, scale: float,
                      out=None, lse=None, num_splits: int = 0, workspace=None, block_size: int = 64,
                      stream=None, return_lse: bool = True, cache_format: int = CACHE_FP8_DS_MLA,
                      swa_kv_cache=None, swa_block_table=None, swa_block_size: int = 64, topk_length=None,
                      compact: bool = False):
    """Run one decode step; returns (out bf16 [T,H,512], lse f32 [T,H] or None).

    The keyword options map to smd_decode_opts: a separate window cache (swa_kv_cache,
    swa_block_table, swa_block_size), a per-token top-k length and compaction."""
    dims = make_dims(q, kv_cache, block_table, req_id, topk_idx, swa_idx, block_size, cache_format)
    opts = make_opts(swa_kv_cache, swa_block_table, swa_block_size, topk_length, compact)
    T, H = dims.num_tokens, dims.num_heads
    dev = q.device
    if out is None:
        out = torch.empty(T, H, LATENT_DIM, dtype=torch.bfloat16, device=dev)
    if lse is None and return_lse:
        lse = torch.empty(T, H, dtype=torch.float32, device=dev)
    if workspace is None:
        nbytes = workspace_size(dims, num_splits, torch.cuda.get_device_properties(dev).multi_processor_count)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    for name, t in (("q", q), ("kv_cache", kv_cache), ("out", out)):
        assert t.is_contiguous(), f"{name} must be contiguous"
    _check(load().smd_sparse_mla_decode_ex(
        ctypes.byref(dims), _opts_ref(opts), _ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(req_id),
        _ptr(topk_idx), _ptr(swa_idx), _ptr(sink), ctypes.c_float(scale), _ptr(out), _ptr(lse), int(num_splits),
        _ptr(workspace), ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream(stream)))
    return out, lse


def attention_dims(T: int, H: int, N: int, num_pages: int, block_size: int = 64, main: int | None = None,
                   cache_format: int = CACHE_FP8_DS_MLA) -> Dims:
    """smd_dims for the attention-only call over converted slots [T, N]; the first ``main``
    entries (default all) are the main scope."""
    K = N if main is None else int(main)
    return Dims(num_tokens=T, num_heads=H, num_requests=1, max_blocks_per_req=1, num_pages=int(num_pages),
                block_size=int(block_size), topk=K, swa=N - K, cache_format=int(cache_format), bt_stride=1,
                topk_stride=max(K, 1), swa_stride=max(N - K, 0))


def sparse_mla_attention(q, kv_cache, gidx, sink, scale: float, num_pages: int | None = None, num_splits: int = 0,
                         out=None, lse=None, o_part=None, lse_part=None, status=None, block_size: int = 64,
                         stream=None, counts=None, main: int | None = None, cache_format: int = CACHE_FP8_DS_MLA,
                         swa_kv_cache=None, swa_block_size: int = 64):
    """Fused gather + dequant + attention over converted slots gidx int32 [T, N].

    ``counts`` int32 [T, 2] (a compacted conversion's per-token counts) or ``main`` (the
    main-scope entries of each row, default all) say which entries read ``swa_kv_cache``.
    One split: returns (out, lse).  Several splits: returns (o_part, lse_part), the
    per-split partials for ``lse_combine``.
    """
    T, N = int(gidx.shape[0]), int(gidx.shape[1])
    H = int(q.shape[1])
    dims = attention_dims(T, H, N, int(kv_cache.shape[0] if num_pages is None else num_pages), block_size, main,
                          cache_format)
    opts = None
    if swa_kv_cache is not None:
        opts = DecodeOpts()
        opts.swa_kv_cache = swa_kv_cache.data_ptr()
        opts.swa_num_pages = int(swa_kv_cache.shape[0])
        opts.swa_block_size = int(swa_block_size)
    sms = torch.cuda.get_device_properties(q.device).multi_processor_count
    S = select_num_splits(dims, num_splits, sms)
    dev = q.device
    if S == 1 and out is None:
        out = torch.empty(T, H, LATENT_DIM, dtype=torch.bfloat16, device=dev)
    if S == 1 and lse is None:
        lse = torch.empty(T, H, dtype=torch.float32, device=dev)
    if S > 1 and o_part is None:
        o_part = torch.empty(T, S, H, LATENT_DIM, dtype=torch.float32, device=dev)
    if S > 1 and lse_part is None:
        lse_part = torch.empty(T, S, H, dtype=torch.float32, device=dev)
    assert gidx.dtype == torch.int32 and gidx.is_contiguous()
    assert counts is None or (counts.dtype == torch.int32 and counts.is_contiguous())
    _check(load().smd_sparse_mla_attention(ctypes.byref(dims), _opts_ref(opts), _ptr(q), _ptr(kv_cache), _ptr(gidx),
                                           _ptr(counts), _ptr(sink), ctypes.c_float(scale), int(num_splits),
                                           _ptr(out), _ptr(lse), _ptr(o_part), _ptr(lse_part), _ptr(status),
                                           _stream(stream)))
    return (out, lse) if S == 1 else (o_part, lse_part)


def convert_req_index(block_table, req_id, topk_idx, swa_idx, num_pages: int, block_size: int = 64,
                      gidx=None, stream=None, topk_length=None, compact: bool = False, swa_block_table=None,
                      swa_num_pages: int = 0, swa_block_size: int = 64, counts=None):
    """Request-local indices -> global slots, int32 [T, K+W] (-1 = invalid).

    With ``compact`` each token's valid slots are packed to the front of its row and the
    call returns (gidx, counts int32 [T, 2] = (valid top-k entries, valid entries)).  A
    window block table (``swa_block_table`` with ``swa_num_pages`` and ``swa_block_size``)
    sends the window entries through the window cache's paging."""
    T = int(req_id.shape[0])
    K = 0 if topk_idx is None else int(topk_idx.shape[1])
    W = 0 if swa_idx is None else int(swa_idx.shape[1])
    dims = Dims(num_tokens=T, num_heads=1, num_requests=int(block_table.shape[0]),
                max_blocks_per_req=int(block_table.shape[1]), num_pages=int(num_pages),
                block_size=int(block_size), topk=K, swa=W, cache_format=0,
                bt_stride=_row_stride(block_table, int(block_table.shape[1])),
                topk_stride=_row_stride(topk_idx, K), swa_stride=_row_stride(swa_idx, W))
    if gidx is None:
        gidx = torch.empty(T, K + W, dtype=torch.int32, device=block_table.device)
    if swa_block_table is None and topk_length is None and not compact:
        _check(load().smd_convert_req_index(ctypes.byref(dims), _ptr(block_table), _ptr(req_id), _ptr(topk_idx),
                                            _ptr(swa_idx), _ptr(gidx), _stream(stream)))
        return gidx
    opts = DecodeOpts()
    if swa_block_table is not None:
        B = int(swa_block_table.shape[1])
        opts.swa_block_table = swa_block_table.data_ptr()
        opts.swa_num_pages = int(swa_num_pages)
        opts.swa_bt_stride = _row_stride(swa_block_table, B)
        opts.swa_block_size = int(swa_block_size)
        opts.swa_max_blocks_per_req = B
    if topk_length is not None:
        assert topk_length.dtype == torch.int32 and topk_length.is_contiguous()
        opts.topk_length = topk_length.data_ptr()
    opts.compact = int(bool(compact))
    if compact and counts is None:
        counts = torch.empty(T, 2, dtype=torch.int32, device=block_table.device)
    _check(load().smd_convert_req_index_ex(ctypes.byref(dims), ctypes.byref(opts), _ptr(block_table), _ptr(req_id),
                                           _ptr(topk_idx), _ptr(swa_idx), _ptr(gidx),
                                           _ptr(counts) if compact else None, _stream(stream)))
    return (gidx, counts) if compact else gidx


def convert_req_index_ragged(block_table, req_id, token_indices, cu_seqlens, block_size: int = 64,
                             total: int | None = None, out=None, stream=None):
    """The pages' ragged conversion: int32 [cu_seqlens[-1]], 0 for an invalid entry.

    ``total`` (= cu_seqlens[-1]) avoids a device read when given."""
    T = int(req_id.shape[0])
    R, B = int(block_table.shape[0]), int(block_table.shape[1])
    ncols = int(token_indices.shape[1])
    dims = Dims(num_tokens=T, num_heads=1, num_requests=R, max_blocks_per_req=B, num_pages=1,
                block_size=int(block_size), bt_stride=_row_stride(block_table, B))
    assert cu_seqlens.dtype == torch.int32 and cu_seqlens.is_contiguous() and cu_seqlens.numel() == T + 1
    if out is None:
        n = int(cu_seqlens[-1].item()) if total is None else int(total)
        out = torch.empty(n, dtype=torch.int32, device=block_table.device)
    _check(load().smd_convert_req_index_ragged(ctypes.byref(dims), _ptr(block_table), _ptr(req_id),
                                               _ptr(token_indices), ncols, _row_stride(token_indices, ncols),
                                               _ptr(cu_seqlens), _ptr(out), _stream(stream)))
    return out


def gather_dequant(kv_cache, gidx, block_size: int = 64, kv_out=None, stream=None,
                   cache_format: int = CACHE_FP8_DS_MLA):
    """Dequantised bf16 latent rows [n, 512] for the global slots in gidx (zero rows if invalid)."""
    flat = gidx.reshape(-1)
    assert flat.dtype == torch.int32 and flat.is_contiguous()
    n = flat.numel()
    if kv_out is None:
        kv_out = torch.empty(n, LATENT_DIM, dtype=torch.bfloat16, device=kv_cache.device)
    dims = Dims(num_tokens=0, num_heads=1, num_requests=1, max_blocks_per_req=1,
                num_pages=int(kv_cache.shape[0]), block_size=int(block_size), cache_format=int(cache_format))
    _check(load().smd_gather_dequant(ctypes.byref(dims), _ptr(kv_cache), _ptr(flat), ctypes.c_int64(n),
                                     _ptr(kv_out), _stream(stream)))
    return kv_out


def lse_combine(o_part, lse_part, sink=None, out=None, lse=None, stream=None):
    """Merge split partials o_part f32 [T,S,H,512], lse_part f32 [T,S,H] -> (out bf16, lse f32)."""
    T, S, H, D = o_part.shape
    assert D == LATENT_DIM and o_part.is_contiguous() and lse_part.is_contiguous()
    if out is None:
        out = torch.empty(T, H, D, dtype=torch.bfloat16, device=o_part.device)
    if lse is None:
        lse = torch.empty(T, H, dtype=torch.float32, device=o_part.device)
    _check(load().smd_lse_combine(T, S, H, _ptr(o_part), _ptr(lse_part), _ptr(sink), _ptr(out), _ptr(lse),
                                  _stream(stream)))
    return out, lse


def read_status(workspace, stream=None) -> int:
    """Device status word of a decode workspace (0 = ok); raises SmdError on a recorded timeout."""
    v = ctypes.c_int32(0)
    _check(load().smd_read_status(_ptr(workspace), ctypes.byref(v), _stream(stream)))
    return v.value


def read_static_scratch_status(stream=None) -> int:
    """Status word of the last allocation-free decode on the current device (0 = ok);
    raises SmdError on a recorded timeout."""
    v = ctypes.c_int32(0)
    _check(load().smd_read_static_scratch_status(ctypes.byref(v), _stream(stream)))
    return v.value


def set_wait_limit_ns(limit_ns: int) -> int:
    """Bound of the attention kernel's pipeline waits for later launches (0 = default 2 s);
    returns the previous bound.  A test hook: a tiny bound makes the waits give up."""
    return int(load().smd_set_wait_limit_ns(ctypes.c_uint64(int(limit_ns))))


# ---------------------------------------------------------------------- indexer step
def indexer_gather_k(cache, block_table, cu_seqlen, token_to_seq, num_batches: int, block_size: int,
                     head_dim: int, layout: int = 0, k_out=None, scale_out=None, stream=None):
    """Key gather of a ragged batch (smd_indexer_gather_k); returns (k u8 [n, head_dim],
    scale f32 [n]).  Entries the rule does not write keep the contents of k_out /
    scale_out (fresh buffers start as zeros)."""
    n = int(token_to_seq.shape[0])
    dev = cache.device
    if k_out is None:
        k_out = torch.zeros(n, head_dim, dtype=torch.uint8, device=dev)
    if scale_out is None:
        scale_out = torch.zeros(n, dtype=torch.float32, device=dev)
    assert cache.is_contiguous() and k_out.is_contiguous() and scale_out.is_contiguous()
    W = int(block_table.shape[1])
    _check(load().smd_indexer_gather_k(
        _ptr(cache), int(cache.shape[0]), int(block_size), int(head_dim), int(layout), _ptr(block_table),
        int(num_batches), W, _row_stride(block_table, W), _ptr(cu_seqlen), _ptr(token_to_seq), n,
        _ptr(k_out), _ptr(scale_out), _stream(stream)))
    return k_out, scale_out


def indexer_mqa_logits(q, weights, cache, block_table, req_id, ctx_lens, max_len: int, block_size: int = 64,
                       logits=None, status=None, stream=None):
    """fp8 paged MQA logits (smd_indexer_mqa_logits): q u8 e4m3 [T, H, 128], weights f32
    [T, H], cache u8 [pages, P * 132] (layout 0); returns logits f32 [T, max_len]."""
    T, H, D = (int(x) for x in q.shape)
    R, W = (int(x) for x in block_table.shape)
    if logits is None:
        logits = torch.empty(T, max_len, dtype=torch.float32, device=q.device)
    for name, t in (("q", q), ("weights", weights), ("cache", cache), ("logits", logits)):
        assert t.is_contiguous(), f"{name} must be contiguous"
    dims = IndexerDims(T, H, D, R, W, int(block_size), int(cache.shape[0]), _row_stride(block_table, W),
                       int(max_len), 0)
    _check(load().smd_indexer_mqa_logits(
        ctypes.byref(dims), _ptr(q), _ptr(weights), _ptr(cache), _ptr(block_table), _ptr(req_id), _ptr(ctx_lens),
        _ptr(logits), _ptr(status), _stream(stream)))
    return logits


def indexer_topk(logits, ctx_lens, k: int, out=None, stream=None):
    """Top-k positions per token (smd_indexer_topk); returns int32 [T, k], -1 padded."""
    T, L = (int(x) for x in logits.shape)
    assert logits.stride(1) == 1, "logits: unit column stride"
    if out is None:
        out = torch.empty(T, k, dtype=torch.int32, device=logits.device)
    assert out.is_contiguous()
    _check(load().smd_indexer_topk(_ptr(logits), T, L, int(logits.stride(0)), _ptr(ctx_lens), int(k), _ptr(out),
                                   _stream(stream)))
    return out
