"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
function include/smd.h declares, and its host-only logic (split selector, workspace
size, argument validation) behaves as documented."""
import ctypes
import os
import re
import subprocess

import pytest

from sparse_mla_decode_req_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load()


def _declared():
    txt = open(os.path.join(ROOT, "include", "smd.h")).read()
    return re.findall(r"SMD_API\s+[\w\s\*]+?\b(smd_\w+)\s*\(", txt)


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(api._SIGS), "binding signatures must mirror the header"


def test_only_abi_symbols_are_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", api.lib_path()], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    ours = {s for s in exported if s.startswith("smd_")}
    assert ours == set(_declared())


def _dims(T=4, H=128, K=2048, W=128, P=64, pages=8192, R=4, B=2048):
    return api.Dims(num_tokens=T, num_heads=H, num_requests=R, max_blocks_per_req=B, num_pages=pages,
                    block_size=P, topk=K, swa=W, cache_format=0, bt_stride=B, topk_stride=K, swa_stride=W)


def test_split_selector_rules(lib):
    # forced counts are honoured exactly
    for s in (1, 2, 7, 32):
        assert api.select_num_splits(_dims(), -s, 152) == s
    # caps are honoured
    for cap in (1, 2, 8, 32):
        assert 1 <= api.select_num_splits(_dims(), cap, 152) <= cap
    # short work: one split per tile when the GPU has room (a CTA's fixed cost outweighs
    # the combine), within the caller's cap
    assert api.select_num_splits(_dims(T=1, H=64, K=512, W=128), 0, 152) == 10
    # long context, low batch: the selector uses many splits to fill the GPU
    s4 = api.select_num_splits(_dims(), 32, 152)
    assert 8 <= s4 <= 32
    # the workloads' automatic choices: single request 5 within its cap of 8 (2 tiles per
    # split; 6 to 8 would leave a split without a tile), batch 32 x 128 heads at 2048
    # entries 2 (128 CTAs, one wave), batch 4 x 128 heads at 2176 entries 17 (136 CTAs,
    # one wave, two tiles per split)
    assert api.select_num_splits(_dims(T=1, H=64, K=512, W=128), 8, 152) == 5
    assert api.select_num_splits(_dims(T=32, H=128, K=2048, W=0), 0, 152) == 2
    assert api.select_num_splits(_dims(T=4, H=128, K=2048, W=128), 32, 152) == 17
    # large batch fills the GPU without splitting
    assert api.select_num_splits(_dims(T=256, H=64, K=512, W=128), 0, 152) == 1
    # every split keeps at least one 64-row tile
    for T in (1, 2, 3, 5, 16):
        for N in (1, 63, 64, 65, 200, 640, 2176):
            d = _dims(T=T, K=N, W=0)
            s = api.select_num_splits(d, 0, 152)
            tiles = -(-N // 64)
            tps = -(-tiles // s)
            assert (s - 1) * tps < tiles
    # depends on shapes and SM count only (graph-safe): repeatable
    assert api.select_num_splits(_dims(), 0, 152) == api.select_num_splits(_dims(), 0, 152)


def test_workspace_size_layout(lib):
    up = lambda x: (x + 255) // 256 * 256
    d = _dims(T=4, H=128, K=2048, W=128)
    s = api.select_num_splits(d, -8, 152)
    T, N, H = 4, 2176, 128
    assert api.workspace_size(d, -8, 152) == (256 + up(T * N * 4) + up(T * 8) + up(T * s * H * 512 * 4)
                                              + up(T * s * H * 4))
    # one split: the status word, the converted slots and the per-token counts only
    d1 = _dims(T=256, H=64, K=512, W=128)
    assert api.workspace_size(d1, 1, 152) == 256 + up(256 * 640 * 4) + up(256 * 8)


@pytest.mark.parametrize("field,value", [("num_heads", 0), ("num_heads", 129), ("block_size", 0),
                                         ("num_pages", 0), ("topk", -1), ("bt_stride", 1),
                                         ("num_tokens", -1), ("num_tokens", 70000), ("cache_format", 2),
                                         ("cache_format", -1)])
def test_invalid_dims_rejected_before_any_launch(lib, field, value):
    d = _dims()
    setattr(d, field, value)
    rc = lib.smd_select_num_splits(ctypes.byref(d), 0, 152)
    assert rc == api.SMD_ERR_INVALID_ARG
    assert api.last_error()
    ws = ctypes.create_string_buffer(64)
    rc = lib.smd_sparse_mla_decode(ctypes.byref(d), None, None, None, None, None, None, None, 1.0, None,
                                   None, 0, ws, 64, None)
    assert rc == api.SMD_ERR_INVALID_ARG


def test_null_pointers_rejected(lib):
    d = _dims(T=2)
    rc = lib.smd_convert_req_index(ctypes.byref(d), None, None, None, None, None, None)
    assert rc == api.SMD_ERR_INVALID_ARG and "required" in api.last_error()
    rc = lib.smd_lse_combine(2, 0, 4, None, None, None, None, None, None)
    assert rc == api.SMD_ERR_INVALID_ARG
    rc = lib.smd_gather_dequant(ctypes.byref(d), None, None, 5, None, None)
    assert rc == api.SMD_ERR_INVALID_ARG
    v = ctypes.c_int32(0)
    assert lib.smd_read_status(None, ctypes.byref(v), None) == api.SMD_ERR_INVALID_ARG


@pytest.mark.parametrize("T,S,H", [(2, 0, 4), (2, 33, 4), (2, 3, 0), (-1, 3, 4)])
def test_combine_bad_shapes_rejected(lib, T, S, H):
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.cast(buf, ctypes.c_void_p)
    rc = lib.smd_lse_combine(T, S, H, p, p, None, p, None, None)
    assert rc == api.SMD_ERR_INVALID_ARG and "combine shape" in api.last_error()


def test_combine_alignment_and_empty_batch(lib):
    buf = ctypes.create_string_buffer(8192)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    al, mis = ctypes.c_void_p(base), ctypes.c_void_p(base + 4)
    for o_part, out in ((mis, al), (al, mis)):
        rc = lib.smd_lse_combine(2, 3, 4, o_part, al, None, out, None, None)
        assert rc == api.SMD_ERR_INVALID_ARG and "aligned" in api.last_error()
    # no tokens: nothing to do, and no pointer is looked at
    assert lib.smd_lse_combine(0, 3, 4, None, None, None, None, None, None) == api.SMD_OK


def test_gather_and_attention_host_checks(lib):
    d = _dims(T=2)
    buf = ctypes.create_string_buffer(8192)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    al, mis = ctypes.c_void_p(base), ctypes.c_void_p(base + 8)
    rc = lib.smd_gather_dequant(ctypes.byref(d), mis, al, 5, al, None)
    assert rc == api.SMD_ERR_INVALID_ARG and "aligned" in api.last_error()
    assert lib.smd_gather_dequant(ctypes.byref(d), None, None, 0, None, None) == api.SMD_OK
    ad = api.attention_dims(2, 64, 640, 100)
    rc = lib.smd_sparse_mla_attention(ctypes.byref(ad), None, al, al, al, None, None, ctypes.c_float(1.0), -33, al,
                                      None, None, None, None, None)
    assert rc == api.SMD_ERR_INVALID_ARG and "num_splits" in api.last_error()
    ad0 = api.attention_dims(0, 64, 640, 100)
    assert lib.smd_sparse_mla_attention(ctypes.byref(ad0), None, None, None, None, None, None, ctypes.c_float(1.0),
                                        0, None, None, None, None, None, None) == api.SMD_OK
    # a misaligned window cache is refused before any launch
    o = api.DecodeOpts()
    o.swa_kv_cache, o.swa_num_pages, o.swa_block_size = base + 8, 10, 64
    rc = lib.smd_sparse_mla_attention(ctypes.byref(ad), ctypes.byref(o), al, al, al, None, None,
                                      ctypes.c_float(1.0), 1, al, None, None, None, None, None)
    assert rc == api.SMD_ERR_INVALID_ARG and "swa_kv_cache" in api.last_error()


def _opts(**kw):
    o = api.DecodeOpts()
    for k, v in kw.items():
        setattr(o, k, v)
    return o


@pytest.mark.parametrize("kw,msg", [
    (dict(swa_kv_cache=4096), "together"),                    # cache without table
    (dict(swa_block_table=4096), "together"),                 # table without cache
    (dict(swa_kv_cache=4096, swa_block_table=4096, swa_block_size=0, swa_num_pages=4,
          swa_max_blocks_per_req=1, swa_bt_stride=1), "swa_block_size"),
    (dict(swa_kv_cache=4096, swa_block_table=4096, swa_block_size=64, swa_num_pages=0,
          swa_max_blocks_per_req=1, swa_bt_stride=1), "swa_num_pages"),
    (dict(swa_kv_cache=4096, swa_block_table=4096, swa_block_size=64, swa_num_pages=1 << 30,
          swa_max_blocks_per_req=1, swa_bt_stride=1), "2^31"),
    (dict(swa_kv_cache=4096, swa_block_table=4096, swa_block_size=64, swa_num_pages=4,
          swa_max_blocks_per_req=8, swa_bt_stride=4), "swa_bt_stride"),
    (dict(swa_kv_cache=4104, swa_block_table=4096, swa_block_size=64, swa_num_pages=4,
          swa_max_blocks_per_req=1, swa_bt_stride=1), "aligned"),
])
def test_decode_options_rejected_before_any_launch(lib, kw, msg):
    d = _dims(T=2)
    ws = ctypes.create_string_buffer(1 << 16)
    wsp = ctypes.c_void_p((ctypes.addressof(ws) + 255) // 256 * 256)
    o = _opts(**kw)
    rc = lib.smd_sparse_mla_decode_ex(ctypes.byref(d), ctypes.byref(o), wsp, wsp, wsp, wsp, wsp, wsp, None,
                                      ctypes.c_float(1.0), wsp, None, 0, wsp, 1 << 15, None)
    assert rc == api.SMD_ERR_INVALID_ARG and msg in api.last_error(), api.last_error()


def test_convert_ex_and_ragged_host_checks(lib):
    d = _dims(T=2)
    p = ctypes.c_void_p(4096)
    # compaction needs the counts array
    rc = lib.smd_convert_req_index_ex(ctypes.byref(d), ctypes.byref(_opts(compact=1)), p, p, p, p, p, None, None)
    assert rc == api.SMD_ERR_INVALID_ARG and "counts" in api.last_error()
    # the conversion reads only the window block table: a table alone is accepted by the
    # checks (no launch happens here: T = 0)
    d0 = _dims(T=0)
    o = _opts(swa_block_table=4096, swa_block_size=32, swa_num_pages=8, swa_max_blocks_per_req=4, swa_bt_stride=4)
    assert lib.smd_convert_req_index_ex(ctypes.byref(d0), ctypes.byref(o), None, None, None, None, None, None,
                                        None) == api.SMD_OK
    # ragged: shape checks, then the empty batch launches nothing
    rc = lib.smd_convert_req_index_ragged(ctypes.byref(d), p, p, p, 5, 4, p, p, None)
    assert rc == api.SMD_ERR_INVALID_ARG and "ti_stride" in api.last_error()
    rc = lib.smd_convert_req_index_ragged(ctypes.byref(d), None, p, p, 5, 5, p, p, None)
    assert rc == api.SMD_ERR_INVALID_ARG and "required" in api.last_error()
    assert lib.smd_convert_req_index_ragged(ctypes.byref(d0), None, None, None, 0, 0, None, None, None) == api.SMD_OK


def test_static_scratch_status_before_any_call(lib):
    assert lib.smd_read_static_scratch_status(None, None) == api.SMD_ERR_INVALID_ARG


def test_version(lib):
    assert lib.smd_version() >= 100


def _idims(T=4, H=64, D=128, R=4, W=16, P=64, pages=64, L=1024, layout=0):
    return api.IndexerDims(num_tokens=T, num_heads=H, head_dim=D, num_requests=R, max_blocks_per_req=W,
                           block_size=P, num_pages=pages, bt_stride=W, max_len=L, layout=layout)


def test_indexer_logits_rejects_shapes_it_does_not_cover(lib):
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    def call(d):
        return lib.smd_indexer_mqa_logits(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake, None, None)
    assert call(_idims(D=64)) == api.SMD_ERR_UNSUPPORTED
    assert call(_idims(H=48)) == api.SMD_ERR_UNSUPPORTED
    for P in (1, 4, 24, 256):
        assert call(_idims(P=P)) == api.SMD_ERR_UNSUPPORTED, P
    assert call(_idims(layout=1)) == api.SMD_ERR_UNSUPPORTED
    assert call(_idims(T=-1)) == api.SMD_ERR_INVALID_ARG
    assert call(_idims(L=-1)) == api.SMD_ERR_INVALID_ARG
    d = _idims()
    d.bt_stride = 3
    assert call(d) == api.SMD_ERR_INVALID_ARG
    assert call(_idims(T=0)) == api.SMD_OK and call(_idims(L=0)) == api.SMD_OK   # nothing to do
    null = lib.smd_indexer_mqa_logits(ctypes.byref(_idims()), None, fake, fake, fake, fake, fake, fake, None, None)
    assert null == api.SMD_ERR_INVALID_ARG
    mis = ctypes.c_void_p((1 << 20) + 4)
    assert lib.smd_indexer_mqa_logits(ctypes.byref(_idims()), mis, fake, fake, fake, fake, fake, fake, None,
                                      None) == api.SMD_ERR_INVALID_ARG


def test_indexer_gather_and_topk_validate_arguments(lib):
    fake = ctypes.c_void_p(1 << 20)
    def gather(D=128, layout=0, n=8, cache=fake, k_out=fake):
        return lib.smd_indexer_gather_k(cache, 64, 64, D, layout, fake, 2, 16, 16, fake, fake, n, k_out, fake, None)
    assert gather(D=6) == api.SMD_ERR_INVALID_ARG
    assert gather(layout=2) == api.SMD_ERR_INVALID_ARG
    assert gather(cache=ctypes.c_void_p((1 << 20) + 8)) == api.SMD_ERR_INVALID_ARG
    assert gather(k_out=ctypes.c_void_p((1 << 20) + 2)) == api.SMD_ERR_INVALID_ARG
    assert gather(n=0) == api.SMD_OK
    assert lib.smd_indexer_topk(fake, 4, 100, 100, fake, 0, fake, None) == api.SMD_ERR_INVALID_ARG
    assert lib.smd_indexer_topk(fake, 4, 100, 99, fake, 8, fake, None) == api.SMD_ERR_INVALID_ARG
    assert lib.smd_indexer_topk(None, 4, 100, 100, fake, 8, fake, None) == api.SMD_ERR_INVALID_ARG
    assert lib.smd_indexer_topk(fake, 0, 100, 100, fake, 8, fake, None) == api.SMD_OK
