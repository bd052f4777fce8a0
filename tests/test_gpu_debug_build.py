"""The SMD_DEBUG range-checking build (libsmd_debug.so) on in-range inputs.

That build re-checks every gathered row address, index read and output write against
the buffer sizes and records a failure in bit 1 of the status word.  On valid calls (every
cache format, page-size alignment class, split mode, both scopes and compaction) no check
may fire and the results must match the oracle as those of the product build do.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.dual_scope import sparse_mla_decode_dual
from sparse_mla_decode_req_gb300 import api, build, synth
from tests.gpu_util import assert_lse_close, assert_out_close, bf16_to_f64, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _debug_lib():
    build.build(debug=True)
    api.use_debug_library(True)
    yield
    api.use_debug_library(False)


def _ws(inp, ns, swa_idx=None):
    dims = api.make_dims(inp.q, inp.kv_cache, inp.block_table, inp.req_id, inp.topk_idx,
                         inp.swa_idx if swa_idx is None else swa_idx, inp.block_size)
    return torch.full((api.workspace_size(dims, ns, 0),), 0xFF, dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("P,ns,compact_", [(64, 1, False), (64, -3, True), (3, 1, False), (5, -2, False)])
def test_debug_build_decode_no_check_fires(P, ns, compact_):
    w = synth.small_workload(num_tokens=3, num_heads=96, topk=400, swa=64, ctx=1200, block_size=P, n_invalid=30)
    inp = synth.make_inputs(w, seed=70 + P, device="cuda")
    ws = _ws(inp, ns)
    out, lse = api.sparse_mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.req_id, inp.topk_idx, inp.swa_idx,
                                     inp.sink, inp.scale, num_splits=ns, workspace=ws, block_size=P,
                                     compact=compact_)
    assert api.read_status(ws) == 0
    ro, rl = oracle_decode(inp)
    assert_out_close(out, ro, f"debug P={P}")
    assert_lse_close(lse, rl, f"debug P={P}")


def test_debug_build_bf16_and_two_caches_no_check_fires():
    wm = synth.Workload("main", 3, 64, 300, 0, 600, 600, block_size=64, n_invalid=9, extra_pages=2)
    ws_ = synth.Workload("swa", 3, 64, 0, 80, 200, 200, block_size=16, n_invalid=3, extra_pages=1)
    a = synth.make_inputs(wm, seed=3, device="cuda")
    b = synth.make_inputs(ws_, seed=4, device="cuda")
    ws = _ws(a, 1, b.swa_idx)
    out, lse = api.sparse_mla_decode(a.q, a.kv_cache, a.block_table, a.req_id, a.topk_idx, b.swa_idx, a.sink,
                                     a.scale, num_splits=1, workspace=ws, swa_kv_cache=b.kv_cache,
                                     swa_block_table=b.block_table, swa_block_size=16)
    assert api.read_status(ws) == 0
    ro, rl = sparse_mla_decode_dual(bf16_to_f64(a.q), a.req_id.cpu().numpy(), a.sink.cpu().double().numpy(),
                                    a.scale, a.kv_cache.cpu().numpy(), a.block_table.cpu().numpy(), 64,
                                    a.topk_idx.cpu().numpy(), b.kv_cache.cpu().numpy(),
                                    b.block_table.cpu().numpy(), 16, b.swa_idx.cpu().numpy())
    assert_out_close(out, ro, "debug dual")
    assert_lse_close(lse, rl, "debug dual")
    # bf16 rows
    cache = synth.make_cache_bf16(a.num_pages, 64, 9, "cuda")
    ws2 = _ws(a, -2)
    api.sparse_mla_decode(a.q, cache, a.block_table, a.req_id, a.topk_idx, None, a.sink, a.scale,
                          num_splits=-2, workspace=ws2, cache_format=api.CACHE_BF16)
    assert api.read_status(ws2) == 0


def test_debug_build_gather_and_ragged_no_check_fires():
    cache = synth.make_cache(30, 64, seed=2, device="cuda")
    slots = torch.randint(-3, 30 * 64 + 5, (500,), generator=torch.Generator().manual_seed(1), dtype=torch.int32)
    kv = api.gather_dequant(cache, slots.cuda(), 64)
    torch.cuda.synchronize()
    ok = (slots >= 0) & (slots < 30 * 64)
    ref = np.zeros((500, 512))
    ref[ok.numpy()] = oracle.dequant_rows(cache.cpu().numpy(), slots[ok].numpy(), 64)
    assert np.array_equal(bf16_to_f64(kv), ref)
