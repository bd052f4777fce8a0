"""The allocation-free decode entry point against the regular one.

smd_sparse_mla_decode_static_scratch serves callers that cannot allocate device memory
(an engine that reserved nearly all HBM for its KV cache and forbids further cudaMalloc,
a plugin inside a process whose allocator owns the device, a latency-critical path that
cannot take cudaMalloc's implicit synchronisation).  It keeps its scratch in a static
device array inside the library.  These checks call it through the C ABI twice in a row
with different shapes (so the second call runs over whatever the first left in the
array) and compare each result with smd_sparse_mla_decode on the same inputs, within the
parity tolerances of the other GPU tests.  The file is named to be collected last and
passes both alone in a fresh process and after the rest of the suite.
"""
import ctypes

import pytest
import torch

from sparse_mla_decode_req_gb300 import api, build, synth
from tests.gpu_util import (OUT_MAX_ABS, OUT_MEAN_REL, assert_lse_close, assert_out_close, bf16_to_f64,
                            oracle_decode)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load()


def _static_call(lib, inp, num_splits):
    w = inp.workload
    topk = inp.topk_idx if w.topk else None
    swa = inp.swa_idx if w.swa else None
    dims = api.make_dims(inp.q, inp.kv_cache, inp.block_table, inp.req_id, topk, swa, w.block_size)
    out = torch.full((w.num_tokens, w.num_heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.num_tokens, w.num_heads), float("nan"), dtype=torch.float32, device="cuda")
    P = api._ptr
    rc = lib.smd_sparse_mla_decode_static_scratch(
        ctypes.byref(dims), P(inp.q), P(inp.kv_cache), P(inp.block_table), P(inp.req_id), P(topk), P(swa),
        P(inp.sink), ctypes.c_float(inp.scale), P(out), P(lse), int(num_splits),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == api.SMD_OK, api.last_error()
    return out, lse


def _regular_call(inp, num_splits):
    w = inp.workload
    return api.sparse_mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.req_id,
                                 inp.topk_idx if w.topk else None, inp.swa_idx if w.swa else None, inp.sink,
                                 inp.scale, num_splits=num_splits, block_size=w.block_size)


def _close(got, ref):
    g, r = bf16_to_f64(got), bf16_to_f64(ref)
    diff = abs(g - r)
    assert diff.max() <= OUT_MAX_ABS
    assert diff.sum() / max(abs(r).sum(), 1e-30) <= OUT_MEAN_REL


def _oracle_close(inp, out, lse):
    ro, rl = oracle_decode(inp)
    assert_out_close(out, ro, "static scratch")
    assert_lse_close(lse, rl, "static scratch")


def test_static_scratch_matches_regular_entry_point_twice(lib):
    cases = [
        (synth.make_inputs(synth.small_workload(num_tokens=3, num_heads=64, topk=600, swa=100, ctx=2000,
                                                n_invalid=21), seed=31, device="cuda"), -5),
        (synth.make_inputs(synth.WORKLOADS[4], device="cuda"), synth.WORKLOADS[4].max_splits),
    ]
    for inp, ns in cases:
        out, lse = _static_call(lib, inp, ns)
        ref_out, ref_lse = _regular_call(inp, ns)
        torch.cuda.synchronize()
        _close(out, ref_out)
        assert torch.allclose(lse, ref_lse, rtol=1e-5, atol=1e-3)
        assert torch.isfinite(out.float()).all()
        _oracle_close(inp, out, lse)
        assert api.read_static_scratch_status() == 0


def test_static_scratch_call_allocates_no_device_memory(lib):
    """After first calls (which load the library's kernels and its static array), further
    calls leave the device's free memory exactly as it was (the outputs the helper makes
    come from torch's caching allocator, which reuses its blocks)."""
    inp = synth.make_inputs(synth.small_workload(num_tokens=2, num_heads=64, topk=300, swa=60, ctx=900,
                                                 n_invalid=7), seed=41, device="cuda")
    inp2 = synth.make_inputs(synth.small_workload(num_tokens=5, num_heads=128, topk=500, swa=0, ctx=1200,
                                                  n_invalid=3), seed=42, device="cuda")
    calls = ((inp, -3), (inp2, 1), (inp2, -7))
    for x, ns in calls:  # also fills torch's caching allocator with the outputs' blocks
        _static_call(lib, x, ns)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        for x, ns in calls:
            _static_call(lib, x, ns)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_static_scratch_rejects_oversized_steps(lib):
    # 32 tokens x 32 splits x 128 heads of fp32 partials = 64 MiB > the static array
    w = synth.Workload("too_big", 32, 128, 2048, 0, 4096, 4096)
    d = api.Dims(num_tokens=w.num_tokens, num_heads=w.num_heads, num_requests=w.num_tokens, max_blocks_per_req=64,
                 num_pages=64 * w.num_tokens, block_size=64, topk=w.topk, swa=0, cache_format=0, bt_stride=64,
                 topk_stride=w.topk, swa_stride=0)
    rc = lib.smd_sparse_mla_decode_static_scratch(ctypes.byref(d), None, None, None, None, None, None, None,
                                                  ctypes.c_float(1.0), None, None, -32, None)
    assert rc == api.SMD_ERR_WORKSPACE
    assert "static scratch" in api.last_error()
