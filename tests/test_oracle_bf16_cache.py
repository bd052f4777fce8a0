"""Pins of the bf16-latent-cache decode oracle (no GPU)."""
import numpy as np
import pytest
import torch

from oracle import dequant_rows, sparse_mla_decode
from oracle.bf16_cache import dequant_rows_bf16, sparse_mla_decode_bf16
from sparse_mla_decode_req_gb300 import synth


def _to_bf16_cache(fp8_cache: np.ndarray, P: int) -> np.ndarray:
    """The fp8 cache's dequantised rows written as bf16 (exact: every finite e4m3 value
    times a power-of-two scale that stays in range is a bf16 value), same slots."""
    pages = fp8_cache.shape[0]
    rows = dequant_rows(fp8_cache, np.arange(pages * P), P)
    assert np.array_equal(torch.from_numpy(rows).to(torch.bfloat16).double().numpy(), rows)
    bits = torch.from_numpy(rows).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return bits.view(np.uint8).reshape(pages, P * 1024)


@pytest.mark.parametrize("P", [64, 1, 5])
def test_bf16_cache_of_the_dequantised_rows_decodes_like_the_fp8_cache(P):
    w = synth.small_workload(num_tokens=3, num_heads=4, topk=30, swa=7, ctx=120, n_invalid=5, block_size=P)
    inp = synth.make_inputs(w, seed=40 + P)
    args = dict(block_table=inp.block_table.numpy(), req_id=inp.req_id.numpy(), topk_idx=inp.topk_idx.numpy(),
                swa_idx=inp.swa_idx.numpy(), sink=inp.sink.double().numpy(), scale=inp.scale, block_size=P)
    q = inp.q.double().numpy()
    ro, rl = sparse_mla_decode(q, inp.kv_cache.numpy(), **args)
    out, lse = sparse_mla_decode_bf16(q, _to_bf16_cache(inp.kv_cache.numpy(), P), **args)
    assert np.array_equal(out, ro) and np.array_equal(lse, rl)


def test_bf16_rows_read_back_through_torch():
    g = torch.Generator().manual_seed(1)
    P, pages = 4, 3
    vals = torch.randn(pages * P, 512, generator=g).to(torch.bfloat16)
    vals[2, 7] = float("nan")
    vals[5, 500] = float("inf")
    cache = vals.view(torch.int16).numpy().view(np.uint8).reshape(pages, P * 1024)
    slots = [11, 0, 5, 2]
    got = dequant_rows_bf16(cache, slots, P)
    want = vals[slots].double().numpy()
    want[~np.isfinite(want)] = 0.0
    assert np.array_equal(got, want)
