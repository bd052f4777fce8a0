"""Shared helpers for the GPU parity tests: oracle calls on CPU copies and tolerances."""
import numpy as np
import torch

import oracle
from sparse_mla_decode_req_gb300 import synth

# Tolerances for bf16 outputs (max abs error, mean relative error = sum|d| / sum|ref|)
# and for the fp32 lse (max abs).
OUT_MAX_ABS = 2e-2
OUT_MEAN_REL = 5e-3
LSE_MAX_ABS = 1e-3
# plus a relative part: fp32 accumulation of a 512-term dot product carries a relative
# error of order 512 * 2^-24 ~ 3e-5 of the score magnitude, which dominates when one
# row's scores are huge (lse ~ 1e12 in the large-scale-code poison case)
LSE_REL = 3e-5


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return oracle.decode_bf16(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def oracle_decode(inp: synth.DecodeInputs, tokens=None):
    """Oracle out/lse for a DecodeInputs (tensors may live on the GPU)."""
    q = bf16_to_f64(inp.q)
    sink = None if inp.sink is None else inp.sink.detach().cpu().double().numpy()
    return oracle.sparse_mla_decode(
        q, inp.kv_cache.cpu().numpy(), inp.block_table.cpu().numpy(), inp.req_id.cpu().numpy(),
        inp.topk_idx.cpu().numpy(), inp.swa_idx.cpu().numpy(), sink, inp.scale, inp.block_size,
        tokens=tokens)


def out_errors(out_gpu: torch.Tensor, ref: np.ndarray):
    got = bf16_to_f64(out_gpu)
    diff = np.abs(got - ref)
    max_abs = float(diff.max()) if diff.size else 0.0
    denom = float(np.abs(ref).sum())
    mean_rel = float(diff.sum() / denom) if denom > 0 else float(diff.sum())
    return got, max_abs, mean_rel


def assert_out_close(out_gpu: torch.Tensor, ref: np.ndarray, what=""):
    got, max_abs, mean_rel = out_errors(out_gpu, ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert max_abs <= OUT_MAX_ABS, f"{what}: max abs error {max_abs:.3e}"
    assert mean_rel <= OUT_MEAN_REL, f"{what}: mean relative error {mean_rel:.3e}"
    return max_abs, mean_rel


def assert_lse_close(lse_gpu: torch.Tensor, ref: np.ndarray, what=""):
    got = lse_gpu.detach().cpu().double().numpy()
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf_ref), f"{what}: -inf pattern differs"
    fin = ~inf_ref
    if fin.any():
        err = np.abs(got[fin] - ref[fin])
        tol = LSE_MAX_ABS + LSE_REL * np.abs(ref[fin])
        worst = int(np.argmax(err - tol))
        assert np.all(err <= tol), f"{what}: lse error {err[worst]:.3e} > {tol[worst]:.3e}"
