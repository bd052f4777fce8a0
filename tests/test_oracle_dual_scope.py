"""Pins of the two-cache (top-k scope + window scope) decode oracle (no GPU).

Checked against the single-cache oracle: with one cache for both scopes, and with the two
caches stacked page by page into one cache whose block table holds both scopes' blocks
(an independent construction of the same rows); and, for caches of different page sizes,
against slots looked up by brute force.
"""
import numpy as np
import pytest

from oracle import attend, dequant_rows, sparse_mla_decode
from oracle.dual_scope import sparse_mla_decode_dual
from sparse_mla_decode_req_gb300 import synth


def _scopes(P_main=16, P_swa=16, T=3, H=4, K=24, W=8, seed=5):
    wm = synth.Workload("main", T, H, K, 0, 150, 150, block_size=P_main, n_invalid=3, extra_pages=2)
    ws = synth.Workload("swa", T, H, 0, W, 60, 60, block_size=P_swa, n_invalid=2, extra_pages=1)
    a = synth.make_inputs(wm, seed=seed)
    b = synth.make_inputs(ws, seed=seed + 100)
    return a, b


def _np(a, b):
    return dict(q=a.q.double().numpy(), req_id=a.req_id.numpy(), sink=a.sink.double().numpy(), scale=a.scale,
                main_cache=a.kv_cache.numpy(), main_block_table=a.block_table.numpy(),
                main_block_size=a.block_size, topk_idx=a.topk_idx.numpy(),
                swa_cache=b.kv_cache.numpy(), swa_block_table=b.block_table.numpy(),
                swa_block_size=b.block_size, swa_idx=b.swa_idx.numpy())


def test_one_cache_for_both_scopes_is_the_single_cache_decode():
    w = synth.small_workload(num_tokens=3, num_heads=4, topk=20, swa=6, ctx=90, n_invalid=4, block_size=8)
    inp = synth.make_inputs(w, seed=3)
    q, cache, bt = inp.q.double().numpy(), inp.kv_cache.numpy(), inp.block_table.numpy()
    sink = inp.sink.double().numpy()
    out, lse = sparse_mla_decode_dual(q, inp.req_id.numpy(), sink, inp.scale, cache, bt, 8, inp.topk_idx.numpy(),
                                      cache, bt, 8, inp.swa_idx.numpy())
    ro, rl = sparse_mla_decode(q, cache, bt, inp.req_id.numpy(), inp.topk_idx.numpy(), inp.swa_idx.numpy(),
                               sink, inp.scale, 8)
    assert np.array_equal(out, ro) and np.array_equal(lse, rl)


@pytest.mark.parametrize("seed", [5, 6])
def test_two_caches_equal_one_stacked_cache(seed):
    """Pages of the window cache appended after the main cache's, the window scope's blocks
    appended to each block-table row, window indices shifted past the main blocks."""
    P = 16
    a, b = _scopes(P, P, seed=seed)
    d = _np(a, b)
    out, lse = sparse_mla_decode_dual(**d)
    n_main = d["main_cache"].shape[0]
    bm, bs = d["main_block_table"], d["swa_block_table"]
    stacked_bt = np.concatenate([bm, np.where(bs >= 0, bs + n_main, -1)], axis=1).astype(np.int32)
    stacked_cache = np.concatenate([d["main_cache"], d["swa_cache"]], axis=0)
    shift = bm.shape[1] * P
    swa = np.where(d["swa_idx"] >= 0, d["swa_idx"] + shift, -1)
    ro, rl = sparse_mla_decode(d["q"], stacked_cache, stacked_bt, d["req_id"], d["topk_idx"], swa,
                               d["sink"], d["scale"], P)
    assert np.array_equal(out, ro) and np.array_equal(lse, rl)


@pytest.mark.parametrize("P_main,P_swa", [(64, 1), (3, 64), (16, 5)])
def test_each_scope_uses_its_own_table_and_page_size(P_main, P_swa):
    a, b = _scopes(P_main, P_swa, seed=P_main * 10 + P_swa)
    d = _np(a, b)
    out, lse = sparse_mla_decode_dual(**d)

    def slots(bt, r, idx, P):
        return [int(bt[r, i // P]) * P + i % P for i in idx if i >= 0 and i // P < bt.shape[1]
                and bt[r, i // P] >= 0]

    for t in range(d["q"].shape[0]):
        r = int(d["req_id"][t])
        km = dequant_rows(d["main_cache"], slots(d["main_block_table"], r, d["topk_idx"][t], P_main), P_main)
        ks = dequant_rows(d["swa_cache"], slots(d["swa_block_table"], r, d["swa_idx"][t], P_swa), P_swa)
        o, l = attend(d["q"][t], np.concatenate([km, ks]), d["sink"], d["scale"])
        assert np.array_equal(o, out[t]) and np.array_equal(l, lse[t])


def test_one_scope_absent():
    a, b = _scopes()
    d = _np(a, b)
    only_main = sparse_mla_decode_dual(**{**d, "swa_idx": None})
    ro = sparse_mla_decode(d["q"], d["main_cache"], d["main_block_table"], d["req_id"], d["topk_idx"], None,
                           d["sink"], d["scale"], d["main_block_size"])
    assert np.array_equal(only_main[0], ro[0]) and np.array_equal(only_main[1], ro[1])
    only_swa = sparse_mla_decode_dual(**{**d, "topk_idx": None})
    rs = sparse_mla_decode(d["q"], d["swa_cache"], d["swa_block_table"], d["req_id"], None, d["swa_idx"],
                           d["sink"], d["scale"], d["swa_block_size"])
    assert np.array_equal(only_swa[0], rs[0]) and np.array_equal(only_swa[1], rs[1])
