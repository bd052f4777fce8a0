"""Pins for the oracle's attention, sink, masking and split combine (CPU only).

The oracle's ``attend`` is compared with torch's float64 ``scaled_dot_product_attention``
(a library route) where the sink is an extra all-zero key/value column whose additive
mask is the sink logit; ``lse`` is recovered from the weights-sum invariant.  Closed
forms (scale 0, one entry, all masked), the brute-force dense case (top-k listing
every context position in a random order, decoded with torch's fp8 dtype), the
duplicate-entry rule and split associativity complete the pins.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attend, dequant_rows, lse_combine, sparse_mla_decode
from sparse_mla_decode_req_gb300 import synth


def _sdpa_with_sink(q, k, sink, scale, extra_mask=None):
    """Library reference: softmax over [scores | sink] with a zero value for the sink."""
    H, D = q.shape
    n = k.shape[0]
    qt = torch.from_numpy(q).view(1, H, 1, D)
    kz = np.concatenate([k, np.zeros((1, D))], axis=0)
    kt = torch.from_numpy(kz).view(1, 1, n + 1, D).expand(1, H, n + 1, D)
    mask = torch.zeros(1, H, 1, n + 1, dtype=torch.float64)
    mask[0, :, 0, n] = torch.from_numpy(np.asarray(sink, dtype=np.float64))
    if extra_mask is not None:
        mask[0, :, 0, :n] += torch.from_numpy(extra_mask)
    out = F.scaled_dot_product_attention(qt, kt, kt, attn_mask=mask, scale=scale)
    return out.view(H, D).numpy()


def _rand_case(rng, H=8, n=37, D=512):
    q = rng.standard_normal((H, D))
    k = rng.standard_normal((n, D))
    sink = rng.standard_normal(H) * 2
    return q, k, sink


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_attend_matches_library_sdpa_with_sink(seed):
    rng = np.random.default_rng(seed)
    q, k, sink = _rand_case(rng)
    k[:, 448] = 1.0                                    # ones column -> weights sum
    scale = 1 / math.sqrt(512)
    out, lse = attend(q, k, sink, scale)
    ref = _sdpa_with_sink(q, k, sink, scale)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)
    # sum of row weights + sink weight = 1; lse recovered from the library output
    w_sink = 1.0 - ref[:, 448]
    assert np.allclose(out[:, 448] + np.exp(sink - lse), 1.0, atol=1e-13)
    assert np.allclose(lse, sink - np.log(w_sink), rtol=1e-10)


def test_no_sink_is_plain_softmax():
    rng = np.random.default_rng(3)
    q, k, _ = _rand_case(rng)
    scale = 0.7
    out, lse = attend(q, k, None, scale)
    ref = _sdpa_with_sink(q, k, np.full(q.shape[0], -np.inf), scale)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)
    k1 = k.copy()
    k1[:, 7] = 1.0
    out1, _ = attend(q, k1, None, scale)
    assert np.allclose(out1[:, 7], 1.0, atol=1e-13)


def test_scale_zero_closed_form():
    rng = np.random.default_rng(4)
    q, k, sink = _rand_case(rng, n=11)
    out, lse = attend(q, k, sink, 0.0)
    n = k.shape[0]
    exp = k.mean(axis=0)[None, :] * (n / (n + np.exp(sink)))[:, None]
    assert np.allclose(out, exp, rtol=1e-12, atol=1e-15)
    assert np.allclose(lse, np.log(n + np.exp(sink)), rtol=1e-13)


def test_single_entry_and_all_masked():
    rng = np.random.default_rng(5)
    q, k, sink = _rand_case(rng, n=1)
    out, lse = attend(q, k, None, 0.3)
    assert np.array_equal(out, np.broadcast_to(k[0], out.shape))
    assert np.allclose(lse, 0.3 * (q @ k[0]), rtol=1e-14)
    out0, lse0 = attend(q, np.zeros((0, 512)), sink, 0.3)
    assert np.all(out0 == 0.0) and np.array_equal(lse0, sink)
    out1, lse1 = attend(q, np.zeros((0, 512)), None, 0.3)
    assert np.all(out1 == 0.0) and np.all(np.isneginf(lse1))


def test_large_scores_stay_finite():
    rng = np.random.default_rng(6)
    q, k, sink = _rand_case(rng, n=20)
    scale = 50.0                                       # scores ~ +-1e3: exp would overflow unshifted
    out, lse = attend(q, k, sink, scale)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    ref = _sdpa_with_sink(q, k, sink, scale)
    assert np.allclose(out, ref, rtol=1e-9, atol=1e-12)


def test_duplicate_entry_doubles_its_weight():
    rng = np.random.default_rng(7)
    q, k, sink = _rand_case(rng, n=9)
    scale = 1 / math.sqrt(512)
    kd = np.concatenate([k, k[4:5]], axis=0)
    out, _ = attend(q, kd, sink, scale)
    bump = np.zeros((q.shape[0], k.shape[0]))
    bump[:, 4] = math.log(2.0)
    ref = _sdpa_with_sink(q, k, sink, scale, extra_mask=bump)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("n_splits", [1, 2, 5, 32])
def test_split_combine_is_exact(n_splits):
    rng = np.random.default_rng(100 + n_splits)
    q, k, sink = _rand_case(rng, n=97)
    scale = 1 / math.sqrt(512)
    full_o, full_l = attend(q, k, sink, scale)
    cuts = np.sort(rng.choice(np.arange(0, 98), size=n_splits - 1, replace=True))
    bounds = [0, *cuts.tolist(), 97]                  # some parts may be empty
    parts = [attend(q, k[a:b], None, scale) for a, b in zip(bounds[:-1], bounds[1:])]
    o = np.stack([p[0] for p in parts])
    l = np.stack([p[1] for p in parts])
    co, cl = lse_combine(o, l, sink)
    assert np.allclose(co, full_o, rtol=1e-12, atol=1e-15)
    assert np.allclose(cl, full_l, rtol=1e-12)
    # all splits empty and no sink -> zero output, -inf lse, never NaN
    eo, el = lse_combine(np.zeros((3, 2, 4)), np.full((3, 2), -np.inf), None)
    assert np.all(eo == 0) and np.all(np.isneginf(el))


def _dense_reference(inp: synth.DecodeInputs, t: int) -> tuple[np.ndarray, np.ndarray]:
    """Dense attention over the token's whole context, decoded with torch's fp8 dtype."""
    P = inp.block_size
    cache = inp.kv_cache
    ctx = inp.ctx_lens[t]
    rows = []
    for pos in range(ctx):
        page = int(inp.block_table[t, pos // P])
        base = page * P * 584
        off = pos % P
        data = cache[page].reshape(-1)[off * 576:off * 576 + 576]
        codes = cache[page].reshape(-1)[P * 576 + off * 8:P * 576 + off * 8 + 7]
        nope = data[:448].view(torch.float8_e4m3fn).to(torch.float64)
        sc = torch.pow(2.0, codes.to(torch.float64) - 127).repeat_interleave(64)
        rope = data[448:].contiguous().view(torch.bfloat16).to(torch.float64)
        rows.append(torch.cat([nope * sc, rope]))
        del base
    kd = torch.stack(rows).numpy()
    q = inp.q[t].to(torch.float64).numpy()
    out = _sdpa_with_sink(q, kd, inp.sink.to(torch.float64).numpy(), inp.scale)
    return out, kd


@pytest.mark.parametrize("P", [64, 1, 16])
def test_full_topk_equals_dense_attention(P):
    """Top-k listing every context position (any order) is dense attention."""
    ctx = 150
    w = synth.Workload("dense", 2, 4, ctx, 0, ctx, ctx, block_size=P)
    inp = synth.make_inputs(w, seed=11 + P)
    g = torch.Generator().manual_seed(P)
    for t in range(2):
        inp.topk_idx[t] = torch.randperm(ctx, generator=g).to(torch.int32)
    out, lse = sparse_mla_decode(inp.q.to(torch.float64).numpy(), inp.kv_cache.numpy(),
                                 inp.block_table.numpy(), inp.req_id.numpy(), inp.topk_idx.numpy(),
                                 inp.swa_idx.numpy(), inp.sink.to(torch.float64).numpy(), inp.scale, P)
    for t in range(2):
        ref, kd = _dense_reference(inp, t)
        assert np.allclose(out[t], ref, rtol=1e-11, atol=1e-13)
        # the dense rows also match the oracle's own decoder slot by slot
        slots = [int(inp.block_table[t, p // P]) * P + p % P for p in range(ctx)]
        assert np.array_equal(dequant_rows(inp.kv_cache.numpy(), slots, P), kd)


def test_invalid_entries_are_masked_and_window_merges():
    """-1 entries contribute nothing; window entries join the same softmax as top-k."""
    w = synth.small_workload(num_tokens=2, num_heads=4, topk=20, swa=8, ctx=100, n_invalid=6)
    inp = synth.make_inputs(w, seed=3)
    args = dict(kv_cache=inp.kv_cache.numpy(), block_table=inp.block_table.numpy(),
                req_id=inp.req_id.numpy(), sink=inp.sink.double().numpy(), scale=inp.scale,
                block_size=w.block_size)
    q = inp.q.double().numpy()
    out, lse = sparse_mla_decode(q, topk_idx=inp.topk_idx.numpy(), swa_idx=inp.swa_idx.numpy(), **args)
    both = np.concatenate([inp.topk_idx.numpy(), inp.swa_idx.numpy()], axis=1)
    for t in range(2):
        keep = both[t][both[t] >= 0]
        o2, l2 = sparse_mla_decode(q[t:t + 1], topk_idx=keep[None, :],
                                   swa_idx=np.zeros((1, 0), np.int32),
                                   **{**args, "req_id": args["req_id"][t:t + 1]})
        assert np.allclose(out[t], o2[0], rtol=1e-13, atol=1e-15)
        assert np.allclose(lse[t], l2[0], rtol=1e-13)


@pytest.mark.parametrize("P", [64, 3])
def test_page_relocation_changes_nothing(P):
    """Moving every page of the cache to another place and rewriting the block table to
    match reads the same rows in the same order: out and lse are bit-identical."""
    w = synth.small_workload(num_tokens=3, num_heads=8, topk=70, swa=12, ctx=260, block_size=P, n_invalid=4,
                             extra_pages=3)
    inp = synth.make_inputs(w, seed=29 + P)
    cache = inp.kv_cache.numpy()
    perm = np.random.default_rng(P).permutation(cache.shape[0])  # page i moves to perm[i]
    moved = np.empty_like(cache)
    moved[perm] = cache
    bt = inp.block_table.numpy()
    bt2 = np.where(bt >= 0, perm[np.clip(bt, 0, None)], bt).astype(np.int32)
    args = dict(req_id=inp.req_id.numpy(), topk_idx=inp.topk_idx.numpy(), swa_idx=inp.swa_idx.numpy(),
                sink=inp.sink.double().numpy(), scale=inp.scale, block_size=P)
    q = inp.q.double().numpy()
    o1, l1 = sparse_mla_decode(q, kv_cache=cache, block_table=bt, **args)
    o2, l2 = sparse_mla_decode(q, kv_cache=moved, block_table=bt2, **args)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
