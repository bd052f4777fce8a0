"""Pins of the indexer oracle (no GPU): the key gather against hand-built pages, the
logits against closed forms, invariances and a direct recomputation from gathered keys,
the top-k selection against a sort."""
import numpy as np
import pytest

import oracle
from oracle.indexer import cp_gather_indexer_k, key_rows, mqa_logits, topk_positions
from sparse_mla_decode_req_gb300 import synth_indexer as si


def _page_cache(num_pages, P, D, layout, rng):
    """Pages whose key bytes name (page, position) and whose scales are distinct floats."""
    cache = np.zeros((num_pages, P * (D + 4)), np.uint8)
    scales = rng.uniform(0.5, 2.0, size=(num_pages, P)).astype(np.float32)
    for pg in range(num_pages):
        for off in range(P):
            # the two layouts written out here, independently of the oracle's offsets
            vo = off * D if layout == 0 else off * (D + 4)
            so = P * D + 4 * off if layout == 0 else vo + D
            cache[pg, vo:vo + D] = (np.arange(D) * 7 + pg * 31 + off * 3) % 251
            cache[pg, so:so + 4] = np.frombuffer(scales[pg, off].tobytes(), np.uint8)
    return cache, scales


@pytest.mark.parametrize("layout", [0, 1])
def test_cp_gather_follows_the_ragged_rule(layout):
    rng = np.random.default_rng(3)
    P, D, num_pages = 4, 16, 9
    cache, scales = _page_cache(num_pages, P, D, layout, rng)
    # three sequences of 6, 0 and 9 tokens; their block tables, one entry past the cache
    cu = np.array([0, 6, 6, 15])
    bt = np.array([[3, 7, -1], [0, 0, 0], [8, 1, 12]])
    tts = np.array([0] * 6 + [2] * 9 + [5, 1, -1])   # three tokens of no valid sequence
    tts[4] = 2                                        # token 4 names a sequence it is not in
    n = tts.shape[0]
    k0 = np.full((n, D), 0xAB, np.uint8)
    s0 = np.full(n, 7.0, np.float32)
    k, s = cp_gather_indexer_k(cache, bt, cu, tts, 3, P, D, layout, k0, s0)
    for tid in range(n):
        b = tts[tid]
        if b not in (0, 2) or not (cu[b] <= tid < cu[b + 1]):
            assert np.all(k[tid] == 0xAB) and s[tid] == 7.0, tid     # untouched
            continue
        pos = tid - cu[b]
        page = bt[b, pos // P]
        if not (0 <= page < num_pages):
            assert np.all(k[tid] == 0xAB) and s[tid] == 0.0, tid      # bytes kept, scale 0
            continue
        assert np.array_equal(k[tid], (np.arange(D) * 7 + page * 31 + (pos % P) * 3) % 251), tid
        assert s[tid] == scales[page, pos % P]
    # the hand-named cases did occur
    assert np.all(k[4] == 0xAB) and np.all(k[15:] == 0xAB)
    assert s[6 + 8] == 0.0                             # sequence 2, position 8: page 12 is past the cache


def test_key_value_is_e4m3_times_scale():
    P, D = 2, 4
    cache = np.zeros((1, P * (D + 4)), np.uint8)
    cache[0, 0:4] = [0x38, 0x40, 0xB8, 0x01]           # 1, 2, -1, 2**-9
    cache[0, P * D:P * D + 4] = np.frombuffer(np.float32(0.25).tobytes(), np.uint8)
    k = key_rows(cache, [(0, 0)], P, D, 0)
    assert np.array_equal(k[0], [0.25, 0.5, -0.25, 2.0 ** -11])


def _hand_case():
    """One token, two heads, D = 4, P = 2, one page; positions 0 and 1."""
    P, D = 2, 4
    cache = np.zeros((1, P * (D + 4)), np.uint8)
    cache[0, 0:4] = [0x40, 0x40, 0x00, 0x00]           # position 0: (2, 2, 0, 0)
    cache[0, 4:8] = [0xB8, 0x00, 0x00, 0x38]           # position 1: (-1, 0, 0, 1)
    cache[0, 8:12] = np.frombuffer(np.float32(0.25).tobytes(), np.uint8)
    cache[0, 12:16] = np.frombuffer(np.float32(4.0).tobytes(), np.uint8)
    q = np.array([[[0x38, 0x38, 0x00, 0x00],           # head 0: (1, 1, 0, 0)
                   [0x00, 0x00, 0x00, 0x40]]], np.uint8)  # head 1: (0, 0, 0, 2)
    return q, cache, np.array([[0]]), P, D


def test_logits_closed_form():
    q, cache, bt, P, D = _hand_case()
    w = np.array([[0.5, 3.0]])
    lg = mqa_logits(q, w, cache, bt, np.array([0]), np.array([2]), P, D)
    # position 0: head 0 dot = (2*1 + 2*1) * 0.25 = 1, head 1 dot = 0 -> 0.5 * 1 + 3 * 0
    # position 1: head 0 dot = -1 * 4 = -4 -> rectified to 0; head 1 dot = 2 * 1 * 4 = 8 -> 3 * 8
    assert np.array_equal(lg, [[0.5, 24.0]])


def test_logits_masks_past_context_and_bad_pages():
    q, cache, _, P, D = _hand_case()
    w = np.array([[1.0, 1.0]])
    lg = mqa_logits(q, w, cache, np.array([[0, 5]]), np.array([0]), np.array([3]), P, D, max_len=4)
    assert lg[0, 0] == 1.0 and lg[0, 1] == 8.0
    assert np.isneginf(lg[0, 2]) and np.isneginf(lg[0, 3])   # page 5 is past the cache; position 3 past ctx


def test_logits_invariances_and_direct_recomputation():
    w = si.small_indexer_workload(num_tokens=4, ctx_lo=90, ctx_hi=260, block_size=16, extra_pages=3)
    inp = si.make_indexer_inputs(w, seed=9)
    q, wt, cache, bt = inp.q.numpy(), inp.weights.numpy().astype(np.float64), inp.cache.numpy(), inp.block_table.numpy()
    req, ctx, P, D = inp.req_id.numpy(), inp.ctx_lens.numpy(), w.block_size, w.head_dim
    base = mqa_logits(q, wt, cache, bt, req, ctx, P, D)
    # weights enter linearly
    w2 = np.random.default_rng(1).normal(size=wt.shape)
    assert np.allclose(mqa_logits(q, wt + w2, cache, bt, req, ctx, P, D),
                       base + mqa_logits(q, w2, cache, bt, req, ctx, P, D), rtol=1e-12, atol=1e-12, equal_nan=True)
    # relabelling the pages (cache rows and block-table entries together) changes nothing
    perm = np.random.default_rng(2).permutation(cache.shape[0])
    inv = np.argsort(perm)
    bt2 = np.where(bt >= 0, inv[np.clip(bt, 0, None)], -1)
    assert np.array_equal(mqa_logits(q, wt, cache[perm], bt2, req, ctx, P, D), base)
    # direct recomputation: gather each token's keys as a ragged batch, then one einsum
    for t in range(w.num_tokens):
        n = int(ctx[t])
        k, s = cp_gather_indexer_k(cache, bt[t:t + 1], np.array([0, n]), np.zeros(n, int), 1, P, D)
        kf = oracle.decode_e4m3(k) * s[:, None].astype(np.float64)
        qf = oracle.decode_e4m3(q[t])
        direct = np.einsum("h,hn->n", wt[t], np.maximum(np.einsum("hd,nd->hn", qf, kf), 0.0))
        assert np.allclose(base[t, :n], direct, rtol=1e-12, atol=1e-12)
        assert np.all(np.isneginf(base[t, n:]))


def test_topk_matches_a_sort_and_pads():
    rng = np.random.default_rng(4)
    lg = rng.normal(size=(3, 50))
    lg[0, 10:] = -np.inf                                # 10 finite logits, K = 16
    lg[1, [3, 7, 9]] = 2.5                              # ties at the top
    K = 16
    tk = topk_positions(lg, K)
    assert tk.shape == (3, K) and tk.dtype == np.int32
    assert sorted(tk[0, :10].tolist()) == list(range(10)) and np.all(tk[0, 10:] == -1)
    for t in (1, 2):
        want = np.argsort(-lg[t], kind="stable")[:K]
        assert tk[t].tolist() == want.tolist()
    assert tk[1, :3].tolist() == [3, 7, 9]              # equal logits: ascending position
    assert np.all(topk_positions(np.full((1, 5), -np.inf), 3) == -1)
