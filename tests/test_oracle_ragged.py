"""Pins of the ragged / length-limited index oracle (no GPU).

Each rule is checked against something other than itself: the top-k length cut against
decoding the truncated index array, the ragged conversion against the dense conversion
(written separately, with its own sentinel), compaction by brute force and by the decode
it must leave unchanged.
"""
import numpy as np
import pytest

from oracle import attend, convert_req_index, dequant_rows, sparse_mla_decode
from oracle.ragged import apply_topk_length, compact, convert_req_index_ragged
from sparse_mla_decode_req_gb300 import synth


def _case(T=4, K=20, W=6, n_invalid=4, seed=9):
    w = synth.small_workload(num_tokens=T, num_heads=4, topk=K, swa=W, ctx=120, n_invalid=n_invalid)
    inp = synth.make_inputs(w, seed=seed)
    args = dict(kv_cache=inp.kv_cache.numpy(), block_table=inp.block_table.numpy(),
                sink=inp.sink.double().numpy(), scale=inp.scale, block_size=w.block_size)
    return w, inp, args


@pytest.mark.parametrize("s_q,lengths", [(1, [0, 3, 20, 11]), (2, [5, 17]), (4, [9])])
def test_topk_length_equals_decoding_the_truncated_columns(s_q, lengths):
    """Cutting column k >= TopkLength[t // s_q] decodes exactly like an index array that
    simply ends at that length (the window scope is untouched)."""
    w, inp, args = _case()
    q = inp.q.double().numpy()
    topk = inp.topk_idx.numpy()
    swa = inp.swa_idx.numpy()
    req = inp.req_id.numpy()
    cut = apply_topk_length(topk, lengths, s_q)
    out, lse = sparse_mla_decode(q, topk_idx=cut, swa_idx=swa, req_id=req, **args)
    for t in range(w.num_tokens):
        L = lengths[t // s_q]
        o2, l2 = sparse_mla_decode(q[t:t + 1], topk_idx=topk[t:t + 1, :L], swa_idx=swa[t:t + 1],
                                   req_id=req[t:t + 1], **args)
        assert np.array_equal(out[t], o2[0]) and np.array_equal(lse[t], l2[0])


def test_topk_length_extremes():
    _, inp, _ = _case()
    topk = inp.topk_idx.numpy()
    assert np.array_equal(apply_topk_length(topk, [topk.shape[1]] * 4), topk)     # no cut
    assert np.all(apply_topk_length(topk, [0] * 4) == -1)                         # everything cut


def _ragged_inputs(seed):
    """Request-local indices whose blocks all map to real pages, plus negative and
    past-the-table entries, and per-token lengths."""
    rng = np.random.default_rng(seed)
    P, R, B, pages = 8, 3, 5, 40
    bt = np.stack([rng.permutation(pages)[:B] for _ in range(R)]).astype(np.int32)
    T, N = 5, 12
    req = rng.integers(0, R, T).astype(np.int32)
    ti = rng.integers(0, B * P, (T, N)).astype(np.int32)
    ti[rng.random((T, N)) < 0.15] = -1
    ti[0, 3] = B * P + 2          # block past the table
    ti[1, 0] = -7                 # other negative
    lens = rng.integers(0, N + 1, T)
    lens[2] = N
    lens[3] = 0
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return P, bt, req, ti, cu, pages


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_ragged_conversion_is_the_dense_one_zero_filled_and_packed(seed):
    P, bt, req, ti, cu, pages = _ragged_inputs(seed)
    got = convert_req_index_ragged(req, bt, ti, cu, P)
    dense = convert_req_index(req, bt, ti, None, P, pages)
    want = []
    for t in range(len(req)):
        row = dense[t, :cu[t + 1] - cu[t]]
        want.extend(np.where(row < 0, 0, row).tolist())
    assert np.array_equal(got, np.asarray(want, dtype=np.int64))
    assert got.shape == (cu[-1],)


def test_ragged_zero_fill_cannot_tell_slot_zero_from_invalid():
    """Why the dense form uses -1: index 0 of a request whose first block is page 0 is the
    real slot 0, and converts to the same value as an invalid entry."""
    P = 4
    bt = np.array([[0, 3]], dtype=np.int32)
    ti = np.array([[0, -1, 5]], dtype=np.int32)
    cu = np.array([0, 3], dtype=np.int32)
    got = convert_req_index_ragged(np.array([0], np.int32), bt, ti, cu, P)
    assert got.tolist() == [0, 0, 3 * P + 1]
    dense = convert_req_index(np.array([0], np.int32), bt, ti, None, P, 8)
    assert dense.tolist() == [[0, -1, 3 * P + 1]]


def test_ragged_form_trusts_the_block_table():
    """The ragged kernel of the pages checks no physical page: an unused table entry (-1)
    yields a negative slot there, where the dense form marks the entry invalid."""
    P = 4
    bt = np.array([[5, -1]], dtype=np.int32)
    ti = np.array([[6]], dtype=np.int32)
    cu = np.array([0, 1], dtype=np.int32)
    assert convert_req_index_ragged(np.array([0], np.int32), bt, ti, cu, P).tolist() == [-1 * P + 2]
    assert convert_req_index(np.array([0], np.int32), bt, ti, None, P, 8).tolist() == [[-1]]


@pytest.mark.parametrize("seed", range(4))
def test_compact_brute_force(seed):
    rng = np.random.default_rng(seed)
    g = rng.integers(-1, 50, (6, 9))
    g[rng.random(g.shape) < 0.4] = -1
    g[2] = -1                                   # a token with nothing valid
    cu, slots = compact(g)
    assert cu[0] == 0 and np.all(np.diff(cu) >= 0) and cu[-1] == (g >= 0).sum()
    for t in range(g.shape[0]):
        assert slots[cu[t]:cu[t + 1]].tolist() == [int(s) for s in g[t] if s >= 0]


def test_decode_over_compacted_slots_is_unchanged():
    """Skipping the invalid rows before the gather leaves every output bit unchanged."""
    w, inp, args = _case(n_invalid=7, seed=21)
    q = inp.q.double().numpy()
    req = inp.req_id.numpy()
    out, lse = sparse_mla_decode(q, topk_idx=inp.topk_idx.numpy(), swa_idx=inp.swa_idx.numpy(), req_id=req, **args)
    dense = convert_req_index(req, args["block_table"], inp.topk_idx.numpy(), inp.swa_idx.numpy(),
                              w.block_size, args["kv_cache"].shape[0])
    cu, slots = compact(dense)
    assert cu[-1] < dense.size                  # something was skipped
    for t in range(w.num_tokens):
        k = dequant_rows(args["kv_cache"], slots[cu[t]:cu[t + 1]], w.block_size)
        o, l = attend(q[t], k, args["sink"], args["scale"])
        assert np.array_equal(o, out[t]) and np.array_equal(l, lse[t])
