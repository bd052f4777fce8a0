"""Host logic of bench.py's end-to-end leg (no GPU): the packed input and result buffers."""
import torch

import bench


def _named():
    g = torch.Generator().manual_seed(5)
    return [("q", torch.randn(3, 64, 512, generator=g).to(torch.bfloat16)),
            ("block_table", torch.randint(-1, 1000, (3, 37), generator=g, dtype=torch.int32)),
            ("req_id", torch.arange(3, dtype=torch.int32)),
            ("topk_idx", torch.randint(-1, 8192, (3, 513), generator=g, dtype=torch.int32)),
            ("swa_idx", torch.zeros(3, 0, dtype=torch.int32)),
            ("lse", torch.randn(3, 64, generator=g))]


def test_pack_layout_offsets_are_aligned_and_disjoint():
    named = _named()
    lay, total = bench.pack_layout(named)
    spans = sorted((o, o + n) for o, n, _, _ in lay.values())
    for (a0, a1), (b0, _) in zip(spans, spans[1:]):
        assert a1 <= b0
    for k, t in named:
        o, n, dt, shape = lay[k]
        assert o % 256 == 0 and n == t.numel() * t.element_size() and dt == t.dtype and shape == tuple(t.shape)
    assert total % 256 == 0 and total >= spans[-1][1]


def test_pack_views_round_trip_bit_exact():
    named = _named()
    lay, total = bench.pack_layout(named)
    buf = torch.zeros(total, dtype=torch.uint8)
    views = bench.pack_views(buf, lay)
    for k, t in named:
        views[k].copy_(t)
    copy = buf.clone()  # stands in for the single transfer to the device
    back = bench.pack_views(copy, lay)
    for k, t in named:
        assert back[k].dtype == t.dtype and back[k].shape == t.shape and back[k].is_contiguous()
        assert torch.equal(back[k].view(torch.uint8) if t.numel() else back[k], t.view(torch.uint8) if t.numel() else t)


def test_pack_layout_of_empty_list():
    lay, total = bench.pack_layout([])
    assert lay == {} and total == 256


def test_e2e_input_sets_keep_the_step_shape_and_draw_new_rows():
    from sparse_mla_decode_req_gb300 import synth
    w = synth.small_workload(num_tokens=4, topk=96, swa=32, ctx=300, n_invalid=5)
    inp = synth.make_inputs(w, seed=11)
    sets = bench.e2e_input_sets(inp, w, 3, seed=3)
    assert len(sets) == 3
    names = bench.e2e_names(w)
    for k in names:  # set 0 is the step's own inputs
        assert torch.equal(sets[0][k], getattr(inp, k).cpu())
    for s in sets[1:]:
        assert set(s) == set(names)
        for k in names:
            assert s[k].shape == sets[0][k].shape and s[k].dtype == sets[0][k].dtype
        for k in ("block_table", "req_id", "swa_idx"):  # pages and window unchanged
            assert torch.equal(s[k], sets[0][k])
        assert not torch.equal(s["q"], sets[0]["q"])
        tk, tk0 = s["topk_idx"], sets[0]["topk_idx"]
        assert torch.equal(tk < 0, tk0 < 0)  # the same -1 entries, so the same valid-row count
        assert not torch.equal(tk, tk0)
        for t in range(tk.shape[0]):
            v = tk[t][tk[t] >= 0]
            assert int(v.min()) >= 0 and int(v.max()) < inp.ctx_lens[t]
            assert v.unique().numel() == v.numel()  # distinct positions, as the workload draws them
    assert not torch.equal(sets[1]["topk_idx"], sets[2]["topk_idx"])
