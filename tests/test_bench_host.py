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
