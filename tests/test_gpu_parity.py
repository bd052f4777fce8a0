"""GPU parity: every step of the CUDA path, called through the C ABI, against the
float64 oracle on the same seeded inputs.

Integer work (index conversion) and the dequantised rows must match bit for bit; bf16
outputs must stay within max abs 2e-2 and mean relative error 5e-3, lse within 1e-3.
The five benchmark workloads run at full size and every output element is compared.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from sparse_mla_decode_req_gb300 import api, build, synth
from tests.gpu_util import assert_lse_close, assert_out_close, bf16_to_f64, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    api.load()


def _run(inp: synth.DecodeInputs, num_splits=None, sink=True, want_lse=True):
    w = inp.workload
    ns = w.max_splits if num_splits is None else num_splits
    out, lse = api.sparse_mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.req_id,
                                     inp.topk_idx if w.topk else None, inp.swa_idx if w.swa else None,
                                     inp.sink if sink else None, inp.scale, num_splits=ns,
                                     block_size=w.block_size, return_lse=want_lse)
    torch.cuda.synchronize()
    return out, lse


# ----------------------------------------------------------------- conversion
@pytest.mark.parametrize("wi", range(len(synth.WORKLOADS)))
def test_convert_bit_exact_on_workloads(wi):
    w = synth.WORKLOADS[wi]
    inp = synth.make_inputs(w, device="cuda")
    g = api.convert_req_index(inp.block_table, inp.req_id, inp.topk_idx if w.topk else None,
                              inp.swa_idx if w.swa else None, inp.num_pages, w.block_size)
    ref = oracle.convert_req_index(inp.req_id.cpu().numpy(), inp.block_table.cpu().numpy(),
                                   inp.topk_idx.cpu().numpy(), inp.swa_idx.cpu().numpy(), w.block_size,
                                   inp.num_pages)
    assert np.array_equal(g.cpu().numpy().astype(np.int64), ref)
    assert int((g >= 0).sum()) == inp.n_valid


@pytest.mark.parametrize("P", [1, 3, 64])
def test_convert_edge_cases(P):
    gen = torch.Generator().manual_seed(P)
    R, B, pages, T, K, W = 5, 9, 20, 7, 50, 13
    bt = torch.randint(-3, pages + 4, (R, B + 3), generator=gen, dtype=torch.int32)  # strided rows
    req = torch.randint(-1, R + 2, (T,), generator=gen, dtype=torch.int32)
    topk = torch.randint(-3, B * P + 5, (T, K + 6), generator=gen, dtype=torch.int32)
    swa = torch.randint(-3, B * P + 5, (T, W), generator=gen, dtype=torch.int32)
    btv, topv = bt[:, :B], topk[:, 2:2 + K]
    g = api.convert_req_index(bt.cuda()[:, :B], req.cuda(), topk.cuda()[:, 2:2 + K], swa.cuda(), pages, P)
    ref = oracle.convert_req_index(req.numpy(), btv.numpy(), topv.numpy(), swa.numpy(), P, pages)
    assert np.array_equal(g.cpu().numpy().astype(np.int64), ref)
    # one scope only, and no tokens at all
    g1 = api.convert_req_index(bt.cuda()[:, :B], req.cuda(), None, swa.cuda(), pages, P)
    assert np.array_equal(g1.cpu().numpy().astype(np.int64), ref[:, K:])
    g0 = api.convert_req_index(bt.cuda()[:, :B], req[:0].cuda(), topk[:0, :K].contiguous().cuda(), None,
                               pages, P)
    assert tuple(g0.shape) == (0, K)


# ----------------------------------------------------------------- gather + dequant
def _poison(cache: torch.Tensor, P: int, slots, kinds=(0, 1, 2, 3)):
    """Write NaN fp8 bytes (kind 0), a NaN scale code (1), non-finite RoPE (2), a code whose
    products overflow bf16 (3) or a large finite code (4) into the given slots."""
    flat = cache.view(-1)
    for i, s in enumerate(slots):
        page, off = divmod(s, P)
        d = page * P * 584 + off * 576
        sc = page * P * 584 + P * 576 + off * 8
        kind = kinds[i % len(kinds)]
        if kind == 0:                         # a NaN byte at each position of a 32-bit word
            flat[d + 300] = 0xFF
            flat[d + 5] = 0x7F
            flat[d + 66] = 0xFF
            flat[d + 131] = 0x7F
        elif kind == 1:
            flat[sc + 2] = 255
        elif kind == 2:
            flat[d + 448 + 6] = 0x80          # bf16 0x7F80 = +inf (little endian)
            flat[d + 448 + 7] = 0x7F
            flat[d + 448 + 20] = 0xC0         # bf16 0xFFC0 = NaN
            flat[d + 448 + 21] = 0xFF
        elif kind == 3:
            flat[sc + 6] = 247                # big code: products overflow bf16 -> scrubbed
            flat[d + 6 * 64 + 1] = 0x7E
        else:
            flat[sc + 3] = 160                # finite but 2^40 larger: this row dominates


@pytest.mark.parametrize("P", [64, 1, 3])
def test_gather_dequant_bit_exact(P):
    pages = 40 if P > 1 else 600
    cache = synth.make_cache(pages, P, seed=5, device="cuda")
    n_slots = pages * P
    _poison(cache, P, [0, 7, 33, n_slots - 1])
    gen = torch.Generator().manual_seed(9)
    slots = torch.randint(-2, n_slots + 3, (1000,), generator=gen, dtype=torch.int32)
    slots[:4] = torch.tensor([0, 7, 33, n_slots - 1], dtype=torch.int32)
    kv = api.gather_dequant(cache, slots.cuda(), P)
    torch.cuda.synchronize()
    got = bf16_to_f64(kv)
    ok = (slots >= 0) & (slots < n_slots)
    ref = np.zeros((1000, 512))
    ref[ok.numpy()] = oracle.dequant_rows(cache.cpu().numpy(), slots[ok].numpy(), P)
    assert np.array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


# ----------------------------------------------------------------- combine
@pytest.mark.parametrize("S", [1, 2, 5, 32])
@pytest.mark.parametrize("with_sink", [True, False])
def test_lse_combine_matches_oracle(S, with_sink):
    gen = torch.Generator().manual_seed(S)
    T, H = 3, 24
    o = torch.randn(T, S, H, 512, generator=gen)
    l = torch.randn(T, S, H, generator=gen) * 3
    if S > 1:
        l[0, 1, :] = -math.inf          # empty split
        l[2, :, 5] = -math.inf          # a head with no entries in any split
    sink = torch.randn(H, generator=gen) if with_sink else None
    out, lse = api.lse_combine(o.cuda(), l.cuda(), None if sink is None else sink.cuda())
    torch.cuda.synchronize()
    ro, rl = oracle.lse_combine(o.double().numpy().transpose(1, 0, 2, 3), l.double().numpy().transpose(1, 0, 2),
                                None if sink is None else sink.double().numpy())
    assert_out_close(out, ro, f"combine S={S}")
    assert_lse_close(lse, rl, f"combine S={S}")


@pytest.mark.parametrize("S", [3, 17])
def test_lse_combine_ignores_rows_of_empty_splits(S):
    """A split with lse -inf has no entries: whatever its partial row holds (NaN here) adds
    nothing.  The oracle gets the same inputs with those rows zeroed."""
    gen = torch.Generator().manual_seed(100 + S)
    T, H = 2, 128
    o = torch.randn(T, S, H, 512, generator=gen)
    l = torch.randn(T, S, H, generator=gen) * 3
    l[0, 1, :] = -math.inf
    l[1, S - 1, :] = -math.inf
    o_clean = o.clone()
    o[0, 1] = math.nan
    o[1, S - 1] = math.nan
    o_clean[0, 1] = 0.0
    o_clean[1, S - 1] = 0.0
    sink = torch.randn(H, generator=gen)
    out, lse = api.lse_combine(o.cuda(), l.cuda(), sink.cuda())
    torch.cuda.synchronize()
    ro, rl = oracle.lse_combine(o_clean.double().numpy().transpose(1, 0, 2, 3), l.double().numpy().transpose(1, 0, 2),
                                sink.double().numpy())
    assert torch.isfinite(out.float()).all()
    assert_out_close(out, ro, f"combine empty splits S={S}")
    assert_lse_close(lse, rl, f"combine empty splits S={S}")


@pytest.mark.parametrize("T,H", [(16, 128), (24, 128), (1, 1216)])
def test_lse_combine_every_warps_per_pair_choice(T, H):
    """The combine launch gives each (token, head) 4, 2 or 1 warps by the pair count
    (here 2048 and 3072 pairs, and 1216, the largest count that takes 4)."""
    gen = torch.Generator().manual_seed(T * 1000 + H)
    S = 5
    o = torch.randn(T, S, H, 512, generator=gen)
    l = torch.randn(T, S, H, generator=gen) * 3
    l[0, 1, :] = -math.inf
    l[T - 1, :, 7] = -math.inf
    sink = torch.randn(H, generator=gen)
    out, lse = api.lse_combine(o.cuda(), l.cuda(), sink.cuda())
    torch.cuda.synchronize()
    ro, rl = oracle.lse_combine(o.double().numpy().transpose(1, 0, 2, 3), l.double().numpy().transpose(1, 0, 2),
                                sink.double().numpy())
    assert_out_close(out, ro, f"combine T={T} H={H}")
    assert_lse_close(lse, rl, f"combine T={T} H={H}")


# ----------------------------------------------------------------- full decode
@pytest.mark.parametrize("wi", range(len(synth.WORKLOADS)))
def test_decode_workloads_full_size(wi):
    w = synth.WORKLOADS[wi]
    inp = synth.make_inputs(w, device="cuda")
    out, lse = _run(inp)
    ro, rl = oracle_decode(inp)
    assert_out_close(out, ro, w.name)
    assert_lse_close(lse, rl, w.name)


@pytest.mark.parametrize("splits", [-1, -2, -3, -8, -32, 0])
def test_decode_forced_splits_match_oracle(splits):
    w = synth.small_workload(num_tokens=3, num_heads=64, topk=600, swa=100, ctx=2000, n_invalid=37)
    inp = synth.make_inputs(w, seed=77, device="cuda")
    out, lse = _run(inp, num_splits=splits)
    ro, rl = oracle_decode(inp)
    assert_out_close(out, ro, f"splits {splits}")
    assert_lse_close(lse, rl, f"splits {splits}")


@pytest.mark.parametrize("H", [1, 16, 64, 128])
@pytest.mark.parametrize("N", [1, 63, 64, 65, 640])
@pytest.mark.parametrize("P", [64, 1])
def test_decode_small_shapes(H, N, P):
    K = N - N // 5
    W = N - K
    w = synth.Workload(f"s{H}_{N}_{P}", 2, H, K, W, 700, 700, block_size=P,
                       n_invalid=min(3, N - 1), extra_pages=2)
    inp = synth.make_inputs(w, seed=H * 1000 + N + P, device="cuda")
    ro, rl = oracle_decode(inp)
    for ns in (1, -3):
        out, lse = _run(inp, num_splits=ns)
        assert_out_close(out, ro, f"H{H} N{N} P{P} splits {ns}")
        assert_lse_close(lse, rl, f"H{H} N{N} P{P} splits {ns}")


@pytest.mark.parametrize("splits", [-32, 0])
def test_decode_long_index_lists(splits):
    """65 573 entries per token (60 000 top-k + 5 573 window, 1 025 tiles, the last ragged),
    1 000 of them -1, over contexts of 70 000 positions: 32 forced splits of 33 tiles, and
    the selector's own choice."""
    w = synth.small_workload(num_tokens=2, num_heads=16, topk=60000, swa=5573, ctx=70000, n_invalid=1000)
    inp = synth.make_inputs(w, seed=4242, device="cuda")
    out, lse = _run(inp, num_splits=splits)
    ro, rl = oracle_decode(inp)
    assert_out_close(out, ro, f"long lists splits {splits}")
    assert_lse_close(lse, rl, f"long lists splits {splits}")


@pytest.mark.parametrize("H", [40, 100, 127])
def test_decode_partial_head_warps(H):
    """Head counts that leave a later softmax warp partly filled (its padding heads get no
    output rows) and, for H <= 96, whole warps of padding; single and split outputs."""
    w = synth.small_workload(num_tokens=3, num_heads=H, topk=520, swa=120, ctx=1500, n_invalid=11)
    inp = synth.make_inputs(w, seed=H, device="cuda")
    ro, rl = oracle_decode(inp)
    for ns in (1, -3, -8):
        out, lse = _run(inp, num_splits=ns)
        assert_out_close(out, ro, f"H{H} splits {ns}")
        assert_lse_close(lse, rl, f"H{H} splits {ns}")


def test_decode_without_sink_and_without_lse():
    w = synth.small_workload(num_tokens=2, num_heads=32, topk=200, swa=30, ctx=500)
    inp = synth.make_inputs(w, seed=4, device="cuda")
    inp_ns = synth.DecodeInputs(**{**inp.__dict__, "sink": None})
    ro, _ = oracle_decode(inp_ns)
    for ns in (1, -4):
        out, lse = _run(inp, num_splits=ns, sink=False, want_lse=False)
        assert lse is None
        assert_out_close(out, ro, f"no sink splits {ns}")


@pytest.mark.parametrize("ns", [1, -5])
def test_decode_all_entries_masked(ns):
    w = synth.small_workload(num_tokens=3, num_heads=16, topk=100, swa=20, ctx=400, n_invalid=0)
    inp = synth.make_inputs(w, seed=6, device="cuda")
    inp.topk_idx[1].fill_(-1)
    inp.swa_idx[1].fill_(-1)
    inp.topk_idx[2].fill_(10 ** 6)          # beyond the block table -> masked too
    inp.swa_idx[2].fill_(-7)
    out, lse = _run(inp, num_splits=ns)
    assert torch.all(out[1:].float() == 0)
    assert torch.equal(lse[1].cpu(), inp.sink.cpu()) and torch.equal(lse[2].cpu(), inp.sink.cpu())
    ro, rl = oracle_decode(inp)
    assert_out_close(out, ro, "all masked")
    assert_lse_close(lse, rl, "all masked")
    out2, lse2 = _run(inp, num_splits=ns, sink=False)
    assert torch.all(out2[1:].float() == 0) and torch.all(torch.isneginf(lse2[1:]))


@pytest.mark.parametrize("kinds", [(0, 1, 2), (0, 1, 2, 4, 0, 1, 2, 0), (4, 0, 1, 4, 2, 0)])
def test_decode_poisoned_rows_are_scrubbed(kinds):
    """NaN bytes, NaN scale codes and non-finite RoPE are zeroed before the dot products.

    Kind 4 (a row whose group-3 scale code is raised to 160, i.e. values about 2^33 times
    larger) dominates its heads' softmax; the third case has two such rows, whose scores
    are both of order 2^33 times the rest and far apart from each other, so the larger one
    takes nearly all the weight on both sides.  Scores are accumulated in fp32 over all
    512 dims inside one CTA, so their error stays a small relative one.

    Kind 3 (code 247: latent values near 2^127) is left to the gather test, where it is
    checked bit for bit: such rows make the fp32 q.k products overflow, a range that fp32
    score accumulation cannot represent and that no writer-produced cache reaches.
    """
    w = synth.small_workload(num_tokens=2, num_heads=64, topk=128, swa=0, ctx=256, n_invalid=0)
    inp = synth.make_inputs(w, seed=8, device="cuda")
    bt = inp.block_table.cpu()
    slots = [int(bt[0, int(inp.topk_idx[0, i]) // 64]) * 64 + int(inp.topk_idx[0, i]) % 64 for i in range(8)]
    _poison(inp.kv_cache, 64, slots, kinds)
    out, lse = _run(inp, num_splits=1)
    ro, rl = oracle_decode(inp)
    assert_out_close(out, ro, "poison")
    assert_lse_close(lse, rl, "poison")


@pytest.mark.parametrize("ns", [1, -3])
def test_page_relocation_is_bit_identical(ns):
    """The cache's pages moved to other places with the block table rewritten to match:
    the same rows are read in the same order, so out and lse are bit for bit the same."""
    w = synth.small_workload(num_tokens=5, num_heads=64, topk=300, swa=40, ctx=1200, n_invalid=9, extra_pages=4)
    inp = synth.make_inputs(w, seed=123, device="cuda")
    perm = torch.randperm(inp.kv_cache.shape[0], generator=torch.Generator().manual_seed(5)).cuda()
    moved = torch.empty_like(inp.kv_cache)
    moved[perm] = inp.kv_cache
    bt = inp.block_table
    bt2 = torch.where(bt >= 0, perm[bt.clamp_min(0).long()].to(torch.int32), bt)
    a_out, a_lse = _run(inp, num_splits=ns)
    b_out, b_lse = api.sparse_mla_decode(inp.q, moved, bt2, inp.req_id, inp.topk_idx, inp.swa_idx, inp.sink,
                                         inp.scale, num_splits=ns, block_size=w.block_size)
    torch.cuda.synchronize()
    assert torch.equal(a_out.view(torch.int16), b_out.view(torch.int16))
    assert torch.equal(a_lse.view(torch.int32), b_lse.view(torch.int32))


def test_duplicates_and_shared_pages_across_tokens():
    """Entries repeated within a token and tokens sharing a request both count as given."""
    w = synth.small_workload(num_tokens=4, num_heads=16, topk=70, swa=10, ctx=300, n_invalid=0)
    inp = synth.make_inputs(w, seed=12, device="cuda")
    inp.topk_idx[0, 10:20] = inp.topk_idx[0, 0]        # duplicates
    inp.req_id[3] = 1                                 # token 3 reads request 1's pages
    out, lse = _run(inp, num_splits=-2)
    ro, rl = oracle_decode(inp)
    assert_out_close(out, ro, "duplicates")
    assert_lse_close(lse, rl, "duplicates")


def test_status_word_clear_after_decode():
    w = synth.small_workload()
    inp = synth.make_inputs(w, seed=1, device="cuda")
    dims = api.make_dims(inp.q, inp.kv_cache, inp.block_table, inp.req_id, inp.topk_idx, inp.swa_idx)
    ws = torch.full((api.workspace_size(dims, -3, 0),), 0xFF, dtype=torch.uint8, device="cuda")
    api.sparse_mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.req_id, inp.topk_idx, inp.swa_idx,
                          inp.sink, inp.scale, num_splits=-3, workspace=ws)
    assert api.read_status(ws) == 0


def test_workspace_too_small_is_rejected():
    w = synth.small_workload()
    inp = synth.make_inputs(w, seed=1, device="cuda")
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.SmdError) as e:
        api.sparse_mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.req_id, inp.topk_idx, inp.swa_idx,
                              inp.sink, inp.scale, num_splits=-4, workspace=ws)
    assert e.value.status == api.SMD_ERR_WORKSPACE


@pytest.mark.parametrize("ns", [1, -4])
def test_staged_calls_match_oracle(ns):
    """convert -> attention -> combine through the three stage entry points."""
    w = synth.small_workload(num_tokens=3, num_heads=128, topk=300, swa=40, ctx=900, n_invalid=9)
    inp = synth.make_inputs(w, seed=21, device="cuda")
    g = api.convert_req_index(inp.block_table, inp.req_id, inp.topk_idx, inp.swa_idx, inp.num_pages)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    a, b = api.sparse_mla_attention(inp.q, inp.kv_cache, g, inp.sink, inp.scale, num_splits=ns, status=status)
    out, lse = (a, b) if ns == 1 else api.lse_combine(a, b, inp.sink)
    torch.cuda.synchronize()
    ro, rl = oracle_decode(inp)
    assert_out_close(out, ro, f"staged splits {ns}")
    assert_lse_close(lse, rl, f"staged splits {ns}")
    assert int(status.item()) == 0


@pytest.mark.parametrize("P", [64, 2, 3])
def test_decode_index_edge_cases(P):
    """The whole decode step over request ids, blocks and pages out of range, negative
    indices and strided index rows, against the oracle."""
    gen = torch.Generator().manual_seed(100 + P)
    R, B, pages, T, K, W, H = 5, 9, 20, 7, 50, 13, 16
    bt = torch.randint(-3, pages + 4, (R, B + 3), generator=gen, dtype=torch.int32)
    req = torch.randint(-1, R + 2, (T,), generator=gen, dtype=torch.int32)
    topk = torch.randint(-3, B * P + 5, (T, K + 6), generator=gen, dtype=torch.int32)
    swa = torch.randint(-3, B * P + 5, (T, W), generator=gen, dtype=torch.int32)
    cache = synth.make_cache(pages, P, seed=7 + P, device="cuda")
    q = (torch.randn(T, H, 512, generator=gen) * 0.5).to(torch.bfloat16)
    sink = torch.randn(H, generator=gen)
    scale = 1.0 / math.sqrt(512)
    btv, topv = bt[:, :B], topk[:, 2:2 + K]
    for ns in (1, -3):
        out, lse = api.sparse_mla_decode(q.cuda(), cache, bt.cuda()[:, :B], req.cuda(), topk.cuda()[:, 2:2 + K],
                                         swa.cuda(), sink.cuda(), scale, num_splits=ns, block_size=P)
        torch.cuda.synchronize()
        ro, rl = oracle.sparse_mla_decode(bf16_to_f64(q), cache.cpu().numpy(), btv.numpy(), req.numpy(),
                                          topv.numpy(), swa.numpy(), sink.double().numpy(), scale, P)
        assert_out_close(out, ro, f"edge P={P} splits {ns}")
        assert_lse_close(lse, rl, f"edge P={P} splits {ns}")


@pytest.mark.parametrize("ns", [1, -3])
def test_decode_replays_in_a_cuda_graph(ns):
    """The decode call captured once in a CUDA graph (its split count depends on shapes
    only) and replayed over two input sets copied into the captured buffers."""
    w = synth.small_workload(num_tokens=4, num_heads=64, topk=200, swa=40, ctx=700, n_invalid=5)
    sets = [synth.make_inputs(w, seed=31 + i, device="cuda") for i in range(2)]
    a = sets[0]
    st = {k: getattr(a, k).clone() for k in ("q", "kv_cache", "block_table", "req_id", "topk_idx", "swa_idx", "sink")}
    dims = api.make_dims(st["q"], st["kv_cache"], st["block_table"], st["req_id"], st["topk_idx"], st["swa_idx"])
    ws = torch.empty(api.workspace_size(dims, ns, 0), dtype=torch.uint8, device="cuda")
    out = torch.empty(w.num_tokens, w.num_heads, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.num_tokens, w.num_heads, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def call():
        api.sparse_mla_decode(st["q"], st["kv_cache"], st["block_table"], st["req_id"], st["topk_idx"],
                              st["swa_idx"], st["sink"], a.scale, out=out, lse=lse, num_splits=ns, workspace=ws,
                              stream=stream)

    with torch.cuda.stream(stream):
        call()  # first call outside the capture (one-time per-device setup)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        call()
    for inp in (sets[1], sets[0]):
        for k, t in st.items():
            t.copy_(getattr(inp, k))
        g.replay()
        torch.cuda.synchronize()
        ro, rl = oracle_decode(inp)
        assert_out_close(out, ro, f"graph replay splits {ns}")
        assert_lse_close(lse, rl, f"graph replay splits {ns}")
        assert api.read_status(ws) == 0


# ----------------------------------------------------------------- bounded waits
def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """With the wait bound shortened to 1 ns through the test hook the attention kernel's
    first wait gives up: the launch records bit 0 in the status word, drains what it has in
    flight and returns, smd_read_status reports SMD_ERR_TIMEOUT, and the next call with the
    default bound on the same workspace clears the word and matches the oracle."""
    w = synth.small_workload(num_tokens=4, num_heads=128, topk=900, swa=100, ctx=3000, n_invalid=20)
    inp = synth.make_inputs(w, seed=61, device="cuda")
    dims = api.make_dims(inp.q, inp.kv_cache, inp.block_table, inp.req_id, inp.topk_idx, inp.swa_idx)
    ws = torch.zeros(api.workspace_size(dims, 1, 0), dtype=torch.uint8, device="cuda")

    def call():
        return api.sparse_mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.req_id, inp.topk_idx,
                                     inp.swa_idx, inp.sink, inp.scale, num_splits=1, workspace=ws)

    call()  # per-device set-up before the bound changes
    torch.cuda.synchronize()
    prev = api.set_wait_limit_ns(1)
    try:
        call()
        torch.cuda.synchronize()
    finally:
        assert api.set_wait_limit_ns(prev) == 1
    word = int(ws[:4].view(torch.int32).item())
    assert word & 1, f"status word {word:#x}"
    with pytest.raises(api.SmdError) as e:
        api.read_status(ws)
    assert e.value.status == api.SMD_ERR_TIMEOUT
    out, lse = call()
    torch.cuda.synchronize()
    assert api.read_status(ws) == 0
    ro, rl = oracle_decode(inp)
    assert_out_close(out, ro, "after a timed-out launch")
    assert_lse_close(lse, rl, "after a timed-out launch")
