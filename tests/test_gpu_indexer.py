"""GPU parity of the indexer step, through the C ABI, against the float64 oracle:

* the key gather of a ragged batch, bit for bit (both cache layouts, untouched entries
  kept);
* the fp8 paged MQA logits (tcgen05 kind::f8f6f4) within a bound derived from float32
  accumulation over the terms' magnitudes, -inf exactly where the oracle has it;
* the top-k selection: the oracle's selection rule applied to the GPU's own float32
  logits (both sides decide in float32) must give the same position sets;
* the indexer's top-k positions fed to the sparse decode.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle.indexer import cp_gather_indexer_k, mqa_logits, topk_positions
from sparse_mla_decode_req_gb300 import api, build, synth, synth_indexer as si
from tests.gpu_util import assert_lse_close, assert_out_close, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    api.load()


def _np(t):
    return t.detach().cpu().numpy()


# ----------------------------------------------------------------- key gather
@pytest.mark.parametrize("layout,P", [(0, 64), (1, 64), (0, 1), (1, 3), (0, 16)])
def test_gather_bit_exact(layout, P):
    w = si.small_indexer_workload(num_tokens=5, ctx_lo=40, ctx_hi=200, block_size=P, extra_pages=2)
    inp = si.make_indexer_inputs(w, seed=11 + P, device="cuda", layout=layout)
    lens = inp.ctx
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n = int(cu[-1]) + 7
    tts = np.concatenate([np.repeat(np.arange(len(lens)), lens), [len(lens) + 3, -1, 1, 0, 2, 4, 3]]).astype(np.int32)
    bt = inp.block_table.clone()
    bt[1, 0] = inp.num_pages + 5          # a page past the cache
    bt[2, 1] = -1                         # an unused entry
    D = w.head_dim
    k0 = torch.full((n, D), 0xAB, dtype=torch.uint8, device="cuda")
    s0 = torch.full((n,), 7.0, dtype=torch.float32, device="cuda")
    k, s = api.indexer_gather_k(inp.cache, bt, torch.tensor(cu, device="cuda"), torch.tensor(tts, device="cuda"),
                                len(lens), P, D, layout, k_out=k0, scale_out=s0)
    torch.cuda.synchronize()
    rk, rs = cp_gather_indexer_k(_np(inp.cache), _np(bt), cu, tts, len(lens), P, D, layout,
                                 np.full((n, D), 0xAB, np.uint8), np.full(n, 7.0, np.float32))
    assert np.array_equal(_np(k), rk)
    assert np.array_equal(_np(s).view(np.uint32), rs.view(np.uint32))


@pytest.mark.parametrize("D,P", [(48, 64), (512, 16), (36, 64), (16, 64), (32, 64), (64, 16), (256, 64)])
def test_gather_head_dims(D, P):
    """Other head sizes: 32 tokens per warp with 1, 2, 4, 16 and 32 16-byte pieces per row
    (D = 16, 32, 64, 256, 512), a 16-byte lane group of 3 (D = 48), and the 4-byte word
    path (D = 36, rows only 4-byte aligned)."""
    w = si.small_indexer_workload(num_tokens=4, ctx_lo=30, ctx_hi=150, head_dim=D, block_size=P, extra_pages=1)
    inp = si.make_indexer_inputs(w, seed=D, device="cuda")
    lens = inp.ctx
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    tts = np.repeat(np.arange(len(lens)), lens).astype(np.int32)
    n = int(cu[-1])
    k0 = torch.full((n, D), 0x5A, dtype=torch.uint8, device="cuda")
    s0 = torch.full((n,), -3.0, dtype=torch.float32, device="cuda")
    k, s = api.indexer_gather_k(inp.cache, inp.block_table, torch.tensor(cu, device="cuda"),
                                torch.tensor(tts, device="cuda"), len(lens), P, D, 0, k_out=k0, scale_out=s0)
    torch.cuda.synchronize()
    rk, rs = cp_gather_indexer_k(_np(inp.cache), _np(inp.block_table), cu, tts, len(lens), P, D, 0)
    assert np.array_equal(_np(k), rk)
    assert np.array_equal(_np(s).view(np.uint32), rs.view(np.uint32))


# ----------------------------------------------------------------- logits
def _abs_bound(inp, max_len):
    """sum_h |w_h| * sum_d |q_hd k_sd| (the magnitude the float32 sums run over)."""
    w = inp.workload
    P, D = w.block_size, w.head_dim
    cache = _np(inp.cache).copy()
    cache[:, : P * D] &= 0x7F                       # key bytes' sign bits (layout 0)
    return mqa_logits(_np(inp.q) & 0x7F, np.abs(_np(inp.weights)), cache, _np(inp.block_table), _np(inp.req_id),
                      _np(inp.ctx_lens), P, D, max_len=max_len)


def _check_logits(got, inp, max_len, tokens=None):
    w = inp.workload
    sel = slice(None) if tokens is None else list(tokens)
    ref = mqa_logits(_np(inp.q)[sel], _np(inp.weights)[sel], _np(inp.cache), _np(inp.block_table),
                     _np(inp.req_id)[sel], _np(inp.ctx_lens)[sel], w.block_size, w.head_dim, max_len=max_len)
    g = _np(got)[sel].astype(np.float64)
    assert np.array_equal(np.isneginf(g), np.isneginf(ref)), "-inf pattern"
    fin = np.isfinite(ref)
    assert np.all(np.isfinite(g[fin]))
    sub = inp if tokens is None else _subset(inp, tokens)
    bound = _abs_bound(sub, max_len)
    err = np.abs(g[fin] - ref[fin])
    assert np.all(err <= 4e-5 * bound[fin] + 1e-30), f"max err/bound {np.max(err / (bound[fin] + 1e-30)):.3g}"
    return ref


def _subset(inp, tokens):
    t = torch.tensor(list(tokens), device=inp.q.device)
    return si.IndexerInputs(inp.workload, inp.q[t], inp.weights[t], inp.cache, inp.block_table, inp.req_id[t],
                            inp.ctx_lens[t], inp.layout, [inp.ctx[i] for i in tokens])


@pytest.mark.parametrize("H,P,T,lo,hi", [(64, 64, 3, 100, 300), (32, 8, 4, 1, 260), (128, 128, 2, 129, 700),
                                         (64, 16, 5, 60, 512)])
def test_logits_match_oracle(H, P, T, lo, hi):
    w = si.small_indexer_workload(num_tokens=T, ctx_lo=lo, ctx_hi=hi, num_heads=H, block_size=P, extra_pages=3)
    inp = si.make_indexer_inputs(w, seed=H + P, device="cuda")
    L = inp.max_len + 37                             # positions past every context, partly in a last tile
    got = api.indexer_mqa_logits(inp.q, inp.weights, inp.cache, inp.block_table, inp.req_id, inp.ctx_lens, L,
                                 block_size=P)
    torch.cuda.synchronize()
    _check_logits(got, inp, L)


def test_logits_masks_bad_pages_requests_and_short_rows():
    w = si.small_indexer_workload(num_tokens=4, ctx_lo=300, ctx_hi=300, block_size=64, extra_pages=1)
    inp = si.make_indexer_inputs(w, seed=5, device="cuda")
    inp.block_table[0, 1] = inp.num_pages + 2        # positions 64..127 of token 0: page past the cache
    inp.block_table[1, 2] = -1                       # positions 128..191 of token 1: unused entry
    inp.req_id[2] = 17                               # token 2: request outside the table
    L = 256                                          # shorter than the contexts: rows cut at L
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = api.indexer_mqa_logits(inp.q, inp.weights, inp.cache, inp.block_table, inp.req_id, inp.ctx_lens, L,
                                 status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g = _np(got)
    assert np.all(np.isneginf(g[0, 64:128])) and np.all(np.isfinite(g[0, :64]))
    assert np.all(np.isneginf(g[1, 128:192])) and np.all(np.isneginf(g[2]))
    _check_logits(got, inp, L)


@pytest.mark.parametrize("which,toks", [(0, [0, 1, "argmax", "argmin", 17, 31]), (1, [0, 1, 128, 255])])
def test_logits_full_size_sampled(which, toks):
    """The mid-batch indexer shape (32 requests, context U[4096, 32768]: CTAs wholly past
    a row's context write -inf only) and the large-batch one (256 requests of 8192), 64
    heads of 128, in the launch the benchmark times: every entry written (the output
    starts as NaN), sampled tokens against the oracle."""
    w = si.INDEXER_WORKLOADS[which]
    inp = si.make_indexer_inputs(w, device="cuda")
    L = inp.max_len
    out = torch.full((w.num_tokens, L), float("nan"), dtype=torch.float32, device="cuda")
    got = api.indexer_mqa_logits(inp.q, inp.weights, inp.cache, inp.block_table, inp.req_id, inp.ctx_lens, L,
                                 logits=out)
    torch.cuda.synchronize()
    assert not bool(torch.isnan(got).any())
    pick = {"argmax": int(np.argmax(inp.ctx)), "argmin": int(np.argmin(inp.ctx))}
    _check_logits(got, inp, L, [pick.get(t, t) for t in toks])


def _inputs_with_contexts(ctx, seed, H=64, P=64):
    """Indexer inputs whose tokens have the given contexts (pages for the longest one each)."""
    top = max(max(ctx), 1)
    w = si.small_indexer_workload(num_tokens=len(ctx), ctx_lo=top, ctx_hi=top, num_heads=H, block_size=P,
                                  extra_pages=2)
    inp = si.make_indexer_inputs(w, seed=seed, device="cuda")
    return dataclasses.replace(inp, ctx_lens=torch.tensor(ctx, dtype=torch.int32, device="cuda"), ctx=list(ctx))


@pytest.mark.parametrize("ctx,L", [([0, 0, 5000, 0], 5000), ([32768], 32768), ([70000, 0, 5], 70000),
                                   ([12000] * 80, 12000), ([1] * 900, 1), ([0] * 40, 300),
                                   ([3000, 128, 129, 127, 1, 0, 2999, 640], 3001)])
def test_logits_ragged_rows_write_every_entry(ctx, L):
    """Ragged rows (empty ones, one position, a partial last tile, rows of 70 000, 900
    tokens): every entry written (the output starts as NaN), sampled rows against the
    oracle."""
    inp = _inputs_with_contexts(ctx, seed=len(ctx) + L % 97)
    out = torch.full((len(ctx), L), float("nan"), dtype=torch.float32, device="cuda")
    got = api.indexer_mqa_logits(inp.q, inp.weights, inp.cache, inp.block_table, inp.req_id, inp.ctx_lens, L,
                                 logits=out)
    torch.cuda.synchronize()
    assert not bool(torch.isnan(got).any())
    _check_logits(got, inp, L, sorted({0, len(ctx) // 2, len(ctx) - 1}))


def test_gather_full_size_prefix():
    """The key gather of every cached position of the large-batch indexer shape (256
    sequences of 8192 positions, 2 097 152 tokens) in the launch the benchmark times; the
    first three sequences' 24 576 tokens against the oracle bit for bit, and no row past
    the batch touched."""
    w = si.INDEXER_WORKLOADS[1]
    inp = si.make_indexer_inputs(w, device="cuda")
    lens = np.asarray(inp.ctx)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    n = int(cu[-1])
    tts = np.repeat(np.arange(len(lens)), lens).astype(np.int32)
    D, P = w.head_dim, w.block_size
    k0 = torch.full((n + 64, D), 0x3C, dtype=torch.uint8, device="cuda")
    s0 = torch.full((n + 64,), 9.0, dtype=torch.float32, device="cuda")
    api.indexer_gather_k(inp.cache, inp.block_table, torch.tensor(cu, device="cuda"), torch.tensor(tts, device="cuda"),
                         len(lens), P, D, 0, k_out=k0[:n], scale_out=s0[:n])
    torch.cuda.synchronize()
    m = int(cu[3])
    rk, rs = cp_gather_indexer_k(_np(inp.cache), _np(inp.block_table), cu[:4], tts[:m], 3, P, D, 0)
    assert np.array_equal(_np(k0[:m]), rk)
    assert np.array_equal(_np(s0[:m]).view(np.uint32), rs.view(np.uint32))
    assert bool((k0[n:] == 0x3C).all()) and bool((s0[n:] == 9.0).all())


# ----------------------------------------------------------------- top-k
def _check_topk(got, logits_gpu, ctx, K):
    lg = _np(logits_gpu).astype(np.float64)
    L = lg.shape[1]
    for t in range(lg.shape[0]):
        n = min(int(ctx[t]), L)
        lg[t, n:] = -np.inf
    lg[np.isnan(lg)] = -np.inf
    ref = topk_positions(lg, K)
    g = _np(got)
    for t in range(g.shape[0]):
        a = g[t][g[t] >= 0]
        b = ref[t][ref[t] >= 0]
        assert a.size == b.size, t
        assert np.array_equal(np.sort(a), np.sort(b)), t
        assert np.all(g[t][a.size:] == -1)
        if a.size == K:  # positions above the K-th value first, each group ascending
            v = lg[t, a]
            above = a[v > v.min()]
            assert np.array_equal(a[:above.size], np.sort(above))
            assert np.all(np.diff(a[above.size:]) > 0)
        else:            # fewer finite logits than K: all of them, ascending
            assert np.all(np.diff(a) > 0)


@pytest.mark.parametrize("T,L,K", [(3, 5000, 512), (2, 300, 400), (4, 70000, 2048), (2, 120000, 2048), (1, 1, 1),
                                   (50, 20000, 1024), (50, 60000, 2048), (80, 3000, 256), (96, 45000, 2048)])
def test_topk_on_synthetic_logits(T, L, K):
    """Few tokens take the clustered kernel (four CTAs per token; on 152 SMs up to 76
    tokens), many tokens or rows past 64 K positions one CTA per token (keys in shared
    memory up to 40 K positions, else read from global memory on every pass)."""
    g = torch.Generator(device="cuda").manual_seed(T * L + K)
    lg = torch.randn(T, L, generator=g, device="cuda")
    if L > 100:
        lg[0, 10:60] = 1.25                          # a run of equal values around the cut
        lg[0, 7] = float("nan")
        lg[0, 8] = -float("inf")
        lg[0, 9] = -0.0
        lg[0, 61] = 0.0
    ctx = torch.tensor([L - 3 * t for t in range(T)], dtype=torch.int32, device="cuda").clamp_min(0)
    got = api.indexer_topk(lg, ctx, K)
    torch.cuda.synchronize()
    _check_topk(got, lg, _np(ctx), K)


@pytest.mark.parametrize("T", [3, 90])
def test_topk_empty_and_short_rows(T):
    """Rows of no position, of fewer finite logits than K, and of only -inf, on the
    clustered (3 tokens) and the single-CTA (90 tokens) kernels."""
    L, K = 2000, 100
    lg = torch.randn(T, L, device="cuda")
    lg[1, :] = -float("inf")
    ctx = torch.full((T,), L, dtype=torch.int32, device="cuda")
    ctx[0] = 0
    ctx[2] = 37
    got = api.indexer_topk(lg, ctx, K)
    torch.cuda.synchronize()
    g = _np(got)
    assert np.all(g[0] == -1) and np.all(g[1] == -1)
    assert g[2, :37].tolist() == list(range(37)) and np.all(g[2, 37:] == -1)
    _check_topk(got, lg, _np(ctx), K)


def test_topk_ties_at_the_cut_take_the_lowest_positions():
    lg = torch.full((1, 4096), -1.0, device="cuda")
    lg[0, 100:200] = 3.0                             # 100 equal values; K = 60 takes the lowest 60 of them
    lg[0, 4000] = 5.0
    got = api.indexer_topk(lg, torch.tensor([4096], dtype=torch.int32, device="cuda"), 61)
    torch.cuda.synchronize()
    assert _np(got)[0].tolist() == [4000] + list(range(100, 160))


@pytest.mark.parametrize("T,L", [(80, 12000), (80, 45000), (3, 30000), (50, 30000)])
def test_topk_rows_of_nearly_equal_logits(T, L):
    """Rows whose logits almost all share the top 12 bits of their key, so that the keys
    under the chosen digit outnumber the single-CTA kernel's 8192 candidate slots (80
    tokens: the last pass then scans the row again, from shared memory at 12 000 positions,
    from global memory at 45 000), and the clustered kernels' slices fill their candidate
    lists (3 and 50 tokens)."""
    g = torch.Generator(device="cuda").manual_seed(T + L)
    lg = 1.0 + torch.rand(T, L, generator=g, device="cuda") * 1e-3   # one exponent, top mantissa bits alike
    lg[:, ::997] = 2.5                                                # a few clear winners
    lg[0, 5:40] = 1.0005                                              # equal values near the cut
    ctx = torch.tensor([L - 7 * t for t in range(T)], dtype=torch.int32, device="cuda")
    for K in (100, 2048):
        got = api.indexer_topk(lg, ctx, K)
        torch.cuda.synchronize()
        _check_topk(got, lg, _np(ctx), K)


def test_topk_ties_at_the_cut_single_cta_kernel():
    """Many tokens (one CTA each): rows whose K-th largest value is shared by a run of
    positions take the lowest of them, rows where it is unique take it alone, and the two
    ordered-pass paths agree with the rule."""
    T, L, K = 80, 3000, 61
    g = torch.Generator(device="cuda").manual_seed(7)
    lg = torch.randn(T, L, generator=g, device="cuda") - 10.0   # all below the planted values
    for t in range(0, T, 2):                                      # even rows: 100 ties at the cut
        lg[t, 100 + t:200 + t] = 3.0
        lg[t, 2900] = 5.0
    for t in range(1, T, 2):                                      # odd rows: distinct planted values
        lg[t, 100:161] = torch.linspace(3.0, 4.0, 61, device="cuda")
    ctx = torch.full((T,), L, dtype=torch.int32, device="cuda")
    got = _np(api.indexer_topk(lg, ctx, K))
    torch.cuda.synchronize()
    for t in range(0, T, 2):
        assert got[t].tolist() == [2900] + list(range(100 + t, 160 + t)), t
    for t in range(1, T, 2):
        assert sorted(got[t].tolist()) == list(range(100, 161)), t
        assert got[t][-1] == 100 and np.all(np.diff(got[t][:-1]) > 0), t   # the K-th largest last
    _check_topk(torch.from_numpy(got), lg, _np(ctx), K)


# ----------------------------------------------------------------- indexer -> decode
def test_indexer_topk_drives_the_decode():
    """Logits and top-k of the indexer over a key cache, then the sparse decode over the
    latent cache of the same requests (same context lengths and page tables) with those
    positions as its top-k list."""
    T, ctx, K = 3, 700, 160
    wi = si.small_indexer_workload(num_tokens=T, ctx_lo=ctx, ctx_hi=ctx, topk=K, extra_pages=0)
    ii = si.make_indexer_inputs(wi, seed=23, device="cuda")
    wd = synth.small_workload(num_tokens=T, num_heads=64, topk=K, swa=32, ctx=ctx, n_invalid=0)
    di = synth.make_inputs(wd, seed=24, device="cuda")
    logits = api.indexer_mqa_logits(ii.q, ii.weights, ii.cache, ii.block_table, ii.req_id, ii.ctx_lens, ctx)
    topk = api.indexer_topk(logits, ii.ctx_lens, K)
    torch.cuda.synchronize()
    _check_topk(topk, logits, ii.ctx, K)
    di.topk_idx.copy_(topk)
    out, lse = api.sparse_mla_decode(di.q, di.kv_cache, di.block_table, di.req_id, di.topk_idx, di.swa_idx,
                                     di.sink, di.scale, num_splits=0)
    torch.cuda.synchronize()
    ro, rl = oracle_decode(di)
    assert_out_close(out, ro, "indexer -> decode")
    assert_lse_close(lse, rl, "indexer -> decode")
