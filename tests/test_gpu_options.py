"""GPU parity of the decode options, through the C ABI, against the float64 oracle:

* a bf16 latent cache (1024-byte rows) instead of fp8_ds_mla;
* two scopes over two caches: top-k entries in the main cache, window entries in a
  window cache with its own block table and page size, one softmax over both;
* a per-token top-k length that masks the top-k columns at and past it;
* compaction: the conversion packs each token's valid slots to the front and the
  attention reads per-token counts instead of masked rows;
* the pages' ragged conversion with 0 for an invalid entry;
* several query tokens per request (multi-token prediction) through req_id.

Integer outputs (slots, counts, ragged output, bf16 rows) are compared bit for bit; the
attention within the tolerances of the other GPU parity tests.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle.bf16_cache import dequant_rows_bf16, sparse_mla_decode_bf16
from oracle.dual_scope import sparse_mla_decode_dual
from oracle.ragged import apply_topk_length, compact, convert_req_index_ragged
from sparse_mla_decode_req_gb300 import api, build, synth
from tests.gpu_util import assert_lse_close, assert_out_close, bf16_to_f64, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    api.load()


def _np(t):
    return t.detach().cpu().numpy()


def _q(inp):
    return bf16_to_f64(inp.q)


def _sink(inp):
    return inp.sink.detach().cpu().double().numpy()


# ----------------------------------------------------------------- bf16 latent cache
def _poison_bf16(cache, P, slots):
    """Non-finite values and a negative zero in the given slots' rows."""
    v = cache.view(torch.int16).reshape(-1)
    for i, s in enumerate(slots):
        base = (s // P) * P * 512 + (s % P) * 512
        v[base + (7 * i) % 512] = 0x7FC0                  # NaN
        v[base + (7 * i + 100) % 512] = 0x7F80            # +inf
        v[base + (7 * i + 450) % 512] = -128              # 0xFF80, -inf
        v[base + (7 * i + 3) % 512] = -32768              # 0x8000, -0.0 (kept)


@pytest.mark.parametrize("P", [64, 1, 3])
def test_gather_bf16_rows_bit_exact(P):
    pages = 40 if P > 1 else 600
    cache = synth.make_cache_bf16(pages, P, seed=5, device="cuda")
    n_slots = pages * P
    _poison_bf16(cache, P, [0, 7, 33, n_slots - 1])
    gen = torch.Generator().manual_seed(19)
    slots = torch.randint(-2, n_slots + 3, (1000,), generator=gen, dtype=torch.int32)
    slots[:4] = torch.tensor([0, 7, 33, n_slots - 1], dtype=torch.int32)
    kv = api.gather_dequant(cache, slots.cuda(), P, cache_format=api.CACHE_BF16)
    torch.cuda.synchronize()
    got = bf16_to_f64(kv)
    ok = (slots >= 0) & (slots < n_slots)
    ref = np.zeros((1000, 512))
    ref[ok.numpy()] = dequant_rows_bf16(_np(cache), slots[ok].numpy(), P)
    assert np.array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


def _bf16_case(w, seed, poison=False):
    inp = synth.make_inputs(w, seed=seed, device="cuda")
    cache = synth.make_cache_bf16(inp.num_pages, w.block_size, seed + 7, "cuda")
    if poison:
        bt = inp.block_table.cpu()
        P = w.block_size
        slots = [int(bt[0, int(inp.topk_idx[0, i]) // P]) * P + int(inp.topk_idx[0, i]) % P for i in range(5)
                 if int(inp.topk_idx[0, i]) >= 0]
        _poison_bf16(cache, P, slots)
    return inp, cache


def _bf16_oracle(inp, cache, tokens=None):
    w = inp.workload
    sel = slice(None) if tokens is None else list(tokens)
    out, lse = sparse_mla_decode_bf16(_q(inp)[sel], _np(cache), _np(inp.block_table), _np(inp.req_id)[sel],
                                      _np(inp.topk_idx)[sel] if w.topk else None,
                                      _np(inp.swa_idx)[sel] if w.swa else None, _sink(inp), inp.scale,
                                      w.block_size)
    return out, lse


@pytest.mark.parametrize("H,N,P,ns", [(64, 200, 64, 1), (128, 330, 16, -3), (16, 70, 3, 1), (96, 640, 64, -5)])
def test_decode_bf16_cache_matches_oracle(H, N, P, ns):
    w = synth.small_workload(num_tokens=3, num_heads=H, topk=N - N // 5, swa=N // 5, ctx=3 * N,
                             block_size=P, n_invalid=N // 9)
    inp, cache = _bf16_case(w, seed=40 + H, poison=True)
    out, lse = api.sparse_mla_decode(inp.q, cache, inp.block_table, inp.req_id, inp.topk_idx, inp.swa_idx,
                                     inp.sink, inp.scale, num_splits=ns, block_size=P,
                                     cache_format=api.CACHE_BF16)
    torch.cuda.synchronize()
    ro, rl = _bf16_oracle(inp, cache)
    assert_out_close(out, ro, f"bf16 H={H} N={N} P={P}")
    assert_lse_close(lse, rl, f"bf16 H={H} N={N} P={P}")


def test_decode_bf16_cache_large_batch_sampled():
    """The large-batch shape (256 tokens x 64 heads, top-k 512 + window 128) over a bf16
    cache, in the launch configuration of the fp8 benchmark (one split); 12 sampled tokens
    against the oracle."""
    w = synth.WORKLOADS[3]
    inp, cache = _bf16_case(w, seed=77)
    out, lse = api.sparse_mla_decode(inp.q, cache, inp.block_table, inp.req_id, inp.topk_idx, inp.swa_idx,
                                     inp.sink, inp.scale, num_splits=1, cache_format=api.CACHE_BF16)
    torch.cuda.synchronize()
    toks = [0, 1, 37, 63, 64, 100, 128, 151, 152, 200, 254, 255]
    ro, rl = _bf16_oracle(inp, cache, toks)
    assert_out_close(out[toks], ro, "bf16 large batch")
    assert_lse_close(lse[toks], rl, "bf16 large batch")


@pytest.mark.parametrize("fmt,ns", [("fp8", 1), ("fp8", -3), ("bf16", 1), ("bf16", -2)])
def test_several_tokens_per_request(fmt, ns):
    """Several query tokens of one request (multi-token prediction): tokens 2r and 2r + 1
    both read request 2r's pages through req_id, each with its own top-k list and window;
    the request rows of the odd tokens go unused."""
    w = synth.small_workload(num_tokens=6, num_heads=64, topk=150, swa=40, ctx=400, n_invalid=11)
    inp = synth.make_inputs(w, seed=91, device="cuda")
    inp.req_id.copy_(torch.tensor([0, 0, 2, 2, 4, 4], dtype=torch.int32))
    if fmt == "fp8":
        out, lse = api.sparse_mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.req_id, inp.topk_idx,
                                         inp.swa_idx, inp.sink, inp.scale, num_splits=ns)
        torch.cuda.synchronize()
        ro, rl = oracle_decode(inp)
    else:
        cache = synth.make_cache_bf16(inp.num_pages, w.block_size, 93, "cuda")
        out, lse = api.sparse_mla_decode(inp.q, cache, inp.block_table, inp.req_id, inp.topk_idx, inp.swa_idx,
                                         inp.sink, inp.scale, num_splits=ns, cache_format=api.CACHE_BF16)
        torch.cuda.synchronize()
        ro, rl = _bf16_oracle(inp, cache)
    assert_out_close(out, ro, f"several tokens per request {fmt}")
    assert_lse_close(lse, rl, f"several tokens per request {fmt}")


# ----------------------------------------------------------------- two caches
def _dual(T, H, K, W, P_main, P_swa, seed, ctx=600, inv_main=7, inv_swa=3):
    wm = synth.Workload("main", T, H, K, 0, ctx, ctx, block_size=P_main, n_invalid=inv_main, extra_pages=2)
    ws = synth.Workload("swa", T, H, 0, W, ctx // 3, ctx // 3, block_size=P_swa, n_invalid=inv_swa, extra_pages=1)
    a = synth.make_inputs(wm, seed=seed, device="cuda")
    b = synth.make_inputs(ws, seed=seed + 100, device="cuda")
    return a, b


def _dual_oracle(a, b, bf16_caches=None):
    if bf16_caches is None:
        return sparse_mla_decode_dual(_q(a), _np(a.req_id), _sink(a), a.scale,
                                      _np(a.kv_cache), _np(a.block_table), a.block_size, _np(a.topk_idx),
                                      _np(b.kv_cache), _np(b.block_table), b.block_size, _np(b.swa_idx))
    # bf16 caches: one stacked list of rows, as the dual-scope oracle builds it
    cm, cs = bf16_caches
    T, H = a.q.shape[0], a.q.shape[1]
    out, lse = np.zeros((T, H, 512)), np.zeros((T, H))
    gm = oracle.convert_req_index(_np(a.req_id), _np(a.block_table), _np(a.topk_idx), None, a.block_size,
                                  cm.shape[0])
    gs = oracle.convert_req_index(_np(a.req_id), _np(b.block_table), None, _np(b.swa_idx), b.block_size,
                                  cs.shape[0])
    q = _q(a)
    for t in range(T):
        k = np.concatenate([dequant_rows_bf16(_np(cm), gm[t][gm[t] >= 0], a.block_size),
                            dequant_rows_bf16(_np(cs), gs[t][gs[t] >= 0], b.block_size)])
        out[t], lse[t] = oracle.attend(q[t], k, _sink(a), a.scale)
    return out, lse


@pytest.mark.parametrize("P_main,P_swa,ns", [(64, 64, 1), (64, 16, 1), (64, 16, -4), (32, 3, 1), (1, 64, -2)])
def test_decode_two_caches_matches_oracle(P_main, P_swa, ns):
    a, b = _dual(T=3, H=64, K=300, W=90, P_main=P_main, P_swa=P_swa, seed=50 + P_swa)
    out, lse = api.sparse_mla_decode(a.q, a.kv_cache, a.block_table, a.req_id, a.topk_idx, b.swa_idx, a.sink,
                                     a.scale, num_splits=ns, block_size=P_main, swa_kv_cache=b.kv_cache,
                                     swa_block_table=b.block_table, swa_block_size=P_swa)
    torch.cuda.synchronize()
    ro, rl = _dual_oracle(a, b)
    assert_out_close(out, ro, f"dual {P_main}/{P_swa}")
    assert_lse_close(lse, rl, f"dual {P_main}/{P_swa}")


def test_decode_two_caches_out_of_range_window_pages():
    """Window block-table entries past the window cache, -1 and negative: masked by the
    window cache's own page range, not the main cache's."""
    a, b = _dual(T=4, H=16, K=100, W=64, P_main=64, P_swa=16, seed=61)
    bt = b.block_table.clone()
    bt[0, :] = b.num_pages + 5            # beyond the window cache
    bt[1, ::2] = -1
    bt[2, 1::3] = -7
    b.block_table = bt
    out, lse = api.sparse_mla_decode(a.q, a.kv_cache, a.block_table, a.req_id, a.topk_idx, b.swa_idx, a.sink,
                                     a.scale, num_splits=1, swa_kv_cache=b.kv_cache, swa_block_table=bt,
                                     swa_block_size=16)
    torch.cuda.synchronize()
    ro, rl = _dual_oracle(a, b)
    assert_out_close(out, ro, "dual window pages")
    assert_lse_close(lse, rl, "dual window pages")


def test_decode_two_bf16_caches_matches_oracle():
    a, b = _dual(T=3, H=128, K=260, W=70, P_main=64, P_swa=8, seed=71)
    cm = synth.make_cache_bf16(a.num_pages, 64, 5, "cuda")
    cs = synth.make_cache_bf16(b.num_pages, 8, 6, "cuda")
    for ns in (1, -3):
        out, lse = api.sparse_mla_decode(a.q, cm, a.block_table, a.req_id, a.topk_idx, b.swa_idx, a.sink, a.scale,
                                         num_splits=ns, cache_format=api.CACHE_BF16, swa_kv_cache=cs,
                                         swa_block_table=b.block_table, swa_block_size=8)
        torch.cuda.synchronize()
        ro, rl = _dual_oracle(a, b, (cm, cs))
        assert_out_close(out, ro, f"dual bf16 splits {ns}")
        assert_lse_close(lse, rl, f"dual bf16 splits {ns}")


def test_two_caches_staged_calls():
    """Conversion with the window block table, then the attention with the window cache
    (the first K entries of each row in the main cache), then the combine."""
    a, b = _dual(T=3, H=64, K=200, W=60, P_main=64, P_swa=16, seed=81)
    g = api.convert_req_index(a.block_table, a.req_id, a.topk_idx, b.swa_idx, a.num_pages,
                              swa_block_table=b.block_table, swa_num_pages=b.num_pages, swa_block_size=16)
    gm = oracle.convert_req_index(_np(a.req_id), _np(a.block_table), _np(a.topk_idx), None, 64, a.num_pages)
    gs = oracle.convert_req_index(_np(a.req_id), _np(b.block_table), None, _np(b.swa_idx), 16, b.num_pages)
    assert np.array_equal(_np(g), np.concatenate([gm, gs], axis=1))
    for ns in (1, -3):
        x, y = api.sparse_mla_attention(a.q, a.kv_cache, g, a.sink, a.scale, num_splits=ns, main=200,
                                        swa_kv_cache=b.kv_cache, swa_block_size=16)
        out, lse = (x, y) if ns == 1 else api.lse_combine(x, y, a.sink)
        torch.cuda.synchronize()
        ro, rl = _dual_oracle(a, b)
        assert_out_close(out, ro, f"dual staged {ns}")
        assert_lse_close(lse, rl, f"dual staged {ns}")


# ----------------------------------------------------------------- top-k length
def _lengths(T, K, seed):
    gen = torch.Generator().manual_seed(seed)
    L = torch.randint(-3, K + 20, (T,), generator=gen, dtype=torch.int32)
    L[0] = 0
    if T > 1:
        L[1] = K
    if T > 2:
        L[2] = K + 100
    return L


@pytest.mark.parametrize("ns,compact_", [(1, False), (-3, False), (1, True), (-3, True)])
def test_decode_topk_length_matches_oracle(ns, compact_):
    w = synth.small_workload(num_tokens=6, num_heads=64, topk=330, swa=64, ctx=1500, n_invalid=20)
    inp = synth.make_inputs(w, seed=91, device="cuda")
    L = _lengths(6, 330, 5)
    out, lse = api.sparse_mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.req_id, inp.topk_idx, inp.swa_idx,
                                     inp.sink, inp.scale, num_splits=ns, topk_length=L.cuda(), compact=compact_)
    torch.cuda.synchronize()
    cut = apply_topk_length(_np(inp.topk_idx), L.numpy())
    ro, rl = oracle.sparse_mla_decode(_q(inp), _np(inp.kv_cache), _np(inp.block_table), _np(inp.req_id), cut,
                                      _np(inp.swa_idx), _sink(inp), inp.scale, 64)
    assert_out_close(out, ro, f"topk_length splits {ns} compact {compact_}")
    assert_lse_close(lse, rl, f"topk_length splits {ns} compact {compact_}")


# ----------------------------------------------------------------- compaction
@pytest.mark.parametrize("P", [64, 5])
def test_compaction_bit_exact(P):
    """Packed slots and counts against the oracle's compaction of its own dense
    conversion; the rest of each row is left as it was."""
    gen = torch.Generator().manual_seed(200 + P)
    R, B, pages, T, K, W = 6, 40, 300, 9, 700, 90
    bt = torch.randint(-2, pages + 3, (R, B), generator=gen, dtype=torch.int32)
    req = torch.randint(-1, R + 1, (T,), generator=gen, dtype=torch.int32)
    topk = torch.randint(-4, B * P + 9, (T, K), generator=gen, dtype=torch.int32)
    swa = torch.randint(-4, B * P + 9, (T, W), generator=gen, dtype=torch.int32)
    topk[3] = -1                                    # a token with no top-k entry
    L = _lengths(T, K, 7)
    gidx = torch.full((T, K + W), -12345, dtype=torch.int32, device="cuda")
    g, counts = api.convert_req_index(bt.cuda(), req.cuda(), topk.cuda(), swa.cuda(), pages, P, gidx=gidx,
                                      topk_length=L.cuda(), compact=True)
    torch.cuda.synchronize()
    dense = oracle.convert_req_index(req.numpy(), bt.numpy(), apply_topk_length(topk.numpy(), L.numpy()),
                                     swa.numpy(), P, pages)
    cu, kept = compact(dense)
    cu_main, _ = compact(dense[:, :K])
    got_g, got_c = _np(g), _np(counts)
    for t in range(T):
        n = int(cu[t + 1] - cu[t])
        assert got_c[t, 1] == n
        assert got_c[t, 0] == int(cu_main[t + 1] - cu_main[t])
        assert np.array_equal(got_g[t, :n], kept[cu[t]:cu[t + 1]])
        assert np.all(got_g[t, n:] == -12345)


def test_compacted_decode_heavily_masked_matches_oracle():
    """Most entries masked (the case compaction is for): the decode with compaction equals
    the oracle, and so does the staged form that hands the counts to the attention."""
    w = synth.small_workload(num_tokens=5, num_heads=128, topk=1024, swa=128, ctx=4000, n_invalid=900)
    inp = synth.make_inputs(w, seed=93, device="cuda")
    ro, rl = oracle.sparse_mla_decode(_q(inp), _np(inp.kv_cache), _np(inp.block_table), _np(inp.req_id),
                                      _np(inp.topk_idx), _np(inp.swa_idx), _sink(inp), inp.scale, 64)
    for ns in (1, -4, 0):
        out, lse = api.sparse_mla_decode(inp.q, inp.kv_cache, inp.block_table, inp.req_id, inp.topk_idx,
                                         inp.swa_idx, inp.sink, inp.scale, num_splits=ns, compact=True)
        torch.cuda.synchronize()
        assert_out_close(out, ro, f"compact splits {ns}")
        assert_lse_close(lse, rl, f"compact splits {ns}")
    g, counts = api.convert_req_index(inp.block_table, inp.req_id, inp.topk_idx, inp.swa_idx, inp.num_pages,
                                      compact=True)
    x, y = api.sparse_mla_attention(inp.q, inp.kv_cache, g, inp.sink, inp.scale, num_splits=-3, counts=counts)
    out, lse = api.lse_combine(x, y, inp.sink)
    torch.cuda.synchronize()
    assert_out_close(out, ro, "compact staged")
    assert_lse_close(lse, rl, "compact staged")


def test_compacted_two_caches_matches_oracle():
    a, b = _dual(T=4, H=64, K=400, W=100, P_main=64, P_swa=16, seed=97, inv_main=250, inv_swa=40)
    out, lse = api.sparse_mla_decode(a.q, a.kv_cache, a.block_table, a.req_id, a.topk_idx, b.swa_idx, a.sink,
                                     a.scale, num_splits=-2, swa_kv_cache=b.kv_cache, swa_block_table=b.block_table,
                                     swa_block_size=16, compact=True)
    torch.cuda.synchronize()
    ro, rl = _dual_oracle(a, b)
    assert_out_close(out, ro, "compact dual")
    assert_lse_close(lse, rl, "compact dual")


# ----------------------------------------------------------------- ragged conversion
@pytest.mark.parametrize("P", [64, 1, 7])
def test_ragged_conversion_bit_exact(P):
    gen = torch.Generator().manual_seed(300 + P)
    R, B, T, C = 5, 30, 11, 700
    bt = torch.randint(0, 5000, (R, B), generator=gen, dtype=torch.int32)
    req = torch.randint(0, R, (T,), generator=gen, dtype=torch.int32)
    ti = torch.randint(-5, B * P + 40, (T, C), generator=gen, dtype=torch.int32)
    lens = torch.randint(0, C + 1, (T,), generator=gen, dtype=torch.int32)
    lens[0], lens[1] = 0, C
    cu = torch.zeros(T + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0)
    out = api.convert_req_index_ragged(bt.cuda(), req.cuda(), ti.cuda(), cu.cuda(), P)
    torch.cuda.synchronize()
    ref = convert_req_index_ragged(req.numpy(), bt.numpy(), ti.numpy(), cu.numpy(), P)
    assert np.array_equal(_np(out).astype(np.int64), ref)


def test_ragged_conversion_guards():
    """Past the index array's columns and for a request id out of range the output is 0
    (cases the pages' kernel would read out of bounds); strided index rows are honoured."""
    P, R, B = 16, 3, 8
    bt = torch.arange(R * B, dtype=torch.int32).reshape(R, B) + 100
    req = torch.tensor([0, 5, -1, 2], dtype=torch.int32)
    wide = torch.randint(0, B * P, (4, 20), generator=torch.Generator().manual_seed(3), dtype=torch.int32)
    ti = wide[:, 2:12]                                  # 10 columns, row stride 20
    cu = torch.tensor([0, 12, 15, 16, 20], dtype=torch.int32)
    out = _np(api.convert_req_index_ragged(bt.cuda(), req.cuda(), wide.cuda()[:, 2:12], cu.cuda(), P))
    torch.cuda.synchronize()
    ref = convert_req_index_ragged(req.numpy()[:1], bt.numpy(), ti.numpy()[:1], np.array([0, 10]), P)
    assert np.array_equal(out[:10].astype(np.int64), ref)
    assert np.all(out[10:12] == 0)                      # columns 10, 11 of a 10-column array
    assert np.all(out[12:16] == 0)                      # request ids 5 and -1
    ref3 = convert_req_index_ragged(req.numpy()[3:], bt.numpy(), ti.numpy()[3:], np.array([0, 4]), P)
    assert np.array_equal(out[16:].astype(np.int64), ref3)
