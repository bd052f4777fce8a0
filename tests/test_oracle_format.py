"""Pins for the oracle's cache-format decoding (CPU only).

The oracle's fp8/UE8M0/bf16 decoders are checked against (a) torch's own dtype
conversions, an independent library route, over every bit pattern, and (b) hand-worked
rows in ``tests/golden/e4m3_ue8m0_hand.txt``.  The dequantised row is checked against
hand-built rows assembled byte by byte here, so that a wrong offset, a swapped byte
order, a wrong scale group or a missing scrub fails.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import decode_bf16, decode_e4m3, decode_ue8m0, dequant_rows, row_offsets
from sparse_mla_decode_req_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_e4m3_matches_torch_for_every_byte():
    b = np.arange(256, dtype=np.uint8)
    ours = decode_e4m3(b)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    assert np.nanmax(ours) == 448.0


def test_ue8m0_decode():
    c = np.arange(256)
    v = decode_ue8m0(c)
    assert np.isnan(v[255])
    for code in (0, 1, 120, 127, 128, 254):
        assert v[code] == math.ldexp(1.0, code - 127)


def test_bf16_matches_torch_for_sampled_patterns():
    rng = np.random.default_rng(0)
    u = np.concatenate([rng.integers(0, 1 << 16, 4096), [0, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x3F80]])
    u = u.astype(np.uint16)
    ours = decode_bf16(u)
    ref = torch.from_numpy(u.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


def _hand_rows():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_ue8m0_hand.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            byte, code, val = int(parts[0], 16), int(parts[1]), parts[2]
            rows.append((byte, code, None if val == "scrub" else float.fromhex(val)))
    return rows


def _build_cache(block_size, rows_spec, num_pages):
    """Assemble a cache by hand: rows_spec maps slot -> (nope bytes[448], codes[7], rope u16[64])."""
    P = block_size
    cache = np.zeros((num_pages, P * 584), dtype=np.uint8)
    flat = cache.reshape(-1)
    for slot, (nope, codes, rope) in rows_spec.items():
        page, off = divmod(slot, P)
        d = page * P * 584 + off * 576
        s = page * P * 584 + P * 576 + off * 8
        flat[d:d + 448] = nope
        rb = np.asarray(rope, dtype=np.uint16)
        flat[d + 448:d + 576:2] = (rb & 0xFF).astype(np.uint8)
        flat[d + 449:d + 576:2] = (rb >> 8).astype(np.uint8)
        flat[s:s + 7] = codes
        flat[s + 7] = 0xAB  # padding byte must be ignored
    return cache


@pytest.mark.parametrize("block_size", [64, 1, 3])
def test_dequant_hand_rows(block_size):
    """Every golden (byte, code) pair placed in a different group and slot of a cache."""
    hand = _hand_rows()
    num_pages = 8
    n_slots = num_pages * block_size
    spec, expect = {}, {}
    for i, (byte, code, val) in enumerate(hand):
        slot = (5 * i + 3) % n_slots
        group = i % 7
        pos = group * 64 + (11 * i) % 64
        nope = np.full(448, 0x38, dtype=np.uint8)          # 1.0 before scaling
        codes = np.full(7, 127, dtype=np.uint8)
        codes[group] = code
        nope[pos] = byte
        rope = np.full(64, 0x3F80, dtype=np.uint16)        # bf16 1.0
        rope[(7 * i) % 64] = 0x4040                        # bf16 3.0
        spec[slot] = (nope, codes, rope)
        e = np.ones(512)
        g0, g1 = group * 64, group * 64 + 64
        scale_val = math.ldexp(1.0, code - 127) if code != 255 else float("nan")
        e[g0:g1] = 1.0 * scale_val
        if code == 255 or not np.isfinite(scale_val):
            e[g0:g1] = 0.0
        elif abs(scale_val) >= float.fromhex("0x1.ffp127"):
            e[g0:g1] = 0.0
        e[pos] = 0.0 if val is None else val
        e[448 + (7 * i) % 64] = 3.0
        expect[slot] = e
    cache = _build_cache(block_size, spec, num_pages)
    slots = np.array(sorted(expect))
    got = dequant_rows(cache, slots, block_size)
    for r, slot in enumerate(slots):
        assert np.array_equal(got[r], expect[slot]), slot
        assert np.array_equal(np.signbit(got[r]), np.signbit(expect[slot])), slot


def test_rope_scrub_and_byte_order():
    P = 64
    nope = np.zeros(448, dtype=np.uint8)
    codes = np.full(7, 127, dtype=np.uint8)
    rope = np.zeros(64, dtype=np.uint16)
    rope[0] = 0x7F80   # +inf
    rope[1] = 0xFFC0   # nan
    rope[2] = 0x4049   # 3.140625
    rope[3] = 0xC000   # -2
    cache = _build_cache(P, {5: (nope, codes, rope)}, 1)
    k = dequant_rows(cache, [5], P)[0]
    assert k[448] == 0.0 and k[449] == 0.0
    assert k[450] == 3.140625 and k[451] == -2.0
    assert np.all(k[:448] == 0.0)


def test_row_offsets_layout():
    # page of 64 slots = 64 data rows of 576 bytes, then 64 scale rows of 8 bytes
    d, s = row_offsets(np.array([0, 1, 63, 64, 130]), 64)
    assert list(d) == [0, 576, 63 * 576, 37376, 2 * 37376 + 2 * 576]
    assert list(s) == [36864, 36872, 36864 + 63 * 8, 37376 + 36864, 2 * 37376 + 36864 + 16]


def test_generator_quantisation_round_trip():
    """Rows written by the generator decode back within e4m3's rounding bound."""
    g = torch.Generator().manual_seed(7)
    n = 257
    x = torch.randn(n, 448, generator=g) * torch.exp(torch.randn(n, 1, generator=g) * 3)
    x[3] = 0.0                                   # amax = 0 group -> code 0, all zeros
    x[4, :64] = 448.0 * 2.0 ** -3                # exact power-of-two amax
    rope = torch.randn(n, 64, generator=g)
    data, scale = synth.quantize_rows(x, rope)
    P = 1
    cache = torch.cat([data, scale], dim=1).numpy()
    k = dequant_rows(cache, np.arange(n), P)
    xs = x.to(torch.float64).numpy()
    codes = scale[:, :7].numpy().astype(np.int64)
    for r in range(n):
        for j in range(7):
            grp = xs[r, 64 * j:64 * j + 64]
            amax = np.abs(grp).max()
            c = int(codes[r, j])
            if amax == 0:
                assert c == 0
                continue
            # the smallest power of two that brings amax under 448
            assert 448.0 * math.ldexp(1.0, c - 127) >= amax
            assert c == 0 or 448.0 * math.ldexp(1.0, c - 128) < amax
            sc = math.ldexp(1.0, c - 127)
            err = np.abs(k[r, 64 * j:64 * j + 64] - grp)
            bound = np.maximum(np.abs(grp) * 2.0 ** -4, sc * 2.0 ** -10)
            assert np.all(err <= bound)
    assert codes[4, 0] == 124
    rope_ref = rope.to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(k[:, 448:], rope_ref)
