"""Pins for the oracle's request-local -> global index conversion (CPU only).

Checked two ways that do not reuse its formula: hand-worked cases from
``tests/golden/convert_hand.txt`` and a brute-force inverse map built from the block
table (every (request, position) a page holds), on tiny random tables.
"""
import os

import numpy as np
import pytest

from oracle import convert_req_index

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_hand():
    bt, cases, P, num_pages = [], [], None, None
    with open(os.path.join(GOLDEN, "convert_hand.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("block_size"):
                P = int(line.split()[1])
            elif line.startswith("num_pages"):
                num_pages = int(line.split()[1])
            elif line.startswith("bt"):
                bt.append([int(x) for x in line.split()[1:]])
            elif line.startswith("case"):
                head, idx, exp = line[4:].split("|")
                cases.append((int(head), [int(x) for x in idx.split()], [int(x) for x in exp.split()]))
    return P, num_pages, np.array(bt, dtype=np.int32), cases


def test_hand_cases():
    P, num_pages, bt, cases = _load_hand()
    for req, idx, exp in cases:
        # split each case between the top-k scope and the window scope
        k = len(idx) // 2
        got = convert_req_index(np.array([req]), bt, np.array([idx[:k]]), np.array([idx[k:]]),
                                P, num_pages)
        assert got.tolist() == [exp], (req, idx)


def test_scope_order_and_empty_scopes():
    P, num_pages, bt, _ = _load_hand()
    got = convert_req_index(np.array([1, 0]), bt, np.array([[0], [1]]), np.array([[4, 5], [5, 0]]),
                            P, num_pages)
    assert got.tolist() == [[20, 0, 1], [13, 5, 12]]
    none_w = convert_req_index(np.array([0]), bt, np.array([[0, 1]]), None, P, num_pages)
    assert none_w.tolist() == [[12, 13]]
    none_k = convert_req_index(np.array([0]), bt, None, np.array([[0, 1]]), P, num_pages)
    assert none_k.tolist() == [[12, 13]]
    empty = convert_req_index(np.array([0]), bt, np.zeros((1, 0)), np.zeros((1, 0)), P, num_pages)
    assert empty.shape == (1, 0)


@pytest.mark.parametrize("P", [1, 2, 4, 64])
def test_brute_force_inverse_map(P):
    rng = np.random.default_rng(P)
    R, max_blocks, num_pages = 3, 5, 9
    bt = rng.integers(-2, num_pages + 3, size=(R, max_blocks)).astype(np.int32)
    # inverse: slot -> list of (request, position) that map there
    slot_of = {}
    for r in range(R):
        for b in range(max_blocks):
            page = int(bt[r, b])
            if 0 <= page < num_pages:
                for o in range(P):
                    slot_of[(r, b * P + o)] = page * P + o
    idx_range = np.arange(-2, max_blocks * P + 3)
    for r in list(range(R)) + [R, -1]:
        got = convert_req_index(np.array([r]), bt, idx_range[None, :], None, P, num_pages)[0]
        exp = [slot_of.get((r, int(i)), -1) for i in idx_range]
        assert got.tolist() == exp
