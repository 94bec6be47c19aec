"""Pins for the oracle's routing (flatten + stable sort + padded layout), CPU."""
import numpy as np
import pytest

from oracle.routing import route
from tests.golden_io import read_table


def _ints(s):
    return [int(v) for v in s.split()]


def test_hand_worked_example():
    g = read_table("route_example.txt")
    T, K, E, A = (int(g[k]) for k in ("T", "K", "E", "A"))
    idx = np.array(_ints(g["topk_idx"])).reshape(T, K)
    r = route(idx, E, A)
    for key in ("counts", "offsets", "perm", "padded_offsets", "inv", "row_slot"):
        assert r[key].tolist() == _ints(g[key]), key


def _naive(idx, E, A):
    """O(S*E) scan: for each expert in order, walk the slots in order."""
    flat = idx.reshape(-1)
    S = flat.size
    inv = [-1] * S
    row_slot = []
    counts = []
    starts = []
    for e in range(E):
        starts.append(len(row_slot))
        c = 0
        for s in range(S):
            if flat[s] == e:
                inv[s] = len(row_slot)
                row_slot.append(s)
                c += 1
        counts.append(c)
        while len(row_slot) % A:
            row_slot.append(-1)
    starts.append(len(row_slot))
    return counts, starts, inv, row_slot


@pytest.mark.parametrize("T,K,E,A,p_skip", [(1, 1, 1, 1, 0.0), (7, 3, 5, 4, 0.2), (33, 8, 16, 128, 0.05),
                                             (64, 2, 8, 16, 0.5), (5, 4, 3, 8, 1.0)])
def test_matches_naive_scan(T, K, E, A, p_skip):
    rng = np.random.default_rng(T * 1000 + E)
    idx = rng.integers(0, E, (T, K))
    idx[rng.random((T, K)) < p_skip] = -1
    r = route(idx, E, A)
    counts, starts, inv, row_slot = _naive(idx, E, A)
    assert r["counts"].tolist() == counts
    assert r["padded_offsets"].tolist() == starts
    assert r["inv"].tolist() == inv
    assert r["row_slot"].tolist() == row_slot


def test_invariants_large():
    rng = np.random.default_rng(11)
    T, K, E, A = 3000, 8, 256, 128
    idx = rng.integers(0, E, (T, K))
    idx[rng.random((T, K)) < 0.05] = -1
    r = route(idx, E, A)
    flat = idx.reshape(-1)
    valid = flat >= 0
    assert r["counts"].sum() == valid.sum()
    assert (r["padded_offsets"] % A == 0).all()
    # every valid slot routed exactly once, into its own expert's group
    rows = r["inv"][valid]
    assert len(set(rows.tolist())) == rows.size
    e = flat[valid]
    assert ((rows >= r["padded_offsets"][e]) & (rows < r["padded_offsets"][e] + r["counts"][e])).all()
    assert (r["inv"][~valid] == -1).all()
    assert (r["row_slot"][rows] == np.flatnonzero(valid)).all()
    # stable: slots ascend inside every group
    for ex in range(E):
        lo, c = r["padded_offsets"][ex], r["counts"][ex]
        grp = r["row_slot"][lo:lo + c]
        assert (np.diff(grp) > 0).all()
    # perm: sorted order of keys, skipped slots last
    assert (np.diff(r["keys"][r["perm"]]) >= 0).all()


def test_invalid_ids_are_skipped_and_counted():
    idx = np.array([[0, 5], [-3, 1], [2, -1]])
    r = route(idx, 3, 1)
    assert r["n_invalid"] == 2
    assert r["inv"].tolist() == [0, -1, -1, 1, 2, -1]
    assert r["counts"].tolist() == [1, 1, 1]


def test_padding_tokens_do_not_move_real_rows():
    g = read_table("route_example.txt")
    rng = np.random.default_rng(12)
    idx = rng.integers(0, 6, (int(g["slice_tokens"]) * 3, 2))
    pad = np.full((int(g["slice_ranks"]) - 1, 2), -1)
    a = route(idx, 6, 8)
    b = route(np.concatenate([idx, pad]), 6, 8)
    n = idx.size
    assert (a["inv"] == b["inv"][:n]).all() and (b["inv"][n:] == -1).all()
    assert (a["counts"] == b["counts"]).all()
