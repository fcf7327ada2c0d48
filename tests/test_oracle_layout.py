"""Pins for the oracle's layout, notify, dispatch index and combine paths.

* a hand-worked example (tests/golden/layout_small.json, derived by hand
  from the article's definitions);
* brute force over every id assignment of tiny problems, against an
  independent route: numpy's stable argsort gives the (token, slot) order
  of each expert's entries, np.bincount the counts;
* invariants the article fixes: counts sum to T*k, prefix-matrix columns are
  non-decreasing with the column totals in the last row, psum entries are
  multiples of the alignment, every routed slot owns exactly one row and
  each segment is sorted by (source rank, token, slot).
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from combine_get_dispatch_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "layout_small.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_golden_layout_and_notify():
    g = _golden()
    idx = np.array(g["topk_idx"], np.int64)
    lay = oracle.layout(idx, g["R"], g["E"])
    assert lay["rc"] == oracle.OK
    for key in ("num_tokens_per_expert", "slot_rank", "is_token_in_rank", "num_tokens_per_rank"):
        assert lay[key].tolist() == g[key], key
    for A, ref in ((1, g["align1"]), (4, g["align4"])):
        n = oracle.notify(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"], g["R"], g["E"], A)
        assert n["rc"] == oracle.OK
        assert n["rank_prefix_matrix"].tolist() == g["rank_prefix_matrix"]
        assert n["expert_prefix"].tolist() == g["expert_prefix"]
        assert n["num_recv_tokens_per_expert"].tolist() == ref["num_recv_tokens_per_expert"]
        assert n["psum"].tolist() == ref["psum"]


def test_golden_dispatch_indices():
    g = _golden()
    R, T_r, E, k = g["R"], g["T_r"], g["E"], g["k"]
    idx = np.array(g["topk_idx"], np.int64)
    H = 8
    x = np.arange(R * T_r * H, dtype=np.uint16).reshape(R, T_r, H)
    lay = oracle.layout(idx, R, E)
    n = oracle.notify(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"], R, E, 1)
    d = oracle.dispatch(x, idx, lay["slot_rank"], n["expert_prefix"], n["psum"], E,
                        oracle.FP8_NONE, g["normal_cap_rows"])
    assert d["rc"] == oracle.OK
    assert d["combine_idx"].tolist() == g["normal_combine_idx"]
    assert d["recv_src_idx"].tolist() == g["normal_recv_src_idx"]
    ll = oracle.ll_dispatch(x, idx, E, g["ll_max_tokens"], oracle.FP8_NONE)
    assert ll["rc"] == oracle.OK
    assert ll["combine_idx"].tolist() == g["ll_combine_idx"]
    assert ll["recv_count"].tolist() == g["ll_recv_count"]
    lr = ll["layout_range"].reshape(E, R)
    assert [[[int(v >> 32), int(v & 0xFFFFFFFF)] for v in row] for row in lr] == g["ll_layout_range"]


def _independent_layout(idx, R, E):
    """Sort-based route: stable argsort by expert id within each rank."""
    _, T_r, k = idx.shape
    E_l = E // R
    slot = np.full(idx.shape, -1, np.int64)
    cnt = np.zeros((R, E), np.int64)
    for i in range(R):
        flat = idx[i].ravel()
        valid = np.nonzero(flat >= 0)[0]
        order = valid[np.argsort(flat[valid], kind="stable")]
        sorted_e = flat[order]
        first = np.searchsorted(sorted_e, sorted_e, side="left")
        s = slot[i].reshape(-1)
        s[order] = np.arange(order.size) - first
        cnt[i] = np.bincount(flat[valid], minlength=E)
    in_rank = np.zeros((R, T_r, R), np.uint8)
    for r in range(R):
        in_rank[:, :, r] = np.any((idx >= 0) & (idx // E_l == r), axis=2)
    return slot, cnt, in_rank, in_rank.sum(axis=1)


def _check_against_independent(idx, R, E):
    lay = oracle.layout(idx, R, E)
    assert lay["rc"] == oracle.OK
    slot, cnt, in_rank, ntpr = _independent_layout(idx, R, E)
    assert np.array_equal(lay["slot_rank"], slot)
    assert np.array_equal(lay["num_tokens_per_expert"], cnt)
    assert np.array_equal(lay["is_token_in_rank"], in_rank)
    assert np.array_equal(lay["num_tokens_per_rank"], ntpr)


@pytest.mark.parametrize("R,T_r,k,E", [(2, 2, 1, 4), (2, 1, 2, 4), (1, 3, 2, 3)])
def test_brute_force_all_assignments(R, T_r, k, E):
    vals = list(range(-1, E))
    n = R * T_r * k
    for assign in itertools.product(vals, repeat=n):
        idx = np.array(assign, np.int64).reshape(R, T_r, k)
        _check_against_independent(idx, R, E)


def test_random_layouts_against_independent_route():
    rng = np.random.default_rng(1)
    for trial in range(200):
        R = int(rng.integers(1, 6))
        E_l = int(rng.integers(1, 5))
        E = R * E_l
        T_r = int(rng.integers(0, 9))
        k = int(rng.integers(1, 5))
        idx = rng.integers(-1, E, size=(R, T_r, k)).astype(np.int64)
        _check_against_independent(idx, R, E)


def _check_invariants(idx, R, E, A):
    _, T_r, k = idx.shape
    E_l = E // R
    lay = oracle.layout(idx, R, E)
    n = oracle.notify(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"], R, E, A)
    valid = (idx >= 0).sum(axis=(1, 2))
    assert np.array_equal(lay["num_tokens_per_expert"].sum(axis=1), valid)
    rpm = n["rank_prefix_matrix"]
    assert np.all(np.diff(rpm, axis=0) >= 0)
    assert np.array_equal(rpm[-1], lay["num_tokens_per_rank"].sum(axis=0))
    assert np.array_equal(rpm[0], lay["num_tokens_per_rank"][0])
    assert np.all(lay["num_tokens_per_rank"].sum(axis=1) <= T_r * min(k, R))
    ep = n["expert_prefix"]
    assert np.array_equal(ep[-1], lay["num_tokens_per_expert"].sum(axis=0))
    assert np.all(n["psum"] % A == 0)
    assert np.array_equal(np.diff(n["psum"], axis=1), n["num_recv_tokens_per_expert"])
    assert np.all(n["num_recv_tokens_per_expert"] >= ep[-1].reshape(R, E_l))
    assert np.all(n["num_recv_tokens_per_expert"] - ep[-1].reshape(R, E_l) < A)
    cap = int(n["psum"][:, -1].max()) + 3
    H = 8
    x = (np.arange(R * T_r, dtype=np.uint16)[:, None] * np.ones(H, np.uint16)).reshape(R, T_r, H)
    d = oracle.dispatch(x, idx, lay["slot_rank"], ep, n["psum"], E, oracle.FP8_NONE, cap)
    assert d["rc"] == oracle.OK
    cidx = d["combine_idx"]
    src = d["recv_src_idx"]
    used = cidx[cidx >= 0]
    assert used.size == (idx >= 0).sum() and np.unique(used).size == used.size
    assert np.array_equal(np.sort(np.nonzero(src.ravel() >= 0)[0]), np.sort(used))
    # round trip: the row of slot (i,t,j) names token i*T_r+t and holds its data
    for i in range(R):
        for t in range(T_r):
            for j in range(k):
                f = cidx[i, t, j]
                if f < 0:
                    continue
                assert src.ravel()[f] == i * T_r + t
                e = idx[i, t, j]
                r, l = divmod(int(e), E_l)
                assert f // cap == r
                row = f % cap
                assert n["psum"][r, l] <= row < n["psum"][r, l] + ep[-1][e]
                assert np.all(d["recv_x"][r, row] == x[i, t])
    # segments sorted by (source rank, token, slot)
    for r in range(R):
        for l in range(E_l):
            e = r * E_l + l
            lo = n["psum"][r, l]
            keys = [(i, t, j) for i in range(R) for t in range(T_r) for j in range(k)
                    if idx[i, t, j] == e]
            rows = [cidx[i, t, j] % cap for (i, t, j) in keys]
            assert rows == list(range(lo, lo + len(keys)))


@pytest.mark.parametrize("A", [1, 4, 128])
def test_invariants_random(A):
    rng = np.random.default_rng(A)
    for trial in range(30):
        R = int(rng.integers(1, 5))
        E = R * int(rng.integers(1, 5))
        T_r = int(rng.integers(0, 7))
        k = int(rng.integers(1, 4))
        idx = rng.integers(-1, E, size=(R, T_r, k)).astype(np.int64)
        _check_invariants(idx, R, E, A)


def test_invariants_tiny_workload():
    w = synth.WORKLOADS["tiny"]
    idx, _ = synth.routing(w)
    assert np.all([len(set(row)) == w.k for row in idx.reshape(-1, w.k)])
    _check_invariants(idx, w.R, w.E, 1)
    _check_invariants(idx, w.R, w.E, 128)


def test_invalid_ids_and_capacity():
    idx = np.array([[[0, 5]]], np.int64)
    assert oracle.layout(idx, 1, 4)["rc"] == oracle.ERR_INVALID_ARG
    idx = np.array([[[0, -2]]], np.int64)
    assert oracle.layout(idx, 1, 4)["rc"] == oracle.ERR_INVALID_ARG
    # num_worst_tokens smaller than the received token count
    idx = np.array([[[0], [0], [1]], [[0], [1], [1]]], np.int64)
    lay = oracle.layout(idx, 2, 2)
    assert oracle.notify(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"], 2, 2, 1, 2)["rc"] \
        == oracle.ERR_CAPACITY
    assert oracle.notify(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"], 2, 2, 1, 3)["rc"] \
        == oracle.OK
    # dispatch capacity: rank 0 receives 3 rows, cap 2
    n = oracle.notify(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"], 2, 2, 1)
    x = np.zeros((2, 3, 8), np.uint16)
    d = oracle.dispatch(x, idx, lay["slot_rank"], n["expert_prefix"], n["psum"], 2, 0, 2)
    assert d["rc"] == oracle.ERR_CAPACITY
    assert (d["combine_idx"] >= 0).sum() == 4
    # low-latency: T_r above the per-rank capacity is rejected
    assert oracle.ll_dispatch(x, idx, 2, 2, 0)["rc"] == oracle.ERR_INVALID_ARG
    # a repeated expert inside one token can overflow R*max rows
    idx2 = np.array([[[0, 0]], [[0, 0]]], np.int64)
    x2 = np.zeros((2, 1, 8), np.uint16)
    ll = oracle.ll_dispatch(x2, idx2, 2, 1, 0)
    assert ll["rc"] == oracle.ERR_CAPACITY and (ll["combine_idx"] >= 0).sum() == 2
