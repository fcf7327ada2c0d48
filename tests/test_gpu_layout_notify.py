"""GPU parity: layout and notify in one launch (ep_layout_notify: the layout
kernel's last CTA computes the notify tables) vs the oracle and vs the two
separate calls, bit-exact, at every workload's full size and on edge
shapes; the host handshake, the fixed-shape capacity check and repeated
calls on one workspace."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_gb300 import ep, synth
from ep_harness import gpu_layout, gpu_notify, np_, poison_, status_word

pytestmark = pytest.mark.gpu

LAYOUT_KEYS = ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "slot_rank")
NOTIFY_KEYS = ("rank_prefix_matrix", "expert_prefix", "num_recv_tokens_per_expert", "psum")


def _fused(idx_dev, E, A, nwt, ws=None, host_rows=None):
    R, T_r, k = idx_dev.shape
    lay = ep.alloc_layout(R, T_r, k, E)
    nt = ep.alloc_notify(R, E)
    for v in list(lay.values()) + list(nt.values()):
        poison_(v)
    ws = ws if ws is not None else ep.alloc_workspace(R, T_r, k, E, 8)
    st = status_word()
    ep.ep_layout_notify(idx_dev, E, A, nwt, lay, nt, ws, host_rows, 10000, st)
    torch.cuda.synchronize()
    return lay, nt, st, ws


def _check(idx, E, A, nwt, lay, nt, st):
    R = idx.shape[0]
    ref = oracle.layout(idx, R, E)
    nref = oracle.notify(ref["num_tokens_per_rank"], ref["num_tokens_per_expert"], R, E, A, nwt)
    for key in LAYOUT_KEYS:
        assert np.array_equal(np_(lay[key]), ref[key]), key
    for key in NOTIFY_KEYS:
        assert np.array_equal(np_(nt[key]), nref[key]), key
    assert ep.ep_read_status(st) == (ref["rc"] if ref["rc"] != oracle.OK else nref["rc"])
    return nref


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_fused_layout_notify_full_size(name):
    w = synth.WORKLOADS[name]
    idx, _ = synth.routing(w)
    idx_dev = torch.from_numpy(idx).cuda()
    for A in (1, 128):
        lay, nt, st, _ = _fused(idx_dev, w.E, A, w.num_worst_tokens)
        _check(idx, w.E, A, w.num_worst_tokens, lay, nt, st)
    # identical to the two separate calls
    lay2 = gpu_layout(idx_dev, w.E)
    nt2 = gpu_notify(lay2, w.E, 128, w.num_worst_tokens)
    torch.cuda.synchronize()
    for key in LAYOUT_KEYS:
        assert torch.equal(lay2[key], lay[key]), key
    for key in NOTIFY_KEYS:
        assert torch.equal(nt2[key], nt[key]), key


@pytest.mark.parametrize("R,T_r,k,E,A", [
    (4, 0, 2, 16, 1),       # no tokens
    (3, 1, 1, 3, 4),        # one token
    (2, 257, 8, 64, 128),   # ragged chunk tail
    (1, 5000, 16, 32, 1),   # one rank, k = 16
    (64, 40, 4, 256, 8),    # many ranks
    (2, 3000, 8, 1024, 1),  # largest expert count
])
def test_fused_layout_notify_edge_shapes(R, T_r, k, E, A):
    rng = np.random.default_rng(R * 1000 + T_r + 7)
    idx = rng.integers(-1, E, size=(R, T_r, k)).astype(np.int64)
    lay, nt, st, _ = _fused(torch.from_numpy(idx).cuda(), E, A, -1)
    _check(idx, E, A, -1, lay, nt, st)


def test_fused_host_handshake_and_capacity():
    w = synth.scaled(synth.WORKLOADS["prefill"], T_r=300)
    idx, _ = synth.routing(w, seed=3)
    idx_dev = torch.from_numpy(idx).cuda()
    host_rows = torch.full((w.R,), -7, dtype=torch.int64).pin_memory()
    lay, nt, st, _ = _fused(idx_dev, w.E, 4, -1, host_rows=host_rows)
    nref = _check(idx, w.E, 4, -1, lay, nt, st)
    assert np.array_equal(host_rows.numpy(), nref["psum"][:, -1])
    # a fixed shape smaller than what a rank receives: EP_ERR_CAPACITY
    lay, nt, st, _ = _fused(idx_dev, w.E, 1, 10)
    assert ep.ep_read_status(st) == ep.EP_ERR_CAPACITY


def test_fused_repeated_calls_on_one_workspace():
    w = synth.scaled(synth.WORKLOADS["skewed"], T_r=64)
    ws = ep.alloc_workspace(w.R, w.T_r, w.k, w.E, 8)
    for seed in range(4):
        idx, _ = synth.routing(w, seed=seed)
        lay, nt, st, _ = _fused(torch.from_numpy(idx).cuda(), w.E, 1, w.num_worst_tokens, ws=ws)
        _check(idx, w.E, 1, w.num_worst_tokens, lay, nt, st)
