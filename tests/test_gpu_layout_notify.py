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
    if st is not None:
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
    (64, 40, 4, 256, 8),    # many ranks (64: the largest bit-mask case), counts staged
    (2, 3000, 8, 1024, 1),  # largest expert count
    (3, 700, 3, 6, 4),      # odd E + R
    (33, 100, 5, 66, 1),    # one chunk per rank, R not a power of two
    (100, 30, 4, 200, 1),   # R > 64 (per-rank loop for is_token_in_rank), counts walked
    (128, 20, 3, 256, 16),  # counts too large to stage: the last CTA walks them in memory
    (8, 2500, 8, 256, 1),   # several chunks per rank (look-back), counts staged
    (4, 40000, 2, 128, 4),  # beyond one wave of 2048-id chunks: 8192-id chunks, ragged
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


def _single_call(w, x_dev, idx_dev, fp8_mode, A, ws=None, status=None):
    cap = w.cap_rows()
    lay = ep.alloc_layout(w.R, w.T_r, w.k, w.E)
    nt = ep.alloc_notify(w.R, w.E)
    d = ep.alloc_dispatch(w.R, w.T_r, w.H, w.k, fp8_mode, cap)
    for v in list(lay.values()) + list(nt.values()) + list(d.values()):
        poison_(v)
    ws = ws if ws is not None else ep.alloc_workspace(w.R, w.T_r, w.k, w.E, w.H)
    st = status if status is not None else status_word()
    ep.ep_layout_notify_dispatch(x_dev, idx_dev, w.E, fp8_mode, A, w.num_worst_tokens, cap, lay,
                                 nt, d, ws, st)
    torch.cuda.synchronize()
    return lay, nt, d, st, cap


@pytest.mark.parametrize("fp8_mode,A", [(0, 1), (1, 1), (2, 128)])
def test_single_call_fixed_shape_matches_the_separate_calls(fp8_mode, A):
    """ep_layout_notify_dispatch (layout + notify, then the dispatch as its
    programmatic dependent) gives exactly the separate calls' outputs."""
    from ep_harness import gpu_dispatch, inputs
    w = synth.scaled(synth.WORKLOADS["skewed"], T_r=96, H=1024, fp8_mode=fp8_mode,
                     num_worst_tokens=32 * 96)
    x_dev, _, idx_dev, idx, _, _ = inputs(w, seed=5)
    lay, nt, d, st, cap = _single_call(w, x_dev, idx_dev, fp8_mode, A)
    assert ep.ep_read_status(st) == ep.EP_OK
    lay2 = gpu_layout(idx_dev, w.E)
    nt2 = gpu_notify(lay2, w.E, A, w.num_worst_tokens)
    d2 = gpu_dispatch(x_dev, idx_dev, lay2, nt2, w.E, fp8_mode, cap)
    torch.cuda.synchronize()
    for key in LAYOUT_KEYS:
        assert torch.equal(lay2[key], lay[key]), key
    for key in NOTIFY_KEYS:
        assert torch.equal(nt2[key], nt[key]), key
    assert torch.equal(d2["combine_idx"], d["combine_idx"])
    assert torch.equal(d2["recv_src_idx"], d["recv_src_idx"])
    rows = torch.nonzero(d["recv_src_idx"].reshape(-1) >= 0).squeeze(1)
    rx, rx2 = d["recv_x"].reshape(w.R * cap, -1), d2["recv_x"].reshape(w.R * cap, -1)
    assert torch.equal(rx[rows].view(torch.uint8), rx2[rows].view(torch.uint8))
    if fp8_mode:
        sc = d["recv_scales"].permute(0, 2, 1).reshape(w.R * cap, -1)
        sc2 = d2["recv_scales"].permute(0, 2, 1).reshape(w.R * cap, -1)
        assert torch.equal(sc[rows], sc2[rows])
    # and the oracle
    from test_gpu_dispatch import _compare_full
    _, x_host, _, _, _, _ = inputs(w, seed=5)
    _compare_full(w, x_host, idx, d, cap, A)


def test_single_call_full_size_skewed_and_repeated():
    from ep_harness import inputs
    from test_gpu_dispatch import _compare_full
    w = synth.WORKLOADS["skewed"]
    ws = ep.alloc_workspace(w.R, w.T_r, w.k, w.E, w.H)
    for seed in (0, 1):
        x_dev, x_host, idx_dev, idx, _, _ = inputs(w, seed=seed)
        lay, nt, d, st, cap = _single_call(w, x_dev, idx_dev, w.fp8_mode, 1, ws=ws)
        assert ep.ep_read_status(st) == ep.EP_OK
        _compare_full(w, x_host, idx, d, cap, 1)


def test_single_call_refuses_the_host_handshake_mode():
    w = synth.scaled(synth.WORKLOADS["prefill"], T_r=8)
    x = torch.zeros((w.R, w.T_r, w.H), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((w.R, w.T_r, w.k), dtype=torch.int64, device="cuda")
    lay = ep.alloc_layout(w.R, w.T_r, w.k, w.E)
    nt = ep.alloc_notify(w.R, w.E)
    d = ep.alloc_dispatch(w.R, w.T_r, w.H, w.k, 0, 64)
    ws = ep.alloc_workspace(w.R, w.T_r, w.k, w.E, w.H)
    with pytest.raises(ep.EPError):
        ep.ep_layout_notify_dispatch(x, idx, w.E, 0, 1, -1, 64, lay, nt, d, ws)


def test_single_call_replays_as_a_cuda_graph():
    from ep_harness import inputs
    w = synth.scaled(synth.WORKLOADS["skewed"], T_r=24, H=512, num_worst_tokens=32 * 24)
    cap = w.cap_rows()
    x_dev, _, idx_dev, _, _, _ = inputs(w)
    lay = ep.alloc_layout(w.R, w.T_r, w.k, w.E)
    nt = ep.alloc_notify(w.R, w.E)
    d = ep.alloc_dispatch(w.R, w.T_r, w.H, w.k, w.fp8_mode, cap)
    for v in d.values():
        poison_(v)   # rows no replay fills keep it
    ws = ep.alloc_workspace(w.R, w.T_r, w.k, w.E, w.H)
    st = status_word()

    def step():
        ep.ep_layout_notify_dispatch(x_dev, idx_dev, w.E, w.fp8_mode, 1, w.num_worst_tokens, cap,
                                     lay, nt, d, ws, st)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    from ep_harness import oracle_normal
    for seed in (7, 8):
        _, x_host, _, idx, _, _ = inputs(w, seed=seed)
        x_dev.copy_(torch.from_numpy(x_host.view(np.int16)).cuda().view(torch.bfloat16))
        idx_dev.copy_(torch.from_numpy(idx).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert ep.ep_read_status(st) == ep.EP_OK
        # rows an earlier replay filled may be unused now: compare the valid ones
        _, _, ref, _ = oracle_normal(x_host, idx, w.E, 1, w.fp8_mode, cap_rows=cap,
                                     num_worst_tokens=w.num_worst_tokens)
        assert np.array_equal(np_(d["combine_idx"]), ref["combine_idx"])
        assert np.array_equal(np_(d["recv_src_idx"]), ref["recv_src_idx"])
        rows = np.nonzero(ref["recv_src_idx"].reshape(-1) >= 0)[0]
        got_x = np_(d["recv_x"]).reshape(w.R * cap, -1)
        assert np.array_equal(got_x[rows], ref["recv_x"].reshape(w.R * cap, -1)[rows])
        r_idx, row_idx = np.divmod(rows, cap)
        gs = np_(d["recv_scales"])
        assert np.array_equal(gs[r_idx, :, row_idx], ref["recv_scales"][r_idx, :, row_idx])


@pytest.mark.parametrize("T_r", [0, 1])
def test_single_call_edge_shapes(T_r):
    """No tokens (every receive row is padding) and one token per rank."""
    from ep_harness import inputs
    w = synth.Workload("edge", R=4, T_r=T_r, H=256, E=16, k=4, routing="uniform", mode="normal",
                       fp8_mode=2, num_worst_tokens=4 * max(T_r, 1))
    x_dev, x_host, idx_dev, idx, _, _ = inputs(w, seed=1)
    lay, nt, d, st, cap = _single_call(w, x_dev, idx_dev, 2, 1)
    assert ep.ep_read_status(st) == ep.EP_OK
    _check(idx, w.E, 1, w.num_worst_tokens, lay, nt, None)   # tables vs the oracle
    from ep_harness import oracle_normal
    _, _, ref, _ = oracle_normal(x_host, idx, w.E, 1, 2, cap_rows=cap,
                                 num_worst_tokens=w.num_worst_tokens)
    assert np.array_equal(np_(d["recv_src_idx"]), ref["recv_src_idx"])
    assert np.array_equal(np_(d["combine_idx"]), ref["combine_idx"])


def test_single_call_reports_invalid_ids():
    from ep_harness import inputs
    w = synth.scaled(synth.WORKLOADS["skewed"], T_r=8, H=512, num_worst_tokens=32 * 8)
    x_dev, _, idx_dev, _, _, _ = inputs(w)
    idx_dev[0, 0, 0] = w.E + 5
    lay, nt, d, st, cap = _single_call(w, x_dev, idx_dev, w.fp8_mode, 1)
    assert ep.ep_read_status(st) == ep.EP_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", ["cap_rows", "scale_alignment"])
def test_single_call_validates_everything_before_launching(bad):
    """A bad dispatch argument (a negative capacity; fp32 scales not 4-byte
    aligned) is refused before the layout kernel runs: the layout outputs
    keep their poison."""
    w = synth.scaled(synth.WORKLOADS["skewed"], T_r=8, H=512, num_worst_tokens=32 * 8)
    x = torch.zeros((w.R, w.T_r, w.H), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((w.R, w.T_r, w.k), dtype=torch.int64, device="cuda")
    lay = ep.alloc_layout(w.R, w.T_r, w.k, w.E)
    nt = ep.alloc_notify(w.R, w.E)
    d = ep.alloc_dispatch(w.R, w.T_r, w.H, w.k, w.fp8_mode, 16)
    for v in lay.values():
        poison_(v)
    ws = ep.alloc_workspace(w.R, w.T_r, w.k, w.E, w.H)
    import ctypes
    L = ep.load()
    P = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off) if t is not None else None
    cap = -1 if bad == "cap_rows" else 16
    off = 2 if bad == "scale_alignment" else 0
    assert w.fp8_mode == 1   # fp32 scales
    rc = L.ep_layout_notify_dispatch(
        P(x), P(idx), w.R, w.T_r, w.H, w.E, w.k, w.fp8_mode, 1, w.num_worst_tokens, cap,
        P(lay["num_tokens_per_rank"]), P(lay["num_tokens_per_expert"]), P(lay["is_token_in_rank"]),
        P(lay["slot_rank"]), P(nt["rank_prefix_matrix"]), P(nt["expert_prefix"]),
        P(nt["num_recv_tokens_per_expert"]), P(nt["psum"]), P(d["recv_x"]), P(d["recv_scales"], off),
        P(d["recv_src_idx"]), P(d["combine_idx"]), P(ws), ws.numel(), None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == ep.EP_ERR_INVALID_ARG
    assert np.all(np_(lay["num_tokens_per_rank"]).view(np.uint8) == 0x5A)
