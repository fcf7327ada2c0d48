"""GPU parity: normal-mode dispatch (contiguous per-expert layout, bf16 or
fused FP8) vs the oracle -- bit-exact rows, scales and indices."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_gb300 import ep, synth
from ep_harness import (POISON, gpu_dispatch, gpu_layout, gpu_notify, inputs, np_, oracle_normal,
                        status_word, to_dev_bf16)

pytestmark = pytest.mark.gpu


def _run_both(w, A=1, cap_rows=None, x_on_device=False):
    x_dev, x_host, idx_dev, idx, _, _ = inputs(w, x_on_device=x_on_device)
    lay = gpu_layout(idx_dev, w.E)
    nt = gpu_notify(lay, w.E, A, w.num_worst_tokens)
    ref_lay = oracle.layout(idx, w.R, w.E)
    ref_nt = oracle.notify(ref_lay["num_tokens_per_rank"], ref_lay["num_tokens_per_expert"], w.R,
                           w.E, A, w.num_worst_tokens)
    if cap_rows is None:
        cap_rows = (w.cap_rows() if w.num_worst_tokens >= 0
                    else max(1, int(ref_nt["psum"][:, -1].max())))
    d = gpu_dispatch(x_dev, idx_dev, lay, nt, w.E, w.fp8_mode, cap_rows)
    return x_dev, x_host, idx, lay, nt, d, cap_rows


def _compare_full(w, x_host, idx, d, cap_rows, A):
    _, _, ref, _ = oracle_normal(x_host, idx, w.E, A, w.fp8_mode, cap_rows=cap_rows,
                                 num_worst_tokens=w.num_worst_tokens)
    assert ref["rc"] == oracle.OK
    assert np.array_equal(np_(d["combine_idx"]), ref["combine_idx"])
    src = np_(d["recv_src_idx"])
    assert np.array_equal(src, ref["recv_src_idx"])
    rows = np.nonzero(src.reshape(-1) >= 0)[0]
    got = np_(d["recv_x"]).reshape(w.R * cap_rows, -1)
    assert np.array_equal(got[rows], ref["recv_x"].reshape(w.R * cap_rows, -1)[rows])
    # rows nobody fills stay untouched (poison)
    unused = np.nonzero(src.reshape(-1) < 0)[0]
    if unused.size:
        assert np.all(got[unused[:4096]].view(np.uint8) == POISON)
    if w.fp8_mode:
        gs = np_(d["recv_scales"])                         # [R, H/128, cap]
        rs = ref["recv_scales"]
        r_idx, row_idx = np.divmod(rows, cap_rows)
        assert np.array_equal(gs[r_idx, :, row_idx], rs[r_idx, :, row_idx])


@pytest.mark.parametrize("fp8_mode", [0, 1, 2])
@pytest.mark.parametrize("A", [1, 128])
def test_dispatch_tiny(fp8_mode, A):
    w = synth.scaled(synth.WORKLOADS["tiny"], fp8_mode=fp8_mode)
    x_dev, x_host, idx, lay, nt, d, cap = _run_both(w, A)
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    _compare_full(w, x_host, idx, d, cap, A)


@pytest.mark.parametrize("name,T_r,fp8_mode", [
    ("prefill", 96, 0), ("prefill", 96, 2), ("skewed", 40, 1), ("large", 80, 2), ("decode", 16, 1),
])
def test_dispatch_scaled_full_compare(name, T_r, fp8_mode):
    base = synth.WORKLOADS[name]
    nwt = base.R * T_r if base.num_worst_tokens >= 0 else -1
    w = synth.scaled(base, T_r=T_r, fp8_mode=fp8_mode, num_worst_tokens=nwt)
    x_dev, x_host, idx, lay, nt, d, cap = _run_both(w, 1)
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    _compare_full(w, x_host, idx, d, cap, 1)


@pytest.mark.parametrize("H", [8, 136, 1032, 1024 + 512 + 8])
def test_dispatch_bf16_ragged_hidden(H):
    w = synth.scaled(synth.WORKLOADS["tiny"], H=H, T_r=33)
    x_dev, x_host, idx, lay, nt, d, cap = _run_both(w, 4)
    _compare_full(w, x_host, idx, d, cap, 4)


@pytest.mark.parametrize("H", [128, 384, 1152])
@pytest.mark.parametrize("fp8_mode", [1, 2])
def test_dispatch_fp8_small_hidden_and_zero_rows(H, fp8_mode):
    w = synth.scaled(synth.WORKLOADS["tiny"], H=H, T_r=20, fp8_mode=fp8_mode)
    x_dev, x_host, idx_dev, idx, _, _ = inputs(w)
    x_host = x_host.copy()
    x_host[0, 3] = 0                                     # all-zero row: amax floor
    x_host[1, 5, :128] = 0x8000                          # -0.0 block
    x_host[2, 7, ::2] = synth.to_bf16_bits(np.float32([3e38]))[0]   # near bf16 max
    x_host[3, 9] = synth.to_bf16_bits(np.float32([1e-30]))[0]       # tiny values
    x_dev = to_dev_bf16(x_host)
    lay = gpu_layout(idx_dev, w.E)
    nt = gpu_notify(lay, w.E, 1)
    cap = int(np_(nt["psum"])[:, -1].max())
    d = gpu_dispatch(x_dev, idx_dev, lay, nt, w.E, fp8_mode, cap)
    _compare_full(w, x_host, idx, d, cap, 1)


def test_dispatch_masked_slots_and_capacity_overflow():
    w = synth.WORKLOADS["tiny"]
    x_dev, x_host, idx_dev, idx, _, _ = inputs(w)
    idx = idx.copy()
    idx[0, :4, 1] = -1
    idx[2, 5, :] = -1
    idx_dev = torch.from_numpy(idx).cuda()
    lay = gpu_layout(idx_dev, w.E)
    nt = gpu_notify(lay, w.E, 1)
    full = int(np_(nt["psum"])[:, -1].max())
    d = gpu_dispatch(x_dev, idx_dev, lay, nt, w.E, 0, full)
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    _compare_full(w, x_host, idx, d, full, 1)
    small = full - 3
    d = gpu_dispatch(x_dev, idx_dev, lay, nt, w.E, 0, small)
    assert ep.ep_read_status(d["status"]) == ep.EP_ERR_CAPACITY
    _, _, ref, _ = oracle_normal(x_host, idx, w.E, 1, 0, cap_rows=small)
    assert ref["rc"] == oracle.ERR_CAPACITY
    assert np.array_equal(np_(d["combine_idx"]), ref["combine_idx"])
    assert np.array_equal(np_(d["recv_src_idx"]), ref["recv_src_idx"])


@pytest.mark.slow
@pytest.mark.parametrize("name", ["prefill", "skewed", "large"])
def test_dispatch_full_size_sampled(name):
    """Full-size workloads in the bench's launch configuration: all index
    outputs compared whole, data rows of a random sample of tokens compared
    against the oracle's per-row definition."""
    w = synth.WORKLOADS[name]
    x_dev, x_host, idx, lay, nt, d, cap = _run_both(w, 1, x_on_device=True)
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    ref_lay = oracle.layout(idx, w.R, w.E)
    ref_nt = oracle.notify(ref_lay["num_tokens_per_rank"], ref_lay["num_tokens_per_expert"], w.R,
                           w.E, 1, w.num_worst_tokens)
    # indices: the oracle's dispatch with zero-width rows (no row data to move)
    x0 = np.zeros((w.R, w.T_r, 0), np.uint16)
    ref = oracle.dispatch(x0, idx, ref_lay["slot_rank"], ref_nt["expert_prefix"], ref_nt["psum"],
                          w.E, 0, cap)
    assert ref["rc"] == oracle.OK
    ref_cidx = ref["combine_idx"]
    assert np.array_equal(np_(d["combine_idx"]), ref_cidx)
    assert np.array_equal(np_(d["recv_src_idx"]), ref["recv_src_idx"])
    # sampled rows
    rng = np.random.default_rng(11)
    toks = rng.choice(w.T, size=min(192, w.T), replace=False)
    recv = d["recv_x"].view(w.R * cap, -1)
    for g in toks:
        i, t = divmod(int(g), w.T_r)
        for j in range(w.k):
            f = int(ref_cidx[i, t, j])
            got = np_(recv[f])
            if w.fp8_mode == 0:
                assert np.array_equal(got, x_host[i, t])
            else:
                q, s = oracle.quantize_row(x_host[i, t], w.fp8_mode)
                assert np.array_equal(got, q)
                rr, rw = divmod(f, cap)
                assert np.array_equal(np_(d["recv_scales"][rr, :, rw]), s)


@pytest.mark.parametrize("fp8_mode", [0, 1])
def test_fixed_shape_normal_path_replays_as_a_cuda_graph(fp8_mode):
    """With num_worst_tokens the normal path needs no host round trip (the
    receive shape is fixed), so layout -> notify -> dispatch -> combine can be
    captured once into a CUDA graph; every replay with new routing and
    activations copied into the captured buffers must match the oracle."""
    w = synth.scaled(synth.WORKLOADS["skewed"], T_r=24, H=512, fp8_mode=fp8_mode,
                     num_worst_tokens=32 * 24)
    cap = w.cap_rows()
    x_dev, _, idx_dev, _, wts_dev, _ = inputs(w)
    ws = ep.alloc_workspace(w.R, w.T_r, w.k, w.E, w.H)
    status = status_word()
    lay = ep.alloc_layout(w.R, w.T_r, w.k, w.E)
    nt = ep.alloc_notify(w.R, w.E)
    d = ep.alloc_dispatch(w.R, w.T_r, w.H, w.k, fp8_mode, cap)
    y = synth.expert_outputs_torch(w.R * cap, w.H, "cuda").view(w.R, cap, w.H)
    out = torch.empty_like(x_dev)

    def step():
        ep.ep_get_dispatch_layout(idx_dev, w.E, lay["num_tokens_per_rank"],
                                  lay["num_tokens_per_expert"], lay["is_token_in_rank"],
                                  lay["slot_rank"], ws, status)
        ep.ep_notify_dispatch(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"], 1,
                              w.num_worst_tokens, nt["rank_prefix_matrix"], nt["expert_prefix"],
                              nt["num_recv_tokens_per_expert"], nt["psum"], None, 10000, status)
        ep.ep_dispatch(x_dev, idx_dev, lay["slot_rank"], nt["expert_prefix"], nt["psum"], w.E,
                       fp8_mode, cap, d["recv_x"], d["recv_scales"], d["recv_src_idx"],
                       d["combine_idx"], ws, status)
        ep.ep_combine(y, wts_dev, d["combine_idx"], cap, out, status)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    y_rows = np_(y).reshape(-1, w.H)
    for seed in (7, 8):
        _, x_host, _, idx, _, wts = inputs(w, seed=seed)
        x_dev.copy_(torch.from_numpy(x_host.view(np.int16)).cuda().view(torch.bfloat16))
        idx_dev.copy_(torch.from_numpy(idx).cuda())
        wts_dev.copy_(torch.from_numpy(wts).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert ep.ep_read_status(status) == ep.EP_OK
        _, _, ref, _ = oracle_normal(x_host, idx, w.E, 1, fp8_mode, cap_rows=cap,
                                     num_worst_tokens=w.num_worst_tokens)
        assert np.array_equal(np_(d["combine_idx"]), ref["combine_idx"])
        assert np.array_equal(np_(d["recv_src_idx"]), ref["recv_src_idx"])
        rows = np.nonzero(ref["recv_src_idx"].reshape(-1) >= 0)[0]
        got_x = np_(d["recv_x"]).reshape(w.R * cap, -1)
        assert np.array_equal(got_x[rows], ref["recv_x"].reshape(w.R * cap, -1)[rows])
        want = oracle.combine(y_rows, wts, ref["combine_idx"], w.H)["out"]
        assert np.array_equal(np_(out).reshape(want.shape), want)


@pytest.mark.parametrize("fp8_mode", [0, 2])
def test_handle_reuse_across_dispatches(fp8_mode):
    """The layout and notify outputs are the dispatch handle (§2.3, §4.3):
    computed once for a routing, they serve any number of dispatches of new
    activations with that routing, with no layout or notify in between
    (each dispatch bit-exact vs the oracle)."""
    w = synth.scaled(synth.WORKLOADS["prefill"], T_r=48, fp8_mode=fp8_mode)
    _, _, idx_dev, idx, _, _ = inputs(w, seed=2)
    lay = gpu_layout(idx_dev, w.E)
    nt = gpu_notify(lay, w.E, 1, -1)
    torch.cuda.synchronize()
    cap = max(1, int(np_(nt["psum"])[:, -1].max()))
    ws = ep.alloc_workspace(w.R, w.T_r, w.k, w.E, w.H)
    for seed in (3, 4, 5):
        x_host = synth.activations(w, seed=seed)
        x_dev = to_dev_bf16(x_host)
        d = gpu_dispatch(x_dev, idx_dev, lay, nt, w.E, fp8_mode, cap, ws=ws)
        torch.cuda.synchronize()
        assert ep.ep_read_status(d["status"]) == ep.EP_OK
        _compare_full(w, x_host, idx, d, cap, 1)


@pytest.mark.parametrize("fp8_mode", [1, 2])
def test_workspace_reused_across_batch_sizes(fp8_mode):
    """One workspace, sized for the largest batch, serves FP8 dispatches of
    several batch sizes in turn (as a serving loop with a varying batch
    does).  The staged scales and the layout's look-back words sit at
    offsets that move with the batch size, so each call finds bytes another
    size left behind; every call must still give the oracle's rows and
    column-major scales."""
    base = synth.scaled(synth.WORKLOADS["skewed"], T_r=64, fp8_mode=fp8_mode)
    ws = ep.alloc_workspace(base.R, 64, base.k, base.E, base.H)
    for i, T_r in enumerate((64, 24, 64, 8, 40, 64)):
        w = synth.scaled(synth.WORKLOADS["skewed"], T_r=T_r, fp8_mode=fp8_mode)
        x_dev, x_host, idx_dev, idx, _, _ = inputs(w, seed=10 + i)
        lay = gpu_layout(idx_dev, w.E)
        nt = gpu_notify(lay, w.E, 1, -1)
        torch.cuda.synchronize()
        cap = max(1, int(np_(nt["psum"])[:, -1].max()))
        d = gpu_dispatch(x_dev, idx_dev, lay, nt, w.E, fp8_mode, cap, ws=ws)
        torch.cuda.synchronize()
        assert ep.ep_read_status(d["status"]) == ep.EP_OK, T_r
        _compare_full(w, x_host, idx, d, cap, 1)


@pytest.mark.parametrize("fp8_mode", [1, 2])
@pytest.mark.parametrize("pad,A", [(16, 1), (16, 4), (2, 1), (1, 1), (0, 128)])
def test_scale_columns_quad_and_single_row_paths(pad, A, fp8_mode):
    """With ue8m0 scales the column pass writes 4 rows per thread (one 4-byte
    store per block) when cap_rows is a multiple of 4, row by row otherwise;
    segment edges inside a quad store byte by byte.  fp32 scales always go
    row by row.  Every path must give the oracle's scales."""
    w = synth.scaled(synth.WORKLOADS["large"], T_r=90, fp8_mode=fp8_mode)
    x_dev, x_host, idx_dev, idx, _, _ = inputs(w, seed=3)
    lay = gpu_layout(idx_dev, w.E)
    nt = gpu_notify(lay, w.E, A, -1)
    _, _, _, cap = oracle_normal(x_host, idx, w.E, A, fp8_mode)
    cap = (cap + 15) // 16 * 16 + pad if pad == 16 else cap + pad
    d = gpu_dispatch(x_dev, idx_dev, lay, nt, w.E, fp8_mode, cap)
    torch.cuda.synchronize()
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    _compare_full(w, x_host, idx, d, cap, A)


def test_fp32_scale_buffer_must_be_word_aligned():
    """fp32 scales are stored as 4-byte words: both dispatches refuse a
    scale buffer that is not 4-byte aligned before launching anything."""
    import ctypes
    w = synth.scaled(synth.WORKLOADS["tiny"], fp8_mode=1)
    x_dev, _, idx_dev, _, _, _ = inputs(w, seed=5)
    lay = gpu_layout(idx_dev, w.E)
    nt = gpu_notify(lay, w.E, 1, -1)
    R, T_r, H = x_dev.shape
    k = idx_dev.shape[2]
    cap = 64
    out = ep.alloc_dispatch(R, T_r, H, k, 1, cap)
    ws = ep.alloc_workspace(R, T_r, k, w.E, H)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    P = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    L = ep.load()
    rc = L.ep_dispatch(P(x_dev), P(idx_dev), P(lay["slot_rank"]), P(nt["expert_prefix"]),
                       P(nt["psum"]), R, T_r, H, w.E, k, 1, cap, P(out["recv_x"]),
                       P(out["recv_scales"], 2), P(out["recv_src_idx"]), P(out["combine_idx"]),
                       P(ws), ws.numel(), P(status), stream)
    assert rc == ep.EP_ERR_INVALID_ARG
    ll = ep.alloc_ll(R, T_r, H, w.E, k, w.max_tokens_per_rank, 1)
    rc = L.ep_ll_dispatch(P(x_dev), P(idx_dev), R, T_r, H, w.E, k, w.max_tokens_per_rank, 1,
                          P(ll["packed_recv_x"]), P(ll["packed_recv_scales"], 2),
                          P(ll["packed_recv_src_info"]), P(ll["layout_range"]),
                          P(ll["recv_count"]), P(ll["combine_idx"]), P(ws), ws.numel(),
                          P(status), stream)
    assert rc == ep.EP_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(status.item()) == ep.EP_OK


def _e4m3_equal(got, want):
    """E4M3 codes equal, a NaN code (S.1111.111) matching a NaN of either sign."""
    got, want = got.view(np.uint8), want.view(np.uint8)
    nan = (want & 0x7F) == 0x7F
    return np.array_equal(got[~nan], want[~nan]) and np.all((got[nan] & 0x7F) == 0x7F)


def _plant_non_finite(x_host):
    x = x_host.copy()
    x[0, 0, 5] = 0x7F80           # +inf in a block of finite values
    x[1, 3, 130] = 0xFF80         # -inf
    x[0, 1, :128] = 0x7F80        # a whole block of +inf
    x[2, 7, 300] = 0x7FC0         # NaN among finite values
    x[3, 15, 511] = 0xFFC1        # NaN with the sign bit set
    x[3, 14, 384:512] = 0xFFC0    # a whole block of NaN (amax stays at the floor)
    return x


@pytest.mark.parametrize("fp8_mode", [1, 2])
def test_dispatch_fp8_non_finite_inputs(fp8_mode):
    """Blocks holding infinities or NaN: amax ignores NaN and saturates an
    infinity to the largest finite float, so scales stay finite and match
    the oracle bit for bit; every NaN input gives an E4M3 NaN code (its sign
    is not specified)."""
    w = synth.scaled(synth.WORKLOADS["tiny"], fp8_mode=fp8_mode, H=512)
    _, x_host, idx_dev, idx, _, _ = inputs(w)
    x_host = _plant_non_finite(x_host)
    x_dev = to_dev_bf16(x_host)
    lay = gpu_layout(idx_dev, w.E)
    nt = gpu_notify(lay, w.E, 1)
    _, _, ref, cap = oracle_normal(x_host, idx, w.E, 1, fp8_mode)
    d = gpu_dispatch(x_dev, idx_dev, lay, nt, w.E, fp8_mode, cap)
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    src = np_(d["recv_src_idx"])
    assert np.array_equal(src, ref["recv_src_idx"])
    rows = np.nonzero(src.reshape(-1) >= 0)[0]
    got = np_(d["recv_x"]).reshape(w.R * cap, -1)[rows]
    want = ref["recv_x"].reshape(w.R * cap, -1)[rows]
    assert _e4m3_equal(got, want)
    r_idx, row_idx = np.divmod(rows, cap)
    gs, rs = np_(d["recv_scales"]), ref["recv_scales"]
    assert np.array_equal(gs[r_idx, :, row_idx], rs[r_idx, :, row_idx])
    # the block of +inf: +448 codes
    assert np.all(want.view(np.uint8).reshape(len(rows), -1)[src.reshape(-1)[rows] == 1, :128] == 0x7E)


@pytest.mark.parametrize("fp8_mode", [1, 2])
def test_ll_dispatch_fp8_non_finite_inputs(fp8_mode):
    """The same non-finite inputs through the single-launch low-latency path."""
    from ep_harness import gpu_ll_dispatch
    w = synth.scaled(synth.WORKLOADS["tiny"], fp8_mode=fp8_mode, H=512)
    _, x_host, idx_dev, idx, _, _ = inputs(w)
    x_host = _plant_non_finite(x_host)
    x_dev = to_dev_bf16(x_host)
    d = gpu_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, fp8_mode)
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    ref = oracle.ll_dispatch(x_host, idx, w.E, w.max_tokens_per_rank, fp8_mode)
    assert np.array_equal(np_(d["recv_count"]), ref["recv_count"])
    S = w.R * w.max_tokens_per_rank
    cnt = ref["recv_count"].reshape(-1)
    px = np_(d["packed_recv_x"]).reshape(w.E, S, -1)
    rpx = ref["packed_recv_x"].reshape(w.E, S, -1)
    ps = np_(d["packed_recv_scales"]).reshape(w.E, w.H // 128, S)
    rps = ref["packed_recv_scales"].reshape(w.E, w.H // 128, S)
    for e in range(w.E):
        assert _e4m3_equal(px[e, :cnt[e]], rpx[e, :cnt[e]]), e
        assert np.array_equal(ps[e, :, :cnt[e]], rps[e, :, :cnt[e]]), e
