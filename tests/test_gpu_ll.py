"""GPU parity: low-latency dispatch into the packed masked layout vs the
oracle (bit-exact rows, scales, counts, ranges, indices), the bounded
device waits of its layout pass, and ep_clean_ll_buffer."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_gb300 import ep, synth
from ep_harness import POISON, gpu_ll_dispatch, inputs, np_, status_word

pytestmark = pytest.mark.gpu


def _compare_ll(w, x_host, idx, d, max_tokens, fp8_mode):
    ref = oracle.ll_dispatch(x_host, idx, w.E, max_tokens, fp8_mode)
    assert ref["rc"] == oracle.OK
    S = w.R * max_tokens
    assert np.array_equal(np_(d["recv_count"]), ref["recv_count"])
    assert np.array_equal(np_(d["layout_range"]), ref["layout_range"])
    assert np.array_equal(np_(d["combine_idx"]), ref["combine_idx"])
    cnt = ref["recv_count"].reshape(-1)
    src = np_(d["packed_recv_src_info"]).reshape(w.E, S)
    px = np_(d["packed_recv_x"]).reshape(w.E, S, -1)
    rsrc = ref["packed_recv_src_info"].reshape(w.E, S)
    rpx = ref["packed_recv_x"].reshape(w.E, S, -1)
    for e in range(w.E):
        c = cnt[e]
        assert np.array_equal(src[e, :c], rsrc[e, :c]), e
        assert np.array_equal(px[e, :c], rpx[e, :c]), e
        if c < S:   # rows past recv_count are untouched
            assert np.all(px[e, c:c + 2].view(np.uint8) == POISON)
            assert np.all(src[e, c:c + 2].view(np.uint8) == POISON)
    if fp8_mode:
        ps = np_(d["packed_recv_scales"]).reshape(w.E, w.H // 128, S)
        rps = ref["packed_recv_scales"].reshape(w.E, w.H // 128, S)
        for e in range(w.E):
            assert np.array_equal(ps[e, :, :cnt[e]], rps[e, :, :cnt[e]]), e


@pytest.mark.parametrize("fp8_mode", [0, 1, 2])
def test_ll_tiny(fp8_mode):
    w = synth.scaled(synth.WORKLOADS["tiny"], fp8_mode=fp8_mode)
    x_dev, x_host, idx_dev, idx, _, _ = inputs(w)
    d = gpu_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, fp8_mode)
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    _compare_ll(w, x_host, idx, d, w.max_tokens_per_rank, fp8_mode)


@pytest.mark.slow
def test_ll_decode_full_size():
    """The decode workload exactly as the benchmark runs it."""
    w = synth.WORKLOADS["decode"]
    x_dev, x_host, idx_dev, idx, _, _ = inputs(w)
    d = gpu_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, w.fp8_mode)
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    _compare_ll(w, x_host, idx, d, w.max_tokens_per_rank, w.fp8_mode)
    # a second call on the same workspace gives identical results
    d2 = gpu_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, w.fp8_mode, ws=d["ws"])
    for key in ("recv_count", "layout_range", "combine_idx"):
        assert torch.equal(d2[key], d[key]), key


@pytest.mark.parametrize("R,T_r,max_tokens,k,E,H,fp8_mode", [
    (16, 100, 128, 8, 256, 1024, 2),   # T_r below the per-rank capacity
    (4, 700, 700, 4, 32, 256, 1),      # several chunks per rank (ragged)
    (8, 1, 1, 1, 8, 128, 0),           # one token per rank, one expert per rank
    (2, 0, 4, 2, 4, 128, 2),           # no tokens at all
    (32, 256, 256, 6, 128, 4096, 1),   # the skewed workload's shape
    (16, 512, 512, 8, 256, 512, 2),    # larger chunks
    (200, 3, 4, 2, 400, 256, 2),       # more ranks than chunks (one chunk per rank)
    (16, 2048, 2048, 8, 256, 128, 2),  # chunks too large: layout kernel with look-back
    (2, 10000, 10000, 8, 16, 128, 0),  # look-back path, ragged chunks
])
def test_ll_shapes(R, T_r, max_tokens, k, E, H, fp8_mode):
    w = synth.Workload("t", R=R, T_r=T_r, H=H, E=E, k=k, routing="uniform", mode="ll",
                       fp8_mode=fp8_mode, max_tokens_per_rank=max_tokens)
    x_dev, x_host, idx_dev, idx, _, _ = inputs(w)
    d = gpu_ll_dispatch(x_dev, idx_dev, E, max_tokens, fp8_mode)
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    _compare_ll(w, x_host, idx, d, max_tokens, fp8_mode)


def test_ll_masked_and_repeated_experts_capacity():
    R, T_r, k, E, H = 2, 2, 2, 4, 128
    w = synth.Workload("t", R=R, T_r=T_r, H=H, E=E, k=k, routing="uniform", mode="ll",
                       fp8_mode=0, max_tokens_per_rank=2)
    x_dev, x_host, _, _, _, _ = inputs(w)
    idx = np.zeros((R, T_r, k), np.int64)      # 8 slots to expert 0, room for 4
    idx[1, 1, 1] = -1
    d = gpu_ll_dispatch(x_dev, torch.from_numpy(idx).cuda(), E, 2, 0)
    assert ep.ep_read_status(d["status"]) == ep.EP_ERR_CAPACITY
    ref = oracle.ll_dispatch(x_host, idx, E, 2, 0)
    assert ref["rc"] == oracle.ERR_CAPACITY
    assert np.array_equal(np_(d["combine_idx"]), ref["combine_idx"])
    assert np.array_equal(np_(d["recv_count"]), ref["recv_count"])


def test_ll_rejects_tokens_above_capacity():
    w = synth.scaled(synth.WORKLOADS["tiny"], T_r=17)
    x_dev, _, idx_dev, _, _, _ = inputs(w)
    with pytest.raises(ep.EPError) as ei:
        gpu_ll_dispatch(x_dev, idx_dev, w.E, 16, 0)
    assert ei.value.code == ep.EP_ERR_INVALID_ARG


def test_ll_bounded_wait_on_a_chunk_that_never_publishes():
    """Host-made fault: the workspace's ticket counter is advanced by one,
    so the CTA for the first chunk never exists and its look-back words are
    never published.  The other CTAs' waits must give up after their bound
    (EP_ERR_TIMEOUT / EP_ERR_STATE in the status word), the kernel must
    finish, and after ep_clean_ll_buffer the same workspace works again."""
    # large enough for the layout kernel with look-back
    w = synth.scaled(synth.WORKLOADS["decode"], T_r=2048, max_tokens_per_rank=2048, H=128,
                     fp8_mode=0)
    x_dev, x_host, idx_dev, idx, _, _ = inputs(w)
    ws = ep.alloc_workspace(w.R, w.T_r, w.k, w.E, w.H)
    ws[:4].view(torch.int32)[0] = 1            # ticket counter := 1
    d = gpu_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, 0, ws=ws)
    torch.cuda.synchronize()
    code = ep.ep_read_status(d["status"])
    assert code in (ep.EP_ERR_TIMEOUT, ep.EP_ERR_STATE)
    ep.ep_clean_ll_buffer(d["recv_count"], w.R, w.E, ws)
    d = gpu_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, 0, ws=ws)
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    _compare_ll(w, x_host, idx, d, w.max_tokens_per_rank, 0)


def test_clean_ll_buffer_zeroes_counts_and_workspace():
    w = synth.WORKLOADS["tiny"]
    x_dev, _, idx_dev, _, _, _ = inputs(w)
    d = gpu_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, 0)
    assert int(d["recv_count"].sum()) == w.T * w.k
    ep.ep_clean_ll_buffer(d["recv_count"], w.R, w.E, d["ws"])
    assert int(d["recv_count"].abs().sum()) == 0
    assert int(d["ws"].sum()) == 0


def test_single_launch_path_reports_an_uncleaned_workspace():
    """Host-made fault on the single-launch path (decode-size batches): the
    workspace's grid-barrier word is left far past the CTA count, as a
    workspace that was never cleaned might hold.  The call must finish,
    report EP_ERR_STATE, and after ep_clean_ll_buffer the same workspace
    must give the oracle's results again."""
    w = synth.scaled(synth.WORKLOADS["tiny"], fp8_mode=2)
    x_dev, x_host, idx_dev, idx, _, _ = inputs(w)
    ws = ep.alloc_workspace(w.R, w.T_r, w.k, w.E, w.H)
    ws[32:36].view(torch.int32)[0] = 0x7FFFFF00      # barrier arrival word
    d = gpu_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, 2, ws=ws)
    torch.cuda.synchronize()
    assert ep.ep_read_status(d["status"]) == ep.EP_ERR_STATE
    ep.ep_clean_ll_buffer(d["recv_count"], w.R, w.E, ws)
    d = gpu_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, 2, ws=ws)
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    _compare_ll(w, x_host, idx, d, w.max_tokens_per_rank, 2)


@pytest.mark.parametrize("fp8_mode", [0, 1, 2])
def test_single_launch_path_repeated_calls_on_one_workspace(fp8_mode):
    """The single-launch path resets its grid-barrier words at the end of
    every call; five calls in a row on one workspace (different routings)
    must each match the oracle."""
    base = synth.scaled(synth.WORKLOADS["decode"], T_r=24, H=1024, fp8_mode=fp8_mode)
    ws = ep.alloc_workspace(base.R, base.T_r, base.k, base.E, base.H)
    for seed in range(5):
        x_dev, x_host, idx_dev, idx, _, _ = inputs(base, seed=seed)
        d = gpu_ll_dispatch(x_dev, idx_dev, base.E, base.max_tokens_per_rank, fp8_mode, ws=ws)
        assert ep.ep_read_status(d["status"]) == ep.EP_OK
        _compare_ll(base, x_host, idx, d, base.max_tokens_per_rank, fp8_mode)


@pytest.mark.parametrize("fp8_mode", [0, 2])
def test_low_latency_dispatch_and_combine_replay_as_a_cuda_graph(fp8_mode):
    """The low-latency path has no host round trip, so a dispatch + combine
    pair can be captured once into a CUDA graph and replayed: every replay
    with new inputs copied into the captured buffers must match the oracle
    (the single-launch kernel's barrier words are reset inside the graph, as
    between eager calls)."""
    w = synth.scaled(synth.WORKLOADS["decode"], T_r=32, H=1024, fp8_mode=fp8_mode)
    S = w.R * w.max_tokens_per_rank
    x_dev, _, idx_dev, _, wts_dev, _ = inputs(w)
    ws = ep.alloc_workspace(w.R, w.T_r, w.k, w.E, w.H)
    status = status_word()
    b = ep.alloc_ll(w.R, w.T_r, w.H, w.E, w.k, w.max_tokens_per_rank, fp8_mode)
    y = synth.expert_outputs_torch(w.E * S, w.H, "cuda").view(w.R, w.E_l, S, w.H)
    out = torch.empty_like(x_dev)

    def step():
        ep.ep_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, fp8_mode, b["packed_recv_x"],
                          b["packed_recv_scales"], b["packed_recv_src_info"], b["layout_range"],
                          b["recv_count"], b["combine_idx"], ws, status)
        ep.ep_ll_combine(y, wts_dev, b["combine_idx"], w.E, w.max_tokens_per_rank, out, status)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                      # eager warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    y_rows = np_(y).reshape(-1, w.H)
    for seed in (3, 4, 5):
        _, x_host, _, idx, _, wts = inputs(w, seed=seed)
        x_dev.copy_(torch.from_numpy(x_host.view(np.int16)).cuda().view(torch.bfloat16))
        idx_dev.copy_(torch.from_numpy(idx).cuda())
        wts_dev.copy_(torch.from_numpy(wts).cuda())
        g.replay()
        torch.cuda.synchronize()
        assert ep.ep_read_status(status) == ep.EP_OK
        ref = oracle.ll_dispatch(x_host, idx, w.E, w.max_tokens_per_rank, fp8_mode)
        assert np.array_equal(np_(b["combine_idx"]), ref["combine_idx"])
        assert np.array_equal(np_(b["recv_count"]), ref["recv_count"])
        assert np.array_equal(np_(b["layout_range"]), ref["layout_range"])
        cnt = ref["recv_count"].reshape(-1)
        px = np_(b["packed_recv_x"]).reshape(w.E, S, -1)
        rpx = ref["packed_recv_x"].reshape(w.E, S, -1)
        for e in range(w.E):
            assert np.array_equal(px[e, :cnt[e]], rpx[e, :cnt[e]]), e
        got = np_(out)
        want = oracle.combine(y_rows, wts, ref["combine_idx"], w.H)["out"]
        assert np.array_equal(got.reshape(want.shape), want)


def _hold_lib(tmp_path):
    """tests/cuda/hold_sms.cu built for this GPU (nvcc), loaded by ctypes."""
    import ctypes
    import os
    import subprocess
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "cuda", "hold_sms.cu")
    so = str(tmp_path / "libhold.so")
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                        "-Xcompiler", "-fPIC", src, "-o", so], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    lib = ctypes.CDLL(so)
    lib.hold_sms.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_longlong, ctypes.c_void_p]
    lib.hold_sms.restype = ctypes.c_int
    return lib


@pytest.mark.slow
@pytest.mark.parametrize("held", ["half", "all"])
def test_ll_dispatch_while_another_stream_holds_sms(tmp_path, held):
    """The single-launch decode kernel waits at a grid barrier, so its CTAs
    must all be resident together.  Here another stream holds half, or all,
    of the SMs for 20 ms (each holding CTA takes 120 KB of shared memory, so
    a dispatch CTA cannot share its SM) while ep_ll_dispatch is issued: the
    call must still return the oracle's results with status EP_OK (the
    kernel starts once its whole grid fits, or the call takes the
    multi-kernel path), not a timed-out barrier."""
    lib = _hold_lib(tmp_path)
    w = synth.WORKLOADS["decode"]
    x_dev, x_host, idx_dev, idx, _, _ = inputs(w)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ws = ep.alloc_workspace(w.R, w.T_r, w.k, w.E, w.H)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    ctas = sms // 2 if held == "half" else sms
    assert lib.hold_sms(ctas, 120 * 1024, 20_000_000, ctypes_stream(side)) == 0
    d = gpu_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, w.fp8_mode, ws=ws)
    torch.cuda.synchronize()
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    _compare_ll(w, x_host, idx, d, w.max_tokens_per_rank, w.fp8_mode)


def ctypes_stream(s):
    import ctypes
    return ctypes.c_void_p(s.cuda_stream)
