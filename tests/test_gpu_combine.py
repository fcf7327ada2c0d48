"""GPU parity: top-k weighted combine (normal and low-latency layouts) vs
the oracle.  Tolerance: at most 1 bf16 ulp of the oracle's fp32-accumulated
result per element (the kernel runs the same fp32 fma chain in the same slot
order, so the observed difference is expected to be 0)."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_gb300 import ep, synth
from ep_harness import (bits_u16, gpu_dispatch, gpu_layout, gpu_ll_dispatch, gpu_notify, inputs,
                        np_, oracle_normal, status_word, to_dev_bf16)

pytestmark = pytest.mark.gpu

MAX_ULP = 1


def assert_bf16_close(got_bits, ref_bits, max_ulp=MAX_ULP):
    got = oracle.bf16_to_f32(got_bits).astype(np.float64)
    ref = oracle.bf16_to_f32(ref_bits).astype(np.float64)
    a = np.abs(ref)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -133)))
    ulp = np.exp2(np.maximum(e, -126) - 7)
    bad = np.abs(got - ref) > max_ulp * ulp
    assert not bad.any(), f"{bad.sum()} elements beyond {max_ulp} ulp"
    return int((got_bits != ref_bits).sum())


def _expert_outputs_dev(n_rows, H, seed=5):
    return synth.expert_outputs_torch(n_rows, H, "cuda", seed)


def _oracle_combine_rows(y_dev_flat, wts, cidx_ref, H):
    """Oracle combine fed only the rows the oracle's own combine_idx names."""
    used = np.unique(cidx_ref[cidx_ref >= 0])
    y_sub = bits_u16(y_dev_flat[torch.from_numpy(used).cuda()])
    remap = np.full(cidx_ref.shape, -1, np.int32)
    m = cidx_ref >= 0
    remap[m] = np.searchsorted(used, cidx_ref[m])
    return oracle.combine(y_sub, wts, remap, H)


def _normal_combine(w, A=1, sample=None, x_on_device=False):
    x_dev, x_host, idx_dev, idx, wts_dev, wts = inputs(w, x_on_device=x_on_device)
    lay = gpu_layout(idx_dev, w.E)
    nt = gpu_notify(lay, w.E, A)
    ref_lay = oracle.layout(idx, w.R, w.E)
    ref_nt = oracle.notify(ref_lay["num_tokens_per_rank"], ref_lay["num_tokens_per_expert"], w.R,
                           w.E, A)
    cap = max(1, int(ref_nt["psum"][:, -1].max()))
    d = gpu_dispatch(x_dev, idx_dev, lay, nt, w.E, 0, cap)
    y = _expert_outputs_dev(w.R * cap, w.H).view(w.R, cap, w.H)
    out = torch.empty((w.R, w.T_r, w.H), dtype=torch.bfloat16, device="cuda")
    st = status_word()
    ep.ep_combine(y, wts_dev, d["combine_idx"], cap, out, st)
    assert ep.ep_read_status(st) == ep.EP_OK
    x0 = np.zeros((w.R, w.T_r, 0), np.uint16)
    ref_d = oracle.dispatch(x0, idx, ref_lay["slot_rank"], ref_nt["expert_prefix"], ref_nt["psum"],
                            w.E, 0, cap)
    cidx_ref = ref_d["combine_idx"]
    assert np.array_equal(np_(d["combine_idx"]), cidx_ref)
    if sample is not None:
        toks = np.random.default_rng(3).choice(w.T, size=sample, replace=False)
        c = _oracle_combine_rows(y.view(-1, w.H), wts.reshape(-1, w.k)[toks],
                                 cidx_ref.reshape(-1, w.k)[toks], w.H)
        return assert_bf16_close(np_(out).reshape(-1, w.H)[toks], c["out"])
    c = _oracle_combine_rows(y.view(-1, w.H), wts, cidx_ref, w.H)
    assert c["rc"] == oracle.OK
    return assert_bf16_close(np_(out), c["out"])


def test_combine_tiny():
    assert _normal_combine(synth.WORKLOADS["tiny"]) == 0


@pytest.mark.parametrize("name,T_r,A", [("prefill", 96, 1), ("skewed", 40, 128),
                                         ("large", 64, 1)])
def test_combine_scaled_full_compare(name, T_r, A):
    w = synth.scaled(synth.WORKLOADS[name], T_r=T_r)
    assert _normal_combine(w, A) == 0


@pytest.mark.parametrize("H,k", [(8, 3), (136, 8), (1032, 16), (520, 9)])
def test_combine_ragged_hidden_and_k(H, k):
    w = synth.scaled(synth.WORKLOADS["tiny"], H=H, k=k, E=16 if k <= 8 else 32, T_r=37)
    assert _normal_combine(w) == 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["prefill", "large"])
def test_combine_full_size_sampled(name):
    w = synth.WORKLOADS[name]
    assert _normal_combine(w, sample=256, x_on_device=True) == 0


def _ll_combine(w, fp8_mode):
    x_dev, x_host, idx_dev, idx, wts_dev, wts = inputs(w)
    d = gpu_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, fp8_mode)
    S = w.R * w.max_tokens_per_rank
    y = _expert_outputs_dev(w.E * S, w.H).view(w.R, w.E_l, S, w.H)
    out = torch.empty((w.R, w.T_r, w.H), dtype=torch.bfloat16, device="cuda")
    st = status_word()
    ep.ep_ll_combine(y, wts_dev, d["combine_idx"], w.E, w.max_tokens_per_rank, out, st)
    assert ep.ep_read_status(st) == ep.EP_OK
    ref = oracle.ll_dispatch(np.zeros((w.R, w.T_r, 0), np.uint16), idx, w.E,
                             w.max_tokens_per_rank, 0)
    assert np.array_equal(np_(d["combine_idx"]), ref["combine_idx"])
    c = _oracle_combine_rows(y.view(-1, w.H), wts, ref["combine_idx"], w.H)
    return assert_bf16_close(np_(out), c["out"])


def test_ll_combine_tiny():
    assert _ll_combine(synth.WORKLOADS["tiny"], 0) == 0


@pytest.mark.slow
def test_ll_combine_decode_full_size():
    w = synth.WORKLOADS["decode"]
    assert _ll_combine(w, w.fp8_mode) == 0


def test_identity_expert_round_trip_on_gpu():
    """dispatch -> (y = received rows) -> combine == bf16(sum_j w_j x)."""
    w = synth.scaled(synth.WORKLOADS["prefill"], T_r=64)
    x_dev, x_host, idx_dev, idx, wts_dev, wts = inputs(w)
    lay = gpu_layout(idx_dev, w.E)
    nt = gpu_notify(lay, w.E, 1)
    cap = int(np_(nt["psum"])[:, -1].max())
    d = gpu_dispatch(x_dev, idx_dev, lay, nt, w.E, 0, cap)
    out = torch.empty_like(x_dev)
    ep.ep_combine(d["recv_x"], wts_dev, d["combine_idx"], cap, out)
    xs = oracle.bf16_to_f32(x_host).astype(np.float64)
    ref = wts.astype(np.float64).sum(axis=2)[..., None] * xs
    got = oracle.bf16_to_f32(np_(out)).astype(np.float64)
    e = np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -133)))
    assert np.all(np.abs(got - ref) <= np.exp2(np.maximum(e, -126) - 7))


def test_combine_special_weights_and_masks():
    w = synth.scaled(synth.WORKLOADS["tiny"], k=1)
    x_dev, x_host, idx_dev, idx, wts_dev, wts = inputs(w)
    lay = gpu_layout(idx_dev, w.E)
    nt = gpu_notify(lay, w.E, 1)
    cap = int(np_(nt["psum"])[:, -1].max())
    d = gpu_dispatch(x_dev, idx_dev, lay, nt, w.E, 0, cap)
    out = torch.empty_like(x_dev)
    ep.ep_combine(d["recv_x"], torch.ones_like(wts_dev), d["combine_idx"], cap, out)
    assert np.array_equal(np_(out), x_host)                 # k = 1, w = 1: exact copy
    ep.ep_combine(d["recv_x"], torch.zeros_like(wts_dev), d["combine_idx"], cap, out)
    assert np.all(np_(out) == 0)                            # +0, not -0
    cidx = d["combine_idx"].clone()
    cidx[:, ::2] = -1
    ep.ep_combine(d["recv_x"], wts_dev, cidx, cap, out)
    assert np.all(np_(out)[:, ::2] == 0)
    # out-of-range indices are reported and skipped, never read
    cidx[0, 1, 0] = w.R * cap
    st = status_word()
    ep.ep_combine(d["recv_x"], wts_dev, cidx, cap, out, st)
    assert ep.ep_read_status(st) == ep.EP_ERR_INVALID_ARG
    assert np.all(np_(out)[0, 1] == 0)


def test_combine_writes_pinned_host_output_directly():
    """out may be pinned host memory: the combine writes the result across
    the host link with no copy; bit-identical to a device output.  Pageable
    host memory is refused before any launch."""
    import ctypes
    w = synth.scaled(synth.WORKLOADS["decode"], T_r=32, H=1024)
    x_dev, _, idx_dev, _, wts_dev, _ = inputs(w)
    d = gpu_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, w.fp8_mode)
    S = w.R * w.max_tokens_per_rank
    y = _expert_outputs_dev(w.E * S, w.H).view(w.R, w.E_l, S, w.H)
    out_dev = torch.empty_like(x_dev)
    out_host = torch.empty(x_dev.shape, dtype=torch.bfloat16).pin_memory()
    ep.ep_ll_combine(y, wts_dev, d["combine_idx"], w.E, w.max_tokens_per_rank, out_dev)
    ep.ep_ll_combine(y, wts_dev, d["combine_idx"], w.E, w.max_tokens_per_rank, out_host)
    torch.cuda.synchronize()
    assert torch.equal(out_host.view(torch.int16), out_dev.cpu().view(torch.int16))
    # rank-level and normal combines take the same path for `out`
    cap = S
    yr = y.reshape(w.R, -1, w.H)[:, :cap].contiguous()
    cidx = torch.where(d["combine_idx"] >= 0, d["combine_idx"] % cap, d["combine_idx"])
    cidx = cidx.to(torch.int32).contiguous()
    ep.ep_rank_combine(yr, cidx, cap, out_dev)
    ep.ep_rank_combine(yr, cidx, cap, out_host)
    torch.cuda.synchronize()
    assert torch.equal(out_host.view(torch.int16), out_dev.cpu().view(torch.int16))
    pageable = np.empty(out_dev.numel(), np.uint16)
    L = ep.load()
    rc = L.ep_ll_combine(ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(wts_dev.data_ptr()),
                         ctypes.c_void_p(d["combine_idx"].data_ptr()), w.R, w.T_r, w.H, w.E, w.k,
                         w.max_tokens_per_rank, ctypes.c_void_p(pageable.ctypes.data), None,
                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == ep.EP_ERR_INVALID_ARG
