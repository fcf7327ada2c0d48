"""GPU parity at the size limits of the entry points: 1024 ranks, 1024
experts (one per rank) and top-16, the largest R, E and k that the C ABI
accepts, through every path -- layout + notify (separate and in one launch),
normal dispatch + combine, the single-call fixed-shape path, the
low-latency single-launch and multi-kernel paths, the once-per-rank layout
-- and a hidden size of 16384 (16 pieces of 1024 channels per token), each
against the oracle: bit-exact, combine within 1 bf16 ulp."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_gb300 import ep, synth
from ep_harness import (gpu_dispatch, gpu_layout, gpu_ll_dispatch, gpu_notify, np_, poison_,
                        status_word, to_dev_bf16)
from test_gpu_combine import _oracle_combine_rows, assert_bf16_close
from test_gpu_dispatch import _compare_full
from test_gpu_layout import NOTIFY_KEYS, _compare_layout
from test_gpu_layout_notify import _check, _fused
from test_gpu_ll import _compare_ll

pytestmark = pytest.mark.gpu

R_MAX, E_MAX, K_MAX = 1024, 1024, 16


def _inputs(seed, R, T_r, H, E, k, masked=0.1):
    """Distinct experts per token, about `masked` of the slots unused (-1)."""
    rng = np.random.default_rng(seed)
    keys = rng.random((R * T_r, E))
    idx = np.argsort(keys, axis=1)[:, :k].astype(np.int64)
    idx[rng.random(idx.shape) < masked] = -1
    idx = idx.reshape(R, T_r, k)
    w = rng.standard_normal((R, T_r, k)).astype(np.float32)
    x = synth.to_bf16_bits(rng.standard_normal((R, T_r, H)).astype(np.float32))
    return idx, w, x


def _normal(seed, R, T_r, H, E, k, fp8_mode, A):
    idx, wts, x_host = _inputs(seed, R, T_r, H, E, k)
    idx_dev = torch.from_numpy(idx).cuda()
    x_dev = to_dev_bf16(x_host)
    lay = gpu_layout(idx_dev, E)
    _compare_layout(idx, E, lay)
    nt = gpu_notify(lay, E, A)
    ref_lay = oracle.layout(idx, R, E)
    ref_nt = oracle.notify(ref_lay["num_tokens_per_rank"], ref_lay["num_tokens_per_expert"], R, E,
                           A)
    for key in NOTIFY_KEYS:
        assert np.array_equal(np_(nt[key]), ref_nt[key]), key
    cap = max(1, int(ref_nt["psum"][:, -1].max()))
    d = gpu_dispatch(x_dev, idx_dev, lay, nt, E, fp8_mode, cap)
    torch.cuda.synchronize()
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    w = synth.Workload("limits", R=R, T_r=T_r, H=H, E=E, k=k, routing="uniform", mode="normal",
                       fp8_mode=fp8_mode)
    _compare_full(w, x_host, idx, d, cap, A)
    y = synth.expert_outputs_torch(R * cap, H, "cuda", seed).view(R, cap, H)
    out = torch.empty((R, T_r, H), dtype=torch.bfloat16, device="cuda")
    st = status_word()
    ep.ep_combine(y, torch.from_numpy(wts).cuda(), d["combine_idx"], cap, out, st)
    assert ep.ep_read_status(st) == ep.EP_OK
    ref = _oracle_combine_rows(y.reshape(-1, H), wts, np_(d["combine_idx"]), H)
    assert ref["rc"] == oracle.OK
    assert_bf16_close(np_(out), ref["out"])


def _low_latency(seed, R, T_r, H, E, k, fp8_mode, max_tokens):
    idx, wts, x_host = _inputs(seed, R, T_r, H, E, k)
    idx_dev = torch.from_numpy(idx).cuda()
    d = gpu_ll_dispatch(to_dev_bf16(x_host), idx_dev, E, max_tokens, fp8_mode)
    torch.cuda.synchronize()
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    w = synth.Workload("limits", R=R, T_r=T_r, H=H, E=E, k=k, routing="uniform", mode="ll",
                       fp8_mode=fp8_mode, max_tokens_per_rank=max_tokens)
    _compare_ll(w, x_host, idx, d, max_tokens, fp8_mode)
    S = R * max_tokens
    y = synth.expert_outputs_torch(E * S, H, "cuda", seed).view(R, E // R, S, H)
    out = torch.empty((R, T_r, H), dtype=torch.bfloat16, device="cuda")
    st = status_word()
    ep.ep_ll_combine(y, torch.from_numpy(wts).cuda(), d["combine_idx"], E, max_tokens, out, st)
    assert ep.ep_read_status(st) == ep.EP_OK
    ref = _oracle_combine_rows(y.reshape(-1, H), wts, np_(d["combine_idx"]), H)
    assert ref["rc"] == oracle.OK
    assert_bf16_close(np_(out), ref["out"])


@pytest.mark.parametrize("fp8_mode,A", [(0, 1), (1, 4), (2, 128)])
def test_normal_path_at_the_rank_expert_and_topk_limits(fp8_mode, A):
    # 3 tokens per rank: one chunk per rank, is_token_in_rank by the per-rank
    # loop (R > 64), notify's counts walked in memory (too large to stage)
    _normal(10 + fp8_mode, R_MAX, 3, 128, E_MAX, K_MAX, fp8_mode, A)


def test_layout_notify_in_one_launch_at_the_limits():
    idx, _, _ = _inputs(20, R_MAX, 3, 8, E_MAX, K_MAX)
    for A, nwt in ((1, -1), (8, R_MAX * 3)):
        lay, nt, st, _ = _fused(torch.from_numpy(idx).cuda(), E_MAX, A, nwt)
        _check(idx, E_MAX, A, nwt, lay, nt, st)


def test_single_call_fixed_shape_at_the_limits():
    R, T_r, H, E, k, A = R_MAX, 3, 128, E_MAX, K_MAX, 4
    idx, _, x_host = _inputs(30, R, T_r, H, E, k)
    nwt = R * T_r
    cap = nwt * min(k, E // R) + (E // R) * (A - 1)
    lay = ep.alloc_layout(R, T_r, k, E)
    nt = ep.alloc_notify(R, E)
    d = ep.alloc_dispatch(R, T_r, H, k, 2, cap)
    for v in list(lay.values()) + list(nt.values()) + list(d.values()):
        poison_(v)
    ws = ep.alloc_workspace(R, T_r, k, E, H)
    st = status_word()
    ep.ep_layout_notify_dispatch(to_dev_bf16(x_host), torch.from_numpy(idx).cuda(), E, 2, A, nwt,
                                 cap, lay, nt, d, ws, st)
    torch.cuda.synchronize()
    assert ep.ep_read_status(st) == ep.EP_OK
    w = synth.Workload("limits", R=R, T_r=T_r, H=H, E=E, k=k, routing="uniform", mode="normal",
                       fp8_mode=2, num_worst_tokens=nwt)
    _compare_full(w, x_host, idx, d, cap, A)


@pytest.mark.parametrize("T_r,fp8_mode", [
    (2, 0),   # 32768 ids: the single-launch path
    (2, 2),
    (5, 1),   # 81920 ids: past the single launch, the multi-kernel path
])
def test_low_latency_path_at_the_rank_expert_and_topk_limits(T_r, fp8_mode):
    _low_latency(40 + T_r, R_MAX, T_r, 128, E_MAX, K_MAX, fp8_mode, T_r)


def test_once_per_rank_path_at_the_limits():
    from test_gpu_rank import _compare, _gpu_rank_path
    idx, wts, x_host = _inputs(50, R_MAX, 3, 128, E_MAX, K_MAX)
    g = _gpu_rank_path(to_dev_bf16(x_host), torch.from_numpy(idx).cuda(),
                       torch.from_numpy(wts).cuda(), E_MAX, 2)
    _compare(x_host, idx, wts, E_MAX, 2, g)


@pytest.mark.parametrize("fp8_mode", [0, 1, 2])
def test_hidden_16384(fp8_mode):
    _normal(60 + fp8_mode, 2, 33, 16384, 8, 4, fp8_mode, 1)
    _low_latency(70 + fp8_mode, 2, 33, 16384, 8, 4, fp8_mode, 40)
