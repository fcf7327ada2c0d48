"""GPU parity over seeded random problem shapes: normal dispatch + combine
and low-latency dispatch + combine (single-launch or multi-kernel path,
whichever the shape takes), all three precisions, odd rank / expert / top-k
counts, ragged hidden sizes and masked slots -- every output vs the oracle
(bit-exact; combine within 1 bf16 ulp)."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_gb300 import ep, synth
from ep_harness import (bits_u16, gpu_dispatch, gpu_layout, gpu_ll_dispatch, gpu_notify, np_,
                        oracle_normal, to_dev_bf16)
from test_gpu_combine import _oracle_combine_rows, assert_bf16_close
from test_gpu_dispatch import _compare_full
from test_gpu_ll import _compare_ll

pytestmark = pytest.mark.gpu


def _shape(seed):
    rng = np.random.default_rng(1000 + seed)
    R = int(rng.choice([1, 2, 3, 4, 8, 16, 24]))
    E_l = int(rng.integers(1, 9))
    E = R * E_l
    k = int(rng.integers(1, min(E, 16) + 1))
    fp8 = int(rng.integers(0, 3))
    H = int(rng.choice([128, 256, 384, 1152, 2048, 3072])) if fp8 else int(rng.choice([8, 72, 264, 1000, 2056]))
    T_r = int(rng.integers(0, 200))
    return rng, R, T_r, H, E, k, fp8


def _inputs(rng, R, T_r, H, E, k):
    # distinct experts per token where possible, then about 10 % of slots masked
    keys = rng.random((R * T_r, E))
    idx = np.argsort(keys, axis=1)[:, :k].astype(np.int64)
    idx[rng.random(idx.shape) < 0.1] = -1
    idx = idx.reshape(R, T_r, k)
    w = rng.standard_normal((R, T_r, k)).astype(np.float32)
    x = synth.to_bf16_bits(rng.standard_normal((R, T_r, H)).astype(np.float32))
    return idx, w, x


@pytest.mark.parametrize("seed", range(32))
def test_random_normal_shapes(seed):
    rng, R, T_r, H, E, k, fp8 = _shape(seed)
    idx, wts, x_host = _inputs(rng, R, T_r, H, E, k)
    A = int(rng.choice([1, 4, 128]))
    idx_dev = torch.from_numpy(idx).cuda()
    x_dev = to_dev_bf16(x_host)
    lay = gpu_layout(idx_dev, E)
    nt = gpu_notify(lay, E, A, -1)
    _, ref_nt, _, cap = oracle_normal(x_host, idx, E, A, fp8)
    d = gpu_dispatch(x_dev, idx_dev, lay, nt, E, fp8, cap)
    torch.cuda.synchronize()
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    w = synth.Workload("rand", R=R, T_r=T_r, H=H, E=E, k=k, routing="uniform", mode="normal",
                       fp8_mode=fp8)
    _compare_full(w, x_host, idx, d, cap, A)
    y = synth.expert_outputs_torch(R * cap, H, "cuda", seed).view(R, cap, H)
    out = torch.empty((R, T_r, H), dtype=torch.bfloat16, device="cuda")
    ep.ep_combine(y, torch.from_numpy(wts).cuda(), d["combine_idx"], cap, out)
    torch.cuda.synchronize()
    ref = _oracle_combine_rows(y.reshape(-1, H), wts, np_(d["combine_idx"]), H)
    assert ref["rc"] == oracle.OK
    assert_bf16_close(np_(out), ref["out"])


@pytest.mark.parametrize("seed", range(32))
def test_random_low_latency_shapes(seed):
    rng, R, T_r, H, E, k, fp8 = _shape(100 + seed)
    T_r = min(T_r, 96)
    max_tokens = T_r + int(rng.integers(1, 40))
    idx, wts, x_host = _inputs(rng, R, T_r, H, E, k)
    idx_dev = torch.from_numpy(idx).cuda()
    x_dev = to_dev_bf16(x_host)
    d = gpu_ll_dispatch(x_dev, idx_dev, E, max_tokens, fp8)
    torch.cuda.synchronize()
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    w = synth.Workload("rand", R=R, T_r=T_r, H=H, E=E, k=k, routing="uniform", mode="ll",
                       fp8_mode=fp8, max_tokens_per_rank=max_tokens)
    _compare_ll(w, x_host, idx, d, max_tokens, fp8)
    S = R * max_tokens
    y = synth.expert_outputs_torch(E * S, H, "cuda", seed).view(R, E // R, S, H)
    out = torch.empty((R, T_r, H), dtype=torch.bfloat16, device="cuda")
    ep.ep_ll_combine(y, torch.from_numpy(wts).cuda(), d["combine_idx"], E, max_tokens, out)
    torch.cuda.synchronize()
    ref = _oracle_combine_rows(y.reshape(-1, H), wts, np_(d["combine_idx"]), H)
    assert ref["rc"] == oracle.OK
    assert_bf16_close(np_(out), ref["out"])


@pytest.mark.parametrize("seed", range(16))
def test_random_once_per_rank_shapes(seed):
    from test_gpu_rank import _compare, _gpu_rank_path
    rng, R, T_r, H, E, k, fp8 = _shape(200 + seed)
    idx, wts, x_host = _inputs(rng, R, T_r, H, E, k)
    g = _gpu_rank_path(to_dev_bf16(x_host), torch.from_numpy(idx).cuda(),
                       torch.from_numpy(wts).cuda(), E, fp8)
    if T_r == 0:   # nothing to place: only the status
        assert ep.ep_read_status(g["status"]) == ep.EP_OK
        return
    _compare(x_host, idx, wts, E, fp8, g)


@pytest.mark.parametrize("seed", range(16))
def test_random_single_call_fixed_shapes(seed):
    from ep_harness import poison_, status_word
    rng, R, T_r, H, E, k, fp8 = _shape(300 + seed)
    idx, wts, x_host = _inputs(rng, R, T_r, H, E, k)
    A = int(rng.choice([1, 4, 128]))
    nwt = R * T_r + int(rng.integers(0, 5))
    cap = max(1, nwt * min(k, E // R))
    # the worst case of the fixed shape, plus the alignment padding of every segment
    cap += (E // R) * (A - 1)
    idx_dev = torch.from_numpy(idx).cuda()
    x_dev = to_dev_bf16(x_host)
    lay = ep.alloc_layout(R, T_r, k, E)
    nt = ep.alloc_notify(R, E)
    d = ep.alloc_dispatch(R, T_r, H, k, fp8, cap)
    for v in list(lay.values()) + list(nt.values()) + list(d.values()):
        poison_(v)
    ws = ep.alloc_workspace(R, T_r, k, E, H)
    st = status_word()
    ep.ep_layout_notify_dispatch(x_dev, idx_dev, E, fp8, A, nwt, cap, lay, nt, d, ws, st)
    torch.cuda.synchronize()
    assert ep.ep_read_status(st) == ep.EP_OK
    w = synth.Workload("rand", R=R, T_r=T_r, H=H, E=E, k=k, routing="uniform", mode="normal",
                       fp8_mode=fp8, num_worst_tokens=nwt)
    _compare_full(w, x_host, idx, d, cap, A)
