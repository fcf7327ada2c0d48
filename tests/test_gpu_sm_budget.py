"""GPU parity under an SM budget (ep_set_num_sms): the data kernels confined
to a few SMs -- the single-launch low-latency path on fewer CTAs, the
multi-kernel low-latency path (the scale-column pass looping over experts),
the normal FP8 path and both combines -- still give the oracle's results
bit for bit (the combines: within 1 bf16 ulp, 0 expected)."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_gb300 import ep, synth
from ep_harness import (bits_u16, gpu_dispatch, gpu_layout, gpu_ll_dispatch, gpu_notify, inputs,
                        np_)
from test_gpu_combine import assert_bf16_close
from test_gpu_dispatch import _compare_full
from test_gpu_ll import _compare_ll

pytestmark = pytest.mark.gpu


@pytest.fixture
def budget():
    def set_budget(n):
        ep.ep_set_num_sms(n)
        return ep.ep_get_num_sms()
    yield set_budget
    ep.ep_set_num_sms(0)


@pytest.mark.parametrize("n_sms,T_r,H", [
    (8, 24, 1024),     # single-launch path on 8 CTAs (48 units each)
    (8, 128, 7168),    # too large for 8 CTAs: layout + scatter + scale columns
    (37, 100, 2048),   # an odd budget
])
def test_ll_dispatch_and_combine_under_a_budget(budget, n_sms, T_r, H):
    assert budget(n_sms) == n_sms
    w = synth.scaled(synth.WORKLOADS["decode"], T_r=T_r, H=H)
    x_dev, x_host, idx_dev, idx, wts_dev, wts = inputs(w, seed=4)
    d = gpu_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, w.fp8_mode)
    torch.cuda.synchronize()
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    _compare_ll(w, x_host, idx, d, w.max_tokens_per_rank, w.fp8_mode)
    S = w.R * w.max_tokens_per_rank
    y = synth.expert_outputs_torch(w.E * S, w.H, "cuda", 3).view(w.R, w.E_l, S, w.H)
    out = torch.empty_like(x_dev)
    ep.ep_ll_combine(y, wts_dev, d["combine_idx"], w.E, w.max_tokens_per_rank, out)
    torch.cuda.synchronize()
    cidx = np_(d["combine_idx"])
    used = np.unique(cidx[cidx >= 0])
    y_flat = y.reshape(-1, w.H)
    sub = bits_u16(y_flat[torch.from_numpy(used).cuda()])
    remap = np.full(cidx.shape, -1, np.int32)
    remap[cidx >= 0] = np.searchsorted(used, cidx[cidx >= 0])
    ref = oracle.combine(sub, wts, remap, w.H)
    assert ref["rc"] == oracle.OK
    assert_bf16_close(np_(out), ref["out"])


@pytest.mark.parametrize("fp8_mode", [0, 1])
def test_normal_dispatch_and_combine_under_a_budget(budget, fp8_mode):
    assert budget(6) == 6
    w = synth.scaled(synth.WORKLOADS["prefill"], T_r=80, fp8_mode=fp8_mode)
    x_dev, x_host, idx_dev, idx, wts_dev, wts = inputs(w, seed=6)
    lay = gpu_layout(idx_dev, w.E)
    nt = gpu_notify(lay, w.E, 1, -1)
    ref_lay = oracle.layout(idx, w.R, w.E)
    ref_nt = oracle.notify(ref_lay["num_tokens_per_rank"], ref_lay["num_tokens_per_expert"], w.R,
                           w.E, 1, -1)
    cap = max(1, int(ref_nt["psum"][:, -1].max()))
    d = gpu_dispatch(x_dev, idx_dev, lay, nt, w.E, fp8_mode, cap)
    torch.cuda.synchronize()
    assert ep.ep_read_status(d["status"]) == ep.EP_OK
    _compare_full(w, x_host, idx, d, cap, 1)
    y = synth.expert_outputs_torch(w.R * cap, w.H, "cuda", 8).view(w.R, cap, w.H)
    out = torch.empty_like(x_dev)
    ep.ep_combine(y, wts_dev, d["combine_idx"], cap, out)
    torch.cuda.synchronize()
    ref = oracle.combine(bits_u16(y), wts, np_(d["combine_idx"]), w.H)
    assert ref["rc"] == oracle.OK
    assert_bf16_close(np_(out), ref["out"])


def test_budget_larger_than_the_gpu_is_the_whole_gpu(budget):
    full = budget(0)
    assert budget(10 ** 6) == full
    assert budget(1) == 1
