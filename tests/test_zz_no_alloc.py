"""ep_get_dispatch_layout_no_alloc: the layout for callers that may not
allocate device memory (allocator callbacks, runtimes that forbid the
library any allocation).  Called through the C ABI and compared
with the oracle and with ep_get_dispatch_layout (caller-provided workspace)
on calls in a row -- each call reuses the static scratch the one before
left behind.
Collected last on purpose, so a failure here cannot hide another test's."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_gb300 import ep, synth

pytestmark = pytest.mark.gpu

_P, _I = ctypes.c_void_p, ctypes.c_int


def _fn():
    f = ep.load().ep_get_dispatch_layout_no_alloc
    f.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]
    f.restype = _I
    return f


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _no_alloc(idx_dev, E):
    R, T_r, k = idx_dev.shape
    out = ep.alloc_layout(R, T_r, k, E)
    for v in out.values():
        v.fill_(-7)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = _fn()(_ptr(idx_dev), R, T_r, k, E, _ptr(out["num_tokens_per_rank"]),
               _ptr(out["num_tokens_per_expert"]), _ptr(out["is_token_in_rank"]),
               _ptr(out["slot_rank"]), _ptr(status), stream)
    assert rc == ep.EP_OK, ep.error_string(rc)
    assert ep.ep_read_status(status) == ep.EP_OK
    return out


def _with_workspace(idx_dev, E):
    R, T_r, k = idx_dev.shape
    out = ep.alloc_layout(R, T_r, k, E)
    ws = ep.alloc_workspace(R, T_r, k, E, 8)
    ep.ep_get_dispatch_layout(idx_dev, E, out["num_tokens_per_rank"], out["num_tokens_per_expert"],
                              out["is_token_in_rank"], out["slot_rank"], ws)
    return out


def test_no_alloc_layout_matches_the_workspace_layout_and_the_oracle():
    """Three calls in a row (prefill, skewed and the large routing, which the
    4 MiB scratch still holds), each compared element by element with the
    oracle's layout and with ep_get_dispatch_layout on the same ids."""
    for name, seed in (("prefill", 0), ("skewed", 1), ("large", 2)):
        w = synth.WORKLOADS[name]
        idx, _ = synth.routing(w, seed)
        idx_dev = torch.from_numpy(idx).cuda()
        got = _no_alloc(idx_dev, w.E)
        ref = _with_workspace(idx_dev, w.E)
        torch.cuda.synchronize()
        want = oracle.layout(idx, w.R, w.E)
        assert want["rc"] == oracle.OK
        for key in ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank",
                    "slot_rank"):
            assert torch.equal(got[key], ref[key]), (name, key)   # integers: exact
            g = got[key].cpu().numpy()
            assert np.array_equal(g.astype(np.int64), want[key].astype(np.int64)), (name, key)


def test_no_alloc_layout_leaves_device_memory_unchanged():
    """After a first (warm) call, a further call changes neither the
    device's free memory nor torch's allocations."""
    w = synth.WORKLOADS["prefill"]
    idx, _ = synth.routing(w, 3)
    idx_dev = torch.from_numpy(idx).cuda()
    out = ep.alloc_layout(w.R, w.T_r, w.k, w.E)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (_ptr(idx_dev), w.R, w.T_r, w.k, w.E, _ptr(out["num_tokens_per_rank"]),
            _ptr(out["num_tokens_per_expert"]), _ptr(out["is_token_in_rank"]),
            _ptr(out["slot_rank"]), _ptr(status), stream)
    assert _fn()(*args) == ep.EP_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    assert _fn()(*args) == ep.EP_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0 and torch.cuda.memory_allocated() == alloc0
    assert ep.ep_read_status(status) == ep.EP_OK
    want = oracle.layout(idx, w.R, w.E)
    assert np.array_equal(out["slot_rank"].cpu().numpy(), want["slot_rank"])


def test_no_alloc_rejects_a_problem_beyond_its_scratch():
    R, T_r, k, E = 8, 65536, 16, 1024       # look-back state far above 4 MiB
    before = ep.ep_launch_count()
    rc = _fn()(None, R, T_r, k, E, None, None, None, None, None, None)
    assert rc == ep.EP_ERR_TOO_LARGE
    assert ep.ep_launch_count() == before
