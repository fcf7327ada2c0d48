"""ep_get_dispatch_layout_no_alloc: the layout for callers that may not
allocate device memory (graph capture, allocator callbacks, runtimes that
forbid the library any allocation).  Called through the C ABI and compared
with ep_get_dispatch_layout (caller-provided workspace) on two calls in a
row -- the second call reuses the static scratch the first one left behind.
Collected last on purpose, so a failure here cannot hide another test's."""
import ctypes

import numpy as np
import pytest
import torch

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


def test_no_alloc_layout_matches_the_workspace_layout_on_two_calls():
    for name, seed in (("prefill", 0), ("skewed", 1)):
        w = synth.WORKLOADS[name]
        idx, _ = synth.routing(w, seed)
        idx_dev = torch.from_numpy(idx).cuda()
        got = _no_alloc(idx_dev, w.E)
        ref = _with_workspace(idx_dev, w.E)
        torch.cuda.synchronize()
        for key in ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank",
                    "slot_rank"):
            assert torch.equal(got[key], ref[key]), (name, key)   # integers: exact


def test_no_alloc_rejects_a_problem_beyond_its_scratch():
    R, T_r, k, E = 8, 65536, 16, 1024       # look-back state far above 4 MiB
    before = ep.ep_launch_count()
    rc = _fn()(None, R, T_r, k, E, None, None, None, None, None, None)
    assert rc == ep.EP_ERR_TOO_LARGE
    assert ep.ep_launch_count() == before
