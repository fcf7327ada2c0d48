"""The C-ABI library builds, loads, and exports every entry point ep.h
declares; host-only entry points behave as documented (no GPU needed)."""
import ctypes
import os
import re
import threading
import time

import pytest
import torch

from combine_get_dispatch_gb300 import _build, ep

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(ep_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol():
    L = ep.load()
    declared = _declared_functions()
    assert {"ep_get_dispatch_layout", "ep_notify_dispatch", "ep_dispatch", "ep_combine",
            "ep_ll_dispatch", "ep_ll_combine", "ep_clean_ll_buffer"} <= declared
    missing = [n for n in sorted(declared) if not hasattr(L, n)]
    assert not missing, missing
    assert set(ep.EXPORTS) <= declared


def test_library_is_built_for_sm_103a_only():
    assert ep.load() is not None
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.ARCH)


def test_sm_budget_setter():
    """ep_set_num_sms: negative budgets are refused, 0 lifts the budget
    (host-only: the budget is read at launch time)."""
    with pytest.raises(ep.EPError):
        ep.ep_set_num_sms(-1)
    ep.ep_set_num_sms(3)
    try:
        assert 1 <= ep.ep_get_num_sms() <= 3
    finally:
        ep.ep_set_num_sms(0)
    assert ep.ep_get_num_sms() >= 1


def test_error_strings_and_launch_counter():
    for code in range(6):
        assert ep.error_string(code)
    assert ep.error_string(99) == "unknown error"
    assert ep.ep_launch_count() >= 0


def test_workspace_size():
    a = ep.ep_workspace_size(16, 128, 8, 256, 7168)
    b = ep.ep_workspace_size(16, 4096, 8, 256, 7168)
    assert a > 0 and b > a and a % 256 == 0
    # the FP8 scale staging grows with the hidden size
    assert ep.ep_workspace_size(16, 128, 8, 256, 4096) < a
    assert ep.ep_workspace_size(0, 1, 1, 1, 128) == 0
    assert ep.ep_workspace_size(2, 1, 17, 4, 128) == 0
    assert ep.ep_workspace_size(2, 1, 1, 4, 0) == 0


def test_host_wait_counters_times_out_and_succeeds():
    c = torch.tensor([3, -1, 0], dtype=torch.int64)
    t0 = time.time()
    assert ep.ep_host_wait_counters(c, 100) == ep.EP_ERR_TIMEOUT
    assert 0.09 <= time.time() - t0 < 2.0
    c[1] = 7
    assert ep.ep_host_wait_counters(c, 100) == ep.EP_OK


def test_host_wait_counters_sees_a_late_writer():
    """A 'rank' that publishes its count after a delay (host-side fault
    model of a slow notify): the wait returns OK once it lands."""
    c = torch.full((4,), -1, dtype=torch.int64)

    def writer():
        time.sleep(0.05)
        for r in range(4):
            c[r] = r

    th = threading.Thread(target=writer)
    th.start()
    rc = ep.ep_host_wait_counters(c, 5000)
    th.join()
    assert rc == ep.EP_OK


def test_argument_validation_returns_invalid_arg_without_launch():
    L = ep.load()
    before = ep.ep_launch_count()
    # E % R != 0, k too large, null pointers: rejected on the host
    assert L.ep_get_dispatch_layout(None, 3, 4, 2, 8, None, None, None, None, None, 0, None,
                                    None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_get_dispatch_layout(None, 2, 4, 17, 8, None, None, None, None, None, 0, None,
                                    None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_notify_dispatch(None, None, 2, 8, 0, -1, None, None, None, None, None, 0, None,
                                None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_dispatch(None, None, None, None, None, 2, 4, 7168, 8, 8, 1, 16, None, None, None,
                         None, None, 0, None, None) == ep.EP_ERR_INVALID_ARG
    # FP8 needs H % 128 == 0
    assert L.ep_dispatch(None, None, None, None, None, 2, 0, 200, 8, 8, 2, 0, None, None, None,
                         None, None, 0, None, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_ll_dispatch(None, None, 2, 8, 256, 8, 2, 4, 0, None, None, None, None, None, None,
                            None, 0, None, None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_combine(None, None, None, 2, 4, 256, 0, 16, None, None,
                        None) == ep.EP_ERR_INVALID_ARG
    assert L.ep_clean_ll_buffer(None, 3, 8, None, 0, None) == ep.EP_ERR_INVALID_ARG
    assert ep.ep_launch_count() == before


def test_binding_rejects_host_tensors():
    idx = torch.zeros((2, 4, 2), dtype=torch.int64)
    with pytest.raises(ValueError):
        ep.ep_get_dispatch_layout(idx, 4, *[torch.zeros(1)] * 4, torch.zeros(1, dtype=torch.uint8))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No CPU or PyTorch fallback: without the built library the binding
    raises instead of computing anything."""
    monkeypatch.setattr(ep, "_lib", None)
    monkeypatch.setattr(_build, "LIB", str(tmp_path / "libep.so"))
    with pytest.raises(RuntimeError, match="libep.so not found"):
        ep.load(build_if_missing=False)
