"""Thin ctypes binding of libep (include/ep.h): argument marshalling only.

Every function below has the name of the C entry point it calls and takes
torch tensors that already live on the GPU; it checks dtype / shape /
contiguity, passes raw pointers and the current CUDA stream, and raises
EPError on a non-zero return code.  Every step of the path runs in libep's
CUDA kernels: there is no CPU or PyTorch fallback, and importing this
module on a machine without the built library raises.

The alloc_* helpers only create output tensors of the documented shapes
(torch is the memory owner); they do no compute.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

EP_OK = 0
EP_ERR_INVALID_ARG = 1
EP_ERR_CAPACITY = 2
EP_ERR_TIMEOUT = 3
EP_ERR_CUDA = 4
EP_ERR_STATE = 5
EP_ERR_TOO_LARGE = 6

EP_FP8_NONE = 0
EP_FP8_E4M3_F32_SCALE = 1
EP_FP8_E4M3_UE8M0 = 2

EXPORTS = (
    "ep_workspace_size", "ep_get_dispatch_layout", "ep_notify_dispatch", "ep_dispatch",
    "ep_combine", "ep_ll_dispatch", "ep_ll_combine", "ep_clean_ll_buffer", "ep_read_status",
    "ep_host_wait_counters", "ep_launch_count", "ep_error_string", "ep_rank_ids",
    "ep_rank_recv_topk", "ep_rank_combine", "ep_set_num_sms", "ep_get_num_sms",
    "ep_format_e4m3", "ep_format_bf16", "ep_layout_notify", "ep_layout_notify_dispatch",
)


class EPError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {error_string(code)} (code {code})")


_lib = None
_P, _I, _I64, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libep.so (building it with nvcc first if it is missing/stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        _build.build()
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"libep.so not found at {_build.LIB}; build it with __graft_entry__.build()")
    L = ctypes.CDLL(_build.LIB)
    L.ep_workspace_size.argtypes = [_I, _I, _I, _I, _I]
    L.ep_workspace_size.restype = _SZ
    L.ep_get_dispatch_layout.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P, _P]
    L.ep_notify_dispatch.argtypes = [_P, _P, _I, _I, _I, _I64, _P, _P, _P, _P, _P, _I, _P, _P]
    L.ep_dispatch.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I64, _P, _P, _P, _P,
                              _P, _SZ, _P, _P]
    L.ep_combine.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I64, _P, _P, _P]
    L.ep_ll_dispatch.argtypes = [_P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                 _SZ, _P, _P]
    L.ep_ll_combine.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P]
    L.ep_clean_ll_buffer.argtypes = [_P, _I, _I, _P, _SZ, _P]
    L.ep_rank_ids.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P]
    L.ep_rank_recv_topk.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I64, _P, _P, _P, _P]
    L.ep_rank_combine.argtypes = [_P, _P, _I, _I, _I, _I, _I64, _P, _P, _P]
    L.ep_read_status.argtypes = [_P, _P, _P]
    L.ep_host_wait_counters.argtypes = [_P, _I, _I]
    L.ep_layout_notify.argtypes = [_P, _I, _I, _I, _I, _I, _I64, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _P, _I, _P, _SZ, _P, _P]
    L.ep_layout_notify.restype = _I
    L.ep_layout_notify_dispatch.argtypes = [_P, _P, _I, _I, _I, _I, _I, _I, _I, _I64, _I64, _P, _P,
                                            _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P,
                                            _P]
    L.ep_layout_notify_dispatch.restype = _I
    L.ep_format_e4m3.argtypes = [_P, _P, _I64, _P]
    L.ep_format_e4m3.restype = _I
    L.ep_format_bf16.argtypes = [_P, _P, _I64, _P]
    L.ep_format_bf16.restype = _I
    L.ep_set_num_sms.argtypes = [_I]
    L.ep_set_num_sms.restype = _I
    L.ep_get_num_sms.argtypes = []
    L.ep_get_num_sms.restype = _I
    L.ep_launch_count.argtypes = []
    L.ep_launch_count.restype = ctypes.c_uint64
    L.ep_error_string.argtypes = [_I]
    L.ep_error_string.restype = ctypes.c_char_p
    for name in ("ep_get_dispatch_layout", "ep_notify_dispatch", "ep_dispatch", "ep_combine",
                 "ep_ll_dispatch", "ep_ll_combine", "ep_clean_ll_buffer", "ep_read_status",
                 "ep_host_wait_counters", "ep_rank_ids", "ep_rank_recv_topk", "ep_rank_combine"):
        getattr(L, name).restype = _I
    _lib = L
    return L


def error_string(code: int) -> str:
    return load().ep_error_string(int(code)).decode()


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor | None, dtype, shape=None, name="tensor", optional=False):
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _need_out(t: torch.Tensor, dtype, shape, name="out"):
    """A combine's output: a CUDA tensor, or a pinned host tensor that the
    kernel writes across the host link."""
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _check(rc: int, where: str):
    if rc != EP_OK:
        raise EPError(rc, where)


def _scale_dtype(fp8_mode: int):
    return torch.float32 if fp8_mode == EP_FP8_E4M3_F32_SCALE else torch.uint8


# ------------------------------------------------------------------ entry points

def ep_workspace_size(R: int, T_r: int, k: int, E: int, H: int) -> int:
    return int(load().ep_workspace_size(R, T_r, k, E, H))


def ep_get_dispatch_layout(topk_idx, num_experts, num_tokens_per_rank, num_tokens_per_expert,
                           is_token_in_rank, slot_rank, workspace, status=None, stream=None):
    R, T_r, k = topk_idx.shape
    E = num_experts
    _need(topk_idx, torch.int64, name="topk_idx")
    _need(num_tokens_per_rank, torch.int32, (R, R), "num_tokens_per_rank")
    _need(num_tokens_per_expert, torch.int32, (R, E), "num_tokens_per_expert")
    _need(is_token_in_rank, torch.uint8, (R, T_r, R), "is_token_in_rank")
    _need(slot_rank, torch.int32, (R, T_r, k), "slot_rank")
    _need(workspace, torch.uint8, name="workspace")
    _need(status, torch.int32, (1,), "status", optional=True)
    rc = load().ep_get_dispatch_layout(_ptr(topk_idx), R, T_r, k, E, _ptr(num_tokens_per_rank),
                                       _ptr(num_tokens_per_expert), _ptr(is_token_in_rank),
                                       _ptr(slot_rank), _ptr(workspace), workspace.numel(),
                                       _ptr(status), _stream(stream))
    _check(rc, "ep_get_dispatch_layout")


def ep_notify_dispatch(num_tokens_per_rank, num_tokens_per_expert, expert_alignment,
                       num_worst_tokens, rank_prefix_matrix, expert_prefix,
                       num_recv_tokens_per_expert, psum, host_recv_rows=None, timeout_ms=10000,
                       status=None, stream=None):
    R, E = num_tokens_per_expert.shape
    E_l = E // R
    _need(num_tokens_per_rank, torch.int32, (R, R), "num_tokens_per_rank")
    _need(num_tokens_per_expert, torch.int32, (R, E), "num_tokens_per_expert")
    _need(rank_prefix_matrix, torch.int32, (R, R), "rank_prefix_matrix")
    _need(expert_prefix, torch.int32, (R + 1, E), "expert_prefix")
    _need(num_recv_tokens_per_expert, torch.int32, (R, E_l), "num_recv_tokens_per_expert")
    _need(psum, torch.int64, (R, E_l + 1), "psum")
    _need(status, torch.int32, (1,), "status", optional=True)
    if host_recv_rows is not None:
        if host_recv_rows.is_cuda or not host_recv_rows.is_pinned() or \
                host_recv_rows.dtype != torch.int64 or host_recv_rows.numel() < R:
            raise ValueError("host_recv_rows must be a pinned host int64 tensor of >= R entries")
    rc = load().ep_notify_dispatch(_ptr(num_tokens_per_rank), _ptr(num_tokens_per_expert), R, E,
                                   expert_alignment, num_worst_tokens, _ptr(rank_prefix_matrix),
                                   _ptr(expert_prefix), _ptr(num_recv_tokens_per_expert),
                                   _ptr(psum), _ptr(host_recv_rows), timeout_ms, _ptr(status),
                                   _stream(stream))
    _check(rc, "ep_notify_dispatch")


def ep_layout_notify(topk_idx, num_experts, expert_alignment, num_worst_tokens, lay, nt,
                     workspace, host_recv_rows=None, timeout_ms=10000, status=None, stream=None):
    """ep_get_dispatch_layout + ep_notify_dispatch in one launch; `lay` and
    `nt` are the dicts of alloc_layout / alloc_notify."""
    R, T_r, k = topk_idx.shape
    E = num_experts
    E_l = E // R
    _need(topk_idx, torch.int64, name="topk_idx")
    _need(lay["num_tokens_per_rank"], torch.int32, (R, R), "num_tokens_per_rank")
    _need(lay["num_tokens_per_expert"], torch.int32, (R, E), "num_tokens_per_expert")
    _need(lay["is_token_in_rank"], torch.uint8, (R, T_r, R), "is_token_in_rank")
    _need(lay["slot_rank"], torch.int32, (R, T_r, k), "slot_rank")
    _need(nt["rank_prefix_matrix"], torch.int32, (R, R), "rank_prefix_matrix")
    _need(nt["expert_prefix"], torch.int32, (R + 1, E), "expert_prefix")
    _need(nt["num_recv_tokens_per_expert"], torch.int32, (R, E_l), "num_recv_tokens_per_expert")
    _need(nt["psum"], torch.int64, (R, E_l + 1), "psum")
    _need(workspace, torch.uint8, name="workspace")
    _need(status, torch.int32, (1,), "status", optional=True)
    if host_recv_rows is not None:
        if host_recv_rows.is_cuda or not host_recv_rows.is_pinned() or \
                host_recv_rows.dtype != torch.int64 or host_recv_rows.numel() < R:
            raise ValueError("host_recv_rows must be a pinned host int64 tensor of >= R entries")
    rc = load().ep_layout_notify(_ptr(topk_idx), R, T_r, k, E, expert_alignment, num_worst_tokens,
                                 _ptr(lay["num_tokens_per_rank"]), _ptr(lay["num_tokens_per_expert"]),
                                 _ptr(lay["is_token_in_rank"]), _ptr(lay["slot_rank"]),
                                 _ptr(nt["rank_prefix_matrix"]), _ptr(nt["expert_prefix"]),
                                 _ptr(nt["num_recv_tokens_per_expert"]), _ptr(nt["psum"]),
                                 _ptr(host_recv_rows), timeout_ms, _ptr(workspace),
                                 workspace.numel(), _ptr(status), _stream(stream))
    _check(rc, "ep_layout_notify")


def ep_layout_notify_dispatch(x, topk_idx, num_experts, fp8_mode, expert_alignment,
                              num_worst_tokens, cap_rows, lay, nt, d, workspace, status=None,
                              stream=None):
    """Fixed-shape normal mode in one call: layout + notify (one launch),
    then the dispatch as its programmatic dependent.  `lay`, `nt`, `d` are
    the dicts of alloc_layout / alloc_notify / alloc_dispatch."""
    R, T_r, H = x.shape
    k = topk_idx.shape[2]
    E = num_experts
    E_l = E // R
    _need(x, torch.bfloat16, (R, T_r, H), "x")
    _need(topk_idx, torch.int64, (R, T_r, k), "topk_idx")
    for key, dt, shape in (("num_tokens_per_rank", torch.int32, (R, R)),
                           ("num_tokens_per_expert", torch.int32, (R, E)),
                           ("is_token_in_rank", torch.uint8, (R, T_r, R)),
                           ("slot_rank", torch.int32, (R, T_r, k))):
        _need(lay[key], dt, shape, key)
    for key, dt, shape in (("rank_prefix_matrix", torch.int32, (R, R)),
                           ("expert_prefix", torch.int32, (R + 1, E)),
                           ("num_recv_tokens_per_expert", torch.int32, (R, E_l)),
                           ("psum", torch.int64, (R, E_l + 1))):
        _need(nt[key], dt, shape, key)
    rdt = torch.bfloat16 if fp8_mode == EP_FP8_NONE else torch.uint8
    _need(d["recv_x"], rdt, (R, cap_rows, H), "recv_x")
    if fp8_mode != EP_FP8_NONE:
        _need(d["recv_scales"], _scale_dtype(fp8_mode), (R, H // 128, cap_rows), "recv_scales")
    _need(d["recv_src_idx"], torch.int32, (R, cap_rows), "recv_src_idx")
    _need(d["combine_idx"], torch.int32, (R, T_r, k), "combine_idx")
    _need(workspace, torch.uint8, name="workspace")
    _need(status, torch.int32, (1,), "status", optional=True)
    rc = load().ep_layout_notify_dispatch(
        _ptr(x), _ptr(topk_idx), R, T_r, H, E, k, fp8_mode, expert_alignment, num_worst_tokens,
        cap_rows, _ptr(lay["num_tokens_per_rank"]), _ptr(lay["num_tokens_per_expert"]),
        _ptr(lay["is_token_in_rank"]), _ptr(lay["slot_rank"]), _ptr(nt["rank_prefix_matrix"]),
        _ptr(nt["expert_prefix"]), _ptr(nt["num_recv_tokens_per_expert"]), _ptr(nt["psum"]),
        _ptr(d["recv_x"]), _ptr(d["recv_scales"]) if fp8_mode != EP_FP8_NONE else None,
        _ptr(d["recv_src_idx"]), _ptr(d["combine_idx"]), _ptr(workspace), workspace.numel(),
        _ptr(status), _stream(stream))
    _check(rc, "ep_layout_notify_dispatch")


def ep_dispatch(x, topk_idx, slot_rank, expert_prefix, psum, num_experts, fp8_mode, cap_rows,
                recv_x, recv_scales, recv_src_idx, combine_idx, workspace=None, status=None,
                stream=None):
    R, T_r, H = x.shape
    k = topk_idx.shape[2]
    E = num_experts
    E_l = E // R
    _need(x, torch.bfloat16, (R, T_r, H), "x")
    _need(topk_idx, torch.int64, (R, T_r, k), "topk_idx")
    _need(slot_rank, torch.int32, (R, T_r, k), "slot_rank")
    _need(expert_prefix, torch.int32, (R + 1, E), "expert_prefix")
    _need(psum, torch.int64, (R, E_l + 1), "psum")
    rdt = torch.bfloat16 if fp8_mode == EP_FP8_NONE else torch.uint8
    _need(recv_x, rdt, (R, cap_rows, H), "recv_x")
    if fp8_mode != EP_FP8_NONE:
        _need(recv_scales, _scale_dtype(fp8_mode), (R, H // 128, cap_rows), "recv_scales")
    _need(recv_src_idx, torch.int32, (R, cap_rows), "recv_src_idx")
    _need(combine_idx, torch.int32, (R, T_r, k), "combine_idx")
    _need(workspace, torch.uint8, name="workspace", optional=fp8_mode == EP_FP8_NONE)
    _need(status, torch.int32, (1,), "status", optional=True)
    rc = load().ep_dispatch(_ptr(x), _ptr(topk_idx), _ptr(slot_rank), _ptr(expert_prefix),
                            _ptr(psum), R, T_r, H, E, k, fp8_mode, cap_rows, _ptr(recv_x),
                            _ptr(recv_scales) if fp8_mode != EP_FP8_NONE else None,
                            _ptr(recv_src_idx), _ptr(combine_idx), _ptr(workspace),
                            0 if workspace is None else workspace.numel(), _ptr(status),
                            _stream(stream))
    _check(rc, "ep_dispatch")


def ep_combine(y, topk_weights, combine_idx, cap_rows, out, status=None, stream=None):
    R, T_r, k = combine_idx.shape
    H = out.shape[2]
    _need(y, torch.bfloat16, (R, cap_rows, H), "y")
    _need(topk_weights, torch.float32, (R, T_r, k), "topk_weights")
    _need(combine_idx, torch.int32, (R, T_r, k), "combine_idx")
    _need_out(out, torch.bfloat16, (R, T_r, H))
    _need(status, torch.int32, (1,), "status", optional=True)
    rc = load().ep_combine(_ptr(y), _ptr(topk_weights), _ptr(combine_idx), R, T_r, H, k, cap_rows,
                           _ptr(out), _ptr(status), _stream(stream))
    _check(rc, "ep_combine")


def ep_ll_dispatch(x, topk_idx, num_experts, max_tokens_per_rank, fp8_mode, packed_recv_x,
                   packed_recv_scales, packed_recv_src_info, layout_range, recv_count, combine_idx,
                   workspace, status=None, stream=None):
    R, T_r, H = x.shape
    k = topk_idx.shape[2]
    E = num_experts
    E_l = E // R
    S = R * max_tokens_per_rank
    _need(x, torch.bfloat16, (R, T_r, H), "x")
    _need(topk_idx, torch.int64, (R, T_r, k), "topk_idx")
    rdt = torch.bfloat16 if fp8_mode == EP_FP8_NONE else torch.uint8
    _need(packed_recv_x, rdt, (R, E_l, S, H), "packed_recv_x")
    if fp8_mode != EP_FP8_NONE:
        _need(packed_recv_scales, _scale_dtype(fp8_mode), (R, E_l, H // 128, S),
              "packed_recv_scales")
    _need(packed_recv_src_info, torch.int32, (R, E_l, S), "packed_recv_src_info")
    _need(layout_range, torch.int64, (R, E_l, R), "layout_range")
    _need(recv_count, torch.int32, (R, E_l), "recv_count")
    _need(combine_idx, torch.int32, (R, T_r, k), "combine_idx")
    _need(workspace, torch.uint8, name="workspace")
    _need(status, torch.int32, (1,), "status", optional=True)
    rc = load().ep_ll_dispatch(_ptr(x), _ptr(topk_idx), R, T_r, H, E, k, max_tokens_per_rank,
                               fp8_mode, _ptr(packed_recv_x),
                               _ptr(packed_recv_scales) if fp8_mode != EP_FP8_NONE else None,
                               _ptr(packed_recv_src_info), _ptr(layout_range), _ptr(recv_count),
                               _ptr(combine_idx), _ptr(workspace), workspace.numel(),
                               _ptr(status), _stream(stream))
    _check(rc, "ep_ll_dispatch")


def ep_ll_combine(y, topk_weights, combine_idx, num_experts, max_tokens_per_rank, out,
                  status=None, stream=None):
    R, T_r, k = combine_idx.shape
    H = out.shape[2]
    E = num_experts
    E_l = E // R
    _need(y, torch.bfloat16, (R, E_l, R * max_tokens_per_rank, H), "y")
    _need(topk_weights, torch.float32, (R, T_r, k), "topk_weights")
    _need(combine_idx, torch.int32, (R, T_r, k), "combine_idx")
    _need_out(out, torch.bfloat16, (R, T_r, H))
    _need(status, torch.int32, (1,), "status", optional=True)
    rc = load().ep_ll_combine(_ptr(y), _ptr(topk_weights), _ptr(combine_idx), R, T_r, H, E, k,
                              max_tokens_per_rank, _ptr(out), _ptr(status), _stream(stream))
    _check(rc, "ep_ll_combine")


def ep_clean_ll_buffer(recv_count, num_ranks, num_experts, workspace, stream=None):
    _need(recv_count, torch.int32, name="recv_count", optional=True)
    _need(workspace, torch.uint8, name="workspace", optional=True)
    rc = load().ep_clean_ll_buffer(_ptr(recv_count), num_ranks, num_experts, _ptr(workspace),
                                   0 if workspace is None else workspace.numel(), _stream(stream))
    _check(rc, "ep_clean_ll_buffer")


def ep_rank_ids(topk_idx, num_experts, rank_ids, status=None, stream=None):
    R, T_r, k = topk_idx.shape
    _need(topk_idx, torch.int64, name="topk_idx")
    _need(rank_ids, torch.int64, (R, T_r, k), "rank_ids")
    _need(status, torch.int32, (1,), "status", optional=True)
    rc = load().ep_rank_ids(_ptr(topk_idx), R, T_r, k, num_experts, _ptr(rank_ids), _ptr(status),
                            _stream(stream))
    _check(rc, "ep_rank_ids")


def ep_rank_recv_topk(topk_idx, topk_weights, combine_idx, num_experts, cap_rows, recv_topk_idx,
                      recv_topk_weights, status=None, stream=None):
    R, T_r, k = topk_idx.shape
    _need(topk_idx, torch.int64, name="topk_idx")
    _need(topk_weights, torch.float32, (R, T_r, k), "topk_weights")
    _need(combine_idx, torch.int32, (R, T_r, k), "combine_idx")
    _need(recv_topk_idx, torch.int64, (R, cap_rows, k), "recv_topk_idx")
    _need(recv_topk_weights, torch.float32, (R, cap_rows, k), "recv_topk_weights")
    _need(status, torch.int32, (1,), "status", optional=True)
    rc = load().ep_rank_recv_topk(_ptr(topk_idx), _ptr(topk_weights), _ptr(combine_idx), R, T_r,
                                  k, num_experts, cap_rows, _ptr(recv_topk_idx),
                                  _ptr(recv_topk_weights), _ptr(status), _stream(stream))
    _check(rc, "ep_rank_recv_topk")


def ep_rank_combine(y, combine_idx, cap_rows, out, status=None, stream=None):
    R, T_r, k = combine_idx.shape
    H = out.shape[2]
    _need(y, torch.bfloat16, (R, cap_rows, H), "y")
    _need(combine_idx, torch.int32, (R, T_r, k), "combine_idx")
    _need_out(out, torch.bfloat16, (R, T_r, H))
    _need(status, torch.int32, (1,), "status", optional=True)
    rc = load().ep_rank_combine(_ptr(y), _ptr(combine_idx), R, T_r, H, k, cap_rows, _ptr(out),
                                _ptr(status), _stream(stream))
    _check(rc, "ep_rank_combine")


def ep_read_status(status, stream=None) -> int:
    _need(status, torch.int32, (1,), "status")
    v = ctypes.c_int32(0)
    rc = load().ep_read_status(_ptr(status), ctypes.byref(v), _stream(stream))
    _check(rc, "ep_read_status")
    return int(v.value)


def ep_host_wait_counters(counters: torch.Tensor, timeout_ms: int) -> int:
    """Bounded host wait on host int64 counters (returns the EP code)."""
    if counters.is_cuda or counters.dtype != torch.int64 or not counters.is_contiguous():
        raise ValueError("counters must be a contiguous host int64 tensor")
    return int(load().ep_host_wait_counters(_ptr(counters), counters.numel(), timeout_ms))


def ep_format_e4m3(x, out, stream=None):
    """fp32 -> E4M3 bytes as the FP8 dispatch casts (x float32, out uint8)."""
    _need(x, torch.float32, name="x")
    _need(out, torch.uint8, tuple(x.shape), "out")
    _check(load().ep_format_e4m3(_ptr(x), _ptr(out), x.numel(), _stream(stream)), "ep_format_e4m3")


def ep_format_bf16(x, out, stream=None):
    """fp32 -> bf16 as the combine rounds (x float32, out bfloat16 or int16)."""
    _need(x, torch.float32, name="x")
    if out.dtype not in (torch.bfloat16, torch.int16):
        raise ValueError("out must be bfloat16 or int16")
    _need(out, None, tuple(x.shape), "out")
    _check(load().ep_format_bf16(_ptr(x), _ptr(out), x.numel(), _stream(stream)), "ep_format_bf16")


def ep_set_num_sms(num_sms: int) -> None:
    """SM budget of the data kernels (0: every SM)."""
    _check(load().ep_set_num_sms(int(num_sms)), "ep_set_num_sms")


def ep_get_num_sms() -> int:
    return int(load().ep_get_num_sms())


def ep_launch_count() -> int:
    return int(load().ep_launch_count())


# ------------------------------------------------------------------ allocation helpers

def alloc_layout(R: int, T_r: int, k: int, E: int, device="cuda"):
    i32 = dict(dtype=torch.int32, device=device)
    return dict(
        num_tokens_per_rank=torch.empty((R, R), **i32),
        num_tokens_per_expert=torch.empty((R, E), **i32),
        is_token_in_rank=torch.empty((R, T_r, R), dtype=torch.uint8, device=device),
        slot_rank=torch.empty((R, T_r, k), **i32),
    )


def alloc_notify(R: int, E: int, device="cuda"):
    i32 = dict(dtype=torch.int32, device=device)
    return dict(
        rank_prefix_matrix=torch.empty((R, R), **i32),
        expert_prefix=torch.empty((R + 1, E), **i32),
        num_recv_tokens_per_expert=torch.empty((R, E // R), **i32),
        psum=torch.empty((R, E // R + 1), dtype=torch.int64, device=device),
    )


def alloc_dispatch(R: int, T_r: int, H: int, k: int, fp8_mode: int, cap_rows: int, device="cuda"):
    rdt = torch.bfloat16 if fp8_mode == EP_FP8_NONE else torch.uint8
    return dict(
        recv_x=torch.empty((R, cap_rows, H), dtype=rdt, device=device),
        recv_scales=(None if fp8_mode == EP_FP8_NONE else
                     torch.empty((R, H // 128, cap_rows), dtype=_scale_dtype(fp8_mode),
                                 device=device)),
        recv_src_idx=torch.empty((R, cap_rows), dtype=torch.int32, device=device),
        combine_idx=torch.empty((R, T_r, k), dtype=torch.int32, device=device),
    )


def alloc_ll(R: int, T_r: int, H: int, E: int, k: int, max_tokens_per_rank: int, fp8_mode: int,
             device="cuda"):
    E_l = E // R
    S = R * max_tokens_per_rank
    rdt = torch.bfloat16 if fp8_mode == EP_FP8_NONE else torch.uint8
    return dict(
        packed_recv_x=torch.empty((R, E_l, S, H), dtype=rdt, device=device),
        packed_recv_scales=(None if fp8_mode == EP_FP8_NONE else
                            torch.empty((R, E_l, H // 128, S), dtype=_scale_dtype(fp8_mode),
                                        device=device)),
        packed_recv_src_info=torch.empty((R, E_l, S), dtype=torch.int32, device=device),
        layout_range=torch.empty((R, E_l, R), dtype=torch.int64, device=device),
        recv_count=torch.zeros((R, E_l), dtype=torch.int32, device=device),
        combine_idx=torch.empty((R, T_r, k), dtype=torch.int32, device=device),
    )


def alloc_workspace(R: int, T_r: int, k: int, E: int, H: int, device="cuda", stream=None):
    """Workspace for layout and dispatch (ep_workspace_size), cleaned and ready."""
    ws = torch.empty((ep_workspace_size(R, T_r, k, E, H),), dtype=torch.uint8, device=device)
    ep_clean_ll_buffer(None, R, E, ws, stream=stream)
    return ws


class LowLatencyBuffers:
    """The low-latency mode's two receive buffers (DeepEP's LL buffer holds
    the results of at most two low-latency calls at once): two sets of
    alloc_ll outputs, each with its own workspace, handed out in turn, so
    the received data of call i stays valid while call i+1 dispatches into
    the other set; call i+2 reuses the first.  Allocation only: the calls
    themselves are the ep_ll_* entry points, issued in stream order (the
    single-launch dispatch needs every SM, so two of them must not run
    concurrently on different streams)."""

    def __init__(self, R: int, T_r: int, H: int, E: int, k: int, max_tokens_per_rank: int,
                 fp8_mode: int, device="cuda", stream=None):
        self.sets = []
        for _ in range(2):
            b = alloc_ll(R, T_r, H, E, k, max_tokens_per_rank, fp8_mode, device=device)
            b["workspace"] = alloc_workspace(R, T_r, k, E, H, device=device, stream=stream)
            self.sets.append(b)
        self._turn = 0

    def next(self) -> dict:
        """The set for the next call (alternates 0, 1, 0, ...)."""
        b = self.sets[self._turn]
        self._turn ^= 1
        return b
