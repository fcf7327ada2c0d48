"""CPU oracle for MoE dispatch / combine -- TEST INFRASTRUCTURE ONLY.

Plain, slow, single-threaded C definitions (ep_oracle.c) wrapped with ctypes
over numpy arrays.  Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg may import this package; the product library
never does, and this package imports nothing from it.

Definitions follow the llm-infra-atlas DeepEP article
(llm-infra-atlas.github.io/moe/06_deepep/): get_dispatch_layout and
notify_dispatch (§2.1), the prefix matrix (§2.3), normal and low-latency
layouts (§1.1, §1.2, §3.2), the EPHandle psum (§4.3); number formats from
the OCP FP8 (E4M3) and bfloat16 definitions.  Every function is pinned by
tests/test_oracle_*.py against things other than itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ep_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libep_oracle.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_CAPACITY = 2

FP8_NONE = 0
FP8_E4M3_F32_SCALE = 1
FP8_E4M3_UE8M0 = 2


def build(force: bool = False) -> str:
    """Compile ep_oracle.c with gcc (no contraction, no fast-math)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib() -> ctypes.CDLL:
    """The oracle library; EP_ORACLE_LIB names another build of it (the
    mutation tests load copies with a planted mistake this way)."""
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(os.environ.get("EP_ORACLE_LIB") or build())
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64


def _declare(L: ctypes.CDLL) -> None:
    L.ep_oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.ep_oracle_bf16_to_f32.restype = ctypes.c_float
    L.ep_oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    L.ep_oracle_f32_to_bf16.restype = ctypes.c_uint16
    L.ep_oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    L.ep_oracle_e4m3_to_f32.restype = ctypes.c_float
    L.ep_oracle_f32_to_e4m3.argtypes = [ctypes.c_float]
    L.ep_oracle_f32_to_e4m3.restype = ctypes.c_uint8
    for name in ("ep_oracle_f32_to_e4m3_batch", "ep_oracle_f32_to_bf16_batch",
                 "ep_oracle_e4m3_to_f32_batch"):
        getattr(L, name).argtypes = [_P, _I64, _P]
        getattr(L, name).restype = None
    L.ep_oracle_quantize_row.argtypes = [_P, _I, _I, _P, _P, _P, _I64]
    L.ep_oracle_quantize_row.restype = None
    L.ep_oracle_layout.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P, _P]
    L.ep_oracle_layout.restype = _I
    L.ep_oracle_notify.argtypes = [_P, _P, _I, _I, _I, _I64, _P, _P, _P, _P]
    L.ep_oracle_notify.restype = _I
    L.ep_oracle_dispatch.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I64,
                                     _P, _P, _P, _P]
    L.ep_oracle_dispatch.restype = _I
    L.ep_oracle_ll_dispatch.argtypes = [_P, _P, _I, _I, _I, _I, _I, _I, _I,
                                        _P, _P, _P, _P, _P, _P]
    L.ep_oracle_ll_dispatch.restype = _I
    L.ep_oracle_combine.argtypes = [_P, _P, _P, _I64, _I64, _I, _I, _P]
    L.ep_oracle_combine.restype = _I
    L.ep_oracle_rank_dispatch.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _I, _I64,
                                          _P, _P, _P, _P, _P, _P]
    L.ep_oracle_rank_dispatch.restype = _I
    L.ep_oracle_rank_combine.argtypes = [_P, _P, _I64, _I64, _I, _I, _P]
    L.ep_oracle_rank_combine.restype = _I
    L.ep_oracle_combine.restype = _I


def _ptr(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


# ---------------------------------------------------------------- formats

def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float32 (exact widening)."""
    return (_c(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(f: np.ndarray) -> np.ndarray:
    f = _c(f, np.float32)
    out = np.empty(f.shape, np.uint16)
    lib().ep_oracle_f32_to_bf16_batch(_ptr(f), f.size, _ptr(out))
    return out


def f32_to_e4m3(f: np.ndarray) -> np.ndarray:
    f = _c(f, np.float32)
    out = np.empty(f.shape, np.uint8)
    lib().ep_oracle_f32_to_e4m3_batch(_ptr(f), f.size, _ptr(out))
    return out


def e4m3_to_f32(b: np.ndarray) -> np.ndarray:
    b = _c(b, np.uint8)
    out = np.empty(b.shape, np.float32)
    lib().ep_oracle_e4m3_to_f32_batch(_ptr(b), b.size, _ptr(out))
    return out


def quantize_row(x_row: np.ndarray, mode: int):
    """One bf16 row [H] -> (E4M3 bytes [H], scales [H/128] fp32 or uint8)."""
    x_row = _c(x_row, np.uint16)
    H = x_row.size
    q = np.empty(H, np.uint8)
    if mode == FP8_E4M3_F32_SCALE:
        s = np.empty(H // 128, np.float32)
        lib().ep_oracle_quantize_row(_ptr(x_row), H, mode, _ptr(q), _ptr(s), None, 1)
    else:
        s = np.empty(H // 128, np.uint8)
        lib().ep_oracle_quantize_row(_ptr(x_row), H, mode, _ptr(q), None, _ptr(s), 1)
    return q, s


# ---------------------------------------------------------------- the path

def layout(topk_idx: np.ndarray, R: int, E: int):
    """topk_idx [R, T_r, k] int64 -> dict of layout arrays (see ep_oracle.c)."""
    idx = _c(topk_idx, np.int64)
    _, T_r, k = idx.shape
    out = dict(
        num_tokens_per_rank=np.zeros((R, R), np.int32),
        num_tokens_per_expert=np.zeros((R, E), np.int32),
        is_token_in_rank=np.zeros((R, T_r, R), np.uint8),
        slot_rank=np.zeros((R, T_r, k), np.int32),
    )
    rc = lib().ep_oracle_layout(_ptr(idx), R, T_r, k, E, _ptr(out["num_tokens_per_rank"]),
                                _ptr(out["num_tokens_per_expert"]), _ptr(out["is_token_in_rank"]),
                                _ptr(out["slot_rank"]))
    out["rc"] = rc
    return out


def notify(num_tokens_per_rank: np.ndarray, num_tokens_per_expert: np.ndarray, R: int, E: int,
           expert_alignment: int = 1, num_worst_tokens: int = -1):
    ntpr = _c(num_tokens_per_rank, np.int32)
    ntpe = _c(num_tokens_per_expert, np.int32)
    E_l = E // R
    out = dict(
        rank_prefix_matrix=np.zeros((R, R), np.int32),
        expert_prefix=np.zeros((R + 1, E), np.int32),
        num_recv_tokens_per_expert=np.zeros((R, E_l), np.int32),
        psum=np.zeros((R, E_l + 1), np.int64),
    )
    rc = lib().ep_oracle_notify(_ptr(ntpr), _ptr(ntpe), R, E, expert_alignment, num_worst_tokens,
                                _ptr(out["rank_prefix_matrix"]), _ptr(out["expert_prefix"]),
                                _ptr(out["num_recv_tokens_per_expert"]), _ptr(out["psum"]))
    out["rc"] = rc
    return out


def _recv_buffers(n_seg: int, seg_rows: int, H: int, fp8_mode: int, fill):
    if fill is None:        # lazily mapped: only rows the oracle writes are touched
        recv = np.empty((n_seg, seg_rows, H), np.uint16 if fp8_mode == FP8_NONE else np.uint8)
        sdt = np.float32 if fp8_mode == FP8_E4M3_F32_SCALE else np.uint8
        scales = None if fp8_mode == FP8_NONE else np.empty((n_seg, H // 128, seg_rows), sdt)
        return recv, scales
    if fp8_mode == FP8_NONE:
        recv = np.full((n_seg, seg_rows, H), fill & 0xFFFF, np.uint16)
        scales = None
    else:
        recv = np.full((n_seg, seg_rows, H), fill & 0xFF, np.uint8)
        sdt = np.float32 if fp8_mode == FP8_E4M3_F32_SCALE else np.uint8
        scales = np.zeros((n_seg, H // 128, seg_rows), sdt)
        scales.view(np.uint8)[...] = fill & 0xFF
    return recv, scales


def dispatch(x: np.ndarray, topk_idx: np.ndarray, slot_rank: np.ndarray,
             expert_prefix: np.ndarray, psum: np.ndarray, E: int, fp8_mode: int,
             cap_rows: int, fill: int = 0):
    """Normal-mode dispatch.  x [R, T_r, H] bf16 bits (uint16)."""
    x = _c(x, np.uint16)
    idx = _c(topk_idx, np.int64)
    R, T_r, H = x.shape
    k = idx.shape[2]
    recv, scales = _recv_buffers(R, cap_rows, H, fp8_mode, fill)
    src = np.zeros((R, cap_rows), np.int32)
    cidx = np.zeros((R, T_r, k), np.int32)
    rc = lib().ep_oracle_dispatch(_ptr(x), _ptr(idx), _ptr(_c(slot_rank, np.int32)),
                                  _ptr(_c(expert_prefix, np.int32)), _ptr(_c(psum, np.int64)),
                                  R, T_r, H, E, k, fp8_mode, cap_rows, _ptr(recv), _ptr(scales),
                                  _ptr(src), _ptr(cidx))
    return dict(rc=rc, recv_x=recv, recv_scales=scales, recv_src_idx=src, combine_idx=cidx)


def ll_dispatch(x: np.ndarray, topk_idx: np.ndarray, E: int, max_tokens_per_rank: int,
                fp8_mode: int, fill: int = 0):
    """Low-latency dispatch into the packed masked layout."""
    x = _c(x, np.uint16)
    idx = _c(topk_idx, np.int64)
    R, T_r, H = x.shape
    k = idx.shape[2]
    E_l = E // R
    seg_rows = R * max_tokens_per_rank
    recv, scales = _recv_buffers(E, seg_rows, H, fp8_mode, fill)
    src = np.full((E, seg_rows), -1, np.int32)
    lrange = np.zeros((E, R), np.int64)
    cnt = np.zeros((E,), np.int32)
    cidx = np.zeros((R, T_r, k), np.int32)
    rc = lib().ep_oracle_ll_dispatch(_ptr(x), _ptr(idx), R, T_r, H, E, k, max_tokens_per_rank,
                                     fp8_mode, _ptr(recv), _ptr(scales), _ptr(src), _ptr(lrange),
                                     _ptr(cnt), _ptr(cidx))
    shape_x = (R, E_l, seg_rows, H)
    out = dict(rc=rc, packed_recv_x=recv.reshape(shape_x),
               packed_recv_src_info=src.reshape(R, E_l, seg_rows),
               layout_range=lrange.reshape(R, E_l, R), recv_count=cnt.reshape(R, E_l),
               combine_idx=cidx)
    out["packed_recv_scales"] = (None if scales is None
                                 else scales.reshape(R, E_l, H // 128, seg_rows))
    return out


def combine(y: np.ndarray, topk_weights: np.ndarray, combine_idx: np.ndarray, H: int):
    """y: bf16 bits viewed [n_rows, H]; weights / combine_idx [..., k]."""
    y = _c(y, np.uint16).reshape(-1, H)
    w = _c(topk_weights, np.float32)
    cidx = _c(combine_idx, np.int32)
    k = cidx.shape[-1]
    n_tokens = cidx.size // k
    out = np.empty(cidx.shape[:-1] + (H,), np.uint16)
    rc = lib().ep_oracle_combine(_ptr(y), _ptr(w), _ptr(cidx), y.shape[0], n_tokens, H, k,
                                 _ptr(out))
    return dict(rc=rc, out=out)


def rank_dispatch(x: np.ndarray, topk_idx: np.ndarray, topk_weights: np.ndarray, E: int,
                  fp8_mode: int, cap_rows: int, fill: int = 0):
    """Once-per-rank receive layout (V1 normal mode).  x [R, T_r, H] bf16
    bits; rows holding no token keep `fill` (recv_topk_* keep -1 / 0)."""
    x = _c(x, np.uint16)
    idx = _c(topk_idx, np.int64)
    w = _c(topk_weights, np.float32)
    R, T_r, H = x.shape
    k = idx.shape[2]
    recv, scales = _recv_buffers(R, cap_rows, H, fp8_mode, fill)
    src = np.zeros((R, cap_rows), np.int32)
    rtk = np.full((R, cap_rows, k), -1, np.int64)
    rtw = np.zeros((R, cap_rows, k), np.float32)
    cidx = np.zeros((R, T_r, k), np.int32)
    rc = lib().ep_oracle_rank_dispatch(_ptr(x), _ptr(idx), _ptr(w), R, T_r, H, E, k, fp8_mode,
                                       cap_rows, _ptr(recv), _ptr(scales), _ptr(src), _ptr(rtk),
                                       _ptr(rtw), _ptr(cidx))
    return dict(rc=rc, recv_x=recv, recv_scales=scales, recv_src_idx=src, recv_topk_idx=rtk,
                recv_topk_weights=rtw, combine_idx=cidx)


def rank_combine(y: np.ndarray, combine_idx: np.ndarray, H: int):
    """Sum over destination ranks of y rows (bf16 bits viewed [n_rows, H])."""
    y = _c(y, np.uint16).reshape(-1, H)
    cidx = _c(combine_idx, np.int32)
    k = cidx.shape[-1]
    n_tokens = cidx.size // k
    out = np.empty(cidx.shape[:-1] + (H,), np.uint16)
    rc = lib().ep_oracle_rank_combine(_ptr(y), _ptr(cidx), y.shape[0], n_tokens, H, k, _ptr(out))
    return dict(rc=rc, out=out)
