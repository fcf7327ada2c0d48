"""Shared plumbing for the GPU parity tests: run a workload through libep
(the CUDA path, via the ctypes binding) and through the oracle (CPU), on the
same seeded inputs.  Nothing here computes any part of the method."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from combine_get_dispatch_gb300 import ep, synth

POISON = 0x5A


def bits_u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns on the host."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def inputs(w: synth.Workload, seed=0, device="cuda", x_on_device=False):
    """(x_dev bf16, x_host uint16 bits, idx_dev, idx_host, wts_dev, wts_host)."""
    idx, wts = synth.routing(w, seed)
    if x_on_device:
        x_dev = synth.activations_torch(w, device, seed)
        x_host = bits_u16(x_dev)
    else:
        x_host = synth.activations(w, seed)
        x_dev = to_dev_bf16(x_host, device)
    return (x_dev, x_host, torch.from_numpy(idx).to(device), idx,
            torch.from_numpy(wts).to(device), wts)


def status_word(device="cuda"):
    return torch.zeros((1,), dtype=torch.int32, device=device)


def poison_(t: torch.Tensor):
    if t is not None:
        t.view(torch.uint8).fill_(POISON)
    return t


def gpu_layout(idx_dev: torch.Tensor, E: int, ws=None, status=None):
    R, T_r, k = idx_dev.shape
    out = ep.alloc_layout(R, T_r, k, E)
    for v in out.values():
        poison_(v)
    ws = ws if ws is not None else ep.alloc_workspace(R, T_r, k, E, 8)
    status = status if status is not None else status_word()
    ep.ep_get_dispatch_layout(idx_dev, E, out["num_tokens_per_rank"], out["num_tokens_per_expert"],
                              out["is_token_in_rank"], out["slot_rank"], ws, status)
    out["status"] = status
    out["ws"] = ws
    return out


def gpu_notify(lay: dict, E: int, A: int = 1, num_worst_tokens: int = -1, host_rows=None,
               status=None):
    R = lay["num_tokens_per_rank"].shape[0]
    out = ep.alloc_notify(R, E)
    for v in out.values():
        poison_(v)
    status = status if status is not None else status_word()
    ep.ep_notify_dispatch(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"], A,
                          num_worst_tokens, out["rank_prefix_matrix"], out["expert_prefix"],
                          out["num_recv_tokens_per_expert"], out["psum"], host_rows, 10000, status)
    out["status"] = status
    return out


def gpu_dispatch(x_dev, idx_dev, lay, nt, E, fp8_mode, cap_rows, status=None, ws=None):
    R, T_r, H = x_dev.shape
    k = idx_dev.shape[2]
    out = ep.alloc_dispatch(R, T_r, H, k, fp8_mode, cap_rows)
    for v in out.values():
        poison_(v)
    status = status if status is not None else status_word()
    ws = ws if ws is not None else ep.alloc_workspace(R, T_r, k, E, H)
    ep.ep_dispatch(x_dev, idx_dev, lay["slot_rank"], nt["expert_prefix"], nt["psum"], E, fp8_mode,
                   cap_rows, out["recv_x"], out["recv_scales"], out["recv_src_idx"],
                   out["combine_idx"], ws, status)
    out["status"] = status
    return out


def gpu_ll_dispatch(x_dev, idx_dev, E, max_tokens, fp8_mode, ws=None, status=None):
    R, T_r, H = x_dev.shape
    k = idx_dev.shape[2]
    out = ep.alloc_ll(R, T_r, H, E, k, max_tokens, fp8_mode)
    for key, v in out.items():
        if key != "recv_count":
            poison_(v)
    ws = ws if ws is not None else ep.alloc_workspace(R, T_r, k, E, H)
    status = status if status is not None else status_word()
    ep.ep_ll_dispatch(x_dev, idx_dev, E, max_tokens, fp8_mode, out["packed_recv_x"],
                      out["packed_recv_scales"], out["packed_recv_src_info"], out["layout_range"],
                      out["recv_count"], out["combine_idx"], ws, status)
    out["status"] = status
    out["ws"] = ws
    return out


def oracle_normal(x_host, idx, E, A, fp8_mode, cap_rows=None, num_worst_tokens=-1):
    R = x_host.shape[0]
    lay = oracle.layout(idx, R, E)
    nt = oracle.notify(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"], R, E, A,
                       num_worst_tokens)
    if cap_rows is None:
        cap_rows = max(1, int(nt["psum"][:, -1].max()))
    d = oracle.dispatch(x_host, idx, lay["slot_rank"], nt["expert_prefix"], nt["psum"], E,
                        fp8_mode, cap_rows)
    return lay, nt, d, cap_rows


def valid_rows(src_idx: np.ndarray) -> np.ndarray:
    """Flat row numbers holding a token (recv_src_idx >= 0)."""
    return np.nonzero(src_idx.reshape(-1) >= 0)[0]


def np_(t):
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return bits_u16(t)
    return t.detach().cpu().numpy()
