"""Seeded synthetic workloads for MoE dispatch / combine.

This module only draws inputs -- token activations x, routing (topk_idx) and
router weights (topk_weights), and stand-in expert outputs -- with the
shapes, sizes and distributions of the workloads the DeepEP article
(llm-infra-atlas.github.io/moe/06_deepep/) discusses: decode batches of a few
hundred tokens per rank, prefill batches of thousands, hidden 7168 with 256
experts and top-8.  It holds none of the dispatch / combine arithmetic; both
the CUDA path and the oracle consume what it returns.

Recipes (seed 0 by default, numpy PCG64 with one spawned stream per tensor):
  * x: N(0, std^2) drawn in fp32, rounded to bf16 (round to nearest even,
    done by torch's dtype conversion); std = 1, or 2 for the skewed workload.
  * "softmax_top": logits ~ N(0,1) [T, E]; the k largest logits (ties to the
    lower id) are the experts, the weights are their softmax probabilities
    over all E experts (not renormalised).
  * "uniform": k distinct experts uniformly at random per token (the k
    smallest of E i.i.d. uniform keys, in key order); weights = softmax of
    k i.i.d. N(0,1) logits.
  * "zipf": expert popularity p_e ~ (e+1)^-s, k experts drawn without
    replacement by sequential renormalised draws (Gumbel top-k on log p);
    weights as for "uniform".
  * expert outputs y: N(0,1) rounded to bf16.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

FP8_NONE = 0
FP8_E4M3_F32_SCALE = 1
FP8_E4M3_UE8M0 = 2


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    R: int            # emulated ranks
    T_r: int          # tokens per rank
    H: int            # hidden size
    E: int            # experts (E / R per rank)
    k: int            # top-k
    routing: str      # "softmax_top" | "uniform" | "zipf"
    mode: str         # "ll" (packed masked) | "normal" (contiguous) | "both"
    fp8_mode: int     # 0 bf16, 1 E4M3 + fp32 scales, 2 E4M3 + ue8m0 scales
    x_std: float = 1.0
    zipf_s: float = 1.2
    max_tokens_per_rank: int = 0     # low-latency capacity per source rank
    num_worst_tokens: int = -1       # fixed-shape normal dispatch (-1 = off)
    expert_alignment: int = 1

    @property
    def E_l(self) -> int:
        return self.E // self.R

    @property
    def T(self) -> int:
        return self.R * self.T_r

    def cap_rows(self) -> int:
        """Per-rank receive rows of the fixed-shape normal layout."""
        assert self.num_worst_tokens >= 0
        return self.num_worst_tokens * min(self.k, self.E_l)


WORKLOADS = {
    "tiny": Workload("tiny", R=4, T_r=16, H=256, E=16, k=2, routing="softmax_top",
                     mode="both", fp8_mode=FP8_NONE, max_tokens_per_rank=16),
    "decode": Workload("decode", R=16, T_r=128, H=7168, E=256, k=8, routing="uniform",
                       mode="ll", fp8_mode=FP8_E4M3_UE8M0, max_tokens_per_rank=128),
    "prefill": Workload("prefill", R=8, T_r=4096, H=7168, E=256, k=8, routing="uniform",
                        mode="normal", fp8_mode=FP8_NONE),
    "skewed": Workload("skewed", R=32, T_r=256, H=4096, E=128, k=6, routing="zipf",
                       mode="normal", fp8_mode=FP8_E4M3_F32_SCALE, x_std=2.0,
                       num_worst_tokens=32 * 256),
    "large": Workload("large", R=8, T_r=16384, H=7168, E=256, k=8, routing="uniform",
                      mode="normal", fp8_mode=FP8_E4M3_UE8M0),
}


def _streams(seed: int, n: int = 4):
    ss = np.random.SeedSequence(seed)
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(n)]


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    p = np.exp(z)
    return p / p.sum(axis=-1, keepdims=True)


def routing(w: Workload, seed: int = 0):
    """Return (topk_idx int64 [R, T_r, k], topk_weights float32 [R, T_r, k])."""
    _, rng_route, rng_w, _ = _streams(seed)
    T, E, k = w.T, w.E, w.k
    if w.routing == "softmax_top":
        logits = rng_route.standard_normal((T, E))
        order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
        probs = _softmax_rows(logits)
        idx = order
        wts = np.take_along_axis(probs, order, axis=1)
    elif w.routing in ("uniform", "zipf"):
        if w.routing == "uniform":
            keys = rng_route.random((T, E), dtype=np.float32)
        else:
            logp = -w.zipf_s * np.log(np.arange(1, E + 1, dtype=np.float64))
            gumbel = -np.log(-np.log(rng_route.random((T, E))))
            keys = -(logp[None, :] + gumbel)
        part = np.argpartition(keys, k - 1, axis=1)[:, :k]
        pk = np.take_along_axis(keys, part, axis=1)
        idx = np.take_along_axis(part, np.argsort(pk, axis=1, kind="stable"), axis=1)
        wts = _softmax_rows(rng_w.standard_normal((T, k)))
    else:
        raise ValueError(w.routing)
    return (idx.astype(np.int64).reshape(w.R, w.T_r, k),
            wts.astype(np.float32).reshape(w.R, w.T_r, k))


def to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even (torch)."""
    t = torch.from_numpy(np.ascontiguousarray(f, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def activations(w: Workload, seed: int = 0) -> np.ndarray:
    """x as bf16 bit patterns [R, T_r, H] (uint16)."""
    rng_x = _streams(seed)[0]
    f = rng_x.standard_normal((w.R, w.T_r, w.H), dtype=np.float32) * np.float32(w.x_std)
    return to_bf16_bits(f)


def activations_torch(w: Workload, device, seed: int = 0) -> torch.Tensor:
    """x [R, T_r, H] bf16 drawn directly on `device` (for sizes where a host
    draw is slow); a different stream from activations(), same recipe."""
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + 17)
    f = torch.randn((w.R, w.T_r, w.H), generator=g, device=device, dtype=torch.float32)
    return (f * w.x_std).to(torch.bfloat16)


def expert_outputs_torch(n_rows: int, H: int, device, seed: int = 0) -> torch.Tensor:
    """Stand-in expert outputs y [n_rows, H] bf16 ~ N(0,1) on `device`."""
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + 29)
    return torch.randn((n_rows, H), generator=g, device=device, dtype=torch.bfloat16)


def expert_outputs(n_rows: int, H: int, seed: int = 0) -> np.ndarray:
    """Stand-in expert outputs y [n_rows, H] as bf16 bits ~ N(0,1) (host)."""
    rng_y = _streams(seed)[3]
    return to_bf16_bits(rng_y.standard_normal((n_rows, H), dtype=np.float32))


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (tests use small T_r)."""
    return dataclasses.replace(w, **changes)
