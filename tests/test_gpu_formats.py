"""The kernels' two number-format conversions (fp32 -> E4M3 as the FP8
dispatch casts, fp32 -> bf16 as the combine rounds) against the oracle's
encoders, written from the OCP FP8 and bfloat16 definitions.

E4M3: every fp32 bit pattern whose exponent can round to a non-zero finite
E4M3 value or to the saturation boundary (2^-12 <= |x| < 2^10, both signs,
all 2^23 mantissas: 369 M inputs), all fp32 subnormals, and a random sample
elsewhere.  bf16: all 2^16 low halves under every sign and exponent with the
kept mantissa at its edges (0, 1, 0x3F, 0x40, 0x7E, 0x7F; 201 M inputs), and a
random sample.  NaN inputs must give a NaN; everything else bit for bit."""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_gb300 import ep

pytestmark = pytest.mark.gpu

_POOL = cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1)))


def _oracle_parallel(fn, x: np.ndarray) -> np.ndarray:
    """The oracle's batch encoder over slices in threads (the C calls drop
    the interpreter lock)."""
    oracle.lib()   # loaded once, before the threads call into it
    parts = np.array_split(x, 32)
    return np.concatenate(list(_POOL.map(fn, parts)))


def _as_f32(bits_i64: torch.Tensor) -> torch.Tensor:
    """uint32 bit patterns held in int64 -> float32 tensor with those bits."""
    b = torch.where(bits_i64 >= 2 ** 31, bits_i64 - 2 ** 32, bits_i64).to(torch.int32)
    return b.view(torch.float32)


def _check_e4m3(bits: torch.Tensor):
    x = _as_f32(bits)
    got = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    ep.ep_format_e4m3(x, got)
    xh = x.cpu().numpy()
    ref = _oracle_parallel(oracle.f32_to_e4m3, xh)
    g = got.cpu().numpy()
    nan = np.isnan(xh)
    assert np.all((g[nan] & 0x7F) == 0x7F)            # E4M3 NaN (S.1111.111)
    bad = (g != ref) & ~nan
    assert not bad.any(), (f"{int(bad.sum())} mismatches, first input bits "
                           f"{hex(int(xh[bad][:1].view(np.uint32)[0]))}")


def _check_bf16(bits: torch.Tensor):
    x = _as_f32(bits)
    got = torch.empty(x.shape, dtype=torch.int16, device="cuda")
    ep.ep_format_bf16(x, got)
    xh = x.cpu().numpy()
    ref = _oracle_parallel(oracle.f32_to_bf16, xh)
    g = got.cpu().numpy().view(np.uint16)
    nan = np.isnan(xh)
    gn = g[nan]
    assert np.all(((gn & 0x7F80) == 0x7F80) & ((gn & 0x007F) != 0))   # a bf16 NaN
    bad = (g != ref) & ~nan
    assert not bad.any(), (f"{int(bad.sum())} mismatches, first input bits "
                           f"{hex(int(xh[bad][:1].view(np.uint32)[0]))}")


def test_e4m3_every_input_near_its_range():
    man = torch.arange(1 << 23, dtype=torch.int64, device="cuda")
    for exp in range(127 - 12, 127 + 10):
        for sign in (0, 1):
            _check_e4m3((sign << 31) | (exp << 23) | man)


def test_e4m3_subnormals_specials_and_a_sample():
    man = torch.arange(1 << 23, dtype=torch.int64, device="cuda")
    _check_e4m3(torch.cat([man, (1 << 31) | man]))                    # fp32 subnormals, zeros
    nan_inf = torch.cat([(255 << 23) | man[:1 << 16], (1 << 31) | (255 << 23) | man[:1 << 16]])
    _check_e4m3(nan_inf)                                              # inf and NaNs
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    _check_e4m3(torch.randint(0, 1 << 32, (1 << 24,), generator=g, device="cuda",
                              dtype=torch.int64))


def test_bf16_every_low_half_at_the_mantissa_edges():
    low = torch.arange(1 << 16, dtype=torch.int64, device="cuda")
    for m7 in (0x00, 0x01, 0x3F, 0x40, 0x7E, 0x7F):
        hi = torch.tensor([(s << 15) | (e << 7) | m7 for s in (0, 1) for e in range(256)],
                          dtype=torch.int64, device="cuda")
        _check_bf16(((hi[:, None] << 16) | low[None, :]).reshape(-1))


def test_bf16_random_sample():
    g = torch.Generator(device="cuda")
    g.manual_seed(12)
    _check_bf16(torch.randint(0, 1 << 32, (1 << 24,), generator=g, device="cuda",
                              dtype=torch.int64))


def test_format_entry_points_reject_odd_lengths():
    x = torch.zeros(3, dtype=torch.float32, device="cuda")
    with pytest.raises(ep.EPError):
        ep.ep_format_e4m3(x, torch.empty(3, dtype=torch.uint8, device="cuda"))
