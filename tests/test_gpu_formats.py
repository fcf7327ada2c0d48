"""The kernels' two number-format conversions (fp32 -> E4M3 as the FP8
dispatch casts, fp32 -> bf16 as the combine rounds) against the oracle's
encoders, written from the OCP FP8 and bfloat16 definitions.

Both conversions are checked on every one of the 2^32 fp32 bit patterns
(in chunks of 2^26, the oracle's encoder run over host threads).  NaN
inputs must give a NaN; everything else bit for bit."""
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


_CHUNK = 1 << 26


@pytest.mark.slow
def test_e4m3_every_fp32_bit_pattern():
    """All 2^32 inputs: zeros, subnormals, every exponent and mantissa of
    both signs, infinities and NaNs."""
    for start in range(0, 1 << 32, _CHUNK):
        _check_e4m3(torch.arange(start, start + _CHUNK, dtype=torch.int64, device="cuda"))


@pytest.mark.slow
def test_bf16_every_fp32_bit_pattern():
    """All 2^32 inputs, each rounded to nearest even on its low 16 bits."""
    for start in range(0, 1 << 32, _CHUNK):
        _check_bf16(torch.arange(start, start + _CHUNK, dtype=torch.int64, device="cuda"))


def test_format_entry_points_reject_odd_lengths():
    x = torch.zeros(3, dtype=torch.float32, device="cuda")
    with pytest.raises(ep.EPError):
        ep.ep_format_e4m3(x, torch.empty(3, dtype=torch.uint8, device="cuda"))
