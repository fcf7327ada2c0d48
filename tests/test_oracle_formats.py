"""Pins for the oracle's number formats and FP8 block quantisation.

The oracle's bf16 and E4M3 encoders are checked against torch's own CPU
dtype conversions (round to nearest even) over every fp32 pattern whose low
12 mantissa bits are one of a set of rounding-relevant patterns (so all
exponents, all kept mantissa bits and every guard/sticky combination are
covered), plus random patterns.  The FP8 block quantiser is pinned by
closed-form properties of the per-128-channel scheme (power-of-two ue8m0
scale, amax mapping to 448, round-trip error within half an E4M3 step).
"""
import numpy as np
import pytest
import torch

import oracle

LOW_PATTERNS = np.array([0x000, 0x001, 0x7FF, 0x800, 0x801, 0xFFF], dtype=np.uint32)


def _patterns(random_extra=1 << 20, seed=0):
    top = np.arange(1 << 20, dtype=np.uint32) << 12
    pats = (top[:, None] | LOW_PATTERNS[None, :]).ravel()
    rnd = np.random.default_rng(seed).integers(0, 1 << 32, random_extra, dtype=np.uint64)
    return np.concatenate([pats, rnd.astype(np.uint32)])


def test_bf16_rne_matches_torch():
    bits = _patterns()
    f = bits.view(np.float32)
    ours = oracle.f32_to_bf16(f)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(ours[nan] == 0x7FFF)


def test_bf16_widening_exact():
    h = np.arange(1 << 16, dtype=np.uint16)
    f = oracle.bf16_to_f32(h)
    ref = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    same = (f.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(f) & np.isnan(ref))
    assert same.all()


def test_e4m3_matches_torch_in_range():
    bits = _patterns()
    f = bits.view(np.float32)
    inrange = np.isfinite(f) & (np.abs(f) <= 448.0)
    fi = f[inrange]
    ours = oracle.f32_to_e4m3(fi)
    ref = torch.from_numpy(fi.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first {fi[bad[:5]]}"


def test_e4m3_saturates_and_nan():
    f = np.array([448.0, 448.0001, 463.9, 464.0, 480.0, 1e6, np.inf, -500.0, -np.inf],
                 dtype=np.float32)
    q = oracle.f32_to_e4m3(f)
    assert list(q) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]
    qn = oracle.f32_to_e4m3(np.array([np.nan, -np.nan], np.float32))
    assert (qn & 0x7F).tolist() == [0x7F, 0x7F]
    assert oracle.f32_to_e4m3(np.array([0.0, -0.0], np.float32)).tolist() == [0x00, 0x80]


def test_e4m3_decode_matches_torch():
    b = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f32(b)
    ref = torch.from_numpy(b.copy()).view(torch.float8_e4m3fn).float().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def _random_rows(n, H, seed, std=1.0):
    rng = np.random.default_rng(seed)
    f = rng.standard_normal((n, H)).astype(np.float32) * np.float32(std)
    # a few rows with wide dynamic range and one all-zero row
    f[1] *= np.float32(1e-6)
    f[2, ::3] *= np.float32(1e3)
    f[3] = 0.0
    return torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("H", [128, 512, 7168])
def test_ue8m0_quantisation_properties(H):
    rows = _random_rows(8, H, seed=H)
    for r in range(rows.shape[0]):
        q, s = oracle.quantize_row(rows[r], oracle.FP8_E4M3_UE8M0)
        x = oracle.bf16_to_f32(rows[r]).astype(np.float64).reshape(-1, 128)
        amax = np.maximum(np.abs(x).max(axis=1), np.float32(1e-4))
        scale = np.ldexp(1.0, s.astype(np.int64) - 127)          # power of two by construction
        # smallest power of two with amax / scale <= 448
        assert np.all(amax / scale <= 448.0)
        assert np.all(amax / (scale / 2) > 448.0 * (1 - 2 ** -23))
        deq = oracle.e4m3_to_f32(q).astype(np.float64).reshape(-1, 128) * scale[:, None]
        xs = np.abs(x / scale[:, None])
        # half an E4M3 step at |x|/scale (subnormal step 2^-9 below 2^-6)
        step = np.where(xs < 2.0 ** -6, 2.0 ** -9, np.exp2(np.floor(np.log2(np.maximum(xs, 1e-300))) - 3))
        assert np.all(np.abs(deq - x) <= 0.5 * step * scale[:, None] + 1e-300)


@pytest.mark.parametrize("H", [128, 4096])
def test_fp32_scale_quantisation_properties(H):
    rows = _random_rows(8, H, seed=7 + H, std=2.0)
    for r in range(rows.shape[0]):
        q, s = oracle.quantize_row(rows[r], oracle.FP8_E4M3_F32_SCALE)
        x = oracle.bf16_to_f32(rows[r]).reshape(-1, 128)
        amax = np.maximum(np.abs(x).max(axis=1), np.float32(1e-4))
        assert np.array_equal(s, (amax / np.float32(448.0)).astype(np.float32))
        qf = oracle.e4m3_to_f32(q).reshape(-1, 128)
        # the block's largest magnitude lands on the E4M3 maximum (unless floored)
        big = np.abs(x).max(axis=1) >= 1e-4
        assert np.all(np.abs(qf[big]).max(axis=1) == 448.0)
        inv = (np.float32(448.0) / amax).astype(np.float32)
        xs = np.abs(x.astype(np.float64) * inv[:, None])
        step = np.where(xs < 2.0 ** -6, 2.0 ** -9, np.exp2(np.floor(np.log2(np.maximum(xs, 1e-300))) - 3))
        err = np.abs(qf.astype(np.float64) - x * inv[:, None].astype(np.float64))
        assert np.all(err <= 0.5 * step * (1 + 2 ** -20) + 1e-30)


def test_all_zero_block_uses_floor():
    x = np.zeros(256, np.uint16)
    q, s = oracle.quantize_row(x, oracle.FP8_E4M3_F32_SCALE)
    assert np.all(q == 0) and np.all(s == np.float32(np.float32(1e-4) / np.float32(448.0)))
    q, s = oracle.quantize_row(x, oracle.FP8_E4M3_UE8M0)
    # 1e-4 / 448 = 2.23e-7 rounds up to 2^-22 -> biased exponent 105
    assert np.all(q == 0) and np.all(s == 105)


def test_quantise_block_holding_an_infinity_or_nan():
    """Non-finite inputs (the article fixes nothing for them; reading: amax
    ignores NaN and is capped at the largest finite float, so scales stay
    finite).  Expected codes derived by hand: FLT_MAX/448 ~ 7.595e35 lies in
    (2^119, 2^120], so the ue8m0 block with an infinity gets 2^120 (byte
    127 + 120 = 247); +-inf saturate to +-448 (0x7E / 0xFE) and the finite
    values, scaled by 2^-120, round to +-0 (0x00 / 0x80).  The NaN block's
    amax is 3.0: 3/448 lies in (2^-8, 2^-7], byte 120, and 3.0 * 2^7 = 384 =
    1.5 * 2^8 is E4M3 0 1111 100 = 0x7C, -1.0 * 2^7 = -2^7 is 1 1110 000 =
    0xF0; the NaN stays a NaN (S.1111.111)."""
    from fractions import Fraction
    inf_bits = {+1: 0x7F80, -1: 0xFF80}                  # bf16 +-infinity
    row = np.zeros(256, np.uint16)
    row[0], row[1] = inf_bits[+1], inf_bits[-1]
    row[2] = 0x3F80                                        # 1.0
    row[3] = 0xC020                                        # -2.5
    row[128] = 0x7FC0                                      # NaN
    row[129] = 0x4040                                      # 3.0
    row[130] = 0xBF80                                      # -1.0
    q, s = oracle.quantize_row(row, oracle.FP8_E4M3_UE8M0)
    assert s.tolist() == [247, 120]
    assert q[0] == 0x7E and q[1] == 0xFE and q[2] == 0x00 and q[3] == 0x80
    assert np.all(q[4:128] == 0x00)
    assert (q[128] & 0x7F) == 0x7F                        # NaN, either sign
    assert q[129] == 0x7C and q[130] == 0xF0 and np.all(q[131:] == 0x00)
    # fp32 scales: the infinity block's scale is FLT_MAX / 448 rounded once
    q, s = oracle.quantize_row(row, oracle.FP8_E4M3_F32_SCALE)
    flt_max = Fraction(2**24 - 1, 2**23) * 2**127
    exact = flt_max / 448
    assert abs(Fraction(float(s[0])) - exact) <= exact * Fraction(1, 2**24)
    assert q[0] == 0x7E and q[1] == 0xFE and q[2] == 0x00 and q[3] == 0x80
    assert abs(Fraction(float(s[1])) - Fraction(3, 448)) <= Fraction(3, 448) * Fraction(1, 2**24)
    assert (q[128] & 0x7F) == 0x7F
    # 3.0 * (448 / 3) = 448 exactly after rounding: the block maximum maps to 448
    assert q[129] == 0x7E
