"""Pins for the oracle's data path: dispatch then combine.

"Combine is dispatch walked backwards" (DeepEP article §4.3, §5): with an
identity expert (y = the dispatched rows) combine must return the router-
weighted sum of the token's own row, bf16(sum_j w_j * x).  The reference sum
is taken in float64 -- each w*x product of an fp32 weight and a bf16 value
is exact there -- and the oracle's fp32 fma chain must land within one bf16
ulp of it.  Special cases: k=1 with weight 1 reproduces x bit for bit; zero
weights and fully masked tokens give +0.  FP8 rows must dequantise to within
half an E4M3 step of x, and the low-latency layout must hold the same rows
as the contiguous layout shifted by the segment starts.
"""
import numpy as np
import pytest

import oracle
from combine_get_dispatch_gb300 import synth


def _bf16_ulp(v):
    v = np.abs(v.astype(np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -133)))
    return np.exp2(np.maximum(e, -126) - 7)


def _normal_path(x, idx, E, fp8_mode, A=1):
    R = x.shape[0]
    lay = oracle.layout(idx, R, E)
    n = oracle.notify(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"], R, E, A)
    cap = int(n["psum"][:, -1].max())
    d = oracle.dispatch(x, idx, lay["slot_rank"], n["expert_prefix"], n["psum"], E, fp8_mode, cap)
    assert d["rc"] == oracle.OK
    return lay, n, d, cap


def _dequant_rows(d, fp8_mode, H):
    """recv rows -> bf16 bits of dequant(q) (the identity expert's output)."""
    q = d["recv_x"]
    R, cap = q.shape[0], q.shape[1]
    s = d["recv_scales"]                       # [R, H/128, cap]
    if fp8_mode == oracle.FP8_E4M3_F32_SCALE:
        scale = s.astype(np.float64)
    else:
        scale = np.ldexp(1.0, s.astype(np.int64) - 127)
    scale = np.repeat(np.transpose(scale, (0, 2, 1)), 128, axis=2)    # [R, cap, H]
    deq = oracle.e4m3_to_f32(q).astype(np.float64) * scale
    return oracle.f32_to_bf16(deq.astype(np.float32))


@pytest.mark.parametrize("fp8_mode", [0, 1, 2])
def test_identity_expert_round_trip(fp8_mode):
    w = synth.WORKLOADS["tiny"]
    w = synth.scaled(w, H=256)
    x = synth.activations(w)
    idx, wts = synth.routing(w)
    _, _, d, cap = _normal_path(x, idx, w.E, fp8_mode)
    y = d["recv_x"] if fp8_mode == 0 else _dequant_rows(d, fp8_mode, w.H)
    c = oracle.combine(y.reshape(-1, w.H), wts, d["combine_idx"], w.H)
    assert c["rc"] == oracle.OK
    out = oracle.bf16_to_f32(c["out"]).astype(np.float64)
    if fp8_mode == 0:
        xv = oracle.bf16_to_f32(x).astype(np.float64)
        ref = wts.astype(np.float64).sum(axis=2)[..., None] * xv
    else:
        # sum_j w_j * dequant(quant(x)) taken from each slot's own row
        yv = oracle.bf16_to_f32(y).reshape(-1, w.H).astype(np.float64)
        ref = np.zeros(out.shape)
        for j in range(w.k):
            ref += wts[..., j:j + 1].astype(np.float64) * yv[d["combine_idx"][..., j]]
        # and dequant(quant(x)) is close to x (half an E4M3 step per block)
        xv = oracle.bf16_to_f32(x).astype(np.float64)
        assert np.max(np.abs(yv[d["combine_idx"][..., 0]] - xv)) <= 0.07 * np.abs(xv).max()
    assert np.all(np.abs(out - ref) <= _bf16_ulp(ref))


def test_k1_weight1_is_exact_copy():
    w = synth.scaled(synth.WORKLOADS["tiny"], k=1)
    x = synth.activations(w)
    idx, _ = synth.routing(w)
    _, _, d, _ = _normal_path(x, idx, w.E, 0)
    c = oracle.combine(d["recv_x"].reshape(-1, w.H), np.ones(idx.shape, np.float32),
                       d["combine_idx"], w.H)
    assert np.array_equal(c["out"], x)


def test_zero_weights_and_masked_tokens_give_plus_zero():
    w = synth.WORKLOADS["tiny"]
    x = synth.activations(w)
    idx, wts = synth.routing(w)
    idx = idx.copy()
    idx[:, 0, :] = -1                     # token 0 of each rank is fully masked
    _, _, d, _ = _normal_path(x, idx, w.E, 0)
    c = oracle.combine(d["recv_x"].reshape(-1, w.H), np.zeros_like(wts), d["combine_idx"], w.H)
    assert np.all(c["out"] == 0)
    c = oracle.combine(d["recv_x"].reshape(-1, w.H), wts, d["combine_idx"], w.H)
    assert np.all(c["out"][:, 0, :] == 0)


def test_combine_single_terms_and_order():
    # acc = fma(w1, y1, fma(w0, y0, 0)): two hand-checkable cases
    H = 8
    y = oracle.f32_to_bf16(np.array([[1.0] * H, [2.0 ** -8] * H], np.float32))
    cidx = np.array([[0, 1]], np.int32)
    c = oracle.combine(y, np.array([[1.0, 1.0]], np.float32), cidx, H)
    # 1 + 2^-8 is a tie between bf16 1.0 and 1.0078125 -> even (1.0)
    assert np.all(c["out"] == 0x3F80)
    c = oracle.combine(y, np.array([[1.0, 1.5]], np.float32), cidx, H)
    # 1 + 1.5*2^-8 rounds up to 1 + 2^-7
    assert np.all(c["out"] == 0x3F81)
    c = oracle.combine(y, np.array([[-1.0, 0.0]], np.float32), np.array([[0, -1]], np.int32), H)
    assert np.all(c["out"] == 0xBF80)


@pytest.mark.parametrize("fp8_mode", [0, 1, 2])
def test_fp8_rows_and_scale_positions(fp8_mode):
    w = synth.scaled(synth.WORKLOADS["tiny"], H=384, fp8_mode=fp8_mode)
    x = synth.activations(w)
    idx, _ = synth.routing(w)
    _, n, d, cap = _normal_path(x, idx, w.E, fp8_mode, A=4)
    for i in range(w.R):
        for t in range(w.T_r):
            for j in range(w.k):
                f = d["combine_idx"][i, t, j]
                r, row = divmod(int(f), cap)
                if fp8_mode == 0:
                    assert np.array_equal(d["recv_x"][r, row], x[i, t])
                else:
                    q, s = oracle.quantize_row(x[i, t], fp8_mode)
                    assert np.array_equal(d["recv_x"][r, row], q)
                    assert np.array_equal(d["recv_scales"][r, :, row], s)


@pytest.mark.parametrize("fp8_mode", [0, 2])
def test_low_latency_matches_contiguous_layout(fp8_mode):
    w = synth.scaled(synth.WORKLOADS["tiny"], fp8_mode=fp8_mode)
    x = synth.activations(w)
    idx, _ = synth.routing(w)
    _, n, d, cap = _normal_path(x, idx, w.E, fp8_mode, A=1)
    ll = oracle.ll_dispatch(x, idx, w.E, w.max_tokens_per_rank, fp8_mode)
    assert ll["rc"] == oracle.OK
    seg = w.R * w.max_tokens_per_rank
    assert np.array_equal(ll["recv_count"].ravel(), n["expert_prefix"][-1])
    for e in range(w.E):
        r, l = divmod(e, w.E_l)
        cnt = ll["recv_count"].ravel()[e]
        lo = n["psum"][r, l]
        px = ll["packed_recv_x"].reshape(w.E, seg, w.H)[e, :cnt]
        assert np.array_equal(px, d["recv_x"][r, lo:lo + cnt])
        assert np.array_equal(ll["packed_recv_src_info"].reshape(w.E, seg)[e, :cnt],
                              d["recv_src_idx"][r, lo:lo + cnt])
        if fp8_mode:
            ps = ll["packed_recv_scales"].reshape(w.E, w.H // 128, seg)[e, :, :cnt]
            assert np.array_equal(ps, d["recv_scales"][r, :, lo:lo + cnt])
    # both combine_idx encodings name the same data
    yn = d["recv_x"].reshape(-1, w.H)
    yl = ll["packed_recv_x"].reshape(-1, w.H)
    m = d["combine_idx"] >= 0
    assert np.array_equal(yn[d["combine_idx"][m]], yl[ll["combine_idx"][m]])
