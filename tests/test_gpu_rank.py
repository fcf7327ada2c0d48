"""GPU parity: the once-per-rank receive layout of V1's normal mode (a token
goes once to every rank holding one of its experts) built from libep's
entry points -- rank ids, layout and notify over ranks, dispatch, local
top-k per received row, rank-level combine -- vs the oracle's direct
definition.  Rows, scales and indices bit-exact; the combine within 1 bf16
ulp (the kernel adds the rows in the same slot order in fp32, so 0 is
expected)."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_gb300 import ep, synth
from ep_harness import (POISON, bits_u16, gpu_dispatch, gpu_layout, gpu_notify, inputs, np_,
                        poison_, status_word)
from test_gpu_combine import assert_bf16_close

pytestmark = pytest.mark.gpu


def _gpu_rank_path(x_dev, idx_dev, wts_dev, E, fp8_mode, num_worst_tokens=-1, y_seed=11):
    R, T_r, k = idx_dev.shape
    H = x_dev.shape[2]
    st = status_word()
    rank_ids = poison_(torch.empty((R, T_r, k), dtype=torch.int64, device="cuda"))
    ep.ep_rank_ids(idx_dev, E, rank_ids, st)
    lay = gpu_layout(rank_ids, R, status=st)
    nt = gpu_notify(lay, R, 1, num_worst_tokens, status=st)
    if num_worst_tokens >= 0:
        cap = max(1, num_worst_tokens)
    else:
        cap = max(1, int(nt["psum"][:, -1].max().item()))
    d = gpu_dispatch(x_dev, rank_ids, lay, nt, R, fp8_mode, cap, status=st)
    rtk = poison_(torch.empty((R, cap, k), dtype=torch.int64, device="cuda"))
    rtw = poison_(torch.empty((R, cap, k), dtype=torch.float32, device="cuda"))
    ep.ep_rank_recv_topk(idx_dev, wts_dev, d["combine_idx"], E, cap, rtk, rtw, st)
    y = synth.expert_outputs_torch(R * cap, H, "cuda", y_seed).view(R, cap, H)
    out = poison_(torch.empty((R, T_r, H), dtype=torch.bfloat16, device="cuda"))
    ep.ep_rank_combine(y, d["combine_idx"], cap, out, st)
    torch.cuda.synchronize()
    return dict(rank_ids=rank_ids, lay=lay, nt=nt, d=d, cap=cap, rtk=rtk, rtw=rtw, y=y, out=out,
                status=st)


def _compare(x_host, idx, wts, E, fp8_mode, g):
    R = idx.shape[0]
    H = x_host.shape[2]
    cap = g["cap"]
    ref = oracle.rank_dispatch(x_host, idx, wts, E, fp8_mode, cap)
    assert ref["rc"] == oracle.OK
    d = g["d"]
    assert np.array_equal(np_(d["combine_idx"]), ref["combine_idx"])
    src = np_(d["recv_src_idx"])
    assert np.array_equal(src, ref["recv_src_idx"])
    rows = np.nonzero(src.reshape(-1) >= 0)[0]
    got = np_(d["recv_x"]).reshape(R * cap, -1)
    assert np.array_equal(got[rows], ref["recv_x"].reshape(R * cap, -1)[rows])
    unused = np.nonzero(src.reshape(-1) < 0)[0]
    if unused.size:
        assert np.all(got[unused[:4096]].view(np.uint8) == POISON)
    if fp8_mode:
        r_idx, row_idx = np.divmod(rows, cap)
        gs = np_(d["recv_scales"])
        assert np.array_equal(gs[r_idx, :, row_idx], ref["recv_scales"][r_idx, :, row_idx])
    k = idx.shape[2]
    assert np.array_equal(np_(g["rtk"]).reshape(-1, k)[rows],
                          ref["recv_topk_idx"].reshape(-1, k)[rows])
    assert np.array_equal(np_(g["rtw"]).reshape(-1, k)[rows].view(np.uint32),
                          ref["recv_topk_weights"].reshape(-1, k)[rows].view(np.uint32))
    rc = oracle.rank_combine(bits_u16(g["y"]), ref["combine_idx"], H)
    assert rc["rc"] == oracle.OK
    assert_bf16_close(np_(g["out"]), rc["out"])
    assert ep.ep_read_status(g["status"]) == ep.EP_OK
    return ref


@pytest.mark.parametrize("name,T_r,fp8_mode", [
    ("tiny", 16, 0), ("tiny", 33, 1), ("prefill", 96, 0), ("prefill", 64, 2), ("large", 80, 2),
    ("skewed", 40, 1), ("decode", 24, 2),
])
def test_rank_layout_matches_the_oracle(name, T_r, fp8_mode):
    base = synth.WORKLOADS[name]
    w = synth.scaled(base, T_r=T_r, fp8_mode=fp8_mode, num_worst_tokens=-1)
    x_dev, x_host, idx_dev, idx, wts_dev, wts = inputs(w, seed=3)
    g = _gpu_rank_path(x_dev, idx_dev, wts_dev, w.E, fp8_mode)
    _compare(x_host, idx, wts, w.E, fp8_mode, g)
    # counting tokens per (source, destination rank) over rank ids is the
    # per-expert layout's num_tokens_per_rank
    lay_e = gpu_layout(idx_dev, w.E)
    torch.cuda.synchronize()
    assert np.array_equal(np_(g["lay"]["num_tokens_per_expert"]),
                          np_(lay_e["num_tokens_per_rank"]))
    assert np.array_equal(np_(g["lay"]["num_tokens_per_rank"]),
                          np_(lay_e["num_tokens_per_rank"]))


def test_rank_layout_with_worst_case_rows_and_masked_slots():
    # skewed routing (few hot experts) and a fixed worst-case row count per
    # rank; a fifth of the slots are unused (-1), some tokens route nowhere
    w = synth.scaled(synth.WORKLOADS["skewed"], T_r=48, num_worst_tokens=32 * 48)
    x_dev, x_host, idx_dev, idx, wts_dev, wts = inputs(w, seed=9)
    rng = np.random.default_rng(4)
    idx = idx.copy()
    idx[rng.random(idx.shape) < 0.2] = -1
    idx[0, :3, :] = -1
    idx_dev = torch.from_numpy(idx).cuda()
    g = _gpu_rank_path(x_dev, idx_dev, wts_dev, w.E, w.fp8_mode, w.num_worst_tokens)
    assert g["cap"] == 32 * 48
    ref = _compare(x_host, idx, wts, w.E, w.fp8_mode, g)
    assert np.all(ref["combine_idx"][0, :3] == -1)
    # tokens that reach no rank combine to +0
    assert np.all(np_(g["out"])[0, :3] == 0)


def test_rank_ids_are_each_tokens_first_slot_per_rank():
    w = synth.scaled(synth.WORKLOADS["tiny"], T_r=40)
    _, _, idx_dev, idx, _, _ = inputs(w, seed=1)
    got = torch.empty_like(idx_dev)
    ep.ep_rank_ids(idx_dev, w.E, got)
    got = np_(got)
    E_l = w.E // w.R
    for i in range(w.R):
        for t in range(w.T_r):
            seen = set()
            for j in range(w.k):
                r = int(idx[i, t, j]) // E_l
                want = -1 if r in seen else r
                seen.add(r)
                assert got[i, t, j] == want


def test_rank_ids_flag_invalid_expert_ids():
    idx = torch.tensor([[[0, 17], [3, -1]], [[-2, 5], [1, 2]]], dtype=torch.int64, device="cuda")
    st = status_word()
    out = torch.empty_like(idx)
    ep.ep_rank_ids(idx, 16, out, st)
    assert ep.ep_read_status(st) == ep.EP_ERR_INVALID_ARG
    o = np_(out)
    assert o[0, 0, 1] == -1 and o[1, 0, 0] == -1 and o[0, 0, 0] == 0


@pytest.mark.parametrize("R,T_r", [(1, 24), (4, 0)])
def test_rank_layout_degenerate_shapes(R, T_r):
    w = synth.Workload("edge", R=R, T_r=T_r, H=256, E=8 * R, k=4, routing="uniform",
                       mode="normal", fp8_mode=2)
    x_dev, x_host, idx_dev, idx, wts_dev, wts = inputs(w, seed=2)
    g = _gpu_rank_path(x_dev, idx_dev, wts_dev, w.E, 2)
    if T_r > 0:
        _compare(x_host, idx, wts, w.E, 2, g)
    else:
        assert ep.ep_read_status(g["status"]) == ep.EP_OK
        assert int(g["nt"]["psum"][:, -1].max().item()) == 0
