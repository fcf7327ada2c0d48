"""Pins of the oracle's once-per-rank receive layout (DeepEP V1 normal mode)
and rank-level combine, against things other than the oracle's own code:

* a hand-worked example (tests/golden/rank_layout_small.json, derived by
  hand from the llm-infra-atlas DeepEP article's definitions, §2.1, §2.3,
  §3.2);
* the already pinned layout / notify oracles: the (token, rank) pairs the
  layout receives are exactly is_token_in_rank, and every source rank's
  segment starts at the previous row of notify's rank_prefix_matrix;
* a bijection / order invariant on random routings with masked and repeated
  experts;
* a closed form for the combine: an identity expert on every rank returns
  bf16(m * x) for a token on m ranks (the fp32 sum of m equal bf16 values is
  exact), and +0 for a token on none.
"""
import json
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rank_layout_small.json")


def _bits(v):
    return torch.tensor(np.asarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(
        np.uint16)


def test_golden_rank_layout_and_combine():
    g = json.load(open(GOLDEN))
    R, T_r, E, k, cap = g["R"], g["T_r"], g["E"], g["k"], g["cap_rows"]
    idx = np.array(g["topk_idx"], np.int64)
    w = np.array([[[(1 + 6 * i + 2 * t + j) / 8 for j in range(k)] for t in range(T_r)]
                  for i in range(R)], np.float32)
    x = np.arange(R * T_r * 8, dtype=np.float32).reshape(R, T_r, 8)
    d = oracle.rank_dispatch(_bits(x), idx, w, E, 0, cap)
    assert d["rc"] == oracle.OK
    assert np.array_equal(d["combine_idx"], np.array(g["combine_idx"]))
    assert np.array_equal(d["recv_src_idx"], np.array(g["recv_src_idx"]))
    src = d["recv_src_idx"]
    valid = src >= 0
    assert np.array_equal(d["recv_topk_idx"][valid], np.array(g["recv_topk_idx"])[valid])
    assert np.array_equal(d["recv_topk_weights"][valid],
                          np.array(g["recv_topk_weights"], np.float32)[valid])
    # every received row holds its source token
    xb = _bits(x).reshape(R * T_r, 8)
    assert np.array_equal(d["recv_x"].reshape(R * cap, 8)[valid.reshape(-1)],
                          xb[src.reshape(-1)[valid.reshape(-1)]])
    lay = oracle.layout(idx, R, E)
    nt = oracle.notify(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"], R, E, 1)
    assert np.array_equal(nt["rank_prefix_matrix"], np.array(g["rank_prefix_matrix"]))
    y = _bits(np.array(g["combine_y"], np.float32)).reshape(-1, 1)
    c = oracle.rank_combine(y, d["combine_idx"], 1)
    assert c["rc"] == oracle.OK
    got = torch.from_numpy(c["out"].view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(got.reshape(R, T_r), np.array(g["combine_out"], np.float32))
    assert c["out"].reshape(-1)[-1] == 0   # +0 for the token with no expert


def _random_idx(rng, R, T_r, k, E):
    idx = rng.integers(0, E, size=(R, T_r, k)).astype(np.int64)   # repeats allowed
    idx[rng.random(idx.shape) < 0.1] = -1
    return idx


def test_rank_layout_matches_is_token_in_rank_and_the_prefix_matrix():
    rng = np.random.default_rng(11)
    for R, T_r, k, E in ((4, 37, 3, 16), (8, 64, 8, 64), (3, 20, 2, 3), (16, 9, 6, 32)):
        idx = _random_idx(rng, R, T_r, k, E)
        w = rng.random((R, T_r, k), dtype=np.float32)
        H = 16
        x = rng.standard_normal((R, T_r, H), dtype=np.float32)
        cap = R * T_r
        d = oracle.rank_dispatch(_bits(x), idx, w, E, 0, cap)
        assert d["rc"] == oracle.OK
        lay = oracle.layout(idx, R, E)
        nt = oracle.notify(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"], R, E, 1)
        rpm = nt["rank_prefix_matrix"]
        src = d["recv_src_idx"]
        E_l = E // R
        for r in range(R):
            rows = src[r]
            n = int(rpm[R - 1, r])
            assert np.all(rows[:n] >= 0) and np.all(rows[n:] == -1)
            for i in range(R):
                lo = 0 if i == 0 else int(rpm[i - 1, r])
                seg = rows[lo:int(rpm[i, r])]
                toks = [t for t in range(T_r) if lay["is_token_in_rank"][i, t, r]]
                assert list(seg) == [i * T_r + t for t in toks]   # token order, once each
        # the slot pointing at each row is the token's first slot on that rank
        cidx = d["combine_idx"]
        for i in range(R):
            for t in range(T_r):
                seen = set()
                for j in range(k):
                    e = idx[i, t, j]
                    if e < 0 or e // E_l in seen:
                        assert cidx[i, t, j] == -1
                        continue
                    r = e // E_l
                    seen.add(r)
                    f = cidx[i, t, j]
                    assert f // cap == r and src.reshape(-1)[f] == i * T_r + t
                    loc = d["recv_topk_idx"].reshape(-1, k)[f]
                    wts = d["recv_topk_weights"].reshape(-1, k)[f]
                    for jj in range(k):
                        on = idx[i, t, jj] >= 0 and idx[i, t, jj] // E_l == r
                        assert loc[jj] == (idx[i, t, jj] - r * E_l if on else -1)
                        assert wts[jj] == (w[i, t, jj] if on else 0.0)


def test_rank_combine_of_an_identity_expert_is_m_times_x():
    rng = np.random.default_rng(5)
    R, T_r, k, E, H = 8, 50, 8, 32, 64
    idx = _random_idx(rng, R, T_r, k, E)
    x = rng.standard_normal((R, T_r, H), dtype=np.float32)
    xb = _bits(x)
    cap = R * T_r
    d = oracle.rank_dispatch(xb, idx, np.ones((R, T_r, k), np.float32), E, 0, cap)
    out = oracle.rank_combine(d["recv_x"].reshape(-1, H), d["combine_idx"], H)["out"]
    E_l = E // R
    m = np.array([[len({e // E_l for e in idx[i, t] if e >= 0}) for t in range(T_r)]
                  for i in range(R)], np.float64)
    xf = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).double().numpy()
    want = _bits((m[..., None] * xf).astype(np.float32))   # m * x exact in fp32
    assert np.array_equal(out, want)
    none = m == 0
    assert np.all(out[none] == 0)


def test_rank_layout_capacity_and_fp8_rows():
    rng = np.random.default_rng(3)
    R, T_r, k, E, H = 4, 12, 4, 16, 256
    idx = _random_idx(rng, R, T_r, k, E)
    x = rng.standard_normal((R, T_r, H), dtype=np.float32)
    d = oracle.rank_dispatch(_bits(x), idx, np.ones((R, T_r, k), np.float32), E, 2, 3)
    assert d["rc"] == oracle.ERR_CAPACITY          # rank buffers of 3 rows overflow
    full = oracle.rank_dispatch(_bits(x), idx, np.ones((R, T_r, k), np.float32), E, 2, R * T_r)
    assert full["rc"] == oracle.OK
    # FP8 rows are the oracle's own per-row quantisation of the source token
    src = full["recv_src_idx"].reshape(-1)
    xb = _bits(x).reshape(R * T_r, H)
    cap = R * T_r
    for f in np.nonzero(src >= 0)[0][:10]:
        q, s = oracle.quantize_row(xb[src[f]], 2)
        assert np.array_equal(full["recv_x"].reshape(-1, H)[f], q)
        r, row = divmod(int(f), cap)   # scales column-major: [R, H/128, cap]
        assert np.array_equal(full["recv_scales"][r, :, row], s)
