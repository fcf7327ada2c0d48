"""GPU parity: get_dispatch_layout and notify_dispatch vs the oracle,
bit-exact, at every workload's full size and on edge cases."""
import numpy as np
import pytest
import torch

import oracle
from combine_get_dispatch_gb300 import ep, synth
from ep_harness import gpu_layout, gpu_notify, np_, status_word

pytestmark = pytest.mark.gpu

LAYOUT_KEYS = ("num_tokens_per_rank", "num_tokens_per_expert", "is_token_in_rank", "slot_rank")
NOTIFY_KEYS = ("rank_prefix_matrix", "expert_prefix", "num_recv_tokens_per_expert", "psum")


def _compare_layout(idx_host, E, lay_gpu):
    R = idx_host.shape[0]
    ref = oracle.layout(idx_host, R, E)
    assert ref["rc"] == oracle.OK
    for key in LAYOUT_KEYS:
        got = np_(lay_gpu[key])
        assert np.array_equal(got, ref[key]), key
    return ref


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_layout_and_notify_full_size(name):
    w = synth.WORKLOADS[name]
    idx, _ = synth.routing(w)
    idx_dev = torch.from_numpy(idx).cuda()
    lay = gpu_layout(idx_dev, w.E)
    ref = _compare_layout(idx, w.E, lay)
    assert ep.ep_read_status(lay["status"]) == ep.EP_OK
    for A in (1, 128):
        nt = gpu_notify(lay, w.E, A, w.num_worst_tokens)
        nref = oracle.notify(ref["num_tokens_per_rank"], ref["num_tokens_per_expert"], w.R, w.E, A,
                             w.num_worst_tokens)
        for key in NOTIFY_KEYS:
            assert np.array_equal(np_(nt[key]), nref[key]), key
        assert ep.ep_read_status(nt["status"]) == nref["rc"]
    # the same workspace again (look-back state reused through the epoch)
    lay2 = gpu_layout(idx_dev, w.E, ws=lay["ws"])
    for key in LAYOUT_KEYS:
        assert torch.equal(lay2[key], lay[key]), key


@pytest.mark.parametrize("R,T_r,k,E", [
    (4, 0, 2, 16),       # no tokens
    (3, 1, 1, 3),        # one token, k = 1, one expert per rank
    (2, 257, 8, 64),     # ragged chunk tail (chunks of 256 tokens at k = 8)
    (5, 1000, 3, 20),    # ragged, odd k
    (1, 5000, 16, 32),   # k = 16 (chunks of 128 tokens), one rank
    (64, 40, 4, 256),    # many ranks
    (2, 3000, 8, 1024),  # largest expert count
    (3, 700, 3, 6),      # odd E + R (shared-memory tables of odd length)
    (33, 100, 5, 66),    # R not a power of two, odd E + R
    (100, 30, 4, 200),   # R > 64: per-rank loop for is_token_in_rank; counts walked in memory
    (96, 12, 2, 192),    # R > 64, notify counts too large to stage
    (3, 110000, 1, 9),   # beyond one wave of 2048-id chunks: 8192-id chunks (k = 1), ragged
    (2, 20000, 8, 64),   # 8192-id chunks at k = 8, look-back over 19 chunks
])
def test_layout_edge_shapes(R, T_r, k, E):
    rng = np.random.default_rng(R * 1000 + T_r)
    idx = rng.integers(-1, E, size=(R, T_r, k)).astype(np.int64)
    lay = gpu_layout(torch.from_numpy(idx).cuda(), E)
    ref = _compare_layout(idx, E, lay)
    assert ep.ep_read_status(lay["status"]) == ep.EP_OK
    # notify on the same counts: column walks over R source ranks in
    # batches (R = 1 .. 64 here, ragged against the batch of 16)
    for A in (1, 8):
        nt = gpu_notify(lay, E, A)
        nref = oracle.notify(ref["num_tokens_per_rank"], ref["num_tokens_per_expert"], R, E, A)
        for key in NOTIFY_KEYS:
            assert np.array_equal(np_(nt[key]), nref[key]), key
        assert ep.ep_read_status(nt["status"]) == ep.EP_OK


def test_layout_all_tokens_to_one_expert():
    R, T_r, k, E = 8, 4096, 1, 256
    idx = np.full((R, T_r, k), 5, np.int64)
    lay = gpu_layout(torch.from_numpy(idx).cuda(), E)
    ref = _compare_layout(idx, E, lay)
    assert ref["num_tokens_per_expert"][:, 5].tolist() == [T_r] * R


def test_layout_invalid_ids_flag_status_and_count_as_unused():
    R, T_r, k, E = 2, 300, 4, 8
    rng = np.random.default_rng(3)
    idx = rng.integers(0, E, size=(R, T_r, k)).astype(np.int64)
    bad = idx.copy()
    bad[1, 17, 2] = E          # out of range
    bad[0, 250, 0] = -5        # negative, not -1
    lay = gpu_layout(torch.from_numpy(bad).cuda(), E)
    assert ep.ep_read_status(lay["status"]) == ep.EP_ERR_INVALID_ARG
    masked = bad.copy()
    masked[1, 17, 2] = -1
    masked[0, 250, 0] = -1
    _compare_layout(masked, E, lay)


def test_notify_host_handshake():
    w = synth.WORKLOADS["prefill"]
    idx, _ = synth.routing(w)
    lay = gpu_layout(torch.from_numpy(idx).cuda(), w.E)
    host_rows = torch.full((w.R,), -7, dtype=torch.int64).pin_memory()
    nt = gpu_notify(lay, w.E, 128, -1, host_rows=host_rows)
    # the call returned only after the kernel published every rank's row count
    assert np.array_equal(host_rows.numpy(), np_(nt["psum"])[:, -1])
    torch.cuda.synchronize()
    assert np.array_equal(host_rows.numpy(), np_(nt["psum"])[:, -1])


def test_notify_num_worst_tokens_capacity():
    R, T_r, k, E = 4, 64, 2, 8
    idx = np.zeros((R, T_r, k), np.int64)
    idx[..., 1] = 1                                   # every token goes to rank 0 only
    lay = gpu_layout(torch.from_numpy(idx).cuda(), E)
    nt = gpu_notify(lay, E, 1, num_worst_tokens=R * T_r)
    assert ep.ep_read_status(nt["status"]) == ep.EP_OK
    nt = gpu_notify(lay, E, 1, num_worst_tokens=R * T_r - 1)
    assert ep.ep_read_status(nt["status"]) == ep.EP_ERR_CAPACITY
