"""The low-latency mode's two receive buffers: consecutive calls alternate
between two buffer sets, so a call's received rows stay valid through the
next call and are replaced only by the one after (bit-exact vs the oracle)."""
import pytest
import torch

from combine_get_dispatch_gb300 import ep, synth
from ep_harness import inputs, poison_
from test_gpu_ll import _compare_ll

pytestmark = pytest.mark.gpu


def _dispatch(w, x_dev, idx_dev, b):
    for key in ("packed_recv_x", "packed_recv_scales", "packed_recv_src_info", "layout_range",
                "combine_idx"):
        poison_(b[key])
    ep.ep_ll_dispatch(x_dev, idx_dev, w.E, w.max_tokens_per_rank, w.fp8_mode, b["packed_recv_x"],
                      b["packed_recv_scales"], b["packed_recv_src_info"], b["layout_range"],
                      b["recv_count"], b["combine_idx"], b["workspace"], b["status"])


@pytest.mark.parametrize("fp8_mode", [0, 2])
def test_two_buffers_alternate(fp8_mode):
    w = synth.scaled(synth.WORKLOADS["decode"], T_r=24, H=1024, fp8_mode=fp8_mode)
    bufs = ep.LowLatencyBuffers(w.R, w.T_r, w.H, w.E, w.k, w.max_tokens_per_rank, fp8_mode)
    batches = [inputs(w, seed=s) for s in range(3)]
    used = []
    for x_dev, _, idx_dev, _, _, _ in batches:
        b = bufs.next()
        b["status"] = torch.zeros(1, dtype=torch.int32, device="cuda")
        _dispatch(w, x_dev, idx_dev, b)
        used.append(b)
    torch.cuda.synchronize()
    assert used[0] is used[2] and used[0] is not used[1]
    for b in used:
        assert ep.ep_read_status(b["status"]) == ep.EP_OK
    # batch 1 is intact after batch 2 went into the other set; batch 2 replaced batch 0
    _, x1, _, idx1, _, _ = batches[1]
    _compare_ll(w, x1, idx1, used[1], w.max_tokens_per_rank, fp8_mode)
    _, x2, _, idx2, _, _ = batches[2]
    _compare_ll(w, x2, idx2, used[2], w.max_tokens_per_rank, fp8_mode)
