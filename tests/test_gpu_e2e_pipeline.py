"""The end-to-end loop the benchmark times (uploads on one copy stream,
dispatch + combine on the compute stream, downloads on another, host buffers
double-buffered, the steps captured as one CUDA graph where the step allows
it): every step's host output must equal a plain device step's output.
measure_e2e raises if it does not."""
import pytest
import torch

import bench
from combine_get_dispatch_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,T_r", [("tiny", 16), ("decode", 32), ("skewed", 24),
                                      ("prefill", 16)])
def test_pipelined_end_to_end_outputs(name, T_r):
    """decode, tiny: low-latency steps (captured); skewed: fixed-shape normal
    steps (captured); prefill: normal steps with a host handshake (eager)."""
    dev = torch.device("cuda:0")
    w = synth.WORKLOADS[name]
    nwt = w.R * T_r if w.num_worst_tokens >= 0 else -1
    w = synth.scaled(w, T_r=T_r, num_worst_tokens=nwt)
    runner = bench.Runner(w, dev)
    flush = torch.empty(1 << 20, dtype=torch.uint8, device=dev)
    for steps in (1, 2, 5):
        res = bench.measure_e2e(runner, steps, 1, flush)
        assert res["ms"] > 0 and res["serial_ms"] > 0
        assert res["h2d_bytes_per_step"] == (runner.x.numel() * 2 + runner.idx.numel() * 8
                                             + runner.wts.numel() * 4)
        assert res["d2h_bytes_per_step"] == runner.out.numel() * 2
