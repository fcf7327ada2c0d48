"""Benchmark: MoE dispatch + combine on one GB300 (R ranks emulated in HBM).

One step = one pass of the hot path over one batch:
  decode (default, low-latency): ep_ll_dispatch (layout + FP8 ue8m0
      scatter into the packed masked layout) + ep_ll_combine;
  prefill / large / skewed (normal mode): ep_get_dispatch_layout +
      ep_notify_dispatch (+ the host handshake unless num_worst_tokens) +
      ep_dispatch + ep_combine.
Inputs are resident in HBM before the timed region; L2 is flushed (512 MiB
write) before every step, outside the per-step CUDA events.  The JSON line
reports the large throughput workload (R=8 x 16384 tokens, H=7168, FP8 ue8m0
dispatch, bf16 combine: the largest configuration on one GPU); the other
workloads are measured in the same run under "workloads", each with its own
roofline object.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workloads large,decode,prefill,skewed,prefill_v1]
  python bench.py --sm-sweep 8,16,32,64,152 [--workloads ...]   (GB/s per SM
                  under an SM budget; one line per workload and budget)

With N > 1 (torchrun) every rank runs an independent replica (the emulated
ranks live inside one GPU; there is no data-path collective): weak scaling,
value = total tokens / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
HEADLINE = "large"
# bench-only workloads: a base workload run through another layout
# ("rank": the once-per-rank receive layout of V1's normal mode)
DERIVED = {"prefill_v1": ("prefill", {"mode": "rank"})}


def workload(name: str, tokens_per_rank: int = 0):
    """A workload by name; tokens_per_rank > 0 scales its T_r (profiling only)."""
    from combine_get_dispatch_gb300 import synth
    if name in DERIVED:
        base, changes = DERIVED[name]
        w = synth.scaled(synth.WORKLOADS[base], name=name, **changes)
    else:
        w = synth.WORKLOADS[name]
    if tokens_per_rank > 0:
        w = synth.scaled(w, T_r=tokens_per_rank,
                         max_tokens_per_rank=max(w.max_tokens_per_rank, tokens_per_rank),
                         num_worst_tokens=(w.R * tokens_per_rank if w.num_worst_tokens >= 0 else -1))
    return w
FLUSH_BYTES = 512 << 20


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workloads", default="large,decode,prefill,skewed,prefill_v1")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    # profiling aids (change the workload; never used for a reported number)
    ap.add_argument("--tokens-per-rank", type=int, default=0,
                    help="override T_r of every selected workload (profiling only)")
    ap.add_argument("--separate-layout-notify", action="store_true",
                    help="normal mode: ep_get_dispatch_layout + ep_notify_dispatch as two "
                         "launches instead of ep_layout_notify (comparison)")
    ap.add_argument("--sm-sweep", default="",
                    help="comma list of SM budgets (ep_set_num_sms): print one line per "
                         "workload and budget with GB/s per SM instead of the headline line")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- distributed

def dist_init(n_gpus: int):
    """(rank, world, local_rank); torch.distributed only when launched by torchrun."""
    if "RANK" in os.environ and "WORLD_SIZE" in os.environ and int(os.environ["WORLD_SIZE"]) > 1:
        import torch.distributed as dist
        backend = os.environ.get("EP_BENCH_BACKEND", "nccl")
        dist.init_process_group(backend=backend)
        return dist.get_rank(), dist.get_world_size(), int(os.environ.get("LOCAL_RANK", 0))
    return 0, 1, 0


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------- workloads

def alg_bytes(w, rows: int):
    """Algorithmic bytes: dispatch reads each source row once and writes one
    row per routed slot (bf16, or E4M3 + scales); combine reads one bf16 row
    per routed slot and writes one bf16 row per token."""
    row_in = 2 * w.H
    if w.fp8_mode == 0:
        row_out = 2 * w.H
    else:
        row_out = w.H + (w.H // 128) * (4 if w.fp8_mode == 1 else 1)
    dispatch = w.T * row_in + rows * row_out
    combine = rows * 2 * w.H + w.T * 2 * w.H
    return dispatch, combine


class Runner:
    """Buffers and one step of one workload on the current GPU."""

    def __init__(self, w, device, fused_layout_notify=True):
        import numpy as np
        import torch

        from combine_get_dispatch_gb300 import ep, synth
        self.w, self.dev, self.ep = w, device, ep
        self.fused_layout_notify = fused_layout_notify
        idx, wts = synth.routing(w)
        self.idx = torch.from_numpy(idx).to(device)
        self.wts = torch.from_numpy(wts).to(device)
        self.x = synth.activations_torch(w, device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.ws = ep.alloc_workspace(w.R, w.T_r, w.k, w.E, w.H, device=device)
        self.out = torch.empty_like(self.x)
        self.rows = int((idx >= 0).sum())
        self.ll = w.mode == "ll"
        self.rank = w.mode == "rank"
        # a step without a host wait can be captured in a CUDA graph
        self.capturable = self.ll or w.num_worst_tokens >= 0
        if self.ll:
            self.buf = ep.alloc_ll(w.R, w.T_r, w.H, w.E, w.k, w.max_tokens_per_rank, w.fp8_mode,
                                   device=device)
            S = w.R * w.max_tokens_per_rank
            self.y = synth.expert_outputs_torch(w.E * S, w.H, device).view(w.R, w.E_l, S, w.H)
        elif self.rank:   # once per (token, destination rank): experts' = ranks
            E_l = w.E // w.R
            r_of = np.where(idx >= 0, idx // E_l, -1)
            self.rows = int(sum(len(set(v[v >= 0].tolist())) for v in r_of.reshape(-1, w.k)))
            self.rank_ids = torch.empty_like(self.idx)
            self.lay = ep.alloc_layout(w.R, w.T_r, w.k, w.R, device=device)
            self.nt = ep.alloc_notify(w.R, w.R, device=device)
            self.host_rows = torch.empty(w.R, dtype=torch.int64).pin_memory()
            self._layout_notify()
            self.cap = (int(self.host_rows.max()) + 15) // 16 * 16
            self.buf = ep.alloc_dispatch(w.R, w.T_r, w.H, w.k, w.fp8_mode, self.cap, device=device)
            self.rtk = torch.empty((w.R, self.cap, w.k), dtype=torch.int64, device=device)
            self.rtw = torch.empty((w.R, self.cap, w.k), dtype=torch.float32, device=device)
            self.y = synth.expert_outputs_torch(w.R * self.cap, w.H, device).view(
                w.R, self.cap, w.H)
        else:
            self.lay = ep.alloc_layout(w.R, w.T_r, w.k, w.E, device=device)
            self.nt = ep.alloc_notify(w.R, w.E, device=device)
            self.host_rows = torch.empty(w.R, dtype=torch.int64).pin_memory()
            if w.num_worst_tokens >= 0:
                self.cap = w.cap_rows()
            else:   # size the receive buffers from one handshake (as the caller would),
                self._layout_notify()   # padded to a multiple of 16 rows
                self.cap = (int(self.host_rows.max()) + 15) // 16 * 16
            self.buf = ep.alloc_dispatch(w.R, w.T_r, w.H, w.k, w.fp8_mode, self.cap, device=device)
            self.y = synth.expert_outputs_torch(w.R * self.cap, w.H, device).view(
                w.R, self.cap, w.H)
        torch.cuda.synchronize()

    def _layout_notify(self, host_wait=True):
        ep, w = self.ep, self.w
        ids, E, A, nwt = self.idx, w.E, w.expert_alignment, w.num_worst_tokens
        if self.rank:   # experts' = ranks, over the per-slot destination ranks
            ep.ep_rank_ids(self.idx, w.E, self.rank_ids, self.status)
            ids, E, A, nwt = self.rank_ids, w.R, 1, -1
        host = self.host_rows if (nwt < 0 and host_wait) else None
        if self.fused_layout_notify:   # one launch (ep_layout_notify)
            ep.ep_layout_notify(ids, E, A, nwt, self.lay, self.nt, self.ws, host, 10000,
                                self.status)
            return
        ep.ep_get_dispatch_layout(ids, E, self.lay["num_tokens_per_rank"],
                                  self.lay["num_tokens_per_expert"], self.lay["is_token_in_rank"],
                                  self.lay["slot_rank"], self.ws, self.status)
        ep.ep_notify_dispatch(self.lay["num_tokens_per_rank"], self.lay["num_tokens_per_expert"],
                              A, nwt, self.nt["rank_prefix_matrix"], self.nt["expert_prefix"],
                              self.nt["num_recv_tokens_per_expert"], self.nt["psum"], host, 10000,
                              self.status)

    def step_single_call(self):
        """Fixed-shape normal mode: ep_layout_notify_dispatch (layout + notify,
        then the dispatch as its programmatic dependent), then the combine."""
        ep, w, b = self.ep, self.w, self.buf
        ep.ep_layout_notify_dispatch(self.x, self.idx, w.E, w.fp8_mode, w.expert_alignment,
                                     w.num_worst_tokens, self.cap, self.lay, self.nt, b, self.ws,
                                     self.status)
        ep.ep_combine(self.y, self.wts, b["combine_idx"], self.cap, self.out, self.status)

    def step(self, ev=None):
        """One pass; ev = (e0, e1, e2, e3) events around dispatch / combine.
        With ev (the per-kernel split), normal mode skips the host wait for
        the receive counts (the buffers are already sized), so the host
        enqueues the whole step at once and no host latency falls between
        the events."""
        ep, w, b = self.ep, self.w, self.buf
        if self.ll:
            if ev:
                ev[0].record()
            ep.ep_ll_dispatch(self.x, self.idx, w.E, w.max_tokens_per_rank, w.fp8_mode,
                              b["packed_recv_x"], b["packed_recv_scales"],
                              b["packed_recv_src_info"], b["layout_range"], b["recv_count"],
                              b["combine_idx"], self.ws, self.status)
            if ev:
                ev[1].record()
                ev[2].record()
            ep.ep_ll_combine(self.y, self.wts, b["combine_idx"], w.E, w.max_tokens_per_rank,
                             self.out, self.status)
            if ev:
                ev[3].record()
        elif self.rank:
            self._layout_notify(host_wait=ev is None)
            if ev:
                ev[0].record()
            ep.ep_dispatch(self.x, self.rank_ids, self.lay["slot_rank"], self.nt["expert_prefix"],
                           self.nt["psum"], w.R, w.fp8_mode, self.cap, b["recv_x"],
                           b["recv_scales"], b["recv_src_idx"], b["combine_idx"], self.ws,
                           self.status)
            ep.ep_rank_recv_topk(self.idx, self.wts, b["combine_idx"], w.E, self.cap, self.rtk,
                                 self.rtw, self.status)
            if ev:
                ev[1].record()
                ev[2].record()
            ep.ep_rank_combine(self.y, b["combine_idx"], self.cap, self.out, self.status)
            if ev:
                ev[3].record()
        else:
            self._layout_notify(host_wait=ev is None)
            if ev:
                ev[0].record()
            ep.ep_dispatch(self.x, self.idx, self.lay["slot_rank"], self.nt["expert_prefix"],
                           self.nt["psum"], w.E, w.fp8_mode, self.cap, b["recv_x"],
                           b["recv_scales"], b["recv_src_idx"], b["combine_idx"], self.ws,
                           self.status)
            if ev:
                ev[1].record()
                ev[2].record()
            ep.ep_combine(self.y, self.wts, b["combine_idx"], self.cap, self.out, self.status)
            if ev:
                ev[3].record()


def workload_desc(w) -> str:
    fp8 = {0: "bf16", 1: "FP8 E4M3 + fp32 per-128 scales", 2: "FP8 E4M3 + ue8m0 per-128 scales"}
    mode = {"ll": "low-latency packed", "rank": "once-per-rank (V1) normal"}.get(
        w.mode, "normal contiguous")
    extra = f", num_worst_tokens={w.num_worst_tokens}" if w.num_worst_tokens >= 0 else ""
    return (f"{w.name}: R={w.R} x {w.T_r} tokens/rank, H={w.H}, E={w.E} ({w.E_l}/rank), "
            f"top-{w.k}, {fp8[w.fp8_mode]} {mode} dispatch + bf16 combine{extra}")


class no_gc:
    """Python's garbage collector off for a timed loop: a collection in the
    middle of it stalls the host for milliseconds, and a step that waits on
    the host for its receive counts then takes the stall on the GPU clock.
    (No collection before it: a full collection made the host-waiting steps
    ~20 us slower, the freed memory being faulted back in by the loop.)"""

    def __enter__(self):
        self.was = gc.isenabled()
        gc.disable()
        return self

    def __exit__(self, *exc):
        if self.was:
            gc.enable()
        return False


def measure(runner, steps: int, warmup: int, world: int, flush, e2e: bool):
    import torch

    ep = runner.ep
    for _ in range(warmup):
        flush.fill_(1)
        runner.step()
    torch.cuda.synchronize()
    code = ep.ep_read_status(runner.status)
    if code != ep.EP_OK:
        raise RuntimeError(f"{runner.w.name}: kernel status {ep.error_string(code)}")
    # the step as a user runs it: events only around it
    outer = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(steps)]
    barrier(world, runner.dev)
    torch.cuda.synchronize()
    launches0 = ep.ep_launch_count()
    with no_gc():
        t_wall = time.perf_counter()
        for s in range(steps):
            flush.fill_(s & 0xFF)
            outer[s][0].record()
            runner.step()
            outer[s][1].record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_wall
    barrier(world, runner.dev)
    launches = ep.ep_launch_count() - launches0
    step_ms = [a.elapsed_time(b) for a, b in outer]
    # the same steps again with events between dispatch and combine (their
    # split; the extra events cost the step a few microseconds; normal mode
    # enqueues the step without the host wait for the receive counts)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    torch.cuda.synchronize()
    with no_gc():
        for s in range(steps):
            flush.fill_(s & 0xFF)
            evs[s][4].record()   # step start: layout + notify run before e[0] in normal mode
            runner.step(evs[s][:4])
        torch.cuda.synchronize()
    disp_ms = [e[0].elapsed_time(e[1]) for e in evs]
    comb_ms = [e[2].elapsed_time(e[3]) for e in evs]
    ln_ms = [e[4].elapsed_time(e[0]) for e in evs]
    def stats_us(v):
        q = sorted(v)
        return {"median": round(statistics.median(q) * 1e3, 2), "min": round(q[0] * 1e3, 2),
                "p90": round(q[min(len(q) - 1, int(0.9 * len(q)))] * 1e3, 2),
                "max": round(q[-1] * 1e3, 2)}

    res = {"step_ms": statistics.mean(step_ms), "step_ms_min": min(step_ms),
           "step_us_stats": stats_us(step_ms), "dispatch_us_stats": stats_us(disp_ms),
           "combine_us_stats": stats_us(comb_ms),
           "dispatch_ms": statistics.mean(disp_ms), "combine_ms": statistics.mean(comb_ms),
           "layout_notify_ms": statistics.mean(ln_ms),
           "launches": launches, "wall_s": wall}
    if e2e:
        res["e2e"] = measure_e2e(runner, steps, world, flush)
    return res


def measure_single_call(runner, steps, flush):
    """The fixed-shape normal step through ep_layout_notify_dispatch: device
    time per step (events around it, L2 flushed before each) and its
    launch-inclusive latency, eager and replayed as a CUDA graph."""
    import torch

    for _ in range(3):
        flush.fill_(1)
        runner.step_single_call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for s in range(steps):
        flush.fill_(s & 0xFF)
        ev[s][0].record()
        runner.step_single_call()
        ev[s][1].record()
    torch.cuda.synchronize()
    code = runner.ep.ep_read_status(runner.status)
    if code != runner.ep.EP_OK:
        raise RuntimeError(f"{runner.w.name}: kernel status {runner.ep.error_string(code)}")
    out = {"step_us": round(statistics.median(a.elapsed_time(b) for a, b in ev) * 1e3, 2)}
    step = runner.step
    runner.step = runner.step_single_call    # the latency helper captures runner.step
    try:
        out.update(measure_launch_latency(runner, steps, flush) or {})
    finally:
        runner.step = step
    return out


def measure_launch_latency(runner, steps, flush):
    """Launch-inclusive latency of one step (host call to completion, after
    a synchronize on both sides): eager through the API, and the same step
    captured once in a CUDA graph and replayed; plus the replay's device time
    (CUDA events).  None for steps that wait on the host (normal mode without
    num_worst_tokens cannot be captured)."""
    import torch

    if not runner.capturable:
        return None

    def wall(fn):
        lat = []
        for s in range(steps):
            flush.fill_(s & 0xFF)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            lat.append((time.perf_counter() - t0) * 1e6)
        return statistics.median(lat)

    eager = wall(runner.step)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        runner.step()              # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        runner.step()
    graph = wall(g.replay)
    dev = []
    for s in range(steps):
        flush.fill_(s & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        dev.append(e0.elapsed_time(e1) * 1e3)
    del g
    code = runner.ep.ep_read_status(runner.status)
    if code != runner.ep.EP_OK:
        raise RuntimeError(f"{runner.w.name}: kernel status {runner.ep.error_string(code)}")
    return {"eager_us": round(eager, 1), "graph_us": round(graph, 1),
            "graph_device_us": round(statistics.median(dev), 1)}


def measure_e2e(runner, steps, world, flush):
    """The step through the public API with its inputs copied from pinned
    host memory and its result copied back to pinned host memory, all inside
    the timed region, two ways:

    * serial: one step at a time (upload, dispatch, combine writing its
      output straight into the pinned buffer -- the API accepts pinned host
      memory for `out` -- so the download is the combine's own stores across
      the host link), timed step by step after an L2 flush: the latency of
      one step with its copies;
    * pipelined (the reported throughput): uploads on one copy stream,
      dispatch + combine (output in HBM) on the compute stream, downloads on
      a second copy stream, inputs and outputs double-buffered, so step s+1's
      upload (queued before step s's own calls) and step s-1's download run
      while step s computes.  Every step
      still moves its own inputs and result across the link.  The K steps
      are captured once as one CUDA graph and replayed (issuing the copies,
      event waits and two API calls of a step from Python takes longer than
      the step itself); steps that wait on the host run the same loop
      eagerly.  No flush: a step's working set (inputs, receive buffers,
      expert outputs, output) is several times the L2.  The last two host
      outputs are checked against a plain device step."""
    import torch

    hx = runner.x.cpu().pin_memory()
    hi = runner.idx.cpu().pin_memory()
    hw = runner.wts.cpu().pin_memory()
    ho = torch.empty(runner.out.shape, dtype=runner.out.dtype).pin_memory()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    dev_out = runner.out
    runner.out = ho
    try:
        barrier(world, runner.dev)
        torch.cuda.synchronize()
        with no_gc():
            for s in range(steps):
                flush.fill_(s & 0xFF)
                evs[s][0].record()
                runner.x.copy_(hx, non_blocking=True)
                runner.idx.copy_(hi, non_blocking=True)
                runner.wts.copy_(hw, non_blocking=True)
                runner.step()
                evs[s][1].record()
            torch.cuda.synchronize()
    finally:
        runner.out = dev_out
    serial_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)

    s_in, s_out = torch.cuda.Stream(runner.dev), torch.cuda.Stream(runner.dev)
    xs = [runner.x, torch.empty_like(runner.x)]
    ids = [runner.idx, torch.empty_like(runner.idx)]
    wts = [runner.wts, torch.empty_like(runner.wts)]
    outs = [runner.out, torch.empty_like(runner.out)]
    hos = [ho, torch.empty_like(ho).pin_memory()]
    in_ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    saved = (runner.x, runner.idx, runner.wts, runner.out)

    def upload(s):
        j = s % 2
        with torch.cuda.stream(s_in):
            if s >= 2:
                s_in.wait_event(in_free[j])         # step s-2 has read this input slot
            xs[j].copy_(hx, non_blocking=True)
            ids[j].copy_(hi, non_blocking=True)
            wts[j].copy_(hw, non_blocking=True)
            in_ready[j].record(s_in)

    def run(n, comp):
        s_in.wait_stream(comp)
        s_out.wait_stream(comp)
        upload(0)
        for s in range(n):
            j = s % 2
            # the next step's upload is queued before this step's API calls:
            # a step that waits on the host for its receive counts then no
            # longer holds the upload stream back while the host wakes up
            if s + 1 < n:
                upload(s + 1)
            comp.wait_event(in_ready[j])
            if s >= 2:
                comp.wait_event(out_free[j])        # step s-2's output has left this slot
            runner.x, runner.idx, runner.wts, runner.out = xs[j], ids[j], wts[j], outs[j]
            runner.step()
            in_free[j].record(comp)
            out_ready[j].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(out_ready[j])
                hos[j].copy_(outs[j], non_blocking=True)
                out_free[j].record(s_out)
        comp.wait_stream(s_in)
        comp.wait_stream(s_out)

    comp = torch.cuda.current_stream()
    try:
        torch.cuda.synchronize()
        run(4, comp)                                # warm-up: pages and streams touched
        torch.cuda.synchronize()
        graph = None
        if runner.capturable:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                run(steps, torch.cuda.current_stream())
            graph.replay()                          # warm-up replay
            torch.cuda.synchronize()
        barrier(world, runner.dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with no_gc():
            t0.record(comp)
            if graph is not None:
                graph.replay()
            else:
                run(steps, comp)
            t1.record(comp)
            torch.cuda.synchronize()
        del graph
    finally:
        runner.x, runner.idx, runner.wts, runner.out = saved
    pipe_ms = t0.elapsed_time(t1) / steps
    runner.step()                                   # the reference result, on the device
    torch.cuda.synchronize()
    ref = runner.out.cpu()
    for h in hos:
        if not torch.equal(h.view(torch.int16), ref.view(torch.int16)):
            raise RuntimeError("pipelined end-to-end step: host output differs from the device step")
    h2d = hx.numel() * hx.element_size() + hi.numel() * 8 + hw.numel() * 4
    d2h = ho.numel() * ho.element_size()
    how = ("the K steps replayed as one CUDA graph" if runner.capturable else
           "issued eagerly: the step waits on the host for its receive counts")
    return {"ms": pipe_ms, "serial_ms": serial_ms, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "mode": ("pipelined: next upload and previous download overlap the kernels "
                     f"(copy streams, double-buffered host I/O, {how}, no L2 flush)")}


def kernel_hash(path: str) -> str:
    """Hash of a kernel source's code: comments and whitespace removed, so
    that a comment edit does not void DRAM counters taken on the same code.
    (A literal holding a comment marker would be cut short; the kernel
    sources hold none that matters to this.)"""
    with open(path, encoding="utf-8") as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    src = " ".join(src.split())
    return hashlib.sha256(src.encode()).hexdigest()[:16]


def load_traffic(kernel: str, workload: str, src: str):
    """dram bytes per launch from the committed ncu summary, if it still
    matches the kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        ent = d[f"{kernel}:{workload}"]
        if ent.get("source_sha") == kernel_hash(src):
            return ent["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        pass
    return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# ---------------------------------------------------------------- CPU oracle

def oracle_step(w, x_bits, idx, wts, y_rows, tokens_per_rank: int):
    """The oracle's dispatch + combine on the first tokens_per_rank tokens of
    every rank (a bounded sample of the workload).  Returns tokens done."""
    import numpy as np

    import oracle
    xs = np.ascontiguousarray(x_bits[:, :tokens_per_rank])
    ids = np.ascontiguousarray(idx[:, :tokens_per_rank])
    ws = np.ascontiguousarray(wts[:, :tokens_per_rank])
    if w.mode == "ll":
        d = oracle.ll_dispatch(xs, ids, w.E, w.max_tokens_per_rank, w.fp8_mode, fill=None)
    elif w.mode == "rank":   # once-per-rank layout: at most one row per (token, rank)
        d = oracle.rank_dispatch(xs, ids, ws, w.E, w.fp8_mode, w.R * tokens_per_rank, fill=None)
        cidx = d["combine_idx"]
        m = cidx >= 0
        remap = np.full(cidx.shape, -1, np.int32)
        remap[m] = np.arange(int(m.sum()), dtype=np.int32)
        oracle.rank_combine(y_rows[: int(m.sum())], remap, w.H)
        return w.R * tokens_per_rank
    else:
        lay = oracle.layout(ids, w.R, w.E)
        nt = oracle.notify(lay["num_tokens_per_rank"], lay["num_tokens_per_expert"], w.R, w.E,
                           w.expert_alignment)
        cap = max(1, int(nt["psum"][:, -1].max()))
        d = oracle.dispatch(xs, ids, lay["slot_rank"], nt["expert_prefix"], nt["psum"], w.E,
                            w.fp8_mode, cap, fill=None)
    cidx = d["combine_idx"]
    # expert outputs for the rows this sample routes to (stand-in values)
    m = cidx >= 0
    remap = np.full(cidx.shape, -1, np.int32)
    remap[m] = np.arange(int(m.sum()), dtype=np.int32)
    oracle.combine(y_rows[: int(m.sum())], ws, remap, w.H)
    return w.R * tokens_per_rank


class one_core:
    """Pin this process to one of its allowed CPUs for the oracle's timing
    (it is single-threaded; the pin makes the core count exact), then
    restore the previous affinity."""

    def __enter__(self):
        self.saved = None
        if hasattr(os, "sched_getaffinity"):
            try:
                self.saved = os.sched_getaffinity(0)
                os.sched_setaffinity(0, {min(self.saved)})
            except OSError:
                self.saved = None
        return self

    def __exit__(self, *exc):
        if self.saved is not None:
            os.sched_setaffinity(0, self.saved)
        return False


def oracle_sample_tokens(w) -> int:
    """Tokens per rank in one oracle sample step: about 512 tokens in all
    (half a second of the single-threaded oracle at H = 7168), at least one
    per rank, never more than the workload has."""
    return max(1, min(w.T_r, 512 // w.R))


def cpu_baseline(w, budget_s: float = 12.0, alg_bytes_per_token: float = 0.0):
    import numpy as np

    import oracle
    from combine_get_dispatch_gb300 import synth
    oracle.build()
    idx, wts = synth.routing(w)
    tpr = oracle_sample_tokens(w)
    sub = synth.scaled(w, T_r=tpr)
    x_bits = synth.activations(sub)
    y_rows = synth.expert_outputs(w.R * tpr * w.k, w.H)
    with one_core():
        done, t0, reps = 0, time.perf_counter(), 0
        while True:
            done += oracle_step(w, x_bits, idx, wts, y_rows, tpr)
            reps += 1
            if time.perf_counter() - t0 >= budget_s or reps >= 500:
                break
        el = time.perf_counter() - t0
    out = {"value": done / el, "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "sample": (f"{reps} x oracle dispatch+combine of the first {tpr} tokens of each of "
                      f"the {w.R} ranks ({w.R * tpr} tokens, 1/{w.T_r // tpr} of the workload), "
                      f"single-threaded C pinned to one core, {el:.1f} s")}
    if alg_bytes_per_token > 0:   # the same algorithmic bytes per token as the GPU line
        out["gbs"] = round(done / el * alg_bytes_per_token / 1e9, 3)
    return out


# ---------------------------------------------------------------- main

def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from combine_get_dispatch_gb300 import synth
    w = synth.WORKLOADS[HEADLINE]
    import numpy as np

    import oracle
    oracle.build()
    idx, wts = synth.routing(w)
    tpr = oracle_sample_tokens(w)
    sub = synth.scaled(w, T_r=tpr)
    x_bits = synth.activations(sub)
    y_rows = synth.expert_outputs(w.R * tpr * w.k, w.H)
    times = []
    with one_core():
        for _ in range(args.warmup):
            oracle_step(w, x_bits, idx, wts, y_rows, tpr)
        for _ in range(args.steps):
            t0 = time.perf_counter()
            n = oracle_step(w, x_bits, idx, wts, y_rows, tpr)
            times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = n / (ms / 1e3)
    sample = (f"oracle (single-threaded C, pinned to one core) dispatch+combine of the first "
              f"{tpr} tokens of each "
              f"of the {w.R} ranks per step ({n} tokens)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": config_of(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_sm_sweep(args, local_rank):
    """Dispatch / combine bandwidth per SM under an SM budget (the kernels
    confined to n SMs), one JSON line per (workload, budget): the per-SM
    read and write rates that size a budget (num_sms = traffic / per-SM
    rate, the bandwidth model of the DeepEP article's §4.6)."""
    import torch

    from combine_get_dispatch_gb300 import ep, synth
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ep.load()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    budgets = [int(b) for b in args.sm_sweep.split(",") if b.strip()]
    try:
        for name in [n.strip() for n in args.workloads.split(",") if n.strip()]:
            w = workload(name, args.tokens_per_rank)
            runner = Runner(w, dev)
            row_in = 2 * w.H
            row_out = (2 * w.H if w.fp8_mode == 0
                       else w.H + (w.H // 128) * (4 if w.fp8_mode == 1 else 1))
            d_rd, d_wr = w.T * row_in, runner.rows * row_out
            c_rd, c_wr = runner.rows * 2 * w.H, w.T * 2 * w.H
            for b in budgets:
                ep.ep_set_num_sms(b)
                n = ep.ep_get_num_sms()
                res = measure(runner, args.steps, args.warmup, 1, flush, e2e=False)
                d_s, c_s = res["dispatch_ms"] * 1e-3, res["combine_ms"] * 1e-3
                print(json.dumps({
                    "sm_sweep": name, "num_sms": n,
                    "dispatch_us": round(d_s * 1e6, 2), "combine_us": round(c_s * 1e6, 2),
                    "dispatch_gbs": round((d_rd + d_wr) / d_s / 1e9, 1),
                    "combine_gbs": round((c_rd + c_wr) / c_s / 1e9, 1),
                    "dispatch_read_gbs_per_sm": round(d_rd / d_s / 1e9 / n, 2),
                    "dispatch_write_gbs_per_sm": round(d_wr / d_s / 1e9 / n, 2),
                    "combine_read_gbs_per_sm": round(c_rd / c_s / 1e9 / n, 2),
                    "combine_write_gbs_per_sm": round(c_wr / c_s / 1e9 / n, 2)}), flush=True)
            del runner
            torch.cuda.empty_cache()
    finally:
        ep.ep_set_num_sms(0)
    return 0


def run_ours(args, rank, world, local_rank):
    import torch

    from combine_get_dispatch_gb300 import ep, synth
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ep.load()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peak, peak_kind = peaks()
    names = [n.strip() for n in args.workloads.split(",") if n.strip()]
    head = names[0]
    results = {}
    clocks = None
    for name in names:
        w = workload(name, args.tokens_per_rank)
        runner = Runner(w, dev, fused_layout_notify=not args.separate_layout_notify)
        sampler = ClockSampler(local_rank) if name == head else None
        if sampler:
            sampler.start()
        res = measure(runner, args.steps, args.warmup, world, flush,
                      e2e=(name == head and not args.no_e2e))
        if sampler:
            clocks = sampler.stop()
        res["step_ms_max"] = max_over_ranks(res["step_ms"], world)
        dbytes, cbytes = alg_bytes(w, runner.rows)
        res["dispatch_alg_bytes"], res["combine_alg_bytes"] = dbytes, cbytes
        res["dispatch_gbs"] = dbytes / (res["dispatch_ms"] * 1e-3) / 1e9
        res["combine_gbs"] = cbytes / (res["combine_ms"] * 1e-3) / 1e9
        res["tokens"] = w.T
        if name == head or name == "skewed":
            res["launch_latency_us"] = measure_launch_latency(runner, args.steps, flush)
        if not runner.ll and not runner.rank and w.num_worst_tokens >= 0:
            res["single_call"] = measure_single_call(runner, args.steps, flush)
        results[name] = (w, runner, res)
        if name != head:
            del runner
            torch.cuda.empty_cache()

    line = assemble_line(args, world, head, results, clocks, peak, peak_kind)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            def per_token(r, wo):
                return (r["dispatch_alg_bytes"] + r["combine_alg_bytes"]) / wo.T
            wh, _, rh = results[head]
            line["cpu_baseline"] = cpu_baseline(wh, alg_bytes_per_token=per_token(rh, wh))
            # every other workload's oracle, once each on a shorter sample
            for name, (wo, _, r) in results.items():
                if name != head:
                    line["workloads"][name]["cpu_baseline"] = cpu_baseline(
                        wo, budget_s=3.0, alg_bytes_per_token=per_token(r, wo))
        print(json.dumps(line), flush=True)
    return 0


def config_of(w, world: int) -> dict:
    """The workload's config object (shared by both arms' lines)."""
    return {"workload": workload_desc(w), "l2": "flushed before every step (512 MiB write)",
            "parallelism": f"{world} replica(s), {w.R} ranks emulated per GPU",
            "data_types": ("x bf16 -> " + {0: "bf16", 1: "E4M3 + fp32 scales",
                                              2: "E4M3 + ue8m0 scales"}[w.fp8_mode]
                           + " dispatch; y bf16 -> bf16 combine, fp32 accumulate")}


def roofline_of(name, w, runner, res, peak, peak_kind):
    """Roofline object of a workload's dominant kernel (the longer of its
    dispatch and combine): algorithmic bytes per launch over the CUDA-event
    time of the launch, against the HBM copy peak; traffic = DRAM bytes per
    launch from the committed ncu summary while the kernel source is
    unchanged since it was taken, else null."""
    dom = "combine" if res["combine_ms"] >= res["dispatch_ms"] else "dispatch"
    kern = {"combine": "k_combine", "dispatch": "k_ll_fused" if runner.ll else "k_scatter"}[dom]
    src = os.path.join(ROOT, "combine_get_dispatch_gb300", "csrc",
                       "combine.cu" if dom == "combine"
                       else ("ll_fused.cu" if runner.ll else "dispatch.cu"))
    achieved = res[f"{dom}_gbs"]
    return {"bound": "hbm", "kernel": kern, "achieved": round(achieved, 1),
            "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "peak_source": f"{peak_kind} hbm_gbs",
            "alg_bytes_per_launch": res[f"{dom}_alg_bytes"],
            "launch_us": round(res[f"{dom}_ms"] * 1e3, 2),
            "traffic": load_traffic(kern, name, src)}


def assemble_line(args, world, head, results, clocks, peak, peak_kind):
    """The contract's JSON line from the per-workload measurements (results:
    name -> (workload, runner, measured dict); the headline first)."""
    w, runner, res = results[head]
    ms = res["step_ms_max"]
    value = world * w.T / (ms * 1e-3)
    e2e = None
    if "e2e" in res:
        e2e_ms = max_over_ranks(res["e2e"]["ms"], world)
        serial_ms = max_over_ranks(res["e2e"]["serial_ms"], world)
        e2e = {"value": world * w.T / (e2e_ms * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": res["e2e"]["h2d_bytes_per_step"],
               "d2h_bytes_per_step": res["e2e"]["d2h_bytes_per_step"], "ms_per_step": e2e_ms,
               "mode": res["e2e"].get("mode", "pipelined"),
               "serial_ms_per_step": serial_ms,
               "serial_value": world * w.T / (serial_ms * 1e-3)}
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": config_of(w, world),
            "hbm_gbs": {"dispatch": round(res["dispatch_gbs"], 1),
                        "combine": round(res["combine_gbs"], 1),
                        "dispatch_frac": round(res["dispatch_gbs"] / peak, 4),
                        "combine_frac": round(res["combine_gbs"] / peak, 4)},
            "clocks": clocks, "e2e": e2e, "gpu_launches": res["launches"],
            "roofline": roofline_of(head, w, runner, res, peak, peak_kind)}
    if "wall_s" in res:
        line["timed_region_s"] = round(res["wall_s"], 4)
    others = {}
    for name, (wo, ro, r) in results.items():
        if name == head:
            continue
        others[name] = {
            "workload": workload_desc(wo), "tokens_per_s": wo.T / (r["step_ms_max"] * 1e-3),
            "ms_per_step": round(r["step_ms_max"], 4),
            "dispatch_ms": round(r["dispatch_ms"], 4), "combine_ms": round(r["combine_ms"], 4),
            "dispatch_gbs": round(r["dispatch_gbs"], 1), "combine_gbs": round(r["combine_gbs"], 1),
            "dispatch_frac": round(r["dispatch_gbs"] / peak, 4),
            "combine_frac": round(r["combine_gbs"] / peak, 4),
            "layout_notify_ms": round(r.get("layout_notify_ms", 0.0), 4),
            "gpu_launches": r["launches"],
            "roofline": roofline_of(name, wo, ro, r, peak, peak_kind)}
        if r.get("launch_latency_us"):
            others[name]["launch_latency_us"] = r["launch_latency_us"]
        if r.get("single_call"):
            others[name]["single_call"] = r["single_call"]
        for key in ("step_us_stats", "dispatch_us_stats", "combine_us_stats"):
            others[name][key] = r[key]
    line["workloads"] = others
    line["kernels_ms"] = {"dispatch": round(res["dispatch_ms"], 5),
                          "combine": round(res["combine_ms"], 5),
                          "layout_notify": round(res.get("layout_notify_ms", 0.0), 5)}
    if res.get("launch_latency_us"):
        line["launch_latency_us"] = res["launch_latency_us"]
    if res.get("single_call"):
        line["single_call"] = res["single_call"]
    for key in ("step_us_stats", "dispatch_us_stats", "combine_us_stats"):
        line[key] = res[key]
    return line


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_init(args.gpus)
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world)
        if args.sm_sweep:
            return run_sm_sweep(args, local_rank) if rank == 0 else 0
        return run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
