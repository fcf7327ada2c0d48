"""The benchmark's multi-process harness (N replicas, one per GPU on a real
node) exercised on CPU with the gloo backend at world size 2: rendezvous on
127.0.0.1, barrier, max-over-ranks timing, and the reference arm's rule that
only rank 0 does work."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), EP_BENCH_BACKEND="gloo")
    try:
        r, w, lr = bench.dist_init(world)
        assert (r, w, lr) == (rank, world, rank)
        bench.barrier(w)
        # each rank "measured" a different step time; the job time is the max
        mx = bench.max_over_ranks(1.0 + rank, w)
        # the reference arm: ranks other than 0 leave without work or output
        args = bench.parse_args(["--impl", "reference", "--gpus", str(world)])
        rc = bench.run_reference(args, r, w) if r != 0 else 0
        bench.barrier(w)
        import torch.distributed as dist
        dist.destroy_process_group()
        q.put((rank, mx, rc))
    except Exception as exc:  # pragma: no cover - reported to the parent
        q.put((rank, repr(exc), -1))


def test_two_rank_gloo_harness():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
    assert [r[0] for r in res] == [0, 1]
    for rank, mx, rc in res:
        assert rc == 0, mx
        assert mx == pytest.approx(2.0)


def test_single_process_defaults():
    for k in ("RANK", "WORLD_SIZE"):
        os.environ.pop(k, None)
    assert bench.dist_init(1) == (0, 1, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
    args = bench.parse_args([])
    assert args.gpus == 1 and args.steps >= 1 and args.warmup >= 3
    # algorithmic bytes of the decode workload (the roofline's numerator)
    from combine_get_dispatch_gb300 import synth
    w = synth.WORKLOADS["decode"]
    d, c = bench.alg_bytes(w, w.T * w.k)
    assert d == 2048 * 14336 + 16384 * (7168 + 56)
    assert c == 16384 * 14336 + 2048 * 14336
