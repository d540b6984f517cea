"""Multi-process host logic of bench.py's N-GPU mode (replicas only): two gloo
ranks on the CPU set up the process group from the torchrun environment, take
the max of their per-rank step times, and report the whole-job value; the
reference arm does its work on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    ms = bench.max_over_ranks(1.5 + rank, w)            # per-rank step times 1.5 and 2.5 ms
    tokens = 4 * 4096
    val = bench.value_of("prefill", ms, tokens, w)       # whole job: all ranks' tokens / max time
    dec = bench.value_of("decode", ms, 64, w)
    out.put((rank, ms, val, dec))

    class A:
        workload = "prefill"
        warmup = 0
        steps = 0
    if rank != 0:
        assert bench.run_reference(A(), rank, w) is None  # non-zero ranks exit without work
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, val, dec in res:
        assert ms == 2.5
        assert val == pytest.approx(2 * 4 * 4096 / 2.5e-3, rel=1e-6)
        assert dec == pytest.approx(2500.0)               # decode: µs per step, not summed
