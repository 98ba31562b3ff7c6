"""Host logic of bench.py's multi-GPU mode, run as two gloo ranks on CPU.

The method has no exchange step (independent (b, h) problems), so N GPUs run N
replicas of the workload; the only cross-rank steps are the barrier and the
maximum of the per-rank times, from which the whole-job throughput is formed.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_setup()
    # each rank timed a different duration; every rank sees the slowest
    t_max = bench.max_over_ranks(10.0 + 5.0 * rank)
    dist.barrier()
    out.put((r, ws, local, t_max))
    dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    sys.path.insert(0, ROOT)
    import bench
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 0, 15.0), (1, 2, 1, 15.0)]
    # 2 replicas of 1e12 FLOP per step, 10 steps, slowest rank 15 ms
    assert bench.throughput_tflops(1e12, 2, 10, 15.0) == pytest.approx(2 * 10 * 1e12 / 0.015 / 1e12)


def test_single_process_max_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
