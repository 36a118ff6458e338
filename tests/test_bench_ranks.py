"""Multi-process host logic of bench.py on CPU: two gloo ranks.

bench.py runs one process per GPU (replicas: every rank times the same
workload, no data-path collective).  What the ranks do share is host logic:
the barrier around the timed region, the maximum of the per-rank times and
the sum of the per-rank work, and rank 0 alone running the CPU reference arm.
Those are exercised here with the gloo backend, world size 2.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    try:
        w, r, _ = bench.dist_setup()
        assert (w, r) == (world, rank)
        assert dist.get_backend() == "gloo"
        bench.barrier(w)
        t_max = bench.max_over_ranks(1.0 + rank, w, "cpu")   # per-rank elapsed times 1.0 and 2.0
        units = bench.sum_over_ranks(10.0 * (rank + 1), w, "cpu")  # per-rank work 10 and 20
        # only rank 0 runs the reference arm; the others return at once
        ref = None
        if rank != 0:
            class A:  # the parsed arguments run_reference would read
                steps, warmup = 1, 3
            ref = bench.run_reference(A(), w, rank)
        bench.barrier(w)
        q.put((rank, t_max, units, ref))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, t_max, units, ref in got:
        assert t_max == 2.0      # the job takes as long as its slowest rank
        assert units == 30.0     # whole-job work is the sum over ranks
        assert ref is None
