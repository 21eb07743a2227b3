"""The N > 1 path of bench.py on the CPU: two gloo ranks, each with its own token batch and no
data-path collective; the timing is reduced with MAX over the ranks and the whole-job rate
counts every rank's tokens over the slowest rank's time.  The reference arm runs on rank 0
alone: the other ranks return without work."""
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


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_env()
        x, lg = bench.make_workload(64, r, torch.device("cpu"))
        # the slowest rank's time decides; every rank sees it
        slowest = bench.max_over_ranks(10.0 + 5.0 * r, w, torch.device("cpu"))
        value = bench.job_throughput(w, 64, 3, slowest)
        ref = bench.run_reference(type("A", (), {})()) if r != 0 else "skipped"
        q.put((r, w, float(x.float().sum()), float(lg.sum()), slowest, value, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(world))
    (r0, w0, x0, l0, s0, v0, ref0), (r1, w1, x1, l1, s1, v1, ref1) = res
    assert (r0, r1) == (0, 1) and w0 == w1 == 2
    assert x0 != x1 and l0 != l1                    # each rank routes its own token batch
    assert s0 == s1 == 15.0                         # MAX over ranks
    assert v0 == v1 == pytest.approx(2 * 64 * 3 / 15e-3)  # all ranks' tokens over the slowest time
    assert ref1 is None                             # rank 1 does no reference work
