"""The benchmark's multi-rank host logic on the CPU: two gloo ranks (the
replicas a `--gpus 2` run launches, minus the GPU work) agree on the
slowest rank's time, count both ranks' products in the job's throughput,
and run the reference arm on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_env()
        slowest = bench.max_over_ranks(10.0 + 5.0 * r, w)  # rank 1 is slower
        dist.barrier()
        ref = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0})(), "laplace2d_64")
        out.put((r, slowest, bench.job_gflops(1000, w, slowest), ref is None))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    got = sorted(out.get() for _ in range(2))
    for rank, slowest, gflops, no_reference in got:
        assert slowest == 15.0                          # the slowest rank's time, on every rank
        assert gflops == pytest.approx(2 * 1000 * 2 / 15e-3 / 1e9)  # both ranks' products
        assert no_reference == (rank != 0)              # the reference arm runs on rank 0 only


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_gflops(500, 1, 1.0) == pytest.approx(2 * 500 / 1e-3 / 1e9)
