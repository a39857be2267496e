"""The benchmark's multi-rank logic on CPU with two gloo ranks: each rank runs
its own batch (no collective on the data path); the job time is the slowest
rank's and the whole-job rate counts every rank's units."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, _ = bench.dist_setup(world)
    assert (w, r) == (world, rank)
    bench.barrier(w)
    t = 0.5 + rank  # rank 1 is the slow one
    slowest = bench.max_over_ranks(t, w)
    rate = bench.whole_job_rate(100.0, w, slowest)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((rank, slowest, rate))


@pytest.mark.parametrize("world", [2])
def test_two_gloo_ranks_take_the_slowest_time(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, slowest, rate in got:
        assert slowest == 1.5
        assert rate == pytest.approx(100.0 * world / 1.5)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import argparse
    import bench
    args = argparse.Namespace(workload="tiny_f32", steps=3, warmup=3, reference_seconds=1.0)
    assert bench.run_reference(args, 2, 1) is None
    line = bench.run_reference(args, 1, 0)
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
