"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): the
timing reduction is a max over ranks, throughput counts every rank's batch,
and the reference arm runs on rank 0 only. The data path has no collective."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        worst = bench.max_over_ranks(10.0 + 5.0 * rank, w)
        tput = bench.job_tokens_per_s(1000, w, worst)
        q.put((r, w, lr, worst, tput))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    for rank, (r, w, lr, worst, tput) in enumerate(got):
        assert (r, w, lr) == (rank, 2, rank)
        assert worst == 15.0                       # slowest rank sets the step time
        assert tput == pytest.approx(2 * 1000 / 15e-3)


def test_reference_arm_only_on_rank_zero(capsys):
    sys.path.insert(0, ROOT)
    import bench
    import synth

    class A:
        steps, warmup = 1, 0
    bench.run_reference(A, synth.get_config("tiny"), rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_index_launch_count_matches_library_rule():
    """bench.py's launch count mirrors the index builder's dispatch."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.index_launches(0, 8) == 1
    assert bench.index_launches(1024, 256) == 1
    assert bench.index_launches(1025, 256) == 3
    assert bench.index_launches(131072, 256) == 3
    assert bench.index_launches(100003, 1000) == 3
