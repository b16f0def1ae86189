"""The multi-GPU bench path is replicas only (no collective on the KDA path):
its host logic -- rank discovery from the launcher's environment, the barrier,
the max over ranks of the per-step time and the whole-job rate -- checked with
two gloo ranks on the CPU, and the reference arm's non-zero ranks exiting
without work."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        env = bench.dist_env()
        ms = bench.max_over_ranks(1.5 * (rank + 1), ws)   # rank r took 1.5 (r + 1) ms per step
        bench.barrier(ws)
        q.put((rank, env, ms, bench.aggregate_rate(1000.0, ms, ws)))
    finally:
        torch.distributed.destroy_process_group()


def test_replicas_max_over_ranks_and_rate():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, env, ms, rate in sorted(out):
        assert env == (ws, rank, rank)
        assert ms == pytest.approx(3.0)                        # the slowest rank's time
        assert rate == pytest.approx(1000.0 / 3e-3 * ws)       # all ranks' units over it


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    bench.barrier(1)
    assert bench.aggregate_rate(500.0, 2.0, 1) == pytest.approx(250000.0)


def test_reference_arm_nonzero_rank_does_no_work(capsys):
    sys.path.insert(0, ROOT)
    import bench
    assert bench.run_reference(None, 2, 1) is None
    assert capsys.readouterr().out == ""
