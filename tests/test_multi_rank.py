"""The benchmark's multi-process path on CPU: two gloo ranks on 127.0.0.1.

The sampler has no cross-canvas exchange, so N GPUs run N independent replicas and the only
collectives are the barrier around the timed region and the max-over-ranks of the elapsed
time.  The whole-job value is the steps of all ranks over the slowest rank's time.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    d = bench.init_dist(w, "gloo")
    bench.barrier(d)
    elapsed = 1.0 + rank          # rank 1 is the slowest
    value, slowest = bench.aggregate(10, elapsed, w, d)
    top = bench.max_over_ranks(d, float(rank * 7), None)
    out[rank] = (r, w, local, value, slowest, top)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_aggregate_uses_slowest_rank():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    for rank in range(2):
        r, w, local, value, slowest, top = out[rank]
        assert (r, w, local) == (rank, 2, rank)
        assert slowest == 2.0                 # max over ranks
        assert value == pytest.approx(20 / 2.0)   # all ranks' steps / slowest time
        assert top == 7.0


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.init_dist(1, "gloo") is None
    value, slowest = bench.aggregate(50, 2.0, 1)
    assert (value, slowest) == (25.0, 2.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    bench.run_reference(args, rank=1, world=2, local=1)
    assert capsys.readouterr().out == ""
