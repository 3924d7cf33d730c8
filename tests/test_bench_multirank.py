"""bench.py's multi-rank plumbing on CPU: two gloo ranks, as torchrun would start them.

Each rank reports its own step time and bytes; the job's time is the slowest rank's and its bytes
are the sum (weak scaling: every rank decodes its own sequences, with no collective on the data
path). Rank seeds differ so that replicas do not decode identical inputs.
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    assert bench.dist_env() == (rank, world, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        t, b = bench.reduce_max_sum(10.0 + 5.0 * rank, 1000.0 * (rank + 1))
        out[rank] = (t, b, bench.rank_seed(1002, rank))
        bench.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_bytes():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True,
                           start_method="spawn")
        got = dict(out)
    assert got[0][:2] == (15.0, 3000.0) and got[1][:2] == (15.0, 3000.0)
    assert got[0][2] == 1002 and got[1][2] != got[0][2]


def test_single_process_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max_sum(3.5, 42.0) == (3.5, 42.0)


def test_self_launch_starts_n_ranks(capfd):
    """`bench.py --gpus N` without WORLD_SIZE re-executes itself under torch.distributed.run with
    N ranks; the same launcher started on a CPU stand-in rank joins N gloo ranks."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    env_world = os.environ.pop("WORLD_SIZE", None)
    try:
        cmd = bench.launch_command(2, ["--gpus", "2", "--steps", "3"],
                                   script=os.path.join(ROOT, "tests", "rank_probe.py"))
        assert cmd[1:3] == ["-m", "torch.distributed.run"]
        assert "--nproc-per-node=2" in cmd and "127.0.0.1" in cmd
        rc = bench.self_launch(2, ["--gpus", "2", "--steps", "3"],
                               script=os.path.join(ROOT, "tests", "rank_probe.py"))
    finally:
        if env_world is not None:
            os.environ["WORLD_SIZE"] = env_world
    assert rc == 0
    lines = [ln for ln in capfd.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    got = json.loads(lines[0])
    assert got["n_gpus"] == 2 and got["max_ms"] == 15.0 and got["bytes"] == 3000.0
    assert got["args"] == ["--gpus", "2", "--steps", "3"]
