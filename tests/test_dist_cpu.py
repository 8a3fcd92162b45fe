"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

The layer partitions over tokens with no exchange step, so `bench.py --gpus N`
runs N independent replicas; the only cross-rank traffic is the timing
barrier and the max-over-ranks reduction of the step time.  These tests run
that logic with the gloo backend on two CPU processes (no GPU), and check that
the reference arm leaves every rank but 0 without work.
"""
import multiprocessing as mp
import os
import socket

import pytest
import torch

import bench


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out) -> None:
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    r, w, local = bench.dist_info()
    dist = bench.dist_init(w, "gloo")
    bench.barrier(w)
    # each rank's "step time": the slowest rank decides the reported time
    slowest = bench.reduce_max(1.5 * (r + 1), w, torch.device("cpu"))
    bench.barrier(w)
    out.put((r, w, local, slowest))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max_step_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 and g[2] == g[0] for g in got)
    assert all(g[3] == 3.0 for g in got)  # max over ranks of 1.5 and 3.0


def test_single_rank_needs_no_process_group():
    assert bench.reduce_max(2.5, 1, torch.device("cpu")) == 2.5
    bench.barrier(1)  # no-op without a process group


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.parse_args(["--impl", "reference", "--workload", "tiny"])
    shape, desc = bench.WORKLOADS["tiny"]
    assert bench.bench_reference(args, shape, desc) is None
    assert capsys.readouterr().out == ""


if __name__ == "__main__":  # pragma: no cover
    pytest.main([__file__, "-q"])
