"""Host-side logic of multi-GPU bench runs, as two gloo ranks on CPU.

Every GPU runs an independent replica of the batch; the reported value is all ranks'
bytes over the slowest rank's time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank], world)
    dist.destroy_process_group()
    queue.put((rank, got))


def test_slowest_rank_sets_the_time_of_all_replicas():
    world = 2
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, queue)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(queue.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0] == results[1] == [2.0, 10.0]


def test_replica_value_counts_every_rank():
    import bench

    assert bench.replica_gbs(10 ** 9, 10, 1, 2.0) == pytest.approx(5.0)
    assert bench.replica_gbs(10 ** 9, 10, 4, 2.0) == pytest.approx(20.0)
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
                "--config", "1"])
    assert capsys.readouterr().out == ""
