"""The multi-GPU form of the benchmark is N independent replicas (the path
shards by problem or kv head, but one GPU runs a whole step): no data-path
collective, the job timed by its slowest rank.  Its host logic runs here as
two gloo processes on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(times[rank], "cpu")
        out[rank] = (t, bench.replica_value(10.0, t, world))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    times = [0.25, 0.4]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        t, v = res[r]
        assert t == 0.4  # every rank reports the slowest time
        assert v == pytest.approx(10.0 * 2 / 0.4)  # all ranks' units over it


def test_single_process_is_the_identity():
    assert bench.max_over_ranks(0.123, "cpu") == 0.123
    assert bench.replica_value(5.0, 0.5, 1) == 10.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    # the other ranks of a torchrun launch exit without work or output
    monkeypatch.setenv("RANK", "1")
    assert bench.reference_arm(None) is None  # (it returns before reading its arguments)
    assert capsys.readouterr().out == ""
