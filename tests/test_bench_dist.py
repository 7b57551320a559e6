"""Multi-rank host logic of bench.py on CPU with gloo (world size 2): the
slowest rank's time is reported, and each rank draws its own batch."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    from exact_tiled_attention_18_gb300 import workloads
    r, w, local = bench.dist_env()
    d = bench.init_dist(r, w, "gloo")
    t = bench.max_over_ranks(10.0 + 5.0 * r, d)
    bench.barrier(d)
    inp = workloads.make_inputs(1, 1, 8, 4, seed=r)
    out[rank] = (t, float(inp["q"].float().sum()))
    dist.destroy_process_group()


def test_two_rank_max_and_independent_batches():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert res[0][1] != res[1][1]


def test_reference_arm_other_ranks_exit_quietly(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert capsys.readouterr().out == ""
