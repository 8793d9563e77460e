"""Host-side logic of bench.py: the max-over-ranks reduction and barrier run
as two gloo ranks on CPU, and the clock-sample parser."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (world, rank, rank)
    bench.barrier(world)
    m = bench.reduce_max(10.0 + rank * 5.0, world, torch.device("cpu"))
    out[rank] = m
    dist.destroy_process_group()


def test_reduce_max_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_clock_summary_parser(tmp_path):
    sys.path.insert(0, ROOT)
    import bench
    c = bench.ClockSampler(0)
    c.path = str(tmp_path / "c.csv")
    with open(c.path, "w") as f:
        f.write("0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 1905, 2070, 1390.2, 0x4, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 1935, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    s = c.summary()
    assert s["sm_mhz"] == 1935 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
