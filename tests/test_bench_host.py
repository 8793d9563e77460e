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


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the CPU oracle on bounded samples) prints
    one JSON line with the keys the benchmark contract asks of that arm; it
    needs no GPU."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"]


def test_kernel_source_digest_ignores_comments_only():
    """The digest that keys the committed DRAM-traffic figures changes with
    any code edit of the kernel sources and with no comment-only edit."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    import tempfile, shutil
    with tempfile.TemporaryDirectory() as d:
        csrc = os.path.join(d, "fp8_mixed_precision_gb300", "csrc")
        shutil.copytree(os.path.join(ROOT, "fp8_mixed_precision_gb300", "csrc"), csrc)
        bench.ROOT = d
        base = bench.kernel_source_digest()
        p = os.path.join(csrc, "glue.cu")
        src = open(p).read()
        open(p, "w").write("// a new comment line\n" + src.replace("\n", "  \n", 3) + "\n/* block\n comment */\n")
        assert bench.kernel_source_digest() == base
        open(p, "w").write(src.replace("kThreads = 256", "kThreads = 128", 1))
        assert bench.kernel_source_digest() != base
