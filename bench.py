"""Benchmark of the FP8 linear hot path on GB300.

Workload (isolated FP8 linear, the reconstruction's timing table): N = 131072
tokens through four linears I->O = 512->512, 512->2048, 2048->512, 512->8192,
current tensorwise scaling, E4M3 X/W and E5M2 dY, fused dual-layout casts,
weight quantization included (every step starts a new accumulation cycle),
fprop + dgrad + wgrad with BF16 outputs.  One step = the four linears' forward
and backward.  value = tokens processed by the linears per second
(4 x 131072 per step), summed over ranks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the
host cores on bounded token samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 linear fwd+bwd tokens/s; cast GB/s & GEMM TFLOP/s vs GB300 roofline"
SHAPES = [(512, 512), (512, 2048), (2048, 512), (512, 8192)]   # (in K, out O)
N_TOKENS = 131072
RECIPE = "tensorwise"
# RTX 4090 fused-layout FP8 medians of the four shapes (ms), the reconstruction's
# isolated-linear table; another machine's numbers, reported as context only.
PAGES_FUSED_MS = [2.0107, 5.4075, 5.4264, 22.7554]
FALLBACK_PEAKS = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0)
FP8_OVER_BF16 = 2.0   # nominal dense FP8 / BF16 tensor rate ratio (4.5 / 2.25 PFLOP/s)


def _peaks():
    """HBM copy bandwidth and dense FP8 tensor peaks (burst: a kernel timed
    alone at full clocks; sustained: a seconds-long loop under the power
    cap), FP8 taken as the measured bf16 GEMM rate x the nominal FP8/BF16
    ratio."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        pk = dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                  bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                  source="measured")
    else:
        pk = dict(FALLBACK_PEAKS, source="fallback")
    pk["fp8_tflops"] = pk["bf16_tflops"] * FP8_OVER_BF16
    pk["fp8_tflops_sustained"] = pk["bf16_tflops_sustained"] * FP8_OVER_BF16
    return pk


def roofline_of(recs, steps: int, peaks: dict) -> dict:
    """Per-instantiation rooflines from the library's per-launch event timing
    (records per kernel name and launch shape).  Each launch is bounded by
    max(flops / FP8 peak, bytes / HBM peak); its bound is the larger term.
    Fractions are against the burst FP8 peak (this region is sub-second at
    full clocks) and, beside it, the sustained one."""
    fb, fs, hbm = peaks["fp8_tflops"], peaks["fp8_tflops_sustained"], peaks["hbm_gbs"]
    tot = sum(r["total_ms"] for r in recs) or 1.0
    inst, roof_ms = [], 0.0
    for r in recs:
        n = r["launches"]
        t = r["total_ms"] / n / 1e3                       # seconds per launch
        fl, by = r["flops"] / n, r["bytes"] / n
        t_fl, t_by = fl / (fb * 1e12), by / (hbm * 1e9)
        roof_ms += n * max(t_fl, t_by) * 1e3 / steps
        if fl > 0 and t_fl >= t_by:
            e = {"bound": "tensor", "achieved": fl / t / 1e12, "unit": "TFLOP/s",
                 "peak_burst": fb, "peak_sustained": fs}
        else:
            e = {"bound": "hbm", "achieved": by / t / 1e9, "unit": "GB/s",
                 "peak_burst": hbm, "peak_sustained": hbm}
        e.update(kernel=r["name"], shape=[r["m"], r["n"], r["k"]],
                 launches_per_step=n / steps, ms_per_launch=t * 1e3,
                 share=r["total_ms"] / tot, frac_burst=e["achieved"] / e["peak_burst"],
                 frac_sustained=e["achieved"] / e["peak_sustained"],
                 roofline_ms_per_launch=max(t_fl, t_by) * 1e3,
                 frac_of_roofline_time=max(t_fl, t_by) / t,
                 traffic=_traffic_for(r["name"], (r["m"], r["n"], r["k"])))
        inst.append(e)
    inst.sort(key=lambda e: -e["share"])
    return {"instances": inst, "roofline_ms_per_step": roof_ms}


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.path is None or not os.path.exists(self.path):
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------- dist
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, world: int, device) -> float:
    """Max over ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- oracle timing
# The CPU oracle, as it stands, timed on the host cores.  Each measurement runs
# in a fresh interpreter whose BLAS thread count is fixed before numpy loads,
# so `cores` states the threads actually used: 1 (single thread) or every
# host core (the oracle's numpy elementwise work - quantizers, encode - is
# single-threaded by nature, so the all-core figures run independent samples
# side by side on a thread pool, numpy releasing the interpreter lock, with
# BLAS on all cores for the fp64 GEMMs).
def _oracle_env(threads: int) -> dict:
    env = dict(os.environ)
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(threads)
    return env


def run_oracle_timing(threads: int, spec: dict, timeout: float = 600.0) -> dict:
    """Run oracle_timing_worker(spec) in a fresh interpreter with `threads`
    BLAS threads; returns its JSON result."""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-timing",
                        json.dumps(dict(spec, threads=threads))],
                       env=_oracle_env(threads), capture_output=True, text=True, timeout=timeout)
    if r.returncode != 0:
        raise RuntimeError(f"oracle timing failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def oracle_timing_worker(spec: dict) -> dict:
    """CPU oracle timings on bounded samples of each workload (called in the
    subprocess).  Every figure names its sample; figures scaled from a
    sample to the full workload say "extrapolated"."""
    from concurrent.futures import ThreadPoolExecutor
    import numpy as np
    import oracle as o
    from fp8_mixed_precision_gb300 import synthetic as syn
    T = int(spec["threads"])
    pool = ThreadPoolExecutor(max_workers=T)
    bits = lambda t: syn.bits(t)
    out = {"threads": T}

    def par(fn, items):
        return list(pool.map(fn, items)) if T > 1 else [fn(x) for x in items]

    def clock(fn):
        t0 = time.perf_counter()
        r = fn()
        return time.perf_counter() - t0, r

    # -- isolated linears (headline workload): n tokens per linear, all four shapes;
    # all-core: T independent samples of n tokens at once
    n = int(spec.get("c1_tokens", 1024))
    lin = []
    for i, (K, O) in enumerate(SHAPES):
        x, w, dy = syn.linear_inputs(n, K, O, layer=i)
        lin.append((bits(x), bits(w), bits(dy)))
    reps = max(1, T)
    one_step = lambda: par(lambda _: [o.linear_fwd_bwd(x, w, dy, RECIPE) for x, w, dy in lin],
                           range(reps))
    for _ in range(int(spec.get("warmup", 0))):
        one_step()
    steps = max(1, int(spec.get("steps", 1)))
    dt, _ = clock(lambda: [one_step() for _ in range(steps)])
    out["c1"] = {"tokens_per_s": steps * reps * len(SHAPES) * n / dt, "seconds": dt,
                 "steps": steps, "sample": f"{reps} x {n} tokens per linear, four shapes"}
    if spec.get("c1_only"):
        return out
    # -- one 512->512 linear at N = 2048 (the whole workload), tensorwise
    x, w, dy = syn.linear_inputs(2048, 512, 512)
    xb, wb, dyb = bits(x), bits(w), bits(dy)
    dt, _ = clock(lambda: o.linear_fwd_bwd(xb, wb, dyb, "tensorwise"))
    out["c0"] = {"ms": 1e3 * dt, "tokens_per_s": 2048 / dt, "sample": "whole workload",
                 "input_sha256": {"X": syn.sha256(x), "W": syn.sha256(w), "dY": syn.sha256(dy)}}
    # -- block MLP d=512/ffn=2048 (fc1, GELU, fc2; fwd + bwd) on a token sample
    nb = int(spec.get("mlp_tokens", 512))
    d, ffn = 512, 2048
    xs = [bits(syn.bf16_normal((nb, d), 1.0, syn.SEED_X + i)) for i in range(reps)]
    dys = [bits(syn.bf16_normal((nb, d), 1e-3, syn.SEED_DY + i)) for i in range(reps)]
    w1 = bits(syn.bf16_normal((ffn, d), 0.02, 43))
    w2 = bits(syn.bf16_normal((d, ffn), 0.02, 44))
    dt, _ = clock(lambda: par(lambda i: o.mlp_fwd_bwd(xs[i], w1, w2, dys[i], "block"), range(reps)))
    mlp_tps = reps * nb / dt
    out["c2"] = {"tokens_per_s": mlp_tps, "ms_per_step_extrapolated": 1e3 * 131072 / mlp_tps,
                 "sample": f"{reps} x {nb} tokens (linear in tokens: extrapolated to 131072)"}
    # -- 8-layer stack, GA = 4: 32 block passes of 131072 tokens + 16 weight quantizations
    dt_w, _ = clock(lambda: par(lambda w: o.quantize(w, "block", "weight"), [w1, w2] * 8))
    step_s = 8 * 4 * 131072 / mlp_tps + dt_w
    out["c3"] = {"ms_per_step_cached_extrapolated": 1e3 * step_s,
                 "ms_per_step_uncached_extrapolated": 1e3 * (step_s + 3 * dt_w),
                 "weight_quantize_ms_16": 1e3 * dt_w,
                 "sample": "block-MLP rate above x 8 layers x 4 microbatches of 131072 tokens "
                           "+ 16 weight quantizations (timed)"}
    # -- large block MLP d=4096/ffn=14336, 16384 tokens: quantizers on row
    # samples and GEMMs on whole 128x128 output tiles, scaled to the workload
    N4, D4, F4 = 16384, 4096, 14336
    rows = 128
    xr = bits(syn.bf16_normal((rows, D4), 1.0, syn.SEED_X, outlier_frac=0.01))
    fr = bits(syn.bf16_normal((rows, F4), 1e-3, syn.SEED_DY))
    wr = bits(syn.bf16_normal((rows, D4), 0.02, syn.SEED_W))
    tq = {}
    tq["act_d"], _ = clock(lambda: o.quantize_1x128(xr, "e4m3"))
    tq["act_f"], _ = clock(lambda: o.quantize_1x128(fr, "e4m3"))
    tq["w"], _ = clock(lambda: o.quantize_128x128(wr, "e4m3"))
    # activations and gradients: X, dY [N, d] and A, dH [N, ffn]; weights W1, W2 [ffn x d]
    q_s = 2 * (N4 / rows) * tq["act_d"] + 2 * (N4 / rows) * tq["act_f"] + 2 * (F4 / rows) * tq["w"]
    # one output tile per GEMM kind, timed on dequantized operands
    def tile_time(kred):
        a = np.random.default_rng(1).standard_normal((128, kred))
        b = np.random.default_rng(2).standard_normal((128, kred))
        t, _ = clock(lambda: a @ b.T)
        return t
    tiles = {"fprop1": (N4 // 128) * (F4 // 128), "fprop2": (N4 // 128) * (D4 // 128)}
    g_s = 0.0
    for kred, ntile in ((D4, tiles["fprop1"]), (F4, tiles["fprop2"]),     # fc1 / fc2 fprop
                        (F4, tiles["fprop2"]), (D4, tiles["fprop1"]),     # fc2 / fc1 dgrad
                        (N4, (F4 // 128) * (D4 // 128)), (N4, (D4 // 128) * (F4 // 128))):  # wgrads
        g_s += ntile * tile_time(kred)
    gelu_s, _ = clock(lambda: o.gelu_fwd(fr))
    out["c4"] = {"ms_per_step_extrapolated": 1e3 * (q_s + g_s + 2 * (N4 / rows) * gelu_s),
                 "quantize_ms_extrapolated": 1e3 * q_s, "gemm_ms_extrapolated": 1e3 * g_s,
                 "tokens_per_s_extrapolated": N4 / (q_s + g_s + 2 * (N4 / rows) * gelu_s),
                 "sample": "quantizers on 128-row samples, one whole 128x128 output tile per GEMM "
                           "(fp64), GELU on a 128-row sample; scaled to the workload"}
    # -- quantizer throughput at the workloads' shapes (algorithmic bytes: 6 B
    # per element tensorwise, 4 B + scales per element for the block recipes)
    qs = {}
    for name, R, C, kind in (("tensorwise 131072x8192", 131072, 8192, "t"),
                             ("1x128 131072x2048", 131072, 2048, "a"),
                             ("1x128 16384x14336", 16384, 14336, "a"),
                             ("128x128 14336x4096", 14336, 4096, "w")):
        r = 256
        xs_q = [bits(syn.bf16_normal((r, C), 1.0, 60 + i)) for i in range(reps)]
        fn = {"t": lambda b: o.quantize_tensorwise(b, "e4m3"),
              "a": lambda b: o.quantize_1x128(b, "e4m3"),
              "w": lambda b: o.quantize_128x128(b, "e4m3")}[kind]
        dt, _ = clock(lambda: par(fn, xs_q))
        per_el = 6.0 if kind == "t" else 4.0 + (16.0 / 128 if kind == "a" else 0.0)
        gbs = reps * r * C * per_el / dt / 1e9
        qs[name] = {"GB/s": gbs, "ms_extrapolated": 1e3 * R * C * per_el / (gbs * 1e9),
                    "sample": f"{reps} x {r} rows"}
    out["quantizers"] = qs
    return out


def run_reference(args):
    """--impl reference: the CPU oracle on bounded samples of the workload,
    every host core in use (independent samples on a thread pool, BLAS on
    all cores), one step = one such sample."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    cores = os.cpu_count() or 1
    # one worker process runs the warm-up and then the timed steps
    r = run_oracle_timing(cores, {"c1_tokens": 256, "c1_only": True, "warmup": args.warmup,
                                  "steps": args.steps})["c1"]
    secs = r["seconds"]
    tps = r["tokens_per_s"]
    toks = tps * secs
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "isolated FP8 linear fwd+bwd, tensorwise, shapes "
                   "512->512/512->2048/2048->512/512->8192",
                   "tokens_per_step": toks / args.steps, "recipe": RECIPE},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{cores} independent samples of 256 tokens per linear per "
                                   f"step (of {N_TOKENS}), one per host thread"},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm
def run_ours(args):
    import torch
    import fp8_mixed_precision_gb300 as fp
    from fp8_mixed_precision_gb300 import synthetic as syn

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fp.lib()

    N = N_TOKENS
    cache = fp.WeightCache()
    layers = []
    hashes = {}
    for i, (K, O) in enumerate(SHAPES):
        x, w, dy = syn.linear_inputs(N, K, O, device=dev, layer=i)
        hashes[f"{K}->{O}"] = {"X": syn.sha256(x), "W": syn.sha256(w), "dY": syn.sha256(dy)}
        h = cache.register(w, RECIPE)
        layers.append(dict(K=K, O=O, x=x, w=w, dy=dy, h=h,
                           y=torch.empty((N, O), dtype=torch.bfloat16, device=dev),
                           dx=torch.empty((N, K), dtype=torch.bfloat16, device=dev),
                           dw=torch.empty((O, K), dtype=torch.bfloat16, device=dev)))
    ws = max((fp.linear_workspace(RECIPE, N, L["K"], L["O"], dev) for L in layers),
             key=lambda t: t.numel())
    ctx = max((fp.LinearContext(fp._empty_bytes(fp._ctx_bytes(RECIPE, N, L["K"]), dev), N, L["K"])
               for L in layers), key=lambda c: c.ctx.numel())
    version = [0]

    def step_serial():
        cache.begin_cycle()
        version[0] += 1
        for L in layers:
            cache.get(L["h"], version[0], True)
            c = fp.LinearContext(ctx.ctx, N, L["K"])
            fp.fp8_linear_fwd(L["x"], cache, L["h"], RECIPE, ws=ws, y=L["y"], ctx=c)
            fp.fp8_linear_bwd(L["dy"], c, cache, L["h"], RECIPE, ws=ws, dx=L["dx"], dw=L["dw"])

    # The same work with the tensorwise amax passes of X and dY (pure HBM
    # reads, almost no shared memory) on a second stream, where their CTAs run
    # beside the GEMM and cast CTAs on the first; each cast waits for its
    # tensor's partial maxima.  The linears run in reverse order, 512->8192
    # first: only its own two amax passes are issued at the start, and the
    # other linears' passes start on the second stream as its backward begins,
    # so that most of them overlap its deep-K dgrad and wgrad (tensor-bound,
    # reading HBM at about half its bandwidth) rather than the HBM-bound casts
    # and K = 512 GEMMs.  Results are bit for bit those of step_serial
    # (checked below on the captured graphs).
    stream = torch.cuda.current_stream()
    aux = torch.cuda.Stream(dev)
    px = [fp.amax_partials_buffer(N, L["K"], dev) for L in layers]
    pdy = [fp.amax_partials_buffer(N, L["O"], dev) for L in layers]
    ev_go = torch.cuda.Event()
    ev_bwd = torch.cuda.Event()
    ev_x = [torch.cuda.Event() for _ in layers]
    ev_dy = [torch.cuda.Event() for _ in layers]
    order = list(reversed(range(len(layers))))

    def amax_on_aux(idx):
        with torch.cuda.stream(aux):
            for i in idx:
                fp.fp8_amax_partials(layers[i]["x"], px[i])
                ev_x[i].record(aux)
                fp.fp8_amax_partials(layers[i]["dy"], pdy[i])
                ev_dy[i].record(aux)

    def step_overlap():
        cur = torch.cuda.current_stream()   # the capture stream while a graph is recorded
        cache.begin_cycle()
        version[0] += 1
        ev_go.record(cur)             # earlier casts are done with the partial buffers
        aux.wait_event(ev_go)
        amax_on_aux(order[:1])
        for n, i in enumerate(order):
            L = layers[i]
            cache.get(L["h"], version[0], True)
            c = fp.LinearContext(ctx.ctx, N, L["K"])
            cur.wait_event(ev_x[i])
            fp.fp8_linear_fwd_after_amax(L["x"], px[i], cache, L["h"], RECIPE, ws, L["y"], c)
            cur.wait_event(ev_dy[i])
            if n == 0:                # the other linears' passes start with this backward
                ev_bwd.record(cur)
                aux.wait_event(ev_bwd)
                amax_on_aux(order[1:])
            fp.fp8_linear_bwd_after_amax(L["dy"], pdy[i], c, cache, L["h"], RECIPE, ws, L["dx"],
                                         L["dw"])

    step = step_overlap if args.schedule == "overlap" else step_serial
    # the first call, cold (per-device kernel attributes and occupancy queries,
    # first touch of every buffer), reported on its own
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    f0.record(stream)
    step()
    f1.record(stream)
    torch.cuda.synchronize()
    first_ms = f0.elapsed_time(f1)
    for _ in range(args.warmup):        # both schedules, so either can be timed warm
        step_overlap()
        step_serial()
    torch.cuda.synchronize()
    st = fp.fp8_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")
    launches_per_step = fp.fp8_launch_count()
    step()
    torch.cuda.synchronize()
    launches_per_step = fp.fp8_launch_count() - launches_per_step

    # One step captured in a CUDA graph: every replay runs the same kernels
    # with the same arguments (the weights are re-quantized each replay, as in
    # the eager step), without the host's per-launch work between them.  Each
    # schedule gets its own graph.
    def capture(fn):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            fn()                        # warm the capture stream
        stream.wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g
    other_fn = step_serial if args.schedule == "overlap" else step_overlap
    graph = capture(step)
    other_graph = capture(other_fn) if args.launch == "graph" else None
    eager_step = step
    timed_step = graph.replay if args.launch == "graph" else eager_step

    # Both schedules, as they are timed, against one eager serial step: every
    # output bit for bit.
    step_serial()
    torch.cuda.synchronize()
    ref = [t.clone() for L in layers for t in (L["y"], L["dx"], L["dw"])]
    schedules_equal = True
    for run in (timed_step, other_graph.replay if other_graph is not None else other_fn):
        for L in layers:
            for t in (L["y"], L["dx"], L["dw"]):
                t.zero_()
        run()
        torch.cuda.synchronize()
        got = [t for L in layers for t in (L["y"], L["dx"], L["dw"])]
        schedules_equal = schedules_equal and all(
            torch.equal(a.view(torch.int16), b.view(torch.int16)) for a, b in zip(ref, got))
    del ref
    if not schedules_equal:
        raise RuntimeError("the two schedules' outputs differ")
    for _ in range(args.warmup):
        timed_step()
    torch.cuda.synchronize()

    # ---- device-resident timing: `value` comes from K steps with no per-kernel
    # events (recording two events around every launch costs a few percent of
    # the step); the per-kernel times for the roofline come from K more steps
    # of the same work with the library's events on.
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        n_launch0 = fp.fp8_launch_count()
        # the K steps in up to 5 groups, an event at each boundary (5 events in
        # all): the spread of the group means is reported with the total
        ngroups = min(5, args.steps)
        bounds = [args.steps * gi // ngroups for gi in range(ngroups + 1)]
        gev = [torch.cuda.Event(enable_timing=True) for _ in range(ngroups - 1)]
        t0.record(stream)
        for gi in range(ngroups):
            for _ in range(bounds[gi + 1] - bounds[gi]):
                timed_step()
            if gi < ngroups - 1:
                gev[gi].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        n_launch = fp.fp8_launch_count() - n_launch0
        if args.launch == "graph":      # replays launch the captured kernels
            n_launch = launches_per_step * args.steps
    clocks = clk.summary()
    marks = [t0] + gev + [t1]
    group_ms = [marks[gi].elapsed_time(marks[gi + 1]) / (bounds[gi + 1] - bounds[gi])
                for gi in range(ngroups)]
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    fp.fp8_profile_begin()
    p0.record(stream)
    for _ in range(args.steps):         # one stream: no kernel shares the GPU with another
        step_serial()
    p1.record(stream)
    torch.cuda.synchronize()
    krecs = fp.fp8_profile_end(by_shape=True)
    profiled_ms_step = p0.elapsed_time(p1) / args.steps
    # the other schedule, for reference (same work, same results), launched
    # the same way
    other = other_graph.replay if other_graph is not None else other_fn
    o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    o0.record(stream)
    for _ in range(args.steps):
        other()
    o1.record(stream)
    torch.cuda.synchronize()
    other_ms_step = reduce_max(o0.elapsed_time(o1), world, dev) / args.steps
    # the other launch mode, for reference
    other_launch = eager_step if args.launch == "graph" else graph.replay
    q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    q0.record(stream)
    for _ in range(args.steps):
        other_launch()
    q1.record(stream)
    torch.cuda.synchronize()
    other_launch_ms = reduce_max(q0.elapsed_time(q1), world, dev) / args.steps
    del graph, other_graph
    ms_local = t0.elapsed_time(t1)
    ms_total = reduce_max(ms_local, world, dev)
    ms_step = ms_total / args.steps
    tokens_per_step = len(SHAPES) * N
    value = world * tokens_per_step / (ms_step / 1e3)

    # ---- rooflines: every kernel instantiation (kernel x launch shape), the
    # dominant one as the headline, and the whole step
    peaks = _peaks()
    rl = roofline_of(krecs, args.steps, peaks)
    agg = {}
    for r in krecs:
        a = agg.setdefault(r["name"], dict(name=r["name"], launches=0, total_ms=0.0, bytes=0.0,
                                           flops=0.0))
        for key in ("launches", "total_ms", "bytes", "flops"):
            a[key] += r[key]
    kstats = sorted(agg.values(), key=lambda k: -k["total_ms"])
    tot_ms = sum(k["total_ms"] for k in kstats) or 1.0
    kernels = []
    for k in kstats:
        gbs = k["bytes"] / (k["total_ms"] / 1e3) / 1e9
        tfs = k["flops"] / (k["total_ms"] / 1e3) / 1e12
        kernels.append({"name": k["name"], "launches": k["launches"] // args.steps,
                        "ms_per_step": k["total_ms"] / args.steps,
                        "share": k["total_ms"] / tot_ms, "GB/s": gbs, "TFLOP/s": tfs,
                        "hbm_frac": gbs / peaks["hbm_gbs"]})
    dom = rl["instances"][0]
    roof = {"bound": dom["bound"], "achieved": dom["achieved"], "peak": dom["peak_burst"],
            "unit": dom["unit"], "frac": dom["frac_burst"], "traffic": dom["traffic"],
            "kernel": dom["kernel"], "shape": dom["shape"],
            "frac_burst": dom["frac_burst"], "frac_sustained": dom["frac_sustained"],
            "peak_sustained": dom["peak_sustained"],
            "peak_source": peaks["source"] + (" bf16 GEMM x 2 (nominal FP8/BF16 ratio); burst, "
                                              "sustained beside it" if dom["bound"] == "tensor"
                                              else " copy bandwidth"),
            "per_instantiation": rl["instances"],
            "step": {"roofline_ms": rl["roofline_ms_per_step"],
                     "measured_ms_graph": ms_step, "measured_ms_profiled": profiled_ms_step,
                     "frac": rl["roofline_ms_per_step"] / ms_step,
                     "note": "sum over the step's launches of max(flops / FP8 burst peak, "
                             "algorithmic bytes / HBM peak), against the measured step time"},
            "timing": ("CUDA events around each launch on its stream, over a second region of "
                       "the same K steps, eager, every kernel on one stream (value comes "
                       "from an event-free region)")}

    # ---- end to end through the C ABI with host buffers
    e2e = run_e2e(fp, layers, cache, ws, ctx, N, dev, world, args, stream)

    # ---- the other workloads: one small linear, weight caching, block MLPs
    workloads = None
    if not args.no_mlp:
        del layers
        workloads = {"c0_linear_512_2048_tokens": run_c0(fp, dev, stream),
                     "quantizers_at_workload_shapes": run_quantizer_workloads(fp, dev, peaks)}
        workloads.update(run_mlp_workloads(fp, dev, stream, peaks))
        lb = workloads["large_block_mlp_4096_14336"]
        lb["gemm_frac_of_fp8_peak_burst"] = lb["gemm_tflops"] / peaks["fp8_tflops"]
        lb["gemm_frac_of_fp8_peak_sustained"] = lb["gemm_tflops"] / peaks["fp8_tflops_sustained"]
        workloads.update(run_plain_and_assay(fp, dev, stream))

    # ---- CPU baselines: the oracle on the host cores (rank 0, one GPU only),
    # single-threaded and on every core, per workload
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        one = run_oracle_timing(1, {"c1_tokens": 512})
        allc = run_oracle_timing(cores, {"c1_tokens": 512})
        cpu = {"value": allc["c1"]["tokens_per_s"], "unit": "tokens/s", "cores": cores,
               "kind": "oracle",
               "sample": allc["c1"]["sample"] + f" (of {N_TOKENS}); {allc['c1']['seconds']:.1f} s",
               "single_thread": {"value": one["c1"]["tokens_per_s"], "cores": 1,
                                 "sample": one["c1"]["sample"]},
               "note": "all cores: independent samples side by side on a thread pool (numpy "
                       "releases the interpreter lock), BLAS on all cores; single thread: one "
                       "sample, BLAS on one thread"}
        if workloads is not None:
            workloads["cpu_baseline_per_workload"] = {"single_thread": one, "all_cores": allc}

    pages_tps = tokens_per_step / (sum(PAGES_FUSED_MS) / 1e3)
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": value / pages_tps,
            "dtype": "fp8 (e4m3/e5m2) x fp8 -> f32 accumulate -> bf16",
            "data": "synthetic (seeded normal bf16 drawn on the host: X~N(0,1), W~N(0,0.02), "
                    "dY~N(0,1e-3))",
            "input_sha256": hashes,
            "config": {"workload": "isolated FP8 linear fwd+bwd, N=131072 tokens, shapes "
                                   "512->512/512->2048/2048->512/512->8192, tensorwise current "
                                   "scaling, fused dual-layout casts, weight quantized every step",
                       "tokens_per_step": tokens_per_step, "recipe": RECIPE,
                       "l2": "inputs larger than L2 (about 9 GB touched per step)",
                       "parallelism": f"dp{world} (replicas, no collective)",
                       "schedule": ("tensorwise amax passes on a second stream beside the "
                                    "GEMMs and casts, linears in reverse order, the other "
                                    "linears' passes started with the first one's backward"
                                    if args.schedule == "overlap" else "one stream"),
                       "launch": ("one step captured as a CUDA graph, replayed"
                                  if args.launch == "graph" else "eager launches"),
                       "programmatic_dependent_launch": os.environ.get("FP8LIN_PDL", "1")[:1] != "0"},
            "other_schedule_ms_per_step": {("serial" if args.schedule == "overlap"
                                            else "overlap"): other_ms_step},
            "schedules_bitwise_equal": schedules_equal,
            "profiled_ms_per_step": profiled_ms_step,
            "other_launch_ms_per_step": {("eager" if args.launch == "graph" else "graph"):
                                         other_launch_ms},
            "step_ms_groups": {"median": statistics.median(group_ms), "min": min(group_ms),
                               "max": max(group_ms), "groups": group_ms},
            "first_call_ms": first_ms,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": n_launch,
            "clocks": clocks,
            "kernels": kernels,
            "workloads": workloads,
            "baseline_note": "vs_baseline divides by the RTX 4090 fused-layout FP8 figures of "
                             "the reconstruction's table (context only)",
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def kernel_source_digest():
    """SHA-256 over the kernel sources with comments and whitespace removed:
    a committed ncu summary stays valid across comment-only edits and goes
    stale on any code change."""
    import hashlib
    import re
    h = hashlib.sha256()
    d = os.path.join(ROOT, "fp8_mixed_precision_gb300", "csrc")
    for fn in sorted(os.listdir(d)):
        with open(os.path.join(d, fn), encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)   # block comments
        src = re.sub(r"//[^\n]*", " ", src)                # line comments
        h.update(fn.encode() + b"\0" + " ".join(src.split()).encode() + b"\0")
    return h.hexdigest()


def _traffic_for(name, shape=None):
    """DRAM bytes per launch from a committed ncu summary, when it still
    matches the current kernel sources (keyed by kernel name and, where the
    summary has it, launch shape "MxNxK")."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("csrc_sha256") != kernel_source_digest():
            return None
        ks = d.get("kernels", {})
        if shape is not None:
            key = f"{name} {shape[0]}x{shape[1]}x{shape[2]}"
            if key in ks:
                return ks[key].get("dram_bytes_per_launch")
        return ks.get(name, {}).get("dram_bytes_per_launch")
    except (OSError, ValueError, KeyError):
        return None


def run_c0(fp, dev, stream):
    """One FP8 linear 512->512 at N = 2048 tokens, tensorwise (the smallest
    workload): fwd + bwd time per call in 5 groups of 25 calls (median of the
    group medians, min and max), eager launches and CUDA-graph replays, the
    cold first call, and the outputs against the CPU oracle on the same
    inputs (relative Frobenius error per output)."""
    import numpy as np
    import torch
    import oracle as o
    from fp8_mixed_precision_gb300 import synthetic as syn
    N, K, O = 2048, 512, 512
    x, w, dy = syn.linear_inputs(N, K, O, device=dev)
    cache = fp.WeightCache()
    h = cache.register(w, "tensorwise")
    ws = fp.linear_workspace("tensorwise", N, K, O, dev)
    ctx = fp.LinearContext(fp._empty_bytes(fp._ctx_bytes("tensorwise", N, K), dev), N, K)
    y = torch.empty((N, O), dtype=torch.bfloat16, device=dev)
    dx = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((O, K), dtype=torch.bfloat16, device=dev)
    ver = [0]

    def step():
        cache.begin_cycle()
        ver[0] += 1
        cache.get(h, ver[0], True)
        fp.fp8_linear_fwd(x, cache, h, "tensorwise", ws=ws, y=y, ctx=ctx)
        fp.fp8_linear_bwd(dy, ctx, cache, h, "tensorwise", ws=ws, dx=dx, dw=dw)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    step()
    e1.record(stream)
    torch.cuda.synchronize()
    first_us = 1e3 * e0.elapsed_time(e1)
    n_l = fp.fp8_launch_count()
    step()
    torch.cuda.synchronize()
    launches = fp.fp8_launch_count() - n_l

    def groups(fn):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        med = []
        for _ in range(5):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(26)]
            ev[0].record(stream)
            for i in range(25):
                fn()
                ev[i + 1].record(stream)
            torch.cuda.synchronize()
            med.append(statistics.median(1e3 * ev[i].elapsed_time(ev[i + 1]) for i in range(25)))
        return {"us_median": statistics.median(med), "us_min": min(med), "us_max": max(med),
                "group_medians_us": med}

    eager = groups(step)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        step()
    graph = groups(g.replay)
    del g
    step()
    torch.cuda.synchronize()
    r = o.linear_fwd_bwd(syn.bits(x), syn.bits(w), syn.bits(dy), "tensorwise")
    rel = {}
    for name, got in (("y", y), ("dx", dx), ("dw", dw)):
        gg = o.bf16_to_f32(syn.bits(got)).astype(np.float64)
        ee = o.bf16_to_f32(r[name]).astype(np.float64)
        rel[name] = float(np.linalg.norm(gg - ee) / max(np.linalg.norm(ee), 1e-30))
    flops = 6.0 * N * K * O
    return {"workload": "one FP8 linear 512->512, N=2048 tokens, tensorwise, fwd+bwd",
            "eager": dict(eager, tokens_per_s=N / (eager["us_median"] / 1e6),
                          tflops=flops / (eager["us_median"] / 1e6) / 1e12),
            "graph_replay": dict(graph, tokens_per_s=N / (graph["us_median"] / 1e6),
                                 tflops=flops / (graph["us_median"] / 1e6) / 1e12),
            "first_call_us": first_us, "launches_per_call": launches,
            "vs_oracle_rel_frobenius": rel,
            "input_sha256": {"X": syn.sha256(x), "W": syn.sha256(w), "dY": syn.sha256(dy)},
            "timing": "5 groups x 25 calls, an event between calls on the launching stream; "
                      "median of the group medians (inputs in L2: the workload is 4 MB)"}


def run_quantizer_workloads(fp, dev, peaks):
    """Every quantizer at the workloads' shapes, launched alone: 12 launches
    per shape rotating over enough input tensors that the bytes read between
    two uses of one input exceed L2, each launch timed by the library's
    events.  GB/s counts algorithmic bytes (bf16 read, both FP8 layouts
    written, scales); hbm_frac is against the measured copy bandwidth."""
    import torch
    from fp8_mixed_precision_gb300 import synthetic as syn
    shapes = [("1x128", "act", 131072, 2048), ("1x128", "act", 16384, 14336),
              ("1x128", "act", 16384, 4096), ("1x128", "act", 131072, 512),
              ("128x128", "weight", 14336, 4096), ("128x128", "weight", 4096, 14336),
              ("128x128", "weight", 2048, 512), ("tensorwise", "act", 131072, 8192),
              ("tensorwise", "act", 131072, 2048)]
    out = {}
    for kind, role, R, C in shapes:
        recipe = "tensorwise" if kind == "tensorwise" else "block"
        copies = max(2, -(-(256 << 20) // (2 * R * C)))   # > 2 x L2 between reuses
        xs = [syn.bf16_normal((R, C), 1.0, 70 + i, device=dev) for i in range(min(copies, 96))]
        fp.fp8_quantize(xs[0], recipe, role)
        torch.cuda.synchronize()
        fp.fp8_profile_begin()
        for i in range(12):
            fp.fp8_quantize(xs[i % len(xs)], recipe, role)
        torch.cuda.synchronize()
        recs = fp.fp8_profile_end(by_shape=True)
        ent = {}
        for r in recs:
            t = r["total_ms"] / r["launches"]
            gbs = r["bytes"] / r["launches"] / (t / 1e3) / 1e9
            ent[r["name"]] = {"ms_per_launch": t, "GB/s": gbs, "hbm_frac": gbs / peaks["hbm_gbs"]}
        tot_b = sum(r["bytes"] for r in recs) / 12
        tot_t = sum(r["total_ms"] for r in recs) / 12
        out[f"{kind} {R}x{C}"] = {"kernels": ent, "ms": tot_t,
                                  "GB/s": tot_b / (tot_t / 1e3) / 1e9,
                                  "hbm_frac": tot_b / (tot_t / 1e3) / 1e9 / peaks["hbm_gbs"],
                                  "inputs_rotated": len(xs)}
        del xs
        torch.cuda.empty_cache()
    return out


def run_mlp_workloads(fp, dev, stream, peaks):
    """The MLP-level workloads, timed with CUDA events on the launching stream:
    weight caching in an 8-layer block-scaled stack under GA = 4 (cached vs
    uncached step time, bitwise comparison of outputs and accumulated
    gradients at full size), the d=512/ffn=2048 block MLP, and the large
    block-scaled MLP (d=4096, ffn=14336, 16384 tokens, 1% x100 outliers)."""
    import torch
    from fp8_mixed_precision_gb300 import synthetic as syn
    from fp8_mixed_precision_gb300.mlp import FP8MLPStack
    out = {}

    def timed(fn, reps):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(reps):
            fn()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / reps

    # ---- weight caching: 8 layers (16 FP8 linears), d=512, ffn=2048, GA=4 x 131072 tokens
    d, ffn, L, N, GA = 512, 2048, 8, 131072, 4
    xs = [syn.bf16_normal((N, d), 1.0, 700 + i, device=dev) for i in range(GA)]
    dys = [syn.bf16_normal((N, d), 1e-3, 800 + i, device=dev) for i in range(GA)]
    stk = FP8MLPStack(d, ffn, L, N, "block", device=dev)
    res, grads = {}, {}
    for use in (False, True):
        stk.step(xs, dys, use, keep_outputs=False)
    times = {False: [], True: []}
    for _ in range(3):                      # interleaved rounds against drift
        for use in (False, True):
            times[use].append(timed(lambda: stk.step(xs, dys, use, keep_outputs=False), 2))
    for use in (False, True):               # full-size bitwise comparison
        outs = stk.step(xs, dys, use, keep_outputs=True)
        res[use] = outs
        grads[use] = [t.clone() for t in stk.dw1 + stk.dw2]
    torch.cuda.synchronize()
    same = all(torch.equal(a.view(torch.int16), b.view(torch.int16))
               for (ya, da), (yb, db) in zip(res[False], res[True]) for a, b in ((ya, yb), (da, db)))
    same = same and all(torch.equal(a.view(torch.int32), b.view(torch.int32))
                        for a, b in zip(grads[False], grads[True]))
    med = {k: statistics.median(v) for k, v in times.items()}
    # the same steps captured once per mode in a CUDA graph and replayed, so
    # host launch jitter cannot swamp a difference of a few tenths of a percent
    graphs = {}
    for use in (False, True):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):       # warm the capture stream's allocator
            stk.step(xs, dys, use, keep_outputs=False)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            stk.step(xs, dys, use, keep_outputs=False)
        graphs[use] = g
    gtimes = {False: [], True: []}
    for _ in range(5):                      # 5 interleaved groups of 2 replays per mode
        for use in (False, True):
            gtimes[use].append(timed(graphs[use].replay, 2))
    gmed = {k: statistics.median(v) for k, v in gtimes.items()}
    del graphs
    # where the difference goes: one eager cycle per mode with per-kernel events
    kb = {}
    for use in (False, True):
        stk.step(xs, dys, use, keep_outputs=False)
        torch.cuda.synchronize()
        fp.fp8_profile_begin()
        stk.step(xs, dys, use, keep_outputs=False)
        torch.cuda.synchronize()
        kb[use] = {k["name"]: (k["total_ms"], k["launches"]) for k in fp.fp8_profile_end()}
    breakdown = {}
    for name in sorted(set(kb[False]) | set(kb[True])):
        u_ms, u_n = kb[False].get(name, (0.0, 0))
        c_ms, c_n = kb[True].get(name, (0.0, 0))
        breakdown[name] = {"uncached_ms": u_ms, "cached_ms": c_ms, "saved_ms": u_ms - c_ms,
                           "uncached_launches": u_n, "cached_launches": c_n}
    # what caching skips: one weight quantization of each fc1 / fc2 shape
    # (device time of its kernels from the library's per-kernel events)
    wq = {}
    for name, (O, K) in (("fc1", (ffn, d)), ("fc2", (d, ffn))):
        wt = syn.bf16_normal((O, K), 0.02, 900, device=dev)
        fp.fp8_quantize(wt, "block", "weight")
        torch.cuda.synchronize()
        fp.fp8_profile_begin()
        for _ in range(50):
            fp.fp8_quantize(wt, "block", "weight")
        torch.cuda.synchronize()
        wq[name] = sum(k["total_ms"] for k in fp.fp8_profile_end()) / 50
    skipped = (GA - 1) * L * (wq["fc1"] + wq["fc2"])
    out["weight_cache_stack"] = {
        "workload": "8-layer MLP stack (16 FP8 linears, d=512, ffn=2048), GA=4 x 131072 tokens, "
                    "block scaling",
        "ms_per_step_uncached": med[False], "ms_per_step_cached": med[True],
        "reduction_pct": 100.0 * (med[False] - med[True]) / med[False],
        "samples_uncached": times[False], "samples_cached": times[True],
        "bitwise_identical": bool(same),
        "weight_quantizations_per_step": {"uncached": 2 * L * GA, "cached": 2 * L},
        "tokens_per_s_cached": GA * N / (med[True] / 1e3),
        "graph_replay": {
            "ms_per_step_uncached": gmed[False], "ms_per_step_cached": gmed[True],
            "reduction_pct": 100.0 * (gmed[False] - gmed[True]) / gmed[False],
            "groups_uncached": gtimes[False], "groups_cached": gtimes[True]},
        "weight_quantize_ms": wq,
        "skipped_weight_quantize_ms_per_step": skipped,
        "skipped_pct_of_uncached_step": 100.0 * skipped / gmed[False],
        "kernel_breakdown_eager": breakdown,
        "input_sha256": {"X": [syn.sha256(t) for t in xs], "dY": [syn.sha256(t) for t in dys],
                         "W1": [syn.sha256(t) for t in stk.w1], "W2": [syn.sha256(t) for t in stk.w2]},
        "kernel_breakdown_note": "one eager cycle per mode, library events around every launch: "
                                 "device time per kernel name, uncached minus cached"}
    del stk, xs, dys, res, grads
    torch.cuda.empty_cache()

    # ---- block MLP d=512, ffn=2048, 131072 tokens (one microbatch, fwd + bwd),
    # unfused and with quantization fused into the GELU producers
    x = syn.bf16_normal((131072, 512), 1.0, syn.SEED_X, device=dev)
    dy = syn.bf16_normal((131072, 512), 1e-3, syn.SEED_DY, device=dev)
    for fused in (False, True):
        blk = FP8MLPStack(512, 2048, 1, 131072, "block", device=dev, fused=fused)
        blk.step([x], [dy], True, keep_outputs=False)
        ms = timed(lambda: blk.step([x], [dy], True, keep_outputs=False), 5)
        fp.fp8_profile_begin()
        blk.step([x], [dy], True, keep_outputs=False)
        torch.cuda.synchronize()
        rl = roofline_of(fp.fp8_profile_end(by_shape=True), 1, peaks)
        out["block_mlp_512_2048" + ("_fused" if fused else "")] = {
            "ms_per_step": ms, "tokens_per_s": 131072 / (ms / 1e3),
            "tflops": 6 * 2 * 131072 * 512 * 2048 / (ms / 1e3) / 1e12,
            "roofline_ms_per_step": rl["roofline_ms_per_step"],
            "per_instantiation": rl["instances"],
            "input_sha256": {"X": syn.sha256(x), "dY": syn.sha256(dy),
                             "W1": syn.sha256(blk.w1[0]), "W2": syn.sha256(blk.w2[0])}}
        del blk
        torch.cuda.empty_cache()
    del x, dy

    # ---- large block MLP d=4096, ffn=14336, 16384 tokens, 1% x100 outliers
    big = FP8MLPStack(4096, 14336, 1, 16384, "block", device=dev, fused=True)
    x = syn.bf16_normal((16384, 4096), 1.0, syn.SEED_X, device=dev, outlier_frac=0.01)
    dy = syn.bf16_normal((16384, 4096), 1e-3, syn.SEED_DY, device=dev)
    big.step([x], [dy], True, keep_outputs=False)
    torch.cuda.synchronize()
    ms_clean = timed(lambda: big.step([x], [dy], True, keep_outputs=False), 3)
    fp.fp8_profile_begin()
    ms = timed(lambda: big.step([x], [dy], True, keep_outputs=False), 3)
    ks_shape = fp.fp8_profile_end(by_shape=True)
    rl = roofline_of(ks_shape, 3, peaks)
    ks = {}
    for r in ks_shape:
        a = ks.setdefault(r["name"], dict(name=r["name"], launches=0, total_ms=0.0, bytes=0.0,
                                          flops=0.0))
        for key in ("launches", "total_ms", "bytes", "flops"):
            a[key] += r[key]
    ks = list(ks.values())
    gemm = [k for k in ks if k["name"].startswith("gemm_fp8")]
    g_ms = sum(k["total_ms"] for k in gemm)
    g_fl = sum(k["flops"] for k in gemm)
    out["large_block_mlp_4096_14336"] = {
        "fused_producers": True,
        "ms_per_step": ms_clean, "tokens_per_s": 16384 / (ms_clean / 1e3),
        "ms_per_step_with_kernel_events": ms,
        "roofline_ms_per_step": rl["roofline_ms_per_step"],
        "per_instantiation": rl["instances"],
        "input_sha256": {"X": syn.sha256(x), "dY": syn.sha256(dy),
                         "W1": syn.sha256(big.w1[0]), "W2": syn.sha256(big.w2[0])},
        "gemm_tflops": g_fl / (g_ms / 1e3) / 1e12,
        "gemm_share": g_ms / sum(k["total_ms"] for k in ks),
        "gemm_kernels": {k["name"]: {"TFLOP/s": k["flops"] / (k["total_ms"] / 1e3) / 1e12,
                                     "ms_per_step": k["total_ms"] / 3} for k in gemm}}
    del big, x, dy
    torch.cuda.empty_cache()
    return out


def run_plain_and_assay(fp, dev, stream):
    """Plain-FP8 arm against the fused path on the isolated-linear shapes, the
    GEMM-only BF16/FP8 assay and memory accounting (the reconstruction's
    isolated-linear table columns, exactness paragraph and component assay).
      plain: every tensor quantized by two separate passes (rowwise-only, then
             transposed-only), GEMMs through fp8_gemm; fused: fp8_linear_fwd/bwd.
      assay: each linear's three GEMMs in FP8 (this library) vs bf16 cuBLAS
             (torch.matmul, context), summed per shape like the page.
      memory: saved-for-backward bytes and peak device memory of one fwd+bwd,
             FP8 (this library) vs a bf16 linear (torch autograd, context)."""
    import torch
    from fp8_mixed_precision_gb300 import synthetic as syn
    N = N_TOKENS
    out = {"plain_vs_fused": {}, "gemm_assay": {}, "memory": {}}

    def timed(fn, reps=5):
        fn()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(reps):
            fn()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / reps

    for i, (K, O) in enumerate(SHAPES):
        x, w, dy = syn.linear_inputs(N, K, O, device=dev, layer=i)
        cache = fp.WeightCache()
        h = cache.register(w, RECIPE)
        ws = fp.linear_workspace(RECIPE, N, K, O, dev)
        res = {}

        def fused():
            cache.begin_cycle()
            cache.get(h, 0, True)
            y, ctx = fp.fp8_linear_fwd(x, cache, h, RECIPE, ws=ws)
            dx, dw = fp.fp8_linear_bwd(dy, ctx, cache, h, RECIPE, ws=ws)
            res["fused"] = (y, dx, dw)

        def plain():
            wr = fp.fp8_quantize(w, RECIPE, "weight", rowwise=True, colwise=False)
            wc = fp.fp8_quantize(w, RECIPE, "weight", rowwise=False, colwise=True)
            xr = fp.fp8_quantize(x, RECIPE, "act", rowwise=True, colwise=False)
            xc = fp.fp8_quantize(x, RECIPE, "act", rowwise=False, colwise=True)
            y = fp.fp8_gemm(xr["row"], "e4m3", xr["row_scale_inv"], wr["row"], "e4m3",
                            wr["row_scale_inv"], "tensor")
            gr = fp.fp8_quantize(dy, RECIPE, "grad", rowwise=True, colwise=False)
            gc = fp.fp8_quantize(dy, RECIPE, "grad", rowwise=False, colwise=True)
            dx = fp.fp8_gemm(gr["row"], "e5m2", gr["row_scale_inv"], wc["col"], "e4m3",
                             wr["row_scale_inv"], "tensor")
            dw = fp.fp8_gemm(gc["col"], "e5m2", gr["row_scale_inv"], xc["col"], "e4m3",
                             xr["row_scale_inv"], "tensor")
            res["plain"] = (y, dx, dw)

        ms_f, ms_p = timed(fused), timed(plain)
        same = all(torch.equal(a.view(torch.int16), b.view(torch.int16))
                   for a, b in zip(res["fused"], res["plain"]))
        out["plain_vs_fused"][f"{K}->{O}"] = {"fused_ms": ms_f, "plain_ms": ms_p,
                                              "fused_speedup": ms_p / ms_f,
                                              "outputs_bitwise_equal": bool(same)}
        # GEMM-only assay: the three GEMMs of the linear, ours (FP8) against bf16
        # cuBLAS and against cuBLAS FP8 on the same operands (library context)
        xq = fp.fp8_quantize(x, RECIPE, "act")
        wq = fp.fp8_quantize(w, RECIPE, "weight")
        gq = fp.fp8_quantize(dy, RECIPE, "grad")

        def g8():
            fp.fp8_gemm(xq["row"], "e4m3", xq["row_scale_inv"], wq["row"], "e4m3", wq["row_scale_inv"], "tensor")
            fp.fp8_gemm(gq["row"], "e5m2", gq["row_scale_inv"], wq["col"], "e4m3", wq["row_scale_inv"], "tensor")
            fp.fp8_gemm(gq["col"], "e5m2", gq["row_scale_inv"], xq["col"], "e4m3", xq["row_scale_inv"], "tensor")

        def g16():
            torch.matmul(x, w.t())
            torch.matmul(dy, w)
            torch.matmul(dy.t(), x)

        def gc8():  # the same FP8 operands and scales through cuBLAS (torch._scaled_mm)
            f8 = lambda t, f: t.view(torch.float8_e4m3fn if f == "e4m3" else torch.float8_e5m2)
            sx, sw, sg = (xq["row_scale_inv"].reshape(()), wq["row_scale_inv"].reshape(()),
                          gq["row_scale_inv"].reshape(()))
            torch._scaled_mm(f8(xq["row"], "e4m3"), f8(wq["row"], "e4m3").t(), scale_a=sx, scale_b=sw,
                             out_dtype=torch.bfloat16)
            torch._scaled_mm(f8(gq["row"], "e5m2"), f8(wq["col"], "e4m3").t(), scale_a=sg, scale_b=sw,
                             out_dtype=torch.bfloat16)
            torch._scaled_mm(f8(gq["col"], "e5m2"), f8(xq["col"], "e4m3").t(), scale_a=sg, scale_b=sx,
                             out_dtype=torch.bfloat16)

        ms8, ms16 = timed(g8), timed(g16)
        ent = {"fp8_ms": ms8, "bf16_cublas_ms": ms16, "bf16_over_fp8": ms16 / ms8}
        try:
            msc = timed(gc8)
            ent.update(cublas_fp8_ms=msc, cublas_fp8_over_ours=msc / ms8)
        except (RuntimeError, AttributeError, TypeError) as e:  # library FP8 path unavailable
            ent.update(cublas_fp8_ms=None, cublas_fp8_note=str(e).splitlines()[0][:120])
        out["gemm_assay"][f"{K}->{O}"] = ent
        # memory: saved for backward and peak of one fwd+bwd
        ctx_b = fp._ctx_bytes(RECIPE, N, K)
        res.clear()
        del xq, wq, gq
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats(dev)
        base = torch.cuda.memory_allocated(dev)
        fused()
        torch.cuda.synchronize()
        peak8 = torch.cuda.max_memory_allocated(dev) - base
        torch.cuda.empty_cache()
        torch.cuda.reset_peak_memory_stats(dev)
        base = torch.cuda.memory_allocated(dev)
        xr_ = x.detach().requires_grad_(True)
        wr_ = w.detach().requires_grad_(True)
        yb = torch.nn.functional.linear(xr_, wr_)
        yb.backward(dy)
        torch.cuda.synchronize()
        peak16 = torch.cuda.max_memory_allocated(dev) - base
        del yb, xr_, wr_
        out["memory"][f"{K}->{O}"] = {"fp8_saved_bytes": ctx_b, "bf16_saved_bytes": 2 * N * K,
                                      "fp8_peak_bytes": peak8, "bf16_peak_bytes": peak16}
        del x, w, dy, cache, ws
        torch.cuda.empty_cache()
    mlp = [f"{k}->{o}" for k, o in SHAPES if k != o]
    sq = [f"{k}->{o}" for k, o in SHAPES if k == o]
    a = out["gemm_assay"]
    out["gemm_assay"]["summed_bf16_over_fp8_mlp_shapes"] = (
        sum(a[s]["bf16_cublas_ms"] for s in mlp) / sum(a[s]["fp8_ms"] for s in mlp))
    out["gemm_assay"]["summed_bf16_over_fp8_square"] = (
        sum(a[s]["bf16_cublas_ms"] for s in sq) / sum(a[s]["fp8_ms"] for s in sq))
    if all(a[s].get("cublas_fp8_ms") for s in mlp + sq):
        out["gemm_assay"]["summed_cublas_fp8_over_ours"] = (
            sum(a[s]["cublas_fp8_ms"] for s in mlp + sq) / sum(a[s]["fp8_ms"] for s in mlp + sq))
    return out


def _link_GBps(dev, nbytes=1 << 30):
    """Host<->device link bandwidth with both directions busy at once (pinned
    buffers, one copy each way), the bound of a copy-limited end-to-end run."""
    import torch
    h1 = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h2 = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d1 = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d2 = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    best = 0.0
    for _ in range(3):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        s1.wait_stream(torch.cuda.current_stream())
        s2.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s1):
            d1.copy_(h1, non_blocking=True)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)
        torch.cuda.current_stream().wait_stream(s1)
        torch.cuda.current_stream().wait_stream(s2)
        b.record()
        torch.cuda.synchronize()
        best = max(best, 2 * nbytes / (a.elapsed_time(b) / 1e3) / 1e9)
    del h1, h2, d1, d2
    return best


def run_e2e(fp, layers, cache, ws, ctx, N, dev, world, args, stream):
    """Same step through the C ABI's host-buffer entry point
    (fp8_linear_step_host): every input is copied from pinned host memory and
    every result copied back by the library, inside the timed region.  One
    pipeline slot per linear: the library's copy-in / compute / copy-out
    streams let the copies of one linear overlap the kernels of another."""
    import torch
    host = []
    h2d = d2h = 0
    for L in layers:
        hb = {"X": torch.empty(L["x"].shape, dtype=torch.bfloat16, pin_memory=True),
              "W": torch.empty(L["w"].shape, dtype=torch.bfloat16, pin_memory=True),
              "dY": torch.empty(L["dy"].shape, dtype=torch.bfloat16, pin_memory=True),
              "Y": torch.empty(L["y"].shape, dtype=torch.bfloat16, pin_memory=True),
              "dX": torch.empty(L["dx"].shape, dtype=torch.bfloat16, pin_memory=True),
              "dW": torch.empty(L["dw"].shape, dtype=torch.bfloat16, pin_memory=True)}
        hb["X"].copy_(L["x"]); hb["W"].copy_(L["w"]); hb["dY"].copy_(L["dy"])
        host.append(hb)
        h2d += 2 * (hb["X"].numel() + hb["W"].numel() + hb["dY"].numel())
        d2h += 2 * (hb["Y"].numel() + hb["dX"].numel() + hb["dW"].numel())
    devs = [{"X": L["x"], "dY": L["dy"], "Y": L["y"], "dX": L["dx"], "dW": L["dw"]}
            for L in layers]
    pipe = fp.HostPipeline(len(layers))
    version = [10 ** 6]

    def step():
        cache.begin_cycle()
        version[0] += 1
        for i, L in enumerate(layers):
            pipe.step(i, host[i], devs[i], ctx, ws, cache, L["h"], RECIPE, version[0])

    k = max(3, min(args.steps, 20))
    step()
    pipe.sync()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0.record(stream)
    pipe.fork(stream)       # no copy or kernel of the timed steps starts before t0
    for _ in range(k):
        step()
    pipe.join(stream)       # the region ends when the last results are on the host
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = reduce_max(t0.elapsed_time(t1), world, dev) / k
    value = world * len(SHAPES) * N / (ms / 1e3)
    link = _link_GBps(dev)
    copy = (h2d + d2h) / (ms / 1e3) / 1e9
    return {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": k, "ms_per_step": ms,
            "copy_GBps": copy, "link_GBps_both_directions": link,
            "copy_frac_of_link": copy / link if link > 0 else None,
            "api": "fp8_linear_step_host (host buffers; library copy-in / compute / "
                   "copy-out streams, one slot per linear)"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--launch", choices=["graph", "eager"], default="graph",
                    help="graph (default): time replays of one step captured as a CUDA graph; "
                         "eager: one library call per linear per step")
    ap.add_argument("--schedule", choices=["serial", "overlap"], default="overlap",
                    help="overlap (default): tensorwise amax passes on a second stream; "
                         "serial: every kernel on one stream")
    ap.add_argument("--no-mlp", action="store_true",
                    help="skip the MLP-level workloads reported beside the main line")
    ap.add_argument("--oracle-timing", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args.oracle_timing is not None:     # internal: one CPU-oracle timing run (subprocess)
        print(json.dumps(oracle_timing_worker(json.loads(args.oracle_timing))), flush=True)
        return 0
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
