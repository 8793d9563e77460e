"""The host-buffer step (fp8_linear_step_host): inputs and results in pinned
host memory, copies made by the library on its own streams, several linears
in flight on different slots.  Its results must equal, bit for bit, those of
fp8_linear_fwd / fp8_linear_bwd on device tensors (which the linear parity
tests check against the oracle), over two steps with a changed weight; one
output is also checked against the oracle directly."""
import numpy as np
import pytest
import torch

import oracle as o
from parity import check_gemm, to_np

pytestmark = pytest.mark.gpu

SHAPES = [(512, 256), (256, 512)]  # (K, O) per slot


@pytest.fixture(scope="module")
def fp():
    from fp8_mixed_precision_gb300 import build
    build.build()
    import fp8_mixed_precision_gb300 as fp
    return fp


def _bits(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("recipe", ["tensorwise", "block"])
def test_host_steps_equal_device_path(fp, recipe):
    from fp8_mixed_precision_gb300 import synthetic as syn
    dev = torch.device("cuda")
    N = 1024
    pipe = fp.HostPipeline(len(SHAPES))
    cache_h, cache_d = fp.WeightCache(), fp.WeightCache()
    # one workspace and one context serve every slot (their kernels are ordered)
    ws = max((fp.linear_workspace(recipe, N, K, O, dev) for K, O in SHAPES), key=lambda t: t.numel())
    ctx = fp.LinearContext(fp._empty_bytes(max(fp._ctx_bytes(recipe, N, K) for K, _ in SHAPES), dev),
                           N, 512)
    slots = []
    for i, (K, O) in enumerate(SHAPES):
        wd_h = torch.empty((O, K), dtype=torch.bfloat16, device=dev)  # filled by the pipeline
        wd_d = torch.empty((O, K), dtype=torch.bfloat16, device=dev)
        slots.append(dict(
            K=K, O=O, h_h=cache_h.register(wd_h, recipe), h_d=cache_d.register(wd_d, recipe),
            wd_d=wd_d,
            dev={"X": torch.empty((N, K), dtype=torch.bfloat16, device=dev),
                 "dY": torch.empty((N, O), dtype=torch.bfloat16, device=dev),
                 "Y": torch.empty((N, O), dtype=torch.bfloat16, device=dev),
                 "dX": torch.empty((N, K), dtype=torch.bfloat16, device=dev),
                 "dW": torch.empty((O, K), dtype=torch.bfloat16, device=dev)}))
    for step in range(2):
        cache_h.begin_cycle()
        cache_d.begin_cycle()
        hosts = []
        for i, s in enumerate(slots):
            K, O = s["K"], s["O"]
            seed = 100 * step + 10 * i
            x = syn.bf16_normal((N, K), 1.0, seed + 1)
            w = syn.bf16_normal((O, K), 0.02, seed + 2)
            dy = syn.bf16_normal((N, O), 1e-3, seed + 3)
            host = {"X": x.pin_memory(), "W": w.pin_memory(), "dY": dy.pin_memory(),
                    "Y": torch.empty((N, O), dtype=torch.bfloat16).pin_memory(),
                    "dX": torch.empty((N, K), dtype=torch.bfloat16).pin_memory(),
                    "dW": torch.empty((O, K), dtype=torch.bfloat16).pin_memory()}
            pipe.step(i, host, s["dev"], ctx, ws, cache_h, s["h_h"], recipe, version=step + 1)
            hosts.append(host)
        pipe.sync()
        for i, (s, host) in enumerate(zip(slots, hosts)):
            s["wd_d"].copy_(host["W"].to(dev))
            cache_d.get(s["h_d"], step + 1, True)
            y, c = fp.fp8_linear_fwd(host["X"].to(dev), cache_d, s["h_d"], recipe)
            dx, dw = fp.fp8_linear_bwd(host["dY"].to(dev), c, cache_d, s["h_d"], recipe)
            torch.cuda.synchronize()
            assert torch.equal(_bits(host["Y"]), _bits(y.cpu())), f"Y slot {i} step {step}"
            assert torch.equal(_bits(host["dX"]), _bits(dx.cpu())), f"dX slot {i} step {step}"
            assert torch.equal(_bits(host["dW"]), _bits(dw.cpu())), f"dW slot {i} step {step}"
    assert fp.fp8_get_device_status() == 0
    # the last step's first slot against the oracle directly
    host = hosts[0]
    r = o.linear_fwd_bwd(to_np(host["X"]), to_np(host["W"]), to_np(host["dY"]), recipe)
    xq, wq = r["xq"], r["wq"]
    A = o.dequantize(xq["row"], xq["row_scale_inv"], "e4m3")
    B = o.dequantize(wq["row"], wq["row_scale_inv"], "e4m3")
    check_gemm(host["Y"], A @ B.T, np.abs(A) @ np.abs(B).T, SHAPES[0][0], "Y (host step)")


def test_host_steps_back_to_back(fp):
    """Three steps enqueued without a sync in between (every slot's device
    buffers reused from step to step, the forward and backward halves of a
    step ordered against the previous step's copies by the pipeline's
    events): every step's host results equal the device path's bit for bit."""
    from fp8_mixed_precision_gb300 import synthetic as syn
    dev = torch.device("cuda")
    recipe, N, steps = "tensorwise", 4096, 3
    pipe = fp.HostPipeline(len(SHAPES))
    cache_h, cache_d = fp.WeightCache(), fp.WeightCache()
    ws = max((fp.linear_workspace(recipe, N, K, O, dev) for K, O in SHAPES), key=lambda t: t.numel())
    ctx = fp.LinearContext(fp._empty_bytes(max(fp._ctx_bytes(recipe, N, K) for K, _ in SHAPES), dev),
                           N, 512)
    slots = []
    for K, O in SHAPES:
        wd_h = torch.empty((O, K), dtype=torch.bfloat16, device=dev)
        wd_d = torch.empty((O, K), dtype=torch.bfloat16, device=dev)
        slots.append(dict(K=K, O=O, h_h=cache_h.register(wd_h, recipe),
                          h_d=cache_d.register(wd_d, recipe), wd_d=wd_d,
                          dev={k: torch.empty(sh, dtype=torch.bfloat16, device=dev) for k, sh in
                               (("X", (N, K)), ("dY", (N, O)), ("Y", (N, O)), ("dX", (N, K)),
                                ("dW", (O, K)))}))
    hosts = []
    for step in range(steps):
        cache_h.begin_cycle()
        row = []
        for i, s in enumerate(slots):
            K, O = s["K"], s["O"]
            seed = 1000 + 100 * step + 10 * i
            host = {"X": syn.bf16_normal((N, K), 1.0, seed + 1).pin_memory(),
                    "W": syn.bf16_normal((O, K), 0.02, seed + 2).pin_memory(),
                    "dY": syn.bf16_normal((N, O), 1e-3, seed + 3).pin_memory(),
                    "Y": torch.empty((N, O), dtype=torch.bfloat16).pin_memory(),
                    "dX": torch.empty((N, K), dtype=torch.bfloat16).pin_memory(),
                    "dW": torch.empty((O, K), dtype=torch.bfloat16).pin_memory()}
            pipe.step(i, host, s["dev"], ctx, ws, cache_h, s["h_h"], recipe, version=step + 1)
            row.append(host)
        hosts.append(row)
    pipe.sync()
    assert fp.fp8_get_device_status() == 0
    for step, row in enumerate(hosts):
        cache_d.begin_cycle()
        for i, (s, host) in enumerate(zip(slots, row)):
            s["wd_d"].copy_(host["W"].to(dev))
            cache_d.get(s["h_d"], step + 1, True)
            y, c = fp.fp8_linear_fwd(host["X"].to(dev), cache_d, s["h_d"], recipe)
            dx, dw = fp.fp8_linear_bwd(host["dY"].to(dev), c, cache_d, s["h_d"], recipe)
            torch.cuda.synchronize()
            for nm, got, exp in (("Y", host["Y"], y), ("dX", host["dX"], dx), ("dW", host["dW"], dw)):
                assert torch.equal(_bits(got), _bits(exp.cpu())), f"{nm} slot {i} step {step}"


def test_host_step_rejects_before_enqueue(fp):
    dev = torch.device("cuda")
    pipe = fp.HostPipeline(1)
    cache = fp.WeightCache()
    h = cache.register(torch.empty((256, 512), dtype=torch.bfloat16, device=dev), "tensorwise")
    N = 128
    host = {"X": torch.empty((N, 512), dtype=torch.bfloat16).pin_memory(),
            "W": torch.empty((256, 512), dtype=torch.bfloat16).pin_memory(),
            "dY": torch.empty((N, 256), dtype=torch.bfloat16).pin_memory(),
            "Y": torch.empty((N, 256), dtype=torch.bfloat16).pin_memory(),
            "dX": None, "dW": torch.empty((256, 512), dtype=torch.bfloat16).pin_memory()}
    devb = {"X": torch.empty((N, 512), dtype=torch.bfloat16, device=dev),
            "dY": torch.empty((N, 256), dtype=torch.bfloat16, device=dev),
            "Y": torch.empty((N, 256), dtype=torch.bfloat16, device=dev), "dX": None,
            "dW": torch.empty((256, 512), dtype=torch.bfloat16, device=dev)}
    ctx = fp.LinearContext(fp._empty_bytes(fp._ctx_bytes("tensorwise", N, 512), dev), N, 512)
    small = torch.empty(16, dtype=torch.uint8, device=dev)
    n0 = fp.fp8_launch_count()
    with pytest.raises(fp.FP8Error) as e:
        pipe.step(0, host, devb, ctx, small, cache, h, "tensorwise", 1)
    assert e.value.status == 8  # workspace too small
    with pytest.raises(fp.FP8Error) as e:
        pipe.step(1, host, devb, ctx, small, cache, h, "tensorwise", 1)
    assert e.value.status == 1  # slot out of range
    with pytest.raises(fp.FP8Error) as e:
        pipe.step(0, host, devb, ctx, small, cache, h, "block", 1)
    assert e.value.status == 1  # recipe differs from the registered one
    assert fp.fp8_launch_count() == n0
