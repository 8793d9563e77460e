"""Overlapped (programmatic dependent) and plain kernel launches give the same
bytes.  Every kernel waits for the kernel before it on the stream before its
first global-memory access; a kernel that did not would race with its
predecessor only under overlapped launch.  The same sequence of library calls,
touching every kernel family (tensorwise amax, cast and GEMMs including the
split-K and CTA-pair paths, the block quantizers and GEMMs, GELU, the fused
GELU quantizers, gradient accumulation, delayed scaling), runs in two child
processes, FP8LIN_PDL=0 and FP8LIN_PDL=1 (the launch mode is read once per
process), and the SHA-256 over all outputs must agree.  Parity of the default
(overlapped) mode with the oracle is covered by the other GPU tests."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))

CHILD = r'''
import hashlib, json, os, sys
import torch
import fp8_mixed_precision_gb300 as fp
from fp8_mixed_precision_gb300 import synthetic as syn
from fp8_mixed_precision_gb300.mlp import FP8MLPStack

dev = "cuda"
h = hashlib.sha256()


def add(*ts):
    for t in ts:
        if t is not None:
            h.update(t.contiguous().view(torch.uint8).cpu().numpy().tobytes())


# tensorwise linears; (N, K, O) chosen so that the wgrad takes the split-K path
# (512 x 512 over 16384 tokens) and the dgrad the CTA-pair path (K = 8192)
for i, (N, K, O) in enumerate([(8192, 512, 2048), (16384, 512, 512), (8192, 512, 8192)]):
    x, w, dy = syn.linear_inputs(N, K, O, device=dev, layer=i)
    cache = fp.WeightCache()
    hw = cache.register(w, "tensorwise")
    cache.begin_cycle()
    cache.get(hw, 1, True)
    y, ctx = fp.fp8_linear_fwd(x, cache, hw, "tensorwise")
    dx, dw = fp.fp8_linear_bwd(dy, ctx, cache, hw, "tensorwise")
    add(y, dx, dw)

# block-scaled MLP stacks, unfused and with GELU fused into the quantizers, two
# microbatches each (gradient accumulation)
for fused in (False, True):
    st = FP8MLPStack(512, 2048, 2, 4096, "block", fused=fused)
    xs = [syn.bf16_normal((4096, 512), 1.0, 42 + m, device=dev) for m in range(2)]
    dys = [syn.bf16_normal((4096, 512), 1e-3, 44 + m, device=dev) for m in range(2)]
    for y, dx in st.step(xs, dys, use_cache=True):
        add(y, dx)
    add(*st.dw1, *st.dw2)

# delayed scaling over three steps (cast, then the history update kernel)
hist = torch.zeros(16, dtype=torch.float32, device=dev)
for s in range(3):
    xd = syn.bf16_normal((2048, 1024), 1.0, 50 + s, device=dev)
    q = fp.fp8_quantize_delayed(xd, "act", hist, s)
    add(q["row"], q["col"], q["scale"], q["scale_inv"], hist)

torch.cuda.synchronize()
print(json.dumps({"status": fp.fp8_get_device_status(), "sha256": h.hexdigest()}))
'''


def _run(tmp_path, pdl):
    script = tmp_path / "launch_mode_child.py"
    script.write_text(CHILD)
    env = dict(os.environ, FP8LIN_PDL=pdl, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, str(script)], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.gpu
def test_overlapped_and_plain_launches_give_the_same_bytes(tmp_path):
    plain = _run(tmp_path, "0")
    overlapped = _run(tmp_path, "1")
    assert plain["status"] == 0 and overlapped["status"] == 0
    assert plain["sha256"] == overlapped["sha256"]
