"""Runs one library kernel on one synthetic case a few times, for profiling
single launches (e.g. under ncu) and timing them with CUDA events.

    python -m fp8_mixed_precision_gb300.kernel_case gemm --M 131072 --N 8192 --K 512 \
        --scaling tensor --reps 3
    python -m fp8_mixed_precision_gb300.kernel_case quantize --M 131072 --N 2048 \
        --recipe tensorwise --role act --reps 3
    python -m fp8_mixed_precision_gb300.kernel_case gelu_bwd --M 131072 --N 2048 --reps 7
"""
from __future__ import annotations

import argparse
import json

import torch

import fp8_mixed_precision_gb300 as fp
from fp8_mixed_precision_gb300 import synthetic as syn


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("kind", choices=["gemm", "quantize", "gelu", "gelu_bwd", "gelu_quant",
                                     "gelu_bwd_quant"])
    ap.add_argument("--M", type=int, required=True)
    ap.add_argument("--N", type=int, required=True)
    ap.add_argument("--K", type=int, default=512)
    ap.add_argument("--scaling", default="tensor", choices=list(fp.SCALING))
    ap.add_argument("--recipe", default="tensorwise", choices=list(fp.RECIPE))
    ap.add_argument("--role", default="act", choices=list(fp.ROLE))
    ap.add_argument("--afmt", default="e4m3", choices=list(fp.FORMAT))
    ap.add_argument("--bfmt", default="e4m3", choices=list(fp.FORMAT))
    ap.add_argument("--reps", type=int, default=3)
    a = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    if a.kind == "gemm":
        # random FP8 codes from a normal draw (valid, finite codes only)
        A = syn.bf16_normal((a.M, a.K), 1.0, 1, device=dev).float().to(torch.float8_e4m3fn)
        B = syn.bf16_normal((a.N, a.K), 1.0, 2, device=dev).float().to(torch.float8_e4m3fn)
        A, B = A.view(torch.uint8), B.view(torch.uint8)
        kb = -(-a.K // 128)
        if a.scaling == "tensor":
            sa, sb = torch.full((1,), 0.01, device=dev), torch.full((1,), 0.02, device=dev)
        elif a.scaling == "1x128_128x128":
            sa = torch.rand((a.M, kb), generator=g, device=dev) * 0.01 + 1e-3
            sb = torch.rand((-(-a.N // 128), kb), generator=g, device=dev) * 0.01 + 1e-3
        else:
            sa = torch.rand((a.M, kb), generator=g, device=dev) * 0.01 + 1e-3
            sb = torch.rand((a.N, kb), generator=g, device=dev) * 0.01 + 1e-3
        C = torch.empty((a.M, a.N), dtype=torch.bfloat16, device=dev)
        run = lambda: fp.fp8_gemm(A, a.afmt, sa, B, a.bfmt, sb, a.scaling, out=C)
        flops = 2.0 * a.M * a.N * a.K
        nbytes = a.M * a.K + a.N * a.K + 2.0 * a.M * a.N
    elif a.kind == "quantize":
        x = syn.bf16_normal((a.M, a.N), 1.0, 3, device=dev)
        run = lambda: fp.fp8_quantize(x, a.recipe, a.role)
        flops = 0.0
        nbytes = (6.0 if a.recipe == "tensorwise" else 4.125) * a.M * a.N
    elif a.kind == "gelu":
        h = syn.bf16_normal((a.M, a.N), 1.0, 4, device=dev)
        out = torch.empty_like(h)
        run = lambda: fp.fp8_gelu_fwd(h, out=out)
        flops = 0.0
        nbytes = 4.0 * a.M * a.N
    elif a.kind == "gelu_bwd":
        h = syn.bf16_normal((a.M, a.N), 1.0, 4, device=dev)
        da = syn.bf16_normal((a.M, a.N), 1.0, 5, device=dev)
        out = torch.empty_like(h)
        run = lambda: fp.fp8_gelu_bwd(da, h, out=out)
        flops = 0.0
        nbytes = 6.0 * a.M * a.N
    else:  # fused GELU (backward) + 1x128 quantization, both layouts
        h = syn.bf16_normal((a.M, a.N), 1.0, 4, device=dev)
        if a.kind == "gelu_quant":
            q = fp.QuantizedTensor(a.M, a.N, "act", dev)
            run = lambda: fp.fp8_gelu_quantize(h, q)
            nbytes = 4.125 * a.M * a.N
        else:
            da = syn.bf16_normal((a.M, a.N), 1.0, 5, device=dev)
            q = fp.QuantizedTensor(a.M, a.N, "grad", dev)
            run = lambda: fp.fp8_gelu_bwd_quantize(da, h, q)
            nbytes = 6.125 * a.M * a.N
        flops = 0.0
    run()
    torch.cuda.synchronize()
    ts = []
    for _ in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    st = fp.fp8_get_device_status()
    ms = min(ts)
    print(json.dumps({"kind": a.kind, "M": a.M, "N": a.N, "K": a.K, "ms_min": ms,
                      "GB/s": nbytes / ms / 1e6, "TFLOP/s": flops / ms / 1e9, "status": st}))
    return 0 if st == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
