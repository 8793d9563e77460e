"""The isolated-linear workload at its full size (N = 131072 tokens; 512->512,
512->2048, 2048->512, 512->8192; tensorwise current scaling), run exactly as
bench.py runs it (one shared workspace and context, fp8_linear_fwd then
fp8_linear_bwd), so every GEMM goes through the tile shape, split count and
CTA-pair configuration the benchmark times.  The oracle computes each
tensor's global amax itself, quantizes only the rows and columns that
sampled 128x128 output tiles of Y, dX and dW need, and checks those tiles."""
import numpy as np
import pytest
import torch

import oracle as o
from parity import check_gemm
from fp8_mixed_precision_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu

N = 131072
SHAPES = [(512, 512), (512, 2048), (2048, 512), (512, 8192)]  # (K, O)


@pytest.fixture(scope="module")
def fp():
    from fp8_mixed_precision_gb300 import build
    build.build()
    import fp8_mixed_precision_gb300 as fp
    return fp


def _scale(bits, fmt):
    return o.scale_from_amax(o.amax_of(o.bf16_to_f32(bits)), fmt)


def _q(bits, s, si, fmt):
    """Dequantized values of a bf16 slice cast with the tensor's scale."""
    return o.decode(o.cast(o.bf16_to_f32(np.ascontiguousarray(bits)), s, fmt), fmt) * np.float64(si)


@pytest.mark.parametrize("layer,K,O", [(i, k, o_) for i, (k, o_) in enumerate(SHAPES)])
def test_bench_linear_sampled_tiles(fp, layer, K, O):
    dev = torch.device("cuda")
    x, w, dy = syn.linear_inputs(N, K, O, device=dev, layer=layer)
    cache = fp.WeightCache()
    h = cache.register(w, "tensorwise")
    ws = max((fp.linear_workspace("tensorwise", N, k, o_, dev) for k, o_ in SHAPES),
             key=lambda t: t.numel())
    ctx = fp.LinearContext(fp._empty_bytes(max(fp._ctx_bytes("tensorwise", N, k) for k, _ in SHAPES),
                                           dev), N, K)
    cache.begin_cycle()
    cache.get(h, 1, True)
    y, _ = fp.fp8_linear_fwd(x, cache, h, "tensorwise", ws=ws, ctx=ctx)
    dx, dw = fp.fp8_linear_bwd(dy, ctx, cache, h, "tensorwise", ws=ws)
    torch.cuda.synchronize()
    assert fp.fp8_get_device_status() == 0
    xb, wb, dyb = syn.bits(x), syn.bits(w), syn.bits(dy)
    sx, sxi = _scale(xb, "e4m3")
    sw, swi = _scale(wb, "e4m3")
    sg, sgi = _scale(dyb, "e5m2")
    rng = np.random.default_rng(layer)
    sl = lambda t: slice(t * 128, (t + 1) * 128)
    tm_last, tn_last, tk_last = N // 128 - 1, O // 128 - 1, K // 128 - 1
    picks = [(0, 0, 0), (tm_last, tn_last, tk_last),
             (int(rng.integers(N // 128)), int(rng.integers(O // 128)), int(rng.integers(K // 128)))]
    for tm, tn, tk in picks:
        # Y tile (tm, tn): X rows x W rows, reduced over K
        A = _q(xb[sl(tm)], sx, sxi, "e4m3")
        B = _q(wb[sl(tn)], sw, swi, "e4m3")
        check_gemm(y[sl(tm), sl(tn)], A @ B.T, np.abs(A) @ np.abs(B).T, K, f"Y tile {tm},{tn}")
        # dX tile (tm, tk): dY rows x W columns, reduced over O
        A = _q(dyb[sl(tm)], sg, sgi, "e5m2")
        B = _q(wb[:, sl(tk)].T, sw, swi, "e4m3")
        check_gemm(dx[sl(tm), sl(tk)], A @ B.T, np.abs(A) @ np.abs(B).T, O, f"dX tile {tm},{tk}")
        # dW tile (tn, tk): dY columns x X columns, reduced over all N tokens
        A = _q(dyb[:, sl(tn)].T, sg, sgi, "e5m2")
        B = _q(xb[:, sl(tk)].T, sx, sxi, "e4m3")
        check_gemm(dw[sl(tn), sl(tk)], A @ B.T, np.abs(A) @ np.abs(B).T, N, f"dW tile {tn},{tk}")
