"""The isolated-linear workload at its full size (N = 131072 tokens; 512->512,
512->2048, 2048->512, 512->8192; tensorwise current scaling), run exactly as
bench.py runs it (one shared workspace and context, fp8_linear_fwd then
fp8_linear_bwd), so every GEMM goes through the tile shape, split count and
CTA-pair configuration the benchmark times.  The oracle computes each
tensor's global amax itself, quantizes only the rows and columns that the
sampled 128x128 output tiles need, and checks for every GEMM the first and
the last tile and 64 seeded random tiles (all tiles of a smaller grid).
The wgrad's tiles, each a reduction over all 131072 tokens, come from a
product set of random tile rows and columns holding at least 64 tiles."""
import numpy as np
import pytest
import torch

import oracle as o
import sampled
from parity import check_gemm, log_margin
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


def _sl(t):
    return slice(t * 128, (t + 1) * 128)


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
    Wd = _q(wb, sw, swi, "e4m3")                     # [O, K], small: whole
    Wa = np.abs(Wd)

    # Y tiles (tm, tn): X rows x W rows, reduced over K
    yt = sampled.tiles(N // 128, O // 128, rng)
    rows = sorted({tm for tm, _ in yt})
    Xr = dict(zip(rows, sampled.pmap(lambda tm: _q(xb[_sl(tm)], sx, sxi, "e4m3"), rows)))
    res = [check_gemm(y[_sl(tm), _sl(tn)], Xr[tm] @ Wd[_sl(tn)].T,
                      np.abs(Xr[tm]) @ Wa[_sl(tn)].T, K, f"Y tile {tm},{tn}") for tm, tn in yt]
    log_margin(f"fprop {N}x{O}x{K} tensorwise", K, res)
    del Xr

    # dX tiles (tm, tk): dY rows x W columns, reduced over O
    dt = sampled.tiles(N // 128, K // 128, rng)
    rows = sorted({tm for tm, _ in dt})
    Gr = dict(zip(rows, sampled.pmap(lambda tm: _q(dyb[_sl(tm)], sg, sgi, "e5m2"), rows)))
    res = [check_gemm(dx[_sl(tm), _sl(tk)], Gr[tm] @ Wd[:, _sl(tk)],
                      np.abs(Gr[tm]) @ Wa[:, _sl(tk)], O, f"dX tile {tm},{tk}") for tm, tk in dt]
    log_margin(f"dgrad {N}x{K}x{O} tensorwise", O, res)
    del Gr

    # dW tiles (tn, tk): dY columns x X columns, reduced over all N tokens
    rn, ck = sampled.tile_grid(O // 128, K // 128, rng)
    Gc = dict(zip(rn, sampled.pmap(lambda tn: _q(dyb[:, _sl(tn)].T, sg, sgi, "e5m2"), rn)))
    Xc = dict(zip(ck, sampled.pmap(lambda tk: _q(xb[:, _sl(tk)].T, sx, sxi, "e4m3"), ck)))
    Xa = {tk: np.abs(v) for tk, v in Xc.items()}
    res = []
    for tn in rn:
        A = Gc.pop(tn)
        Aa = np.abs(A)
        for tk in ck:
            res.append(check_gemm(dw[_sl(tn), _sl(tk)], A @ Xc[tk].T, Aa @ Xa[tk].T, N,
                                  f"dW tile {tn},{tk}"))
    log_margin(f"wgrad {O}x{K}x{N} tensorwise", N, res)
