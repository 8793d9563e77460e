"""The block-scaled MLP workloads at their full sizes, run through
FP8MLPStack exactly as bench.py runs them.

* Block MLP d=512, ffn=2048 at N = 131072 tokens (fc1 -> GELU -> fc2, fwd +
  bwd, Float8BlockScaling reading: 1x128 blocks for activations and
  gradients, 128x128 for weights).  Every GEMM of both linears - fprop,
  dgrad and the 1x128 x 1x128 wgrad reduced over all 131072 tokens, through
  the plan and split the benchmark uses - is checked against the oracle on
  its first and last 128x128 output tile and 64 seeded random tiles (every
  tile when the output has no more).  Checks are stage-wise: a GEMM fed by
  an earlier GEMM's or the GELU's bf16 output gets the GPU's own copy of that
  tensor as the oracle's input, so each stage is held to the single-GEMM
  bound (rel. Frobenius 2e-3 and 2 bf16 ulp).
* Weight caching under gradient accumulation: the 8-layer stack (16 FP8
  linears, d=512, ffn=2048), GA = 4 microbatches of 131072 tokens, one
  cycle cached (is_first_microbatch True/False) and one uncached (None):
  outputs and accumulated gradients bitwise identical (TransformerEngine
  issue #2852, maintainer reply), each cached weight's FP8 bytes and scales
  equal to the oracle's."""
import numpy as np
import pytest
import torch

import oracle as o
import sampled
from parity import assert_bytes_equal, assert_f32_equal, bf16_ulp
from fp8_mixed_precision_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp():
    from fp8_mixed_precision_gb300 import build
    build.build()
    import fp8_mixed_precision_gb300 as fp
    return fp


def test_block_mlp_full_size_sampled_tiles(fp):
    from fp8_mixed_precision_gb300.mlp import FP8MLPStack
    N, d, ffn = 131072, 512, 2048
    st = FP8MLPStack(d, ffn, 1, N, "block")
    x = syn.bf16_normal((N, d), 1.0, syn.SEED_X, device="cuda")
    dy = syn.bf16_normal((N, d), 1e-3, syn.SEED_DY, device="cuda")
    st.step([x], [dy], use_cache=True)
    torch.cuda.synchronize()
    assert fp.fp8_get_device_status() == 0
    xb, dyb = syn.bits(x), syn.bits(dy)
    Hb, Ab = syn.bits(st.H[0]), syn.bits(st.A[0])          # fc1 output, GELU output
    dAb, dHb = syn.bits(st.dA), syn.bits(st.dH)            # fc2 dgrad, GELU backward
    w1q = o.quantize_128x128(syn.bits(st.w1[0]), "e4m3")    # [ffn, d]
    w2q = o.quantize_128x128(syn.bits(st.w2[0]), "e4m3")    # [d, ffn]
    e1, e2 = st.cache.entries[st.h1[0]], st.cache.entries[st.h2[0]]
    for e, wq, nm in ((e1, w1q, "W1"), (e2, w2q, "W2")):
        assert_bytes_equal(e.row, wq["row"], f"{nm}q row")
        assert_bytes_equal(e.col, wq["col"], f"{nm}q col")
        assert_f32_equal(e.row_scale_inv, wq["row_scale_inv"], f"{nm}q row scale_inv")
    W1r = o.dequantize(w1q["row"], w1q["row_scale_inv"], "e4m3")   # fc1 fprop B [ffn, d]
    W1c = o.dequantize(w1q["col"], w1q["col_scale_inv"], "e4m3")   # fc1 dgrad B [d, ffn]
    W2r = o.dequantize(w2q["row"], w2q["row_scale_inv"], "e4m3")   # fc2 fprop B [d, ffn]
    W2c = o.dequantize(w2q["col"], w2q["col_scale_inv"], "e4m3")   # fc2 dgrad B [ffn, d]
    dw1 = st.dwb1.clone()   # bf16 dW of the single microbatch, before accumulation
    dw2 = st.dwb2.clone()
    rng = np.random.default_rng(2)
    sampled.check_fwd_like(st.H[0], xb, "e4m3", W1r, d, f"fc1 fprop {N}x{ffn}x{d} block", rng)
    sampled.check_fwd_like(st.Y[0], Ab, "e4m3", W2r, ffn, f"fc2 fprop {N}x{d}x{ffn} block", rng)
    sampled.check_fwd_like(st.dA, dyb, "e5m2", W2c, d, f"fc2 dgrad {N}x{ffn}x{d} block", rng)
    sampled.check_fwd_like(st.g[0], dHb, "e5m2", W1c, ffn, f"fc1 dgrad {N}x{d}x{ffn} block", rng)
    sampled.check_wgrad(dw2, dyb, "e5m2", Ab, "e4m3", f"fc2 wgrad {d}x{ffn}x{N} block 1x128x1x128", rng)
    sampled.check_wgrad(dw1, dHb, "e5m2", xb, "e4m3", f"fc1 wgrad {ffn}x{d}x{N} block 1x128x1x128", rng)
    # the fp32 accumulators of the single microbatch hold exactly the bf16 dW
    assert torch.equal(st.dw1[0], dw1.float()) and torch.equal(st.dw2[0], dw2.float())
    # the GELU stages on 2^20 sampled entries: within 1 bf16 ulp of the fp64 oracle
    idx = rng.choice(Hb.size, size=1 << 20, replace=False)
    h_s, da_s = Hb.reshape(-1)[idx], dAb.reshape(-1)[idx]
    for got, exp, nm in ((Ab.reshape(-1)[idx], o.gelu_fwd(h_s), "A = GELU(H)"),
                         (dHb.reshape(-1)[idx], o.gelu_bwd(da_s, h_s), "dH = dA GELU'(H)")):
        g = o.bf16_to_f32(got).astype(np.float64)
        e = o.bf16_to_f32(exp).astype(np.float64)
        bad = np.abs(g - e) > bf16_ulp(e)
        assert not bad.any(), f"{nm}: {int(bad.sum())} sampled entries beyond 1 bf16 ulp"


def test_weight_cache_stack_full_size_bitwise(fp):
    from fp8_mixed_precision_gb300.mlp import FP8MLPStack
    d, ffn, L, N, GA = 512, 2048, 8, 131072, 4
    xs = [syn.bf16_normal((N, d), 1.0, 700 + i, device="cuda") for i in range(GA)]
    dys = [syn.bf16_normal((N, d), 1e-3, 800 + i, device="cuda") for i in range(GA)]
    res = {}
    for use in (False, True):
        st = FP8MLPStack(d, ffn, L, N, "block")
        q0 = st.requantized
        outs = st.step(xs, dys, use)
        torch.cuda.synchronize()
        assert fp.fp8_get_device_status() == 0
        res[use] = (outs, [t.clone() for t in st.dw1 + st.dw2], st.requantized - q0)
        if use:   # the FP8 copies the cached cycle made on microbatch 0 and reused
            for l in range(L):
                for w, hd, nm in ((st.w1[l], st.h1[l], "W1"), (st.w2[l], st.h2[l], "W2")):
                    wq = o.quantize_128x128(syn.bits(w), "e4m3")
                    e = st.cache.entries[hd]
                    assert_bytes_equal(e.row, wq["row"], f"layer {l} {nm}q row")
                    assert_bytes_equal(e.col, wq["col"], f"layer {l} {nm}q col")
                    assert_f32_equal(e.row_scale_inv, wq["row_scale_inv"], f"layer {l} {nm} sinv")
        del st
        torch.cuda.empty_cache()
    (o_u, g_u, q_u), (o_c, g_c, q_c) = res[False], res[True]
    assert q_u == 2 * L * GA and q_c == 2 * L
    for i, ((y1, dx1), (y2, dx2)) in enumerate(zip(o_u, o_c)):
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16)), f"Y, microbatch {i}"
        assert torch.equal(dx1.view(torch.int16), dx2.view(torch.int16)), f"dX, microbatch {i}"
    for i, (a, b) in enumerate(zip(g_u, g_c)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"accumulated dW {i}"
