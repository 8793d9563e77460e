"""GPU parity of the MLP-level workloads: the block-scaled MLP block (fc1 ->
GELU -> fc2, fwd + bwd), the weight cache under gradient accumulation in a
stack (cached vs uncached bitwise identical, one weight quantization per
cycle), and the large block-scaled linear with 1% x100 outliers checked on
sampled output tiles at its full size."""
import numpy as np
import pytest
import torch

import oracle as o
import sampled
from fp8_mixed_precision_gb300 import synthetic as syn
from parity import assert_bytes_equal, assert_f32_equal, bf16_ulp, check_gemm, to_np

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def fp():
    from fp8_mixed_precision_gb300 import build
    build.build()
    import fp8_mixed_precision_gb300 as fp
    return fp


def _rel(got, exp_bits_or_f32):
    g = o.bf16_to_f32(to_np(got)).astype(np.float64) if got.dtype == torch.bfloat16 \
        else to_np(got).astype(np.float64)
    e = exp_bits_or_f32
    e = o.bf16_to_f32(e).astype(np.float64) if e.dtype == np.uint16 else e.astype(np.float64)
    return float(np.linalg.norm(g - e) / max(np.linalg.norm(e), 1e-300))


def _oracle_stack(xb, w1b, w2b, dyb, recipe):
    """Oracle chain for a stack of MLP blocks, one microbatch."""
    L = len(w1b)
    w1q = [o.quantize(w, recipe, "weight") for w in w1b]
    w2q = [o.quantize(w, recipe, "weight") for w in w2b]
    h, saved = xb, []
    for l in range(L):
        f1 = o.linear_fwd(h, w1q[l], recipe)
        a = o.gelu_fwd(f1["y"])
        f2 = o.linear_fwd(a, w2q[l], recipe)
        saved.append((f1, a, f2))
        h = f2["y"]
    y = h
    g = dyb
    dw1, dw2 = [None] * L, [None] * L
    for l in reversed(range(L)):
        f1, a, f2 = saved[l]
        b2 = o.linear_bwd(g, f2, w2q[l], recipe)
        dh = o.gelu_bwd(b2["dx"], f1["y"])
        b1 = o.linear_bwd(dh, f1, w1q[l], recipe)
        dw1[l], dw2[l] = b1["dw"], b2["dw"]
        g = b1["dx"]
    return dict(y=y, dx=g, dw1=dw1, dw2=dw2, h0=saved[0][0]["y"], xq0=saved[0][0]["xq"])


def _stage_fwd(got, a_bits, wq, recipe, K, what):
    """One linear's forward as a stage: the oracle quantizes the GPU's own
    bf16 input and multiplies it with the oracle's FP8 weight; the GPU's
    output must be within the single-GEMM bound.  Returns the oracle's
    forward context for the backward stage."""
    f = o.linear_fwd(a_bits, wq, recipe)
    xq = f["xq"]
    A = o.dequantize(xq["row"], xq["row_scale_inv"], "e4m3")
    B = o.dequantize(wq["row"], wq["row_scale_inv"], "e4m3")
    check_gemm(got, A @ B.T, np.abs(A) @ np.abs(B).T, K, what)
    return f


def _stage_bwd(dx_got, dw_got, g_bits, ctx, wq, recipe, O, N, what):
    """One linear's backward as a stage, from the GPU's own incoming bf16
    gradient: dgrad and wgrad within the single-GEMM bound."""
    gq = o.quantize(g_bits, recipe, "grad")
    A = o.dequantize(gq["row"], gq["row_scale_inv"], "e5m2")
    B = o.dequantize(wq["col"], wq["col_scale_inv"], "e4m3")
    check_gemm(dx_got, A @ B.T, np.abs(A) @ np.abs(B).T, O, what + " dgrad")
    A = o.dequantize(gq["col"], gq["col_scale_inv"], "e5m2")
    xq = ctx["xq"]
    B = o.dequantize(xq["col"], xq["col_scale_inv"], "e4m3")
    check_gemm(dw_got, A @ B.T, np.abs(A) @ np.abs(B).T, N, what + " wgrad")


def _within_ulp(got, exp_bits, what):
    g = o.bf16_to_f32(to_np(got)).astype(np.float64)
    e = o.bf16_to_f32(exp_bits).astype(np.float64)
    bad = ~(np.abs(g - e) <= bf16_ulp(e))
    assert not bad.any(), f"{what}: {int(bad.sum())} entries beyond 1 bf16 ulp"


# End-to-end sanity bound for outputs several re-quantized stages away from
# the synthetic inputs.  Two evaluations of the same FP8 chain that differ
# only by 1 bf16 ulp in a few GELU outputs re-quantize later tensors onto
# different codes and block scales (E5M2 gradients keep 2 mantissa bits), so
# their end-to-end results differ by a few percent at four stages, while the
# FP8 chain itself is about 10% away from unquantized arithmetic.  Every
# stage is held to the exact bounds separately (stage-wise checks); this
# bound only catches gross errors.
E2E_TOL = 5e-2


@pytest.mark.parametrize("recipe", ["block", "tensorwise"])
@pytest.mark.parametrize("N", [4096, 400])
def test_mlp_block_parity(fp, recipe, N):
    """One MLP block fwd + bwd, every stage against the oracle fed the GPU's
    own inputs for that stage: both linears' forward, dgrad and wgrad within
    the single-GEMM bound, both GELU stages within 1 bf16 ulp, the saved
    FP8 input bytes exact; end-to-end outputs against the oracle's chain
    within the sanity bound."""
    from fp8_mixed_precision_gb300.mlp import FP8MLPStack
    d, ffn = 512, 2048
    st = FP8MLPStack(d, ffn, 1, N, recipe)
    x = syn.bf16_normal((N, d), 1.0, syn.SEED_X, device="cuda")
    dy = syn.bf16_normal((N, d), 1e-3, syn.SEED_DY, device="cuda")
    st.step([x], [dy], use_cache=True)
    torch.cuda.synchronize()
    assert fp.fp8_get_device_status() == 0
    xb, dyb = syn.bits(x), syn.bits(dy)
    Hb, Ab, dAb, dHb = syn.bits(st.H[0]), syn.bits(st.A[0]), syn.bits(st.dA), syn.bits(st.dH)
    w1q = o.quantize(syn.bits(st.w1[0]), recipe, "weight")
    w2q = o.quantize(syn.bits(st.w2[0]), recipe, "weight")
    f1 = _stage_fwd(st.H[0], xb, w1q, recipe, d, "fc1 fprop")
    xq_col = st.ctx1[0].ctx[:N * d].view(d, N)
    assert_bytes_equal(xq_col, f1["xq"]["col"], "Xq colwise (fc1 context)")
    _within_ulp(st.A[0], o.gelu_fwd(Hb), "A = GELU(H)")
    f2 = _stage_fwd(st.Y[0], Ab, w2q, recipe, ffn, "fc2 fprop")
    _stage_bwd(st.dA, st.dwb2, dyb, f2, w2q, recipe, d, N, "fc2")
    _within_ulp(st.dH, o.gelu_bwd(dAb, Hb), "dH = dA GELU'(H)")
    _stage_bwd(st.g[0], st.dwb1, dHb, f1, w1q, recipe, ffn, N, "fc1")
    # end to end against the oracle's own chain: sanity bound only
    r = _oracle_stack(xb, [syn.bits(st.w1[0])], [syn.bits(st.w2[0])], dyb, recipe)
    rels = {"Y": _rel(st.Y[0], r["y"]), "dX": _rel(st.g[0], r["dx"]),
            "dW1": _rel(st.dw1[0], o.bf16_to_f32(r["dw1"][0])),
            "dW2": _rel(st.dw2[0], o.bf16_to_f32(r["dw2"][0]))}
    for k, v in rels.items():
        assert v <= E2E_TOL, f"{k}: end-to-end relative Frobenius error {v:.3g}"


@pytest.mark.parametrize("recipe", ["block", "tensorwise"])
def test_stack_weight_cache_bitwise(fp, recipe):
    """Two-layer stack, GA = 4: is_first_microbatch True/False against None
    gives bitwise identical outputs and accumulated gradients over two
    cycles; the cached run quantizes each of the 4 weights once per cycle."""
    from fp8_mixed_precision_gb300.mlp import FP8MLPStack
    d, ffn, N, L, GA = 512, 2048, 1024, 2, 4
    xs = [syn.bf16_normal((N, d), 1.0, 500 + i, device="cuda") for i in range(GA)]
    dys = [syn.bf16_normal((N, d), 1e-3, 600 + i, device="cuda") for i in range(GA)]
    res = {}
    for use in (False, True):
        st = FP8MLPStack(d, ffn, L, N, recipe)
        n0 = fp.fp8_launch_count()
        outs = [st.step(xs, dys, use) for _ in range(2)]
        torch.cuda.synchronize()
        res[use] = (outs, [t.clone() for t in st.dw1 + st.dw2], st.requantized,
                    fp.fp8_launch_count() - n0)
    (o_u, g_u, q_u, l_u), (o_c, g_c, q_c, l_c) = res[False], res[True]
    assert q_u == 2 * GA * 2 * L and q_c == 2 * 2 * L
    assert l_c < l_u
    for cyc_u, cyc_c in zip(o_u, o_c):
        for (y1, dx1), (y2, dx2) in zip(cyc_u, cyc_c):
            assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
            assert torch.equal(dx1.view(torch.int16), dx2.view(torch.int16))
    for a, b in zip(g_u, g_c):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    # the last stage of the last microbatch against the oracle fed the GPU's
    # own inputs: layer 0's fc1 wgrad from its dH and that microbatch's X
    w1q0 = o.quantize(syn.bits(st.w1[0]), recipe, "weight")
    f1 = o.linear_fwd(syn.bits(xs[-1]), w1q0, recipe)
    gq = o.quantize(syn.bits(st.dH), recipe, "grad")
    A = o.dequantize(gq["col"], gq["col_scale_inv"], "e5m2")
    B = o.dequantize(f1["xq"]["col"], f1["xq"]["col_scale_inv"], "e4m3")
    check_gemm(st.dwb1, A @ B.T, np.abs(A) @ np.abs(B).T, N, "layer 0 fc1 wgrad, last microbatch")
    # the accumulated gradients against the oracle's chain + fp32
    # accumulation: end-to-end sanity bound (see E2E_TOL)
    w1b = [syn.bits(w) for w in st.w1]      # the stack's synthetic weights (generator output)
    w2b = [syn.bits(w) for w in st.w2]
    acc1 = [np.zeros((ffn, d), np.float32) for _ in range(L)]
    for i in range(GA):
        r = _oracle_stack(syn.bits(xs[i]), w1b, w2b, syn.bits(dys[i]), recipe)
        for l in range(L):
            acc1[l] = o.grad_accumulate(acc1[l], r["dw1"][l])
    for l in range(L):
        rel = _rel(g_c[l], acc1[l])
        assert rel <= E2E_TOL, f"dW1[{l}] accumulated: end-to-end relative Frobenius error {rel:.3g}"


@pytest.mark.parametrize("K,O", [(4096, 14336), (14336, 4096)])
def test_large_block_linear_sampled_tiles(fp, K, O):
    """fc1 (4096 -> 14336) and fc2 (14336 -> 4096) of the large block-scaled
    MLP at full size (16384 tokens, 1% of X entries x100): GPU fwd + bwd,
    oracle on the first, the last and 64 seeded random 128x128 tiles of Y, dX
    and dW."""
    N = 16384
    x = syn.bf16_normal((N, K), 1.0, syn.SEED_X, device="cuda", outlier_frac=0.01)
    w = syn.bf16_normal((O, K), 0.02, syn.SEED_W, device="cuda")
    dy = syn.bf16_normal((N, O), 1e-3, syn.SEED_DY, device="cuda")
    cache = fp.WeightCache()
    h = cache.register(w, "block")
    cache.begin_cycle()
    cache.get(h, 0, True)
    y, ctx = fp.fp8_linear_fwd(x, cache, h, "block")
    dx, dw = fp.fp8_linear_bwd(dy, ctx, cache, h, "block")
    torch.cuda.synchronize()
    assert fp.fp8_get_device_status() == 0
    xb, wb, dyb = syn.bits(x), syn.bits(w), syn.bits(dy)
    wq = o.quantize_128x128(wb, "e4m3")
    e = cache.entries[h]
    assert_bytes_equal(e.row, wq["row"], "Wq row")
    assert_bytes_equal(e.col, wq["col"], "Wq col")
    assert_f32_equal(e.col_scale_inv, wq["col_scale_inv"], "Wq col scale_inv")
    rng = np.random.default_rng(3)
    Wr = o.dequantize(wq["row"], wq["row_scale_inv"], "e4m3")    # fprop B [O, K]
    Wc = o.dequantize(wq["col"], wq["col_scale_inv"], "e4m3")    # dgrad B [K, O]
    # first, last and 64 random output tiles of each GEMM (X rows and dY rows
    # in 1x128 blocks along the reduction; the wgrad's operands are the
    # transposed layouts, 1x128 blocks along the 16384 tokens)
    sampled.check_fwd_like(y, xb, "e4m3", Wr, K, f"fprop {N}x{O}x{K} block 1x128x128x128", rng)
    sampled.check_fwd_like(dx, dyb, "e5m2", Wc, O, f"dgrad {N}x{K}x{O} block 1x128x128x128", rng)
    sampled.check_wgrad(dw, dyb, "e5m2", xb, "e4m3", f"wgrad {O}x{K}x{N} block 1x128x1x128", rng)


@pytest.mark.parametrize("N", [1024, 400])
def test_fused_gelu_quantize_equals_unfused(fp, N):
    """Quantization fused into the GELU producers gives the bytes and scales
    of the unfused sequence (GELU to bf16, then quantize) bit for bit."""
    F = 384
    h = syn.bf16_normal((N, F), 2.0, 81, device="cuda", outlier_frac=0.01)
    da = syn.bf16_normal((N, F), 1e-3, 82, device="cuda")
    qf = fp.fp8_gelu_quantize(h, fp.QuantizedTensor(N, F, "act", "cuda"))
    ref = fp.fp8_quantize(fp.fp8_gelu_fwd(h), "block", "act")
    gf = fp.fp8_gelu_bwd_quantize(da, h, fp.QuantizedTensor(N, F, "grad", "cuda"))
    gref = fp.fp8_quantize(fp.fp8_gelu_bwd(da, h), "block", "grad")
    torch.cuda.synchronize()
    for got, exp in ((qf, ref), (gf, gref)):
        assert torch.equal(got.row, exp["row"]) and torch.equal(got.col, exp["col"])
        for k in ("row_scale", "row_scale_inv", "col_scale", "col_scale_inv"):
            assert torch.equal(getattr(got, k).view(torch.int32), exp[k].view(torch.int32)), k


@pytest.mark.parametrize("N,F", [(1024, 384), (400, 400)])
def test_fused_gelu_quantize_oracle(fp, N, F):
    """Quantization fused into the GELU producers against the oracle,
    stage-wise (GELU is held to 1 bf16 ulp of the fp64 oracle, not bitwise):
    the oracle's 1x128 quantizer, fed the GPU's bf16 GELU output (forward)
    or dA * GELU'(H) (backward), gives the fused kernel's row and transposed
    bytes and all four scale arrays bit for bit.  1% of H entries are x100
    outliers; (400, 400) has ragged 128-blocks in both dimensions."""
    h = syn.bf16_normal((N, F), 2.0, 83, device="cuda", outlier_frac=0.01)
    da = syn.bf16_normal((N, F), 1e-3, 84, device="cuda")
    qf = fp.fp8_gelu_quantize(h, fp.QuantizedTensor(N, F, "act", "cuda"))
    gf = fp.fp8_gelu_bwd_quantize(da, h, fp.QuantizedTensor(N, F, "grad", "cuda"))
    a = fp.fp8_gelu_fwd(h)
    dh = fp.fp8_gelu_bwd(da, h)
    torch.cuda.synchronize()
    hb, dab = syn.bits(h), syn.bits(da)
    for got_bf16, exp_bits, nm in ((a, o.gelu_fwd(hb), "GELU"), (dh, o.gelu_bwd(dab, hb), "GELU'")):
        g = o.bf16_to_f32(syn.bits(got_bf16)).astype(np.float64)
        e = o.bf16_to_f32(exp_bits).astype(np.float64)
        assert (np.abs(g - e) <= bf16_ulp(e)).all(), f"{nm} beyond 1 bf16 ulp"
    for q, stage, fmt, nm in ((qf, a, "e4m3", "fused GELU + quantize"),
                              (gf, dh, "e5m2", "fused GELU backward + quantize")):
        r = o.quantize_1x128(syn.bits(stage), fmt)
        assert_bytes_equal(q.row, r["row"], f"{nm}: row bytes")
        assert_bytes_equal(q.col, r["col"], f"{nm}: transposed bytes")
        for k in ("row_scale", "row_scale_inv", "col_scale", "col_scale_inv"):
            assert_f32_equal(getattr(q, k), r[k], f"{nm}: {k}")


def test_fused_mlp_stack_equals_unfused(fp):
    from fp8_mixed_precision_gb300.mlp import FP8MLPStack
    d, ffn, N, L, GA = 512, 1024, 768, 2, 2
    xs = [syn.bf16_normal((N, d), 1.0, 900 + i, device="cuda") for i in range(GA)]
    dys = [syn.bf16_normal((N, d), 1e-3, 910 + i, device="cuda") for i in range(GA)]
    res = {}
    for fused in (False, True):
        st = FP8MLPStack(d, ffn, L, N, "block", fused=fused)
        outs = st.step(xs, dys, True)
        torch.cuda.synchronize()
        res[fused] = (outs, [t.clone() for t in st.dw1 + st.dw2])
    for (y1, dx1), (y2, dx2) in zip(res[False][0], res[True][0]):
        assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
        assert torch.equal(dx1.view(torch.int16), dx2.view(torch.int16))
    for a, b in zip(res[False][1], res[True][1]):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
