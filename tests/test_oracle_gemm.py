"""Pins of the oracle's GEMM, linear layer, weight-cache model and GELU:
brute force with exactly rounded sums, closed forms, the transpose identity,
finite differences for the backward operands and orientations, and library
routines for GELU."""
import math

import numpy as np
import pytest
import torch

import oracle as o
from fp8_mixed_precision_gb300 import synthetic as syn


def _rand_q(shape, seed):
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, shape).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x11                  # drop NaN codes (both formats)
    q[(q & 0x7C) == 0x7C] = 0x21                  # drop E5M2 inf/NaN codes
    return q


def _scale_at(s, m, k, rows):
    """scale_inv of element (m, k): explicit lookup, independent of the oracle."""
    s = np.asarray(s)
    if s.size == 1:
        return float(s.reshape(-1)[0])
    if s.shape[0] == rows:                       # 1x128 blocks along k
        return float(s[m, k // 128])
    return float(s[m // 128, k // 128])          # 128x128 tiles


def _brute_entry(aq, asi, af, bq, bsi, bf, m, n):
    """One output by a plain loop: decode each byte, apply its scale, exact
    sum with math.fsum, one rounding to bf16."""
    K = aq.shape[1]
    terms = [o.decode_byte(int(aq[m, k]), af) * _scale_at(asi, m, k, aq.shape[0]) *
             o.decode_byte(int(bq[n, k]), bf) * _scale_at(bsi, n, k, bq.shape[0])
             for k in range(K)]
    return o.round_to_bf16(np.array([math.fsum(terms)]))[0]


@pytest.mark.parametrize("M,N,K,scales", [(128, 128, 128, "tensor"), (128, 256, 384, "block"),
                                          (256, 128, 256, "mixed")])
def test_gemm_matches_brute_force(M, N, K, scales):
    rng = np.random.default_rng(M + N + K)
    aq, bq = _rand_q((M, K), 1), _rand_q((N, K), 2)
    if scales == "tensor":
        asi = np.float32([0.0123]); bsi = np.float32([3.5e-4])
    elif scales == "block":         # A 1x128 blocks, B 128x128 tiles (fprop / dgrad)
        asi = rng.uniform(1e-4, 1e-2, (M, K // 128)).astype(np.float32)
        bsi = rng.uniform(1e-4, 1e-2, (N // 128, K // 128)).astype(np.float32)
    else:                           # both 1x128 blocks along k (wgrad)
        asi = rng.uniform(1e-4, 1e-2, (M, K // 128)).astype(np.float32)
        bsi = rng.uniform(1e-4, 1e-2, (N, K // 128)).astype(np.float32)
    got = o.gemm(aq, asi, "e5m2", bq, bsi, "e4m3")
    picks = [(0, 0), (M - 1, N - 1), (127, 128 % N), (M // 2 + 3, N - 5)]
    picks += [tuple(p) for p in zip(rng.integers(0, M, 12), rng.integers(0, N, 12))]
    for m, n in picks:
        assert got[m, n] == _brute_entry(aq, asi, "e5m2", bq, bsi, "e4m3", m, n), (m, n)


def test_gemm_deep_k_brute_force():
    # wgrad-like reduction depth
    K = 131072
    aq, bq = _rand_q((128, K), 5), _rand_q((128, K), 6)
    rng = np.random.default_rng(0)
    asi = rng.uniform(1e-4, 1e-2, (128, K // 128)).astype(np.float32)
    bsi = rng.uniform(1e-4, 1e-2, (128, K // 128)).astype(np.float32)
    got = o.gemm(aq, asi, "e5m2", bq, bsi, "e4m3")
    A = o.dequantize(aq, asi, "e5m2")
    B = o.dequantize(bq, bsi, "e4m3")
    for (m, n) in [(0, 0), (5, 77), (127, 127), (64, 3)]:
        ref = o.round_to_bf16(np.array([math.fsum(A[m] * B[n])]))[0]
        assert got[m, n] == ref


def test_gemm_closed_form_integer_sums():
    # small-integer FP8 values with power-of-two scales: every sum is an
    # integer times 2^-j and exactly representable in bf16 -> exact result
    K = 256
    a_vals = np.array([1, 2, -1, 0, 3, -2], dtype=np.float32)
    rng = np.random.default_rng(1)
    A = rng.choice(a_vals, (128, K))
    B = np.zeros((128, K), np.float32)
    B[np.arange(128), np.arange(128)] = 1.0
    B[np.arange(128), np.arange(128) + 1] = -1.0
    aq, bq = o.encode(A, "e4m3"), o.encode(B, "e4m3")
    y = o.gemm(aq, np.float32([0.25]), "e4m3", bq, np.float32([2.0]), "e4m3")
    expect = (A[:, :128] - A[:, 1:129]) * 0.5
    assert np.array_equal(o.bf16_to_f32(y), expect.astype(np.float32))


def test_gemm_scaled_identity_weight():
    # W = c*I with c = 448*2^-5: tensorwise scale 2^5, W decodes to c exactly,
    # so Y = bf16(decode(Xq) * sx_inv * c)
    c = 448.0 * 2.0 ** -5
    W = np.eye(128, dtype=np.float32) * c
    wb = (W.view(np.uint32) >> 16).astype(np.uint16)
    wq = o.quantize_tensorwise(wb, "e4m3")
    assert wq["row_scale"][0] == 32.0
    x = syn.bits(syn.bf16_normal((256, 128), 1.0, 1))
    xq = o.quantize_tensorwise(x, "e4m3")
    y = o.gemm(xq["row"], xq["row_scale_inv"], "e4m3", wq["row"], wq["row_scale_inv"], "e4m3")
    exp = o.round_to_bf16(o.decode(xq["row"], "e4m3") * float(xq["row_scale_inv"][0]) * c)
    assert np.array_equal(y, exp)


def test_gemm_transpose_identity():
    aq, bq = _rand_q((256, 256), 3), _rand_q((128, 256), 4)
    rng = np.random.default_rng(2)
    asi = rng.uniform(1e-3, 1e-1, (256, 2)).astype(np.float32)
    bsi = rng.uniform(1e-3, 1e-1, (128, 2)).astype(np.float32)
    ab = o.gemm(aq, asi, "e5m2", bq, bsi, "e4m3")
    ba = o.gemm(bq, bsi, "e4m3", aq, asi, "e5m2")
    assert np.array_equal(ab.T, ba)


@pytest.mark.parametrize("recipe", ["tensorwise", "block"])
def test_linear_backward_by_finite_differences(recipe):
    # f(X) = sum(Y(X) * G) with G the dequantized incoming gradient.  Y is linear
    # in X, so f(Xd + E_ij) - f(Xd) is exactly sum_o G[i,o] Wd[o,j] = dX[i,j]
    # before rounding; likewise for W.  The difference is taken with the
    # oracle's *forward* GEMM, so a wrong operand, layout or orientation in
    # the backward GEMMs shows up here.
    N, K, O = 256, 256, 128
    x, w, dy = syn.linear_inputs(N, K, O)
    x, w, dy = syn.bits(x), syn.bits(w), syn.bits(dy)
    r = o.linear_fwd_bwd(x, w, dy, recipe)
    Xd = o.dequantize(r["xq"]["row"], r["xq"]["row_scale_inv"], "e4m3")
    Wd = o.dequantize(r["wq"]["row"], r["wq"]["row_scale_inv"], "e4m3")
    Gd_row = o.dequantize(r["gq"]["row"], r["gq"]["row_scale_inv"], "e5m2")
    Gd_col = o.dequantize(r["gq"]["col"], r["gq"]["col_scale_inv"], "e5m2").T
    Xd_col = o.dequantize(r["xq"]["col"], r["xq"]["col_scale_inv"], "e4m3").T
    Wd_col = o.dequantize(r["wq"]["col"], r["wq"]["col_scale_inv"], "e4m3").T
    if recipe == "tensorwise":      # one scale: both layouts hold the same values
        assert np.array_equal(Xd_col, Xd) and np.array_equal(Gd_col, Gd_row)
    assert np.array_equal(Wd_col, Wd)   # weights: byte transpose with transposed scales
    f = lambda X, W, G: float(np.sum((X @ W.T) * G))
    rng = np.random.default_rng(0)
    for _ in range(6):
        i, j = rng.integers(N), rng.integers(K)
        E = np.zeros_like(Xd); E[i, j] = 1.0
        fd = f(Xd + E, Wd_col, Gd_row) - f(Xd, Wd_col, Gd_row)
        assert o.round_to_bf16(np.array([fd]))[0] == r["dx"][i, j] or \
            abs(o.bf16_to_f32(r["dx"][i:i+1, j])[0] - fd) <= 2 ** -7 * abs(fd) + 1e-30
        p, q = rng.integers(O), rng.integers(K)
        E = np.zeros_like(Wd); E[p, q] = 1.0
        fd = f(Xd_col, Wd + E, Gd_col) - f(Xd_col, Wd, Gd_col)
        assert abs(o.bf16_to_f32(r["dw"][p:p+1, q])[0] - fd) <= 2 ** -7 * abs(fd) + 1e-30
        # exact fp64 value of the same entries from explicit sums
        assert o.round_to_bf16(np.array([math.fsum(Gd_col[:, p] * Xd_col[:, q])]))[0] == r["dw"][p, q]
        assert o.round_to_bf16(np.array([math.fsum(Gd_row[i, :] * Wd_col[:, j])]))[0] == r["dx"][i, j]


def test_weight_cache_model_bitwise_and_counts():
    x, w, dy = syn.linear_inputs(256, 256, 128)
    w = syn.bits(w)
    outs = {}
    for use in (False, True):
        c = o.WeightCache("block")
        c.register("fc", w)
        ys = []
        for cycle in range(2):
            c.begin_cycle()
            for mb in range(4):
                xb = syn.bits(syn.bf16_normal((256, 256), 1.0, 100 + mb))
                ys.append(o.linear_fwd(xb, c.get("fc", use), "block")["y"])
        outs[use] = (ys, c.quantize_calls)
    assert all(np.array_equal(a, b) for a, b in zip(outs[False][0], outs[True][0]))
    assert outs[False][1] == 8 and outs[True][1] == 2


def test_gelu_pins():
    assert o.gelu_f64(np.array([0.0]))[0] == 0.0
    assert o.gelu_grad_f64(np.array([0.0]))[0] == 0.5
    assert abs(o.gelu_f64(np.array([10.0]))[0] - 10.0) < 1e-12
    assert abs(o.gelu_f64(np.array([-10.0]))[0]) < 1e-12
    # 50-digit evaluation of h * Phi(h) and Phi(h) + h phi(h) (mpmath), including
    # the far negative tail where 1 + erf(h/sqrt 2) would cancel in fp64
    import mpmath as mp
    mp.mp.dps = 50
    hs = np.concatenate([np.linspace(-14, 8, 221), [-7.8125, -7.875, -3.0, -1e-3, 1e-3]])
    for h in hs:
        H = mp.mpf(float(h))
        cdf = mp.ncdf(H)
        pdf = mp.npdf(H)
        g = float(H * cdf)
        d = float(cdf + H * pdf)
        assert abs(o.gelu_f64(np.array([h]))[0] - g) <= 1e-13 * abs(g) + 1e-300
        assert abs(o.gelu_grad_f64(np.array([h]))[0] - d) <= 1e-12 * abs(d) + 1e-300
    # torch's fp64 GELU (library routine) where its erf form has no cancellation
    h = np.linspace(-3, 8, 2001)
    ht = torch.from_numpy(h).requires_grad_(True)
    yt = torch.nn.functional.gelu(ht)
    yt.sum().backward()
    assert np.allclose(o.gelu_f64(h), yt.detach().numpy(), rtol=1e-12, atol=1e-15)
    assert np.allclose(o.gelu_grad_f64(h), ht.grad.numpy(), rtol=1e-12, atol=1e-15)
    # bf16 wrappers round once
    hb = syn.bits(syn.bf16_normal((4, 128), 2.0, 3))
    assert np.array_equal(o.gelu_fwd(hb), o.round_to_bf16(o.gelu_f64(o.bf16_to_f32(hb))))


def test_grad_accumulate_fp32():
    acc = np.zeros(4, np.float32)
    d = np.array([0x3F80, 0x3F80, 0xBF80, 0x0000], np.uint16)   # 1, 1, -1, 0
    acc = o.grad_accumulate(acc, d)
    acc = o.grad_accumulate(acc, d)
    assert list(acc) == [2.0, 2.0, -2.0, 0.0]
    big = np.array([2.0 ** 24], np.float32)
    assert o.grad_accumulate(big, np.array([0x3F80], np.uint16))[0] == 2.0 ** 24   # fp32 RNE tie-to-even


def test_mlp_gelu_stage_by_central_differences():
    # In the MLP backward, dH = dA * GELU'(H) with H the bf16 fc1 output and
    # dA the fc2 dgrad output.  Check that wiring (H, not A; dA, not dY) with a
    # central difference of the fp64 GELU, independent of gelu_grad_f64.
    N, d, ffn = 256, 128, 256
    x = syn.bits(syn.bf16_normal((N, d), 1.0, 61))
    w1 = syn.bits(syn.bf16_normal((ffn, d), 0.02, 62))
    w2 = syn.bits(syn.bf16_normal((d, ffn), 0.02, 63))
    dy = syn.bits(syn.bf16_normal((N, d), 1e-3, 64))
    r = o.mlp_fwd_bwd(x, w1, w2, dy, "block")
    h = o.bf16_to_f32(r["h"]).astype(np.float64)
    da = o.bf16_to_f32(r["da"]).astype(np.float64)
    dh = o.bf16_to_f32(r["dh"]).astype(np.float64)
    rng = np.random.default_rng(7)
    for _ in range(64):
        i, j = int(rng.integers(N)), int(rng.integers(ffn))
        hv = h[i, j]
        eps = 1e-5 * max(1.0, abs(hv))
        slope = (o.gelu_f64(np.array([hv + eps])) - o.gelu_f64(np.array([hv - eps])))[0] / (2 * eps)
        want = da[i, j] * slope
        # dH is rounded once to bf16: within one bf16 ulp of the product (plus
        # the difference quotient's own error)
        assert abs(dh[i, j] - want) <= 2.0 ** -8 * abs(want) + 1e-12 * abs(da[i, j]) + 1e-30, \
            (i, j, dh[i, j], want)
    # the forward stage: A = bf16(GELU(H)) from the same H
    a = o.bf16_to_f32(r["a"]).astype(np.float64)
    ref = o.gelu_f64(h)
    assert np.all(np.abs(a - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30)
