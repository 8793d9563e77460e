"""GPU parity of DelayedScaling (amax-history ring): bytes, scales and the
history ring bit-exact against the oracle over a sequence of tensors, the
weight cache under delayed scaling matching the oracle in both caching modes
(and the two modes differing, the documented non-bitwise behaviour), and a
delayed-scaling linear layer."""
import numpy as np
import pytest
import torch

import oracle as o
from fp8_mixed_precision_gb300 import synthetic as syn
from parity import assert_bytes_equal, assert_f32_equal, check_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp():
    from fp8_mixed_precision_gb300 import build
    build.build()
    import fp8_mixed_precision_gb300 as fp
    return fp


@pytest.mark.parametrize("role,shape", [("act", (512, 384)), ("grad", (272, 144))])
def test_delayed_sequence_parity(fp, role, shape):
    fmt = o.ROLE_FORMAT[role]
    H = 3
    hist_gpu = torch.zeros(H, dtype=torch.float32, device="cuda")
    hist = np.zeros(H, np.float32)
    for step, (std, seed) in enumerate([(1.0, 1), (4.0, 2), (0.25, 3), (2.0, 4), (0.5, 5)]):
        std = std * (1e-3 if role == "grad" else 1.0)
        x = syn.bf16_normal(shape, std, seed, device="cuda", outlier_frac=0.01)
        got = fp.fp8_quantize_delayed(x, role, hist_gpu, step)
        torch.cuda.synchronize()
        exp = o.quantize_delayed(syn.bits(x), fmt, hist, step)
        hist = exp["history"]
        assert_bytes_equal(got["row"], exp["row"], f"step {step} row")
        assert_bytes_equal(got["col"], exp["col"], f"step {step} col")
        assert_f32_equal(got["scale"], exp["row_scale"], f"step {step} scale")
        assert_f32_equal(got["scale_inv"], exp["row_scale_inv"], f"step {step} scale_inv")
        assert_f32_equal(hist_gpu, hist, f"step {step} history")


def test_delayed_weight_cache_matches_oracle_and_is_not_neutral(fp):
    """The weight changes between cycles (as after an optimizer step).  Under
    delayed scaling each quantization pushes the weight's amax into its
    history, so is_first_microbatch True/False and None give different FP8
    weights; both match the oracle's cache model bit for bit."""
    O, K, GA = 256, 384, 3
    ws0 = [syn.bf16_normal((O, K), 0.02 * (1.5 ** c), 70 + c, device="cuda") for c in range(3)]
    got, exp = {}, {}
    for use in (False, True):
        w = ws0[0].clone()
        cache = fp.WeightCache()
        h = cache.register(w, "delayed", history_len=4)
        oc = o.WeightCache("delayed", history_len=4)
        oc.register("w", syn.bits(w))
        g_rows, e_rows = [], []
        for cyc in range(3):
            w.copy_(ws0[cyc])                       # weight update between cycles
            oc.update("w", syn.bits(ws0[cyc]))
            cache.begin_cycle()
            oc.begin_cycle()
            for mb in range(GA):
                cache.get(h, cyc, use)
                g_rows.append(cache.entries[h].row.clone())
                e_rows.append(oc.get("w", use)["row"].copy())
        torch.cuda.synchronize()
        for i, (g, e) in enumerate(zip(g_rows, e_rows)):
            assert_bytes_equal(g, e, f"{'cached' if use else 'uncached'} quantization {i}")
        assert_f32_equal(cache.entries[h].history, oc.entries["w"]["history"], "history")
        got[use] = g_rows
    assert not all(torch.equal(a, b) for a, b in zip(got[False], got[True]))


def test_delayed_linear(fp):
    N, K, O = 512, 256, 384
    x, w, dy = syn.linear_inputs(N, K, O, device="cuda")
    cache = fp.WeightCache()
    h = cache.register(w, "delayed", history_len=2)
    cache.begin_cycle()
    cache.get(h, 0, True)          # first quantization: empty history -> scale 1
    cache.begin_cycle()
    cache.get(h, 1, True)          # second: scale from the recorded amax
    y, ctx = fp.fp8_linear_fwd(x, cache, h, "delayed")
    dx, dw = fp.fp8_linear_bwd(dy, ctx, cache, h, "delayed")
    torch.cuda.synchronize()
    wb = syn.bits(w)
    r0 = o.quantize_delayed(wb, "e4m3", np.zeros(2, np.float32), 0)
    wq = o.quantize_delayed(wb, "e4m3", r0["history"], 1)
    assert_bytes_equal(cache.entries[h].row, wq["row"], "Wq")
    xq = o.quantize_tensorwise(syn.bits(x), "e4m3")
    gq = o.quantize_tensorwise(syn.bits(dy), "e5m2")
    A = o.dequantize(xq["row"], xq["row_scale_inv"], "e4m3")
    B = o.dequantize(wq["row"], wq["row_scale_inv"], "e4m3")
    check_gemm(y, A @ B.T, np.abs(A) @ np.abs(B).T, K, "Y")
    G = o.dequantize(gq["row"], gq["row_scale_inv"], "e5m2")
    check_gemm(dx, G @ B, np.abs(G) @ np.abs(B), O, "dX")
    check_gemm(dw, G.T @ A, np.abs(G).T @ np.abs(A), N, "dW")
