"""GPU parity of the FP8 linear layer (fwd + bwd through the C ABI) and of
the weight cache: quantized X/W/dY bytes and scales bit-exact, Y/dX/dW within
the GEMM tolerance, cached vs uncached outputs bitwise identical."""
import numpy as np
import pytest
import torch

import oracle as o
from fp8_mixed_precision_gb300 import synthetic as syn
from parity import bf16_ulp, assert_bytes_equal, assert_f32_equal, check_gemm, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp():
    from fp8_mixed_precision_gb300 import build
    build.build()
    import fp8_mixed_precision_gb300 as fp
    return fp


def _gemm_ref(aq, asi, af, bq, bsi, bf):
    A = o.dequantize(aq, asi, af)
    B = o.dequantize(bq, bsi, bf)
    return A @ B.T, np.abs(A) @ np.abs(B).T


@pytest.mark.parametrize("recipe", ["tensorwise", "block"])
@pytest.mark.parametrize("N,K,O", [(2048, 512, 512), (400, 272, 144), (1024, 512, 2048)])
def test_linear_parity(fp, recipe, N, K, O):
    x, w, dy = syn.linear_inputs(N, K, O, device="cuda")
    cache = fp.WeightCache()
    h = cache.register(w, recipe)
    cache.begin_cycle()
    assert cache.get(h, 0, True)
    y, ctx = fp.fp8_linear_fwd(x, cache, h, recipe)
    dx, dw = fp.fp8_linear_bwd(dy, ctx, cache, h, recipe)
    torch.cuda.synchronize()
    assert fp.fp8_get_device_status() == 0
    r = o.linear_fwd_bwd(syn.bits(x), syn.bits(w), syn.bits(dy), recipe)
    e = cache.entries[h]
    assert_bytes_equal(e.row, r["wq"]["row"], "Wq row")
    assert_bytes_equal(e.col, r["wq"]["col"], "Wq col")
    assert_f32_equal(e.row_scale_inv, r["wq"]["row_scale_inv"], "W scale_inv")
    xq, gq, wq = r["xq"], r["gq"], r["wq"]
    ref, ab = _gemm_ref(xq["row"], xq["row_scale_inv"], "e4m3", wq["row"], wq["row_scale_inv"], "e4m3")
    check_gemm(y, ref, ab, K, "Y")
    ref, ab = _gemm_ref(gq["row"], gq["row_scale_inv"], "e5m2", wq["col"], wq["col_scale_inv"], "e4m3")
    check_gemm(dx, ref, ab, O, "dX")
    ref, ab = _gemm_ref(gq["col"], gq["col_scale_inv"], "e5m2", xq["col"], xq["col_scale_inv"], "e4m3")
    check_gemm(dw, ref, ab, N, "dW")


@pytest.mark.parametrize("recipe", ["block", "tensorwise"])
def test_weight_cache_bitwise_and_launches(fp, recipe):
    """GA=4 microbatches, 2 cycles: is_first_microbatch True/False vs None give
    bitwise identical outputs and gradients; the cached run quantizes each
    weight once per cycle."""
    N, K, O = 1024, 512, 1024
    w = syn.bf16_normal((O, K), 0.02, 43, device="cuda")
    xs = [syn.bf16_normal((N, K), 1.0, 100 + i, device="cuda") for i in range(4)]
    dys = [syn.bf16_normal((N, O), 1e-3, 200 + i, device="cuda") for i in range(4)]
    outs = {}
    for use in (False, True):
        cache = fp.WeightCache()
        h = cache.register(w, recipe)
        ws = fp.linear_workspace(recipe, N, K, O, "cuda")
        res, nq = [], 0
        for cycle in range(2):
            cache.begin_cycle()
            for mb in range(4):
                nq += cache.get(h, cycle, use)
                y, ctx = fp.fp8_linear_fwd(xs[mb], cache, h, recipe, ws=ws)
                dx, dw = fp.fp8_linear_bwd(dys[mb], ctx, cache, h, recipe, ws=ws)
                res.append((y.clone(), dx.clone(), dw.clone()))
        torch.cuda.synchronize()
        outs[use] = (res, nq)
    assert outs[False][1] == 8 and outs[True][1] == 2
    for a, b in zip(outs[False][0], outs[True][0]):
        for t1, t2 in zip(a, b):
            assert torch.equal(t1.view(torch.int16), t2.view(torch.int16))


def test_weight_cache_stale_version(fp):
    w = syn.bf16_normal((256, 256), 0.02, 1, device="cuda")
    cache = fp.WeightCache()
    h = cache.register(w, "block")
    cache.begin_cycle()
    assert cache.get(h, 7, True) is True
    assert cache.get(h, 7, True) is False
    with pytest.raises(fp.FP8Error) as ei:
        cache.get(h, 8, True)
    assert ei.value.status == 4
    cache.begin_cycle()
    assert cache.get(h, 8, True) is True
    assert cache.get(h, 8, False) is True   # is_first_microbatch=None always re-quantizes


def test_gelu_and_accumulate(fp):
    hb = syn.bits(syn.bf16_normal((512, 256), 2.0, 11))
    hb[0, :6] = [0x0000, 0x8000, 0x4120, 0xC120, 0x3F80, 0xBF80]   # 0, -0, 10, -10, 1, -1
    h = syn.from_bits(hb, "cuda")
    a = fp.fp8_gelu_fwd(h)
    dab = syn.bits(syn.bf16_normal((512, 256), 1e-3, 12))
    da = syn.from_bits(dab, "cuda")
    dh = fp.fp8_gelu_bwd(da, h)
    torch.cuda.synchronize()
    for got, exp in ((a, o.gelu_fwd(hb)), (dh, o.gelu_bwd(dab, hb))):
        g = o.bf16_to_f32(to_np(got)).astype(np.float64)
        e = o.bf16_to_f32(exp).astype(np.float64)
        ulp = np.ldexp(1.0, (np.maximum(np.frexp(np.abs(e))[1] - 1, -126) - 7).astype(np.int32))
        assert np.all(np.abs(g - e) <= ulp), "GELU beyond 1 bf16 ulp"
    acc = torch.zeros((512, 256), dtype=torch.float32, device="cuda")
    exp = np.zeros((512, 256), np.float32)
    for i in range(3):
        db = syn.bits(syn.bf16_normal((512, 256), 1e-3, 30 + i))
        fp.fp8_grad_accumulate(acc, syn.from_bits(db, "cuda"))
        exp = o.grad_accumulate(exp, db)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(acc).view(np.uint32), exp.view(np.uint32))


def test_gelu_every_bf16_value(fp):
    """GELU forward and backward on every finite bf16 value (the whole input
    domain of the bf16 stage): within 1 bf16 ulp of the fp64 oracle.  The
    backward runs with dA = 1 (dH is then GELU'(H) rounded once) and with a
    seeded random dA."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    fin = np.isfinite(o.bf16_to_f32(allb))
    hb = allb[fin].reshape(-1, 128)     # 65280 finite patterns (256 are inf or NaN)
    h = syn.from_bits(hb, "cuda")
    ones = syn.from_bits(np.full(hb.shape, 0x3F80, np.uint16), "cuda")
    dab = syn.bits(syn.bf16_normal(hb.shape, 1e-3, 13))
    a = fp.fp8_gelu_fwd(h)
    d1 = fp.fp8_gelu_bwd(ones, h)
    d2 = fp.fp8_gelu_bwd(syn.from_bits(dab, "cuda"), h)
    torch.cuda.synchronize()
    for got, exp, nm in ((a, o.gelu_fwd(hb), "GELU"),
                         (d1, o.gelu_bwd(np.full(hb.shape, 0x3F80, np.uint16), hb), "GELU'"),
                         (d2, o.gelu_bwd(dab, hb), "dA GELU'")):
        g = o.bf16_to_f32(to_np(got)).astype(np.float64)
        e = o.bf16_to_f32(exp).astype(np.float64)
        bad = ~(np.abs(g - e) <= bf16_ulp(e))
        assert not bad.any(), (f"{nm}: {int(bad.sum())} inputs beyond 1 bf16 ulp, first "
                               f"{hb.reshape(-1)[np.argmax(bad.reshape(-1))]:#06x}")


def test_bounded_wait_reports_timeout_and_context_survives(fp):
    """A device-side wait that nothing satisfies gives up after its limit,
    records FP8_ERR_TIMEOUT (read and cleared by fp8_get_device_status), and
    the context keeps working: no trap, no fault, no hang."""
    import time
    t0 = time.perf_counter()
    fp.fp8_debug_wait_timeout(50_000_000)          # 50 ms
    assert fp.fp8_get_device_status() == 5          # FP8_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert fp.fp8_get_device_status() == 0          # cleared
    with pytest.raises(fp.FP8Error):
        fp.fp8_debug_wait_timeout(0)
    # the context is still usable: a GEMM runs and agrees with an exact case
    a = torch.full((128, 128), 0x38, dtype=torch.uint8, device="cuda")   # E4M3 1.0
    one = torch.ones(1, device="cuda")
    c = fp.fp8_gemm(a, "e4m3", one, a, "e4m3", one, "tensor")
    torch.cuda.synchronize()
    assert torch.all(c.float() == 128.0)
    assert fp.fp8_get_device_status() == 0


@pytest.mark.parametrize("recipe", ["tensorwise", "block"])
def test_fused_equals_plain_fp8(fp, recipe):
    """Exactness of the fused dual-layout path ("Native FP8 MLP reconstruction",
    exactness paragraph: fused output/dX/dW equal plain FP8 exactly): the
    plain arm quantizes every tensor in two separate passes (rowwise only,
    then transposed only) and calls the GEMMs directly; all bytes, scales and
    outputs equal the fused fp8_linear_fwd/bwd bit for bit."""
    N, K, O = 1024, 512, 768
    x, w, dy = syn.linear_inputs(N, K, O, device="cuda")
    cache = fp.WeightCache()
    h = cache.register(w, recipe)
    cache.begin_cycle()
    cache.get(h, 0, True)
    y, ctx = fp.fp8_linear_fwd(x, cache, h, recipe)
    dx, dw = fp.fp8_linear_bwd(dy, ctx, cache, h, recipe)
    q = lambda t, role, r, c: fp.fp8_quantize(t, recipe, role, rowwise=r, colwise=c)
    wr, wc = q(w, "weight", True, False), q(w, "weight", False, True)
    xr, xc = q(x, "act", True, False), q(x, "act", False, True)
    gr, gc = q(dy, "grad", True, False), q(dy, "grad", False, True)
    e = cache.entries[h]
    assert torch.equal(wr["row"], e.row) and torch.equal(wc["col"], e.col)
    blk = recipe == "block"
    y2 = fp.fp8_gemm(xr["row"], "e4m3", xr["row_scale_inv"], wr["row"], "e4m3", wr["row_scale_inv"],
                     "1x128_128x128" if blk else "tensor")
    dx2 = fp.fp8_gemm(gr["row"], "e5m2", gr["row_scale_inv"], wc["col"], "e4m3",
                      wc["col_scale_inv"] if blk else wc["row_scale_inv"],
                      "1x128_128x128" if blk else "tensor")
    dw2 = fp.fp8_gemm(gc["col"], "e5m2", gc["col_scale_inv"] if blk else gc["row_scale_inv"],
                      xc["col"], "e4m3", xc["col_scale_inv"] if blk else xc["row_scale_inv"],
                      "1x128_1x128" if blk else "tensor")
    torch.cuda.synchronize()
    for a, b, name in ((y, y2, "Y"), (dx, dx2, "dX"), (dw, dw2, "dW")):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name


@pytest.mark.parametrize("recipe", ["tensorwise", "delayed"])
def test_split_amax_pass_equals_one_call(fp, recipe):
    """fp8_amax_partials on a second stream, then the *_after_amax linear calls
    on the first: bit for bit the results of fp8_linear_fwd / fp8_linear_bwd."""
    N, K, O = 2048, 512, 1024
    x, w, dy = syn.linear_inputs(N, K, O, device="cuda")
    outs = {}
    for split in (False, True):
        cache = fp.WeightCache()
        h = cache.register(w, recipe)
        cache.begin_cycle()
        cache.get(h, 0, True)
        ws = fp.linear_workspace(recipe, N, K, O, "cuda")
        ctx = fp.LinearContext(fp._empty_bytes(fp._ctx_bytes(recipe, N, K), "cuda"), N, K)
        y = torch.empty((N, O), dtype=torch.bfloat16, device="cuda")
        dx = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
        dw = torch.empty((O, K), dtype=torch.bfloat16, device="cuda")
        if split:
            aux = torch.cuda.Stream()
            aux.wait_stream(torch.cuda.current_stream())
            px, pdy = fp.amax_partials_buffer(N, K, "cuda"), fp.amax_partials_buffer(N, O, "cuda")
            ex, ed = torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(aux):
                fp.fp8_amax_partials(x, px)
                ex.record(aux)
                fp.fp8_amax_partials(dy, pdy)
                ed.record(aux)
            torch.cuda.current_stream().wait_event(ex)
            fp.fp8_linear_fwd_after_amax(x, px, cache, h, recipe, ws, y, ctx)
            torch.cuda.current_stream().wait_event(ed)
            fp.fp8_linear_bwd_after_amax(dy, pdy, ctx, cache, h, recipe, ws, dx, dw)
        else:
            fp.fp8_linear_fwd(x, cache, h, recipe, ws=ws, y=y, ctx=ctx)
            fp.fp8_linear_bwd(dy, ctx, cache, h, recipe, ws=ws, dx=dx, dw=dw)
        torch.cuda.synchronize()
        outs[split] = (y, dx, dw)
    assert fp.fp8_get_device_status() == 0
    for a, b, name in zip(outs[False], outs[True], ("Y", "dX", "dW")):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name


def test_split_amax_pass_refuses_block_recipe(fp):
    N, K, O = 256, 256, 256
    x, w, dy = syn.linear_inputs(N, K, O, device="cuda")
    cache = fp.WeightCache()
    h = cache.register(w, "block")
    cache.begin_cycle()
    cache.get(h, 0, True)
    ws = fp.linear_workspace("block", N, K, O, "cuda")
    ctx = fp.LinearContext(fp._empty_bytes(fp._ctx_bytes("block", N, K), "cuda"), N, K)
    px = fp.amax_partials_buffer(N, K, "cuda")
    y = torch.empty((N, O), dtype=torch.bfloat16, device="cuda")
    n0 = fp.fp8_launch_count()
    with pytest.raises(fp.FP8Error) as e:
        fp.fp8_linear_fwd_after_amax(x, px, cache, h, "block", ws, y, ctx)
    assert e.value.status == 7
    assert fp.fp8_launch_count() == n0
