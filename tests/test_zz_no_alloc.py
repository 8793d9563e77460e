"""The allocation-free tensorwise quantizer, called through the C ABI.

It exists for callers that cannot allocate device memory: code running inside
a device allocator or memory-pool hook (allocating there would re-enter the
allocator), paths that must not call cudaMalloc/cudaFree because those can
synchronise the device, and plugins whose host framework owns all device
memory and hands them only inputs and outputs.  Its scratch is a fixed array
inside the library, shared by every call.

GPU checks: the same FP8 bytes and scales as fp8_quantize (bit for bit, the
tolerance every quantizer test uses) on two calls in a row, the second
running with the first call's leftovers in the shared array; the same bytes
and scales as the oracle; a transposed-only E5M2 call.  CPU checks: argument
errors are answered before anything is launched.

Collected last on purpose, so that a run stopping at its first failure has
already run every other test; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as o
from parity import assert_bytes_equal, assert_f32_equal


def _bind(fp):
    L = fp.lib()
    f = L.fp8_quantize_tensorwise_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return f


@pytest.fixture(scope="module")
def fp():
    from fp8_mixed_precision_gb300 import build
    build.build()
    import fp8_mixed_precision_gb300 as fp
    _bind(fp)
    return fp


def _noalloc(fp, x, role, rowwise=True, colwise=True):
    R, C = x.shape
    row = torch.empty((R, C), dtype=torch.uint8, device="cuda") if rowwise else None
    col = torch.empty((C, R), dtype=torch.uint8, device="cuda") if colwise else None
    s = torch.empty(1, dtype=torch.float32, device="cuda")
    si = torch.empty(1, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ptr = lambda t: ctypes.c_void_p(t.data_ptr() if t is not None else None)
    st = fp.lib().fp8_quantize_tensorwise_noalloc(
        ctypes.c_void_p(x.data_ptr()), R, C, fp.ROLE[role], ptr(row), ptr(col), ptr(s), ptr(si),
        stream)
    assert st == 0, st
    return row, col, s, si


@pytest.mark.gpu
def test_noalloc_matches_workspace_quantizer_twice(fp):
    from fp8_mixed_precision_gb300 import synthetic as syn
    cases = [((4096, 1024), 1.0, "act", 11), ((2048, 768), 1e-3, "grad", 12)]
    for (shape, std, role, seed) in cases:          # two calls in a row
        x = syn.bf16_normal(shape, std, seed, device="cuda", outlier_frac=0.01)
        row, col, s, si = _noalloc(fp, x, role)
        ref = fp.fp8_quantize(x, "tensorwise", role)
        torch.cuda.synchronize()
        assert torch.equal(row, ref["row"])
        assert torch.equal(col, ref["col"])
        assert torch.equal(s.view(torch.int32), ref["row_scale"].reshape(-1).view(torch.int32))
        assert torch.equal(si.view(torch.int32), ref["row_scale_inv"].reshape(-1).view(torch.int32))
    # the second call must not depend on the first: a small tensor after a large one
    x = syn.bf16_normal((64, 64), 1.0, 13, device="cuda")
    row, col, s, si = _noalloc(fp, x, "act")
    ref = fp.fp8_quantize(x, "tensorwise", "act")
    torch.cuda.synchronize()
    assert torch.equal(row, ref["row"]) and torch.equal(col, ref["col"])
    assert torch.equal(s.view(torch.int32), ref["row_scale"].reshape(-1).view(torch.int32))


@pytest.mark.gpu
def test_noalloc_matches_oracle(fp):
    """Bytes of both layouts and both scales equal the oracle's tensorwise
    quantizer (E4M3 activations, 1% x100 outliers, a ragged 144-column
    tensor)."""
    from fp8_mixed_precision_gb300 import synthetic as syn
    x = syn.bf16_normal((1024, 144), 1.0, 14, device="cuda", outlier_frac=0.01)
    row, col, s, si = _noalloc(fp, x, "act")
    torch.cuda.synchronize()
    r = o.quantize_tensorwise(syn.bits(x), "e4m3")
    assert_bytes_equal(row, r["row"], "rowwise bytes")
    assert_bytes_equal(col, r["col"], "transposed bytes")
    assert_f32_equal(s, r["row_scale"], "scale")
    assert_f32_equal(si, r["row_scale_inv"], "scale_inv")


@pytest.mark.gpu
def test_noalloc_transposed_only_e5m2(fp):
    """rowwise_out NULL: only the transposed E5M2 layout is written, equal to
    fp8_quantize's bit for bit."""
    from fp8_mixed_precision_gb300 import synthetic as syn
    x = syn.bf16_normal((512, 256), 1e-3, 15, device="cuda")
    row, col, s, si = _noalloc(fp, x, "grad", rowwise=False, colwise=True)
    ref = fp.fp8_quantize(x, "tensorwise", "grad", rowwise=False, colwise=True)
    torch.cuda.synchronize()
    assert row is None
    assert torch.equal(col, ref["col"])
    assert torch.equal(s.view(torch.int32), ref["col_scale"].reshape(-1).view(torch.int32))
    assert torch.equal(si.view(torch.int32), ref["col_scale_inv"].reshape(-1).view(torch.int32))


def test_noalloc_argument_errors_without_gpu():
    """Argument errors return before anything is launched (the pointers
    below are never dereferenced): NULL scale, a misaligned input, rows not
    a multiple of 16, no output layout at all."""
    from fp8_mixed_precision_gb300 import build
    build.build()
    import fp8_mixed_precision_gb300 as fp
    f = _bind(fp)
    P = ctypes.c_void_p
    buf, odd = P(4096), P(4096 + 8)
    assert f(buf, 128, 128, 0, buf, buf, None, buf, None) == 1          # FP8_ERR_INVALID_ARG
    assert f(buf, 128, 128, 0, buf, buf, buf, None, None) == 1
    assert f(odd, 128, 128, 0, buf, buf, buf, buf, None) == 3           # FP8_ERR_ALIGN
    assert f(buf, 128, 128, 0, odd, None, buf, buf, None) == 3
    assert f(buf, 100, 128, 0, buf, buf, buf, buf, None) == 2           # FP8_ERR_SHAPE
    assert f(buf, 128, 128, 0, None, None, buf, buf, None) == 1
    assert f(buf, 128, 128, 9, buf, buf, buf, buf, None) == 1           # unknown role
