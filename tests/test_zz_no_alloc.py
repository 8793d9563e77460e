"""The allocation-free tensorwise quantizer, called through the C ABI, must
give the same FP8 bytes and scales as fp8_quantize (bit for bit, the
tolerance every quantizer test uses) on two calls in a row.  The second call
runs with the first call's leftovers in the library's fixed scratch array.

Collected last on purpose: the entry point exists for callers that cannot
allocate device memory (allocator hooks, plugins whose framework owns all
memory, paths that must avoid cudaMalloc/cudaFree), and this test must pass
both alone in a fresh process and after every other test."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp():
    from fp8_mixed_precision_gb300 import build
    build.build()
    import fp8_mixed_precision_gb300 as fp
    L = fp.lib()
    f = L.fp8_quantize_tensorwise_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return fp


def _noalloc(fp, x, role):
    R, C = x.shape
    row = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    col = torch.empty((C, R), dtype=torch.uint8, device="cuda")
    s = torch.empty(1, dtype=torch.float32, device="cuda")
    si = torch.empty(1, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = fp.lib().fp8_quantize_tensorwise_noalloc(
        ctypes.c_void_p(x.data_ptr()), R, C, fp.ROLE[role], ctypes.c_void_p(row.data_ptr()),
        ctypes.c_void_p(col.data_ptr()), ctypes.c_void_p(s.data_ptr()),
        ctypes.c_void_p(si.data_ptr()), stream)
    assert st == 0, st
    return row, col, s, si


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
