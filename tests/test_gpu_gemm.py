"""GPU parity of the tcgen05 FP8 GEMM against the oracle's fp64 GEMM:
relative Frobenius <= 2e-3 and <= 2 bf16 ulp per element (with the fp32
summation-bound exception counted), for every scaling layout, mixed E5M2 x
E4M3 operands, several tiles with ragged tails, split-K depths, and
closed-form exact cases."""
import numpy as np
import pytest
import torch

import oracle as o
from parity import check_gemm, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp():
    from fp8_mixed_precision_gb300 import build
    build.build()
    import fp8_mixed_precision_gb300 as fp
    return fp


def _rand_q(shape, fmt, rng, spread=True):
    """Random valid FP8 codes of a realistic magnitude mix."""
    v = rng.standard_normal(shape).astype(np.float32)
    if spread:
        v *= np.float32(2.0) ** rng.integers(-6, 7, shape).astype(np.float32)
    return o.encode(np.clip(v, -o.FMAX[fmt], o.FMAX[fmt]), fmt)


def _scales(kind, rows, K, rng, tile_rows=False):
    nkb = -(-K // 128)
    if kind == "tensor":
        return rng.uniform(1e-3, 1e-1, (1,)).astype(np.float32)
    if tile_rows:
        return rng.uniform(1e-3, 1e-1, (-(-rows // 128), nkb)).astype(np.float32)
    return rng.uniform(1e-3, 1e-1, (rows, nkb)).astype(np.float32)


def _run(fp, M, N, K, scaling, afmt="e5m2", bfmt="e4m3", seed=0):
    rng = np.random.default_rng(seed)
    aq, bq = _rand_q((M, K), afmt, rng), _rand_q((N, K), bfmt, rng)
    akind = "tensor" if scaling == "tensor" else "block"
    asi = _scales(akind, M, K, rng)
    bsi = _scales(akind, N, K, rng, tile_rows=(scaling == "1x128_128x128"))
    dev = "cuda"
    C = fp.fp8_gemm(torch.from_numpy(aq).to(dev), afmt, torch.from_numpy(asi).to(dev),
                    torch.from_numpy(bq).to(dev), bfmt, torch.from_numpy(bsi).to(dev), scaling)
    torch.cuda.synchronize()
    ref = o.gemm_f64(aq, asi, afmt, bq, bsi, bfmt)
    absref = np.abs(o.dequantize(aq, asi, afmt)) @ np.abs(o.dequantize(bq, bsi, bfmt)).T
    return check_gemm(C, ref, absref, K, f"gemm {M}x{N}x{K} {scaling}")


@pytest.mark.parametrize("scaling", ["tensor", "1x128_128x128", "1x128_1x128"])
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 512), (272, 144, 400),
                                   (16, 16, 16), (1024, 512, 1024), (128, 256, 8192),
                                   (512, 512, 2048)])
def test_gemm_parity(fp, M, N, K, scaling):
    _run(fp, M, N, K, scaling)


@pytest.mark.parametrize("M,N,K", [(8192, 512, 512), (8320, 400, 496), (16384, 2048, 256),
                                   (8192, 2176, 512), (4224, 8192, 384)])
def test_gemm_short_k_many_tiles(fp, M, N, K):
    # output-bound shapes: many M tiles over a short (ragged) K; 2176 = 8.5
    # 256-wide N tiles (a half-filled last tile), 8192 x 384 a ragged M
    _run(fp, M, N, K, "tensor", "e4m3", "e4m3", seed=M + N)


@pytest.mark.parametrize("M,N,K", [(4096, 2048, 4096), (8400, 768, 4096), (8320, 768, 4096),
                                   (4096, 768, 16384)])
def test_gemm_deep_k_tensor(fp, M, N, K):
    # deep-K tensor-scaled shapes (256-row tiles of two M halves); ragged last
    # tiles with a partial second half (8400) and a second half past M (8320);
    # split-K over such tiles (K = 16384)
    _run(fp, M, N, K, "tensor", "e4m3", "e5m2", seed=K + M)


@pytest.mark.parametrize("M,N,K", [(4224, 304, 1024), (384, 256, 640), (4224, 304, 32768),
                                   (3072, 2048, 8192), (4224, 2048, 8192)])
def test_gemm_tensor_ragged_tiles(fp, M, N, K):
    # an odd number of M tiles, and N = 304: the last 256-wide N tile holds
    # 48 valid columns, its second 128-column half none.  The K >= 8192
    # cases run 256-row tiles as CTA pairs (cta_group::2), split over K
    # (32768) or not (8192), with the last pair's second tile past M (4224)
    _run(fp, M, N, K, "tensor", "e5m2", "e4m3", seed=N + K)


@pytest.mark.parametrize("M,N,K", [(4224, 304, 8192), (384, 256, 640), (2048, 512, 32768),
                                   (1152, 1040, 2048)])
def test_gemm_block_block_ragged(fp, M, N, K):
    # 1x128 x 1x128 (wgrad scaling; 16 epilogue warps of 32 columns, 16x256b
    # TMEM reads): an odd M tile count, ragged N and K tails, split-K (32768)
    _run(fp, M, N, K, "1x128_1x128", "e5m2", "e4m3", seed=M + K)


@pytest.mark.parametrize("afmt,bfmt", [("e4m3", "e4m3"), ("e5m2", "e4m3"), ("e4m3", "e5m2"),
                                       ("e5m2", "e5m2")])
def test_gemm_formats(fp, afmt, bfmt):
    _run(fp, 256, 256, 384, "tensor", afmt, bfmt)
    _run(fp, 256, 256, 384, "1x128_1x128", afmt, bfmt, seed=1)


def test_gemm_deep_k_split(fp):
    # wgrad depth with few output tiles: exercises split-K and its ordered reduction
    r = _run(fp, 256, 256, 32768, "1x128_1x128", seed=3)
    assert r["rel_frob"] < 2e-3
    _run(fp, 256, 256, 32768, "tensor", seed=4)


def test_gemm_exact_closed_form(fp):
    # small integers with power-of-two scales: exact in fp32 and in bf16
    rng = np.random.default_rng(5)
    M, N, K = 256, 256, 512
    a = rng.integers(-3, 4, (M, K)).astype(np.float32)
    b = rng.integers(-2, 3, (N, K)).astype(np.float32)
    aq, bq = o.encode(a, "e4m3"), o.encode(b, "e4m3")
    C = fp.fp8_gemm(torch.from_numpy(aq).cuda(), "e4m3", torch.tensor([0.5]).cuda(),
                    torch.from_numpy(bq).cuda(), "e4m3", torch.tensor([0.25]).cuda(), "tensor")
    exp = o.round_to_bf16((a.astype(np.float64) @ b.T.astype(np.float64)) * 0.125)
    assert np.array_equal(to_np(C), exp)


def test_gemm_empty_and_degenerate(fp):
    e = torch.empty((0, 128), dtype=torch.uint8, device="cuda")
    b = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    s = torch.ones(1, device="cuda")
    C = fp.fp8_gemm(e, "e4m3", s, b, "e4m3", s, "tensor")
    assert C.shape == (0, 128)
    # all-zero operands -> exact zeros
    z = torch.zeros((128, 256), dtype=torch.uint8, device="cuda")
    C = fp.fp8_gemm(z, "e4m3", s, z, "e4m3", s, "tensor")
    assert torch.count_nonzero(C.float()).item() == 0
