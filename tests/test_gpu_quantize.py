"""GPU parity of the fused quantizers against the oracle: FP8 bytes and
scales bit-exact, every recipe and role, tiles with ragged tails, special
values, every finite bf16 bit pattern, and sampled tiles at full size."""
import numpy as np
import pytest
import torch

import oracle as o
from fp8_mixed_precision_gb300 import synthetic as syn
from parity import assert_bytes_equal, assert_f32_equal

pytestmark = pytest.mark.gpu

CASES = [("tensorwise", "act"), ("tensorwise", "weight"), ("tensorwise", "grad"),
         ("block", "act"), ("block", "weight"), ("block", "grad")]


@pytest.fixture(scope="module")
def fp():
    from fp8_mixed_precision_gb300 import build
    build.build()
    import fp8_mixed_precision_gb300 as fp
    return fp


def _check(fp, xb, recipe, role, rowwise=True, colwise=True):
    x = syn.from_bits(xb, "cuda")
    got = fp.fp8_quantize(x, recipe, role, rowwise=rowwise, colwise=colwise)
    torch.cuda.synchronize()
    exp = o.quantize(xb, recipe, role)
    if rowwise:
        assert_bytes_equal(got["row"], exp["row"], f"{recipe}/{role} row bytes")
    if rowwise or recipe == "tensorwise":
        assert_f32_equal(got["row_scale"], exp["row_scale"], "row_scale")
        assert_f32_equal(got["row_scale_inv"], exp["row_scale_inv"], "row_scale_inv")
    if colwise:
        assert_bytes_equal(got["col"], exp["col"], f"{recipe}/{role} col bytes")
        assert_f32_equal(got["col_scale"], exp["col_scale"], "col_scale")
        assert_f32_equal(got["col_scale_inv"], exp["col_scale_inv"], "col_scale_inv")


@pytest.mark.parametrize("recipe,role", CASES)
@pytest.mark.parametrize("shape", [(256, 384), (144, 272), (16, 16), (400, 48), (1024, 640)])
def test_quantize_parity(fp, recipe, role, shape):
    std = 1e-3 if role == "grad" else (0.02 if role == "weight" else 1.0)
    xb = syn.bits(syn.bf16_normal(shape, std, 7 + shape[0], outlier_frac=0.01))
    _check(fp, xb, recipe, role)


@pytest.mark.parametrize("recipe,role", CASES)
def test_single_layout_requests(fp, recipe, role):
    xb = syn.bits(syn.bf16_normal((256, 256), 1.0, 5))
    _check(fp, xb, recipe, role, rowwise=True, colwise=False)
    _check(fp, xb, recipe, role, rowwise=False, colwise=True)


@pytest.mark.parametrize("recipe,role", CASES)
def test_special_values(fp, recipe, role):
    xb = syn.bits(syn.bf16_normal((256, 256), 1.0, 9))
    xb[0, :8] = [0x7FC0, 0xFFC1, 0x8000, 0x0000, 0x0001, 0x8001, 0x7F7F, 0xFF7F]  # NaN, -0, tiny, max
    xb[130:258, 5] = 0                    # an all-zero column block
    xb[3, 128:256] = 0x8000               # a row block of -0
    xb[200, 7] = 0x7F80                   # +inf in another block
    _check(fp, xb, recipe, role)


@pytest.mark.parametrize("fmt_role", ["act", "grad"])
def test_every_finite_bf16_pattern(fp, fmt_role):
    # all 65536 bf16 bit patterns minus non-finite ones, 128 per row: every
    # 1x128 block sees a different amax, exercising rounding across binades
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    b[(b & 0x7F80) == 0x7F80] = 0x3F80
    xb = np.ascontiguousarray(b.reshape(512, 128))
    _check(fp, xb, "block", fmt_role)
    _check(fp, np.ascontiguousarray(xb.T), "block", fmt_role)


@pytest.mark.parametrize("shape,role,std", [((131072, 512), "act", 1.0), ((131072, 2048), "act", 1.0),
                                            ((131072, 8192), "grad", 1e-3),
                                            ((16384, 14336), "act", 1.0)])
@pytest.mark.parametrize("recipe", ["tensorwise", "block"])
def test_full_size_sampled_tiles(fp, shape, role, std, recipe):
    """Workload sizes: the whole tensor is quantized on the GPU; the oracle
    recomputes sampled 128x128 tiles (tensorwise: with the oracle's global
    amax over the whole tensor)."""
    x = syn.bf16_normal(shape, std, 42, device="cuda", outlier_frac=0.01 if shape[0] == 16384 else 0)
    got = fp.fp8_quantize(x, recipe, role)
    torch.cuda.synchronize()
    xb = syn.bits(x)
    fmt = o.ROLE_FORMAT[role]
    R, C = shape
    rng = np.random.default_rng(0)
    tiles = [(0, 0), (R // 128 - 1, C // 128 - 1)] + \
        [(int(a), int(b)) for a, b in zip(rng.integers(0, R // 128, 6), rng.integers(0, C // 128, 6))]
    if recipe == "tensorwise":
        s, si = o.scale_from_amax(o.amax_of(o.bf16_to_f32(xb)), fmt)
        assert_f32_equal(got["row_scale"], np.array([s], np.float32), "scale")
        assert_f32_equal(got["row_scale_inv"], np.array([si], np.float32), "scale_inv")
    row = got["row"]
    col = got["col"]
    for (tr, tc) in tiles:
        sl = xb[tr * 128:(tr + 1) * 128, tc * 128:(tc + 1) * 128]
        if recipe == "tensorwise":
            q = o.cast(o.bf16_to_f32(sl), s, fmt)
            qc = q.T
        else:
            e = o.quantize(np.ascontiguousarray(sl), recipe, role)
            q, qc = e["row"], e["col"]
            gs = got["row_scale"][tr * 128:(tr + 1) * 128, tc:tc + 1]
            assert_f32_equal(gs, e["row_scale"], "row_scale tile")
            gcs = got["col_scale_inv"][tc * 128:(tc + 1) * 128, tr:tr + 1]
            assert_f32_equal(gcs, e["col_scale_inv"], "col_scale_inv tile")
        assert_bytes_equal(row[tr * 128:(tr + 1) * 128, tc * 128:(tc + 1) * 128], q, f"row tile {tr},{tc}")
        assert_bytes_equal(col[tc * 128:(tc + 1) * 128, tr * 128:(tr + 1) * 128], np.ascontiguousarray(qc),
                           f"col tile {tr},{tc}")
