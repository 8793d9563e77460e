"""Pins of the oracle's quantizers: hand-worked blocks (tests/golden), the
amax-maps-to-fmax invariant, a lossless power-of-two special case, layout
identities and the special scale cases."""
import os

import numpy as np
import pytest

import oracle as o
from fp8_mixed_precision_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    d = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            d[k] = v
    return d


@pytest.mark.parametrize("name", ["worked_block_e4m3.txt", "worked_block_e5m2.txt"])
def test_worked_block(name):
    g = _read_golden(name)
    fmt = g["fmt"][0]
    x = np.zeros((128, 128), np.uint16)
    vals = [int(v, 16) for v in g["x_bf16_bits"]]
    x[0, :len(vals)] = vals
    q = o.quantize_tensorwise(x, fmt)
    assert int(q["row_scale"].view(np.uint32)[0]) == int(g["scale_bits"][0], 16)
    assert int(q["row_scale_inv"].view(np.uint32)[0]) == int(g["scale_inv_bits"][0], 16)
    assert [int(b) for b in q["row"][0, :len(vals)]] == [int(v, 16) for v in g["q"]]
    # the same block alone in a 1x128 row block and a 128x128 tile gives the same bytes
    b = o.quantize_1x128(x, fmt)
    assert np.array_equal(b["row"][0], q["row"][0])
    assert int(b["row_scale"].view(np.uint32)[0, 0]) == int(g["scale_bits"][0], 16)
    t = o.quantize_128x128(x, fmt)
    assert np.array_equal(t["row"], q["row"])


def _inputs(R, C, std, seed, outliers=0.0):
    return syn.bits(syn.bf16_normal((R, C), std, seed, outlier_frac=outliers))


@pytest.mark.parametrize("recipe,role", [("tensorwise", "act"), ("tensorwise", "grad"),
                                         ("block", "act"), ("block", "grad"), ("block", "weight")])
def test_amax_element_encodes_to_fmax(recipe, role):
    x = _inputs(256, 384, 1e-3 if role == "grad" else 1.0, 3, outliers=0.01)
    fmt = o.ROLE_FORMAT[role]
    top = {"e4m3": 0x7E, "e5m2": 0x7B}[fmt]
    q = o.quantize(x, recipe, role)
    xf = o.bf16_to_f32(x)
    # every block: the element(s) of largest magnitude encode to +-fmax
    if recipe == "tensorwise" or role == "weight":
        bs = (x.shape[0], x.shape[1]) if recipe == "tensorwise" else (128, 128)
        for i in range(0, x.shape[0], bs[0]):
            for j in range(0, x.shape[1], bs[1]):
                blk = np.abs(xf[i:i + bs[0], j:j + bs[1]])
                qb = q["row"][i:i + bs[0], j:j + bs[1]]
                assert np.all((qb[blk == blk.max()] & 0x7F) == top)
    else:
        for i in range(x.shape[0]):
            for j in range(0, x.shape[1], 128):
                blk = np.abs(xf[i, j:j + 128])
                assert np.all((q["row"][i, j:j + 128][blk == blk.max()] & 0x7F) == top)
        for j in range(x.shape[1]):
            for i in range(0, x.shape[0], 128):
                blk = np.abs(xf[i:i + 128, j])
                assert np.all((q["col"][j, i:i + 128][blk == blk.max()] & 0x7F) == top)
    # nothing exceeds fmax
    assert not np.any(np.abs(o.decode(q["row"], fmt)) > o.FMAX[fmt])


@pytest.mark.parametrize("k", [0, 3, 9])
def test_lossless_power_of_two_block(k):
    # x drawn from E4M3 values times 2^-k with amax = 448 * 2^-k: scale = 2^k
    # exactly, so decode(q) * scale_inv reproduces x bit for bit.
    rng = np.random.default_rng(k)
    codes = rng.integers(0, 0x7F, (128, 256)).astype(np.uint8)
    codes[codes == 0x7F] = 0
    codes[5, 7] = 0x7E
    sign = (rng.random((128, 256)) < 0.5).astype(np.uint8) << 7
    vals = o.decode(codes | sign, "e4m3") * 2.0 ** -k
    xb = (vals.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(o.bf16_to_f32(xb).astype(np.float64), vals)  # exact in bf16
    for qz in (o.quantize_tensorwise(xb, "e4m3"), o.quantize_128x128(xb, "e4m3")):
        s = qz["row_scale"].reshape(-1)
        assert np.all(s[np.isfinite(s)][:1] == np.float32(2.0 ** k))
        back = o.dequantize(qz["row"], qz["row_scale_inv"], "e4m3")
        assert np.array_equal(back, vals)


def test_layout_identities():
    x = _inputs(384, 256, 1.0, 9, outliers=0.01)
    for fmt in ("e4m3", "e5m2"):
        t = o.quantize_tensorwise(x, fmt)
        assert np.array_equal(t["col"], t["row"].T)
        w = o.quantize_128x128(x, fmt)
        assert np.array_equal(w["col"], w["row"].T)
        assert np.array_equal(w["col_scale"], w["row_scale"].T)
        # 1x128: colwise of x is the rowwise quantization of x^T (independent code path)
        b = o.quantize_1x128(x, fmt)
        bt = o.quantize_1x128(np.ascontiguousarray(x.T), fmt)
        assert np.array_equal(b["col"], bt["row"])
        assert np.array_equal(b["col_scale"], bt["row_scale"])
        assert np.array_equal(b["col_scale_inv"], bt["row_scale_inv"])
        assert b["row_scale"].shape == (384, 2) and b["col_scale"].shape == (256, 3)
        # in general colwise is NOT the byte transpose of rowwise for 1x128 blocks
        assert not np.array_equal(b["col"], b["row"].T)


def test_special_scale_cases():
    z = np.zeros((128, 128), np.uint16)
    z[0, 1] = 0x8000                                        # -0
    q = o.quantize_tensorwise(z, "e4m3")
    assert q["row_scale"][0] == 1.0 and q["row_scale_inv"][0] == 1.0
    assert q["row"][0, 1] == 0x80 and q["row"][0, 0] == 0
    # tiny amax: fmax/amax overflows -> FLT_MAX
    t = np.zeros((128, 128), np.uint16)
    t[0, 0] = 0x0001                                        # smallest bf16 subnormal
    q = o.quantize_tensorwise(t, "e4m3")
    assert q["row_scale"][0] == np.finfo(np.float32).max
    # NaN ignored by amax; inf amax -> scale 0 -> inf*0 = NaN byte, finite -> +-0
    n = np.zeros((128, 128), np.uint16)
    n[0, 0] = 0x7FC0                                        # NaN
    n[0, 1] = 0x4000                                        # 2.0
    q = o.quantize_tensorwise(n, "e4m3")
    assert q["amax"] == 2.0 and q["row"][0, 0] == 0x7F and q["row"][0, 1] == 0x7E
    n[0, 2] = 0x7F80                                        # +inf
    n[0, 3] = 0xC000                                        # -2.0
    q = o.quantize_tensorwise(n, "e5m2")
    assert q["row_scale"][0] == 0.0 and np.isinf(q["row_scale_inv"][0])
    assert list(q["row"][0, :4]) == [0x7F, 0x00, 0x7F, 0x80]


@pytest.mark.parametrize("R,C", [(144, 272), (16, 128), (128, 16), (400, 48)])
def test_ragged_tail_blocks(R, C):
    # a ragged tail block is quantized exactly like a standalone tensor made of
    # the elements present (tensorwise quantization of that slice)
    x = _inputs(R, C, 1.0, 21, outliers=0.02)
    for fmt in ("e4m3", "e5m2"):
        b = o.quantize_1x128(x, fmt)
        assert b["row_scale"].shape == (R, -(-C // 128))
        assert b["col_scale"].shape == (C, -(-R // 128))
        c0 = (C - 1) // 128 * 128
        i = R - 1
        t = o.quantize_tensorwise(np.ascontiguousarray(x[i:i + 1, c0:]), fmt)
        assert np.array_equal(b["row"][i, c0:], t["row"][0])
        assert b["row_scale"][i, -1] == t["row_scale"][0]
        r0 = (R - 1) // 128 * 128
        j = C - 1
        t = o.quantize_tensorwise(np.ascontiguousarray(x[r0:, j:j + 1]), fmt)
        assert np.array_equal(b["col"][j, r0:], t["row"][:, 0])
        assert b["col_scale_inv"][j, -1] == t["row_scale_inv"][0]
        w = o.quantize_128x128(x, fmt)
        t = o.quantize_tensorwise(np.ascontiguousarray(x[r0:, c0:]), fmt)
        assert np.array_equal(w["row"][r0:, c0:], t["row"])
        assert w["row_scale"][-1, -1] == t["row_scale"][0]
        assert np.array_equal(w["col"], w["row"].T)


def test_delayed_scaling_pins():
    x = _inputs(256, 128, 1.0, 31)
    xf = o.bf16_to_f32(x)
    cur = o.quantize_tensorwise(x, "e4m3")
    # empty history: scale 1 (amax 0 rule); the tensor's amax lands at step % H
    r = o.quantize_delayed(x, "e4m3", np.zeros(4, np.float32), 6)
    assert r["row_scale"][0] == 1.0 and r["row_scale_inv"][0] == 1.0
    assert np.array_equal(r["row"], o.encode(xf, "e4m3"))
    assert list(r["history"]) == [0.0, 0.0, float(cur["amax"]), 0.0]
    # a history whose maximum equals this tensor's amax reduces to current scaling
    h = np.array([0.5, cur["amax"], 0.25], np.float32)
    r = o.quantize_delayed(x, "e4m3", h, 1)
    assert np.array_equal(r["row"], cur["row"]) and r["row_scale"][0] == cur["row_scale"][0]
    # the scale follows the history's maximum, not the current tensor
    h = np.array([float(cur["amax"]) * 4], np.float32)
    r = o.quantize_delayed(x, "e4m3", h, 0)
    assert r["row_scale"][0] == np.float32(448.0) / np.float32(float(cur["amax"]) * 4)
    assert r["history"][0] == cur["amax"]
    assert np.array_equal(r["col"], r["row"].T)


def test_delayed_weight_cache_is_not_bitwise_neutral():
    # With an amax history, re-quantizing the same weight inside a cycle uses
    # a scale the cached copy never saw: the two runs differ (the TE
    # documentation's warning), unlike the non-delayed recipes.
    w = _inputs(256, 256, 0.02, 5)
    outs = {}
    for use in (False, True):
        c = o.WeightCache("delayed", history_len=4)
        c.register("w", w)
        got = []
        for cyc in range(2):
            c.begin_cycle()
            for mb in range(3):
                got.append(c.get("w", use)["row"].copy())
        outs[use] = got
    assert not all(np.array_equal(a, b) for a, b in zip(outs[False], outs[True]))
    assert np.array_equal(outs[False][0], outs[True][0])   # first quantization agrees
