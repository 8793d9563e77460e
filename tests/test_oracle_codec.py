"""Pins of the oracle's FP8 codec and bf16 rounding against facts fixed by the
format definitions, exhaustive enumeration, exact rational arithmetic and
torch's own FP8/bf16 casts (library routines) where those apply."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as o


# ----------------------------------------------------------------- decode
@pytest.mark.parametrize("fmt,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_decode_all_256_bytes_match_torch(fmt, tdt):
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(tdt).to(torch.float64).numpy()
    got = o.decode(np.arange(256, dtype=np.uint8), fmt)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])
    # sign symmetry incl. -0
    assert np.array_equal(np.signbit(ref[m]), np.signbit(got[m]))


def test_decode_anchors():
    d4 = lambda b: o.decode_byte(b, "e4m3")
    d5 = lambda b: o.decode_byte(b, "e5m2")
    assert d4(0x7E) == 448.0 and d4(0xFE) == -448.0
    assert np.isnan(d4(0x7F)) and np.isnan(d4(0xFF))
    assert d4(0x01) == 2.0 ** -9 and d4(0x08) == 2.0 ** -6 and d4(0x07) == 7 * 2.0 ** -9
    assert d4(0x38) == 1.0 and d4(0x00) == 0.0
    assert d5(0x7B) == 57344.0 and d5(0x7C) == float("inf") and d5(0xFC) == float("-inf")
    assert all(np.isnan(d5(b)) for b in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF))
    assert d5(0x01) == 2.0 ** -16 and d5(0x04) == 2.0 ** -14 and d5(0x3C) == 1.0
    # exactly one NaN pair in E4M3, six NaN codes in E5M2
    assert sum(np.isnan(o.decode(np.arange(256, dtype=np.uint8), "e4m3"))) == 2
    assert sum(np.isnan(o.decode(np.arange(256, dtype=np.uint8), "e5m2"))) == 6


# ----------------------------------------------------------------- encode
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_encode_roundtrip_every_finite_byte(fmt):
    b = np.arange(256, dtype=np.uint8)
    v = o.decode(b, fmt)
    fin = np.isfinite(v)
    assert np.array_equal(o.encode(v[fin].astype(np.float32), fmt), b[fin])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_encode_midpoints_tie_to_even_and_neighbours(fmt):
    codes = [b for b in range(0x80) if np.isfinite(o.decode_byte(b, fmt))]
    vals = [o.decode_byte(b, fmt) for b in codes]
    for (b_lo, v_lo), (b_hi, v_hi) in zip(zip(codes, vals), zip(codes[1:], vals[1:])):
        mid = (v_lo + v_hi) / 2
        m32 = np.float32(mid)
        assert float(m32) == mid  # midpoints of FP8 values are exact in fp32
        even = b_lo if (b_lo & 1) == 0 else b_hi
        assert o.encode(np.float32([mid]), fmt)[0] == even
        assert o.encode(np.float32([-mid]), fmt)[0] == (even | 0x80)
        up = np.nextafter(m32, np.float32(np.inf))
        dn = np.nextafter(m32, np.float32(0))
        assert o.encode(np.float32([up]), fmt)[0] == b_hi
        assert o.encode(np.float32([dn]), fmt)[0] == b_lo


def test_encode_saturation_and_specials():
    e4 = o.encode(np.float32([448, 449, 463.99, 464, 480, 1e6, np.inf]), "e4m3")
    assert list(e4) == [0x7E] * 7
    e4n = o.encode(np.float32([-448, -449, -464, -480, -1e6, -np.inf]), "e4m3")
    assert list(e4n) == [0xFE] * 6
    e5 = o.encode(np.float32([57344, 61439, 61440, 1e9, np.inf]), "e5m2")
    assert list(e5) == [0x7B] * 5
    assert list(o.encode(np.float32([-np.inf, -1e9]), "e5m2")) == [0xFB] * 2
    assert o.encode(np.float32([np.nan]), "e4m3")[0] == 0x7F
    assert o.encode(np.float32([-np.nan]), "e5m2")[0] == 0x7F
    # sign of zero survives; negative values that round to zero give 0x80
    assert list(o.encode(np.float32([0.0, -0.0, -1e-30, 1e-30]), "e4m3")) == [0, 0x80, 0x80, 0]
    # smallest subnormal: half of it ties to zero (even), just above goes up
    assert o.encode(np.float32([2.0 ** -10]), "e4m3")[0] == 0x00
    assert o.encode(np.float32([np.nextafter(np.float32(2.0 ** -10), np.float32(1))]), "e4m3")[0] == 0x01
    assert o.encode(np.float32([1.5 * 2.0 ** -9]), "e4m3")[0] == 0x02   # tie between 1 and 2 -> even 2


@pytest.mark.parametrize("fmt,tdt,lim", [("e4m3", torch.float8_e4m3fn, 448.0),
                                         ("e5m2", torch.float8_e5m2, 57344.0)])
def test_encode_in_range_matches_torch_cast(fmt, tdt, lim):
    # torch's cast does not saturate (E4M3 470 -> NaN, E5M2 1e6 -> inf), so only
    # in-range values are compared; in range both are round-to-nearest-even.
    rng = np.random.default_rng(7)
    parts = [rng.standard_normal(20000) * s for s in (1e-4, 1e-2, 1.0, 30.0, lim / 8)]
    v = np.concatenate(parts).astype(np.float32)
    v = v[np.abs(v) <= lim]
    ref = torch.from_numpy(v).to(tdt).view(torch.uint8).numpy()
    assert np.array_equal(o.encode(v, fmt), ref)
    # torch really does not saturate: the reason out-of-range is excluded
    assert torch.tensor([470.0]).to(torch.float8_e4m3fn).float().isnan().item()


# ----------------------------------------------------------------- bf16 rounding
def _bf16_nearest_exact(x: float) -> int:
    """Brute-force RNE to bf16 with exact rationals (finite, in range)."""
    f = np.float32(x)
    # bracket x between two adjacent bf16 values using fp32 bit patterns
    b = int(np.float32(abs(x)).view(np.uint32)) >> 16
    cands = [b - 1, b, b + 1, b + 2]
    best = None
    X = Fraction(abs(x))
    for c in cands:
        if c < 0 or c > 0x7F7F:
            continue
        v = Fraction(float(np.uint32(c << 16).view(np.float32)))
        d = abs(v - X)
        key = (d, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    sign = 0x8000 if np.signbit(x) else 0
    return best[1] | sign


def test_round_to_bf16_matches_exact_rational_rounding():
    rng = np.random.default_rng(11)
    xs = list(rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000))
    # exact midpoints between adjacent bf16 values and their fp64 neighbours
    for c in rng.integers(0x0001, 0x7F7E, 500):
        lo = float(np.uint32(int(c) << 16).view(np.float32))
        hi = float(np.uint32((int(c) + 1) << 16).view(np.float32))
        mid = (lo + hi) / 2
        xs += [mid, np.nextafter(mid, np.inf), np.nextafter(mid, 0.0), -mid]
    xs = np.array(xs, dtype=np.float64)
    got = o.round_to_bf16(xs)
    ref = np.array([_bf16_nearest_exact(x) for x in xs], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_round_to_bf16_is_single_rounding():
    # 1 + 2^-8 + 2^-30 is above the bf16 midpoint 1 + 2^-8 and must round up;
    # rounding via fp32 first would land on the midpoint and tie down to 1.0.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert o.round_to_bf16(np.array([x]))[0] == 0x3F81
    assert o.round_to_bf16(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80
    assert o.round_to_bf16(np.array([3.4e38]))[0] == 0x7F80
    assert o.round_to_bf16(np.array([-np.inf, np.nan]))[0] == 0xFF80


def test_bf16_to_f32_matches_torch():
    b = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = o.bf16_to_f32(b)
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m]) and np.array_equal(np.isnan(got), ~m)
