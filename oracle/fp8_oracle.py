"""CPU oracle for the FP8 linear layer: quantizers, FP8 GEMMs, linear fwd/bwd,
weight-cache model, GELU and gradient accumulation.

TEST INFRASTRUCTURE ONLY.  This module is the slow, plainly written statement
of what the CUDA library computes.  Only the test suite, the package smoke
check and the benchmark's CPU-baseline leg may import it; the library itself
never does, and this module imports nothing from the library.

Sources, cited by page title and section:
  [NFP8]  "Native FP8 MLP reconstruction: frozen-model memory savings,
          full-budget quality test underway" (rstation.ai general_pretraining
          post 23).  Implementation paragraph: current tensorwise amax, E4M3
          inputs/weights, E5M2 incoming gradients, BF16 GEMM outputs,
          use_fast_accum=False, fused cast writing ordinary + transposed
          layouts, detached scales, forward-rounded X/W reused in backward,
          received gradient rounded separately.  Exactness paragraph after the
          isolated-linear table: fused output/dX/dW equal plain FP8 exactly.
  [TE2852] "FP8 weight caching shows no speedup (sometimes slowdown) and
          causes training curve differences under Float8BlockScaling"
          (TransformerEngine issue #2852).  Opening post: is_first_microbatch
          True/False under gradient accumulation, blockwise Float8BlockScaling
          without amax history.  Maintainer reply: with non-delayed recipes
          cached and uncached runs give exactly the same results.

Readings where the pages are silent (the library's recipe definition):
  * block recipe = 1x128 blocks for activations and gradients, 128x128 blocks
    for weights; every scale is fp32 scale = fmax / amax (IEEE division,
    round-to-nearest-even), scale_inv = 1 / scale (fp32, RNE);
  * the cast is one fp32 multiply x * scale followed by a saturating
    round-to-nearest-even conversion to the 8-bit format;
  * amax == 0 gives scale = scale_inv = 1; fmax / amax overflowing gives
    scale = FLT_MAX; NaN inputs are ignored by amax (fmaxf semantics);
  * a NaN value encodes to the canonical NaN byte 0x7F in both formats;
  * the transposed (colwise) layout of a 1x128-block tensor has its own
    1x128 blocks along its own contiguous dimension (128 tokens);
  * GEMM: operands decoded exactly, multiplied by their scale_inv in fp64,
    summed in fp64, rounded once to bf16 (round-to-nearest-even, directly
    from fp64);
  * GELU is the exact erf form, evaluated in fp64 and rounded once to bf16.

Numbers are carried as numpy arrays: bf16 tensors as uint16 bit patterns,
FP8 tensors as uint8 bytes, scales as float32.
"""
from __future__ import annotations

import numpy as np
from scipy.special import erfc as _erfc

# ---------------------------------------------------------------------------
# FP8 formats  ([NFP8] implementation paragraph names E4M3 and E5M2; the bit
# layouts are the OCP 8-bit floating point definitions)
# ---------------------------------------------------------------------------
E4M3 = "e4m3"
E5M2 = "e5m2"

_FMT = {
    # exponent bits, mantissa bits, exponent bias, largest finite value
    E4M3: dict(ebits=4, mbits=3, bias=7, fmax=448.0),
    E5M2: dict(ebits=5, mbits=2, bias=15, fmax=57344.0),
}

FMAX = {E4M3: 448.0, E5M2: 57344.0}
NAN_BYTE = 0x7F

ROLE_FORMAT = {"act": E4M3, "weight": E4M3, "grad": E5M2}   # [NFP8] impl. paragraph


def decode_byte(b: int, fmt: str) -> float:
    """Exact value of one FP8 byte, from the format definition."""
    p = _FMT[fmt]
    ebits, mbits, bias = p["ebits"], p["mbits"], p["bias"]
    sign = -1.0 if (b >> 7) & 1 else 1.0
    e = (b >> mbits) & ((1 << ebits) - 1)
    m = b & ((1 << mbits) - 1)
    emax_field = (1 << ebits) - 1
    if fmt == E4M3:
        if e == emax_field and m == (1 << mbits) - 1:
            return float("nan")          # S.1111.111 is the only NaN, no infinities
    else:
        if e == emax_field:
            return sign * float("inf") if m == 0 else float("nan")
    if e == 0:                             # subnormal: m * 2^(1 - bias - mbits)
        return sign * m * 2.0 ** (1 - bias - mbits)
    return sign * (1.0 + m / (1 << mbits)) * 2.0 ** (e - bias)


_DECODE_TABLE = {f: np.array([decode_byte(b, f) for b in range(256)], dtype=np.float64)
                 for f in _FMT}


def decode(q: np.ndarray, fmt: str) -> np.ndarray:
    """Exact fp64 values of an array of FP8 bytes."""
    return _DECODE_TABLE[fmt][np.asarray(q, dtype=np.uint8)]


def _positive_codes(fmt: str):
    """Finite non-negative codes in increasing order with their values."""
    codes = [b for b in range(0x80) if np.isfinite(_DECODE_TABLE[fmt][b])]
    vals = _DECODE_TABLE[fmt][codes]
    assert np.all(np.diff(vals) > 0)
    return np.array(codes, dtype=np.uint8), vals


_POS = {f: _positive_codes(f) for f in _FMT}


def encode(v, fmt: str) -> np.ndarray:
    """Saturating round-to-nearest-even of fp32 values to FP8 bytes.

    |v| is rounded to the nearest representable magnitude; on a tie the
    candidate with an even mantissa wins (this holds across the subnormal
    range too, whose spacing equals that of the lowest binade).  Magnitudes
    at or above fmax, infinities included, become fmax.  The sign is kept,
    so negative values that round to zero give 0x80.  NaN gives 0x7F.
    """
    p = _FMT[fmt]
    mbits, bias, fmax = p["mbits"], p["bias"], p["fmax"]
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v.astype(np.float64))
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    # binade exponent floor(log2 a), clamped to the smallest normal exponent
    _, ex = np.frexp(a)
    e = np.maximum(ex.astype(np.int64) - 1, 1 - bias)
    quantum = np.ldexp(1.0, (e - mbits).astype(np.int32))
    # a / quantum is exact (power-of-two division of a 24-bit value in fp64);
    # np.rint rounds half to even, i.e. the even multiple of the quantum
    # wins a tie, which is the even mantissa.
    r = np.rint(a / quantum) * quantum
    r = np.minimum(r, fmax)                       # saturation to the largest finite
    codes, vals = _POS[fmt]
    idx = np.searchsorted(vals, r)
    idx = np.minimum(idx, len(vals) - 1)
    assert np.all(vals[idx] == r), "rounded value is not representable"
    out = codes[idx].astype(np.uint8)
    out = out | (np.signbit(v).astype(np.uint8) << 7)
    out = np.where(nan, np.uint8(NAN_BYTE), out)
    return out.astype(np.uint8)


# ---------------------------------------------------------------------------
# bf16 helpers
# ---------------------------------------------------------------------------
def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact float32 values."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values once to bf16 (round-to-nearest-even), return bit patterns.

    bf16 has 8 exponent bits and 7 stored mantissa bits, so the rounding
    quantum in the binade [2^e, 2^(e+1)) is 2^(e-7), with e clamped at the
    smallest normal exponent -126.  Magnitudes that round to 2^128 or above
    become infinity.  NaN gives the quiet NaN 0x7FC0.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    nan = np.isnan(a)
    inf_in = np.isinf(a)
    a = np.where(nan | inf_in, 0.0, a)
    _, ex = np.frexp(a)
    e = np.maximum(ex.astype(np.int64) - 1, -126)
    quantum = np.ldexp(1.0, (e - 7).astype(np.int32))
    r = np.rint(a / quantum) * quantum
    over = (r >= 2.0 ** 128) | inf_in
    r = np.where(over, 0.0, r)
    bits = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bits = np.where(over, np.uint16(0x7F80), bits)
    bits = bits | (np.signbit(x).astype(np.uint16) << 15)
    bits = np.where(nan, np.uint16(0x7FC0), bits)
    return bits.astype(np.uint16)


# ---------------------------------------------------------------------------
# Scales  (library recipe definition: fp32 scale = fmax / amax)
# ---------------------------------------------------------------------------
FLT_MAX = np.float32(np.finfo(np.float32).max)


def amax_of(xf: np.ndarray, axis=None) -> np.ndarray:
    """max |x| ignoring NaN, starting from 0 (fmaxf semantics)."""
    a = np.abs(np.asarray(xf, dtype=np.float32))
    a = np.where(np.isnan(a), np.float32(0), a)
    return np.max(a, axis=axis, initial=np.float32(0)).astype(np.float32)


def scale_from_amax(amax: np.ndarray, fmt: str):
    """(scale, scale_inv) in fp32 for an array of amax values."""
    amax = np.asarray(amax, dtype=np.float32)
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        s = np.float32(FMAX[fmt]) / amax
        s = np.where(amax == 0, np.float32(1.0), s)
        s = np.where(np.isinf(s), FLT_MAX, s).astype(np.float32)
        s_inv = (np.float32(1.0) / s).astype(np.float32)
    return s, s_inv


def cast(xf: np.ndarray, scale: np.ndarray, fmt: str) -> np.ndarray:
    """q = sat_RNE_fp8(fp32(x) * scale): one fp32 multiply, then encode."""
    with np.errstate(invalid="ignore", over="ignore"):
        y = (np.asarray(xf, dtype=np.float32) * np.asarray(scale, dtype=np.float32)).astype(np.float32)
    return encode(y, fmt)


# ---------------------------------------------------------------------------
# Quantizers.  Each returns a dict with
#   row: uint8 [R, C]           rowwise bytes
#   col: uint8 [C, R]           transposed-layout bytes
#   row_scale, row_scale_inv    float32 scale arrays for `row`
#   col_scale, col_scale_inv    float32 scale arrays for `col`
# ---------------------------------------------------------------------------
def quantize_tensorwise(x_bits: np.ndarray, fmt: str) -> dict:
    """Current tensorwise scaling ([NFP8] implementation paragraph): one amax
    over the whole tensor, one scale, one cast written in both layouts."""
    xf = bf16_to_f32(x_bits)
    amax = amax_of(xf)
    s, s_inv = scale_from_amax(amax, fmt)
    q = cast(xf, s, fmt)
    s1 = np.array([s], dtype=np.float32).reshape(1)
    si1 = np.array([s_inv], dtype=np.float32).reshape(1)
    return dict(row=q, col=np.ascontiguousarray(q.T), row_scale=s1, row_scale_inv=si1,
                col_scale=s1.copy(), col_scale_inv=si1.copy(), amax=amax)


def _pad128(xf: np.ndarray) -> np.ndarray:
    """Zero-pad both dimensions up to multiples of 128.  Zeros never raise an
    amax, so a ragged tail block's amax covers exactly the elements present;
    padded outputs are cropped away."""
    R, C = xf.shape
    Rp, Cp = -(-R // 128) * 128, -(-C // 128) * 128
    if (Rp, Cp) == (R, C):
        return xf
    out = np.zeros((Rp, Cp), dtype=xf.dtype)
    out[:R, :C] = xf
    return out


def quantize_1x128(x_bits: np.ndarray, fmt: str) -> dict:
    """1x128 block scaling for activations and gradients.

    Rowwise: each row's 128-column slices are blocks; scales [R, ceil(C/128)].
    Colwise: each column's 128-row slices are blocks; the bytes are stored
    transposed, [C, R], with scales [C, ceil(R/128)].
    """
    R, C = x_bits.shape
    xf = _pad128(bf16_to_f32(x_bits))
    Rp, Cp = xf.shape
    # rowwise blocks: x[i, 128b : 128b+128]
    xr = xf.reshape(Rp, Cp // 128, 128)
    amax_r = amax_of(xr, axis=2)                       # [Rp, Cp/128]
    s_r, si_r = scale_from_amax(amax_r, fmt)
    q_row = cast(xr, s_r[:, :, None], fmt).reshape(Rp, Cp)[:R, :C]
    # colwise blocks: x[128b : 128b+128, j]
    xc = xf.reshape(Rp // 128, 128, Cp)
    amax_c = amax_of(xc, axis=1)                       # [Rp/128, Cp]
    s_c, si_c = scale_from_amax(amax_c, fmt)
    q_c = cast(xc, s_c[:, None, :], fmt).reshape(Rp, Cp)[:R, :C]
    return dict(row=np.ascontiguousarray(q_row), col=np.ascontiguousarray(q_c.T),
                row_scale=np.ascontiguousarray(s_r[:R]), row_scale_inv=np.ascontiguousarray(si_r[:R]),
                col_scale=np.ascontiguousarray(s_c.T[:C]), col_scale_inv=np.ascontiguousarray(si_c.T[:C]))


def quantize_128x128(x_bits: np.ndarray, fmt: str) -> dict:
    """128x128 block scaling for weights: one scale per 128x128 tile, scales
    [ceil(R/128), ceil(C/128)]; the transposed layout is the byte transpose
    with the transposed scale grid."""
    R, C = x_bits.shape
    xf = _pad128(bf16_to_f32(x_bits))
    Rp, Cp = xf.shape
    xt = xf.reshape(Rp // 128, 128, Cp // 128, 128)
    amax_t = amax_of(xt, axis=(1, 3))                  # [Rp/128, Cp/128]
    s, si = scale_from_amax(amax_t, fmt)
    q = cast(xt, s[:, None, :, None], fmt).reshape(Rp, Cp)[:R, :C]
    return dict(row=np.ascontiguousarray(q), col=np.ascontiguousarray(q.T), row_scale=s,
                row_scale_inv=si, col_scale=np.ascontiguousarray(s.T),
                col_scale_inv=np.ascontiguousarray(si.T))


def quantize_delayed(x_bits: np.ndarray, fmt: str, history: np.ndarray, step: int) -> dict:
    """DelayedScaling (TE2852 opening post: DelayedScaling keeps amax_history
    state; Float8BlockScaling does not).  Reading, margin 0: the scale comes
    from the largest amax recorded in the history *before* this tensor is
    seen, scale = fp32(fmax / max(history)) with the same special cases as
    current scaling; the tensor is cast with it; then this tensor's own amax
    is written into the ring at position step mod len(history)."""
    hist = np.array(history, dtype=np.float32, copy=True)
    s, s_inv = scale_from_amax(amax_of(hist), fmt)
    xf = bf16_to_f32(x_bits)
    q = cast(xf, s, fmt)
    hist[int(step) % len(hist)] = amax_of(xf)
    s1 = np.array([s], dtype=np.float32).reshape(1)
    si1 = np.array([s_inv], dtype=np.float32).reshape(1)
    return dict(row=q, col=np.ascontiguousarray(q.T), row_scale=s1, row_scale_inv=si1,
                col_scale=s1.copy(), col_scale_inv=si1.copy(), history=hist)


def quantize(x_bits: np.ndarray, recipe: str, role: str) -> dict:
    """Dispatch on recipe ('tensorwise' | 'block') and role ('act' | 'weight' | 'grad')."""
    fmt = ROLE_FORMAT[role]
    if recipe == "tensorwise":
        return quantize_tensorwise(x_bits, fmt)
    if recipe == "block":
        return quantize_128x128(x_bits, fmt) if role == "weight" else quantize_1x128(x_bits, fmt)
    raise ValueError(recipe)


# ---------------------------------------------------------------------------
# GEMM: C[M, N] = sum_k A[m, k] * B[n, k], both operands K-major
# ---------------------------------------------------------------------------
def expand_scale(s_inv: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Per-element fp64 scale_inv for a [rows, cols] operand whose scale array
    is [1] (tensorwise), [rows, ceil(cols/128)] (1x128 blocks along cols) or
    [ceil(rows/128), ceil(cols/128)] (128x128 tiles)."""
    s = np.asarray(s_inv, dtype=np.float64)
    nb_c = -(-cols // 128)
    nb_r = -(-rows // 128)
    if s.size == 1:
        return np.full((rows, cols), float(s.reshape(-1)[0]))
    if s.shape == (rows, nb_c):
        return np.repeat(s, 128, axis=1)[:, :cols]
    if s.shape == (nb_r, nb_c):
        return np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)[:rows, :cols]
    raise ValueError(f"scale shape {s.shape} for operand {rows}x{cols}")


def dequantize(q: np.ndarray, s_inv: np.ndarray, fmt: str) -> np.ndarray:
    """decode(q) * scale_inv of its block, in fp64 (exact: <=4 + 24 significant bits)."""
    R, C = q.shape
    return decode(q, fmt) * expand_scale(s_inv, R, C)


def gemm_f64(a_q, a_sinv, a_fmt, b_q, b_sinv, b_fmt) -> np.ndarray:
    """Unrounded fp64 product of the dequantized operands, [M, N]."""
    return dequantize(a_q, a_sinv, a_fmt) @ dequantize(b_q, b_sinv, b_fmt).T


def gemm(a_q, a_sinv, a_fmt, b_q, b_sinv, b_fmt) -> np.ndarray:
    """FP8 GEMM with fp64 accumulation rounded once to bf16 (bit patterns)."""
    return round_to_bf16(gemm_f64(a_q, a_sinv, a_fmt, b_q, b_sinv, b_fmt))


# ---------------------------------------------------------------------------
# Linear layer  ([NFP8] implementation paragraph)
#   X [N, K] (tokens x in), W [O, K] (out x in), Y = X W^T [N, O]
# ---------------------------------------------------------------------------
def linear_fwd(x_bits, wq: dict, recipe: str) -> dict:
    """Forward: quantize X (E4M3, both layouts), fprop GEMM with the rowwise
    FP8 weight.  Returns Y (bf16 bits) and the saved context."""
    xq = quantize(x_bits, recipe, "act")
    y = gemm(xq["row"], xq["row_scale_inv"], E4M3, wq["row"], wq["row_scale_inv"], E4M3)
    return dict(y=y, xq=xq)


def linear_bwd(dy_bits, ctx: dict, wq: dict, recipe: str) -> dict:
    """Backward: dY gets its own amax and an E5M2 cast in both layouts; dgrad
    reuses the forward-rounded W (transposed layout), wgrad reuses the
    forward-rounded X (transposed layout).  Scales are constants."""
    gq = quantize(dy_bits, recipe, "grad")
    dx = gemm(gq["row"], gq["row_scale_inv"], E5M2, wq["col"], wq["col_scale_inv"], E4M3)
    xq = ctx["xq"]
    dw = gemm(gq["col"], gq["col_scale_inv"], E5M2, xq["col"], xq["col_scale_inv"], E4M3)
    return dict(dx=dx, dw=dw, gq=gq)


def linear_fwd_bwd(x_bits, w_bits, dy_bits, recipe: str) -> dict:
    wq = quantize(w_bits, recipe, "weight")
    f = linear_fwd(x_bits, wq, recipe)
    b = linear_bwd(dy_bits, f, wq, recipe)
    return dict(wq=wq, xq=f["xq"], y=f["y"], gq=b["gq"], dx=b["dx"], dw=b["dw"])


# ---------------------------------------------------------------------------
# Weight cache model  ([TE2852] opening post and maintainer reply)
# ---------------------------------------------------------------------------
class WeightCache:
    """is_first_microbatch semantics: with use_cache the weight is quantized on
    the first get() of a cycle and the FP8 copy is returned afterwards;
    without it every get() re-quantizes."""

    def __init__(self, recipe: str, history_len: int = 16):
        self.recipe = recipe
        self.entries = {}
        self.quantize_calls = 0
        self.history_len = history_len

    def register(self, name, w_bits):
        self.entries[name] = dict(w=w_bits, q=None,
                                  history=np.zeros(self.history_len, np.float32), steps=0)

    def update(self, name, w_bits):
        """The bf16 weight changed (e.g. an optimizer step between cycles)."""
        self.entries[name]["w"] = w_bits

    def begin_cycle(self):
        for e in self.entries.values():
            e["q"] = None

    def get(self, name, use_cache: bool) -> dict:
        e = self.entries[name]
        if not use_cache or e["q"] is None:
            if self.recipe == "delayed":
                r = quantize_delayed(e["w"], E4M3, e["history"], e["steps"])
                e["history"] = r["history"]
                e["steps"] += 1
                e["q"] = r
            else:
                e["q"] = quantize(e["w"], self.recipe, "weight")
            self.quantize_calls += 1
        return e["q"]


# ---------------------------------------------------------------------------
# MLP glue: GELU (exact erf form) and gradient accumulation
# ---------------------------------------------------------------------------
def _normal_cdf(h: np.ndarray) -> np.ndarray:
    """Phi(h) = erfc(-h / sqrt(2)) / 2.  The erfc form keeps full relative
    precision for negative h, where 1 + erf(h / sqrt(2)) would cancel."""
    return 0.5 * _erfc(-np.asarray(h, dtype=np.float64) / np.sqrt(2.0))


def gelu_f64(h: np.ndarray) -> np.ndarray:
    """GELU(h) = h * Phi(h), Phi the standard normal CDF."""
    h = np.asarray(h, dtype=np.float64)
    return h * _normal_cdf(h)


def gelu_grad_f64(h: np.ndarray) -> np.ndarray:
    """d GELU / dh = Phi(h) + h * phi(h)."""
    h = np.asarray(h, dtype=np.float64)
    pdf = np.exp(-0.5 * h * h) / np.sqrt(2.0 * np.pi)
    return _normal_cdf(h) + h * pdf


def gelu_fwd(h_bits: np.ndarray) -> np.ndarray:
    """bf16 in -> GELU in fp64 -> bf16 out (bit patterns)."""
    return round_to_bf16(gelu_f64(bf16_to_f32(h_bits)))


def gelu_bwd(da_bits: np.ndarray, h_bits: np.ndarray) -> np.ndarray:
    """dH = bf16(dA * GELU'(H)), evaluated in fp64."""
    return round_to_bf16(bf16_to_f32(da_bits).astype(np.float64) * gelu_grad_f64(bf16_to_f32(h_bits)))


def grad_accumulate(acc_f32: np.ndarray, dw_bits: np.ndarray) -> np.ndarray:
    """acc += float(dW) in fp32 (one IEEE add per element)."""
    return (np.asarray(acc_f32, dtype=np.float32) + bf16_to_f32(dw_bits)).astype(np.float32)


def mlp_fwd_bwd(x_bits, w1_bits, w2_bits, dy_bits, recipe: str = "block") -> dict:
    """fc1 -> GELU -> fc2 and its backward, each stage through the oracle."""
    w1q = quantize(w1_bits, recipe, "weight")
    w2q = quantize(w2_bits, recipe, "weight")
    f1 = linear_fwd(x_bits, w1q, recipe)
    a = gelu_fwd(f1["y"])
    f2 = linear_fwd(a, w2q, recipe)
    b2 = linear_bwd(dy_bits, f2, w2q, recipe)
    dh = gelu_bwd(b2["dx"], f1["y"])
    b1 = linear_bwd(dh, f1, w1q, recipe)
    return dict(h=f1["y"], a=a, y=f2["y"], da=b2["dx"], dw2=b2["dw"], dh=dh,
                dx=b1["dx"], dw1=b1["dw"])
