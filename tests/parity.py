"""Comparison helpers shared by the GPU parity tests (no FP8 arithmetic here:
the expected values always come from the oracle)."""
import json
import os

import numpy as np
import torch

import oracle as o

FROB_TOL = 2e-3      # relative Frobenius error bound for GEMM outputs
ULP_TOL = 2          # per-element bound in bf16 ulps of the oracle's value


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def assert_bytes_equal(got: torch.Tensor, exp: np.ndarray, what: str):
    g = to_np(got)
    assert g.shape == exp.shape, (what, g.shape, exp.shape)
    if not np.array_equal(g, exp):
        bad = np.argwhere(g != exp)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} mismatches, first at {i}: got {g[i]:#x} "
                             f"expected {exp[i]:#x}")


def assert_f32_equal(got: torch.Tensor, exp: np.ndarray, what: str):
    g = to_np(got).astype(np.float32).reshape(exp.shape)
    gb, eb = g.view(np.uint32), np.ascontiguousarray(exp, dtype=np.float32).view(np.uint32)
    if not np.array_equal(gb, eb):
        bad = np.argwhere(gb != eb)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} mismatches, first at {i}: got {g[i]!r} "
                             f"expected {exp[i]!r}")


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (the subnormal spacing 2^-133 below
    2^-126, zero included)."""
    a = np.abs(v.astype(np.float64))
    _, ex = np.frexp(a)
    e = np.where(a == 0, -126, np.maximum(ex.astype(np.int64) - 1, -126))
    return np.ldexp(1.0, (e - 7).astype(np.int32))


def check_gemm(got: torch.Tensor, ref_f64: np.ndarray, abs_f64: np.ndarray, K: int, what: str):
    """GEMM output check: relative Frobenius <= 2e-3, and <= 2 bf16 ulps of the
    oracle's bf16 value per element, except elements whose error is still
    inside the fp32 summation bound gamma_K * sum|a_k b_k| (+1 ulp for the
    final roundings); those are counted and must stay rare."""
    g = o.bf16_to_f32(to_np(got)).astype(np.float64)
    ref_b = o.bf16_to_f32(o.round_to_bf16(ref_f64)).astype(np.float64)
    denom = np.linalg.norm(ref_f64)
    rel = np.linalg.norm(g - ref_f64) / denom if denom > 0 else np.linalg.norm(g)
    assert rel <= FROB_TOL, f"{what}: relative Frobenius error {rel:.3g}"
    ulp = bf16_ulp(ref_b)
    err = np.abs(g - ref_b)
    over = err > ULP_TOL * ulp
    if over.any():
        u = 2.0 ** -24
        gamma = K * u / (1 - K * u)
        allowed = gamma * abs_f64 + ulp
        hard = over & (np.abs(g - ref_f64) > allowed)
        assert not hard.any(), (f"{what}: {int(hard.sum())} elements beyond 2 ulp and the fp32 "
                                f"summation bound, first at {tuple(np.argwhere(hard)[0])}")
        assert over.mean() < 1e-3, f"{what}: {int(over.sum())} elements beyond 2 ulp"
    nz = ulp > 0
    max_ulp = float(np.max(err[nz] / ulp[nz])) if nz.any() else 0.0
    return dict(rel_frob=float(rel), over_2ulp=int(over.sum()), max_ulp=max_ulp,
                elements=int(g.size))


def log_margin(what: str, K: int, results) -> dict:
    """Aggregate check_gemm results of one GEMM (several tiles): worst
    relative Frobenius error, total elements beyond 2 ulp, worst ulp error.
    Appended as one JSON line to the file named by FP8_PARITY_LOG, if set."""
    results = list(results)
    agg = dict(gemm=what, K=int(K), tiles=len(results),
               elements=sum(r["elements"] for r in results),
               rel_frob_max=max(r["rel_frob"] for r in results),
               over_2ulp=sum(r["over_2ulp"] for r in results),
               max_ulp=max(r["max_ulp"] for r in results))
    path = os.environ.get("FP8_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(agg) + "\n")
    return agg
