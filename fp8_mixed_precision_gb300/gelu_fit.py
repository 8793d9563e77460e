"""Coefficients of the erfc approximation used by the GELU kernels.

erfc(z) = exp(-z^2) * erfcx(z) for z >= 0, and erfcx(z) is approximated as
t * Q(t) with t = 1 / (1 + z/2) (t runs over (0, 1] as z runs over [0, inf))
and Q a polynomial of degree 7.  Q is fitted here by least squares on the
relative error over z in [0, 1e6], reweighted a few times toward the largest
errors; the reference values come from scipy.special.erfcx.  The kernels
evaluate t * Q(t) / 2 (the 1/2 of Phi folded in), so the float literals that
csrc/common.cuh holds are the fitted float32 coefficients halved, an exact
scaling; they are printed lowest degree first, with the fit's maximum
relative error (about 3e-6, far below the 2^-9 that one bf16 ulp allows).

    python -m fp8_mixed_precision_gb300.gelu_fit
"""
from __future__ import annotations

import numpy as np

DEGREE = 7


def fit(degree: int = DEGREE):
    from scipy.special import erfcx
    z = np.concatenate([np.linspace(0, 4, 200001), np.linspace(4, 40, 200001),
                        np.geomspace(40, 1e6, 20001)])
    t = 1.0 / (1.0 + 0.5 * z)
    y = erfcx(z) / t
    extra = np.ones_like(t)
    best = (np.inf, None)
    for _ in range(20):
        w = extra / y
        V = np.vander(t, degree + 1, increasing=True) * w[:, None]
        c, *_ = np.linalg.lstsq(V, y * w, rcond=None)
        r = np.abs(np.polynomial.polynomial.polyval(t, c) / y - 1)
        if r.max() < best[0]:
            best = (float(r.max()), c)
        extra = np.minimum(extra * (1 + r / r.max()), 1e3)
    return best[1].astype(np.float32), best[0]


if __name__ == "__main__":
    c, err = fit()
    print(f"max relative error {err:.3g}")
    for i, v in enumerate(c / np.float32(2)):
        print(f"  {float(v)!r}f,  // t^{i}")
