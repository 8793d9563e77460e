"""Helpers for the full-size parity tests: which 128x128 output tiles to
check, a thread pool that runs independent oracle calls (each on its own
slice of an operand) side by side - the oracle's numpy work releases the
interpreter lock, so threads use all host cores - and the sampled-tile GEMM
checks built on them.  Expected values come from the oracle: its quantizer
and dequantizer on the operand slices a tile needs, then the fp64 product
(the oracle's GEMM definition) of those slices."""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle as o
from parity import check_gemm, log_margin

N_RANDOM = 64   # seeded random output tiles per GEMM, besides the first and the last

_POOL = None


def pmap(fn, items):
    """fn over items on the host cores, results in order."""
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1))
    return list(_POOL.map(fn, items))


def tiles(n_rows: int, n_cols: int, rng) -> list[tuple[int, int]]:
    """The first tile, the last tile and N_RANDOM distinct random tiles of an
    n_rows x n_cols tile grid (every tile when the grid has no more)."""
    total = n_rows * n_cols
    if total <= N_RANDOM + 2:
        return [(i, j) for i in range(n_rows) for j in range(n_cols)]
    first, last = 0, total - 1
    pick = rng.choice(np.arange(1, total - 1), size=N_RANDOM, replace=False)
    ids = [first] + sorted(int(p) for p in pick) + [last]
    return [(i // n_cols, i % n_cols) for i in ids]


def tile_grid(n_rows: int, n_cols: int, rng) -> tuple[list[int], list[int]]:
    """Tile rows and tile columns whose product set holds at least N_RANDOM
    tiles (every tile when the grid has no more), always with the first and
    the last tile.  For GEMMs whose operands are expensive per tile row or
    column (a reduction over all tokens), so that few distinct operand
    slices serve many tiles."""
    if n_rows * n_cols <= N_RANDOM + 2:
        return list(range(n_rows)), list(range(n_cols))
    a = min(n_rows, 8)
    b = min(n_cols, math.ceil(N_RANDOM / a))
    a = min(n_rows, max(a, math.ceil(N_RANDOM / b)))

    def choose(n, k):
        mid = rng.choice(np.arange(1, n - 1), size=max(0, k - 2), replace=False) if n > 2 else []
        return sorted({0, n - 1, *(int(m) for m in mid)})
    return choose(n_rows, a), choose(n_cols, b)


def _sl(t):
    return slice(t * 128, (t + 1) * 128)


def rows_1x128(bits, fmt):
    """Dequantized rows of a bf16 slice under 1x128 rowwise blocks."""
    q = o.quantize_1x128(np.ascontiguousarray(bits), fmt)
    return o.dequantize(q["row"], q["row_scale_inv"], fmt)


def cols_1x128(bits, fmt):
    """Dequantized transposed layout of a [tokens, 128] bf16 column slice
    under 1x128 blocks along the tokens: [128, tokens]."""
    q = o.quantize_1x128(np.ascontiguousarray(bits), fmt)
    return o.dequantize(q["col"], q["col_scale_inv"], fmt)


def check_fwd_like(got, a_bits, a_fmt, B, K, what, rng):
    """C = A B^T with A's rows quantized 1x128 from a_bits [M, K] and B the
    dequantized [N, K] operand (whole): sampled tiles."""
    M, Nc = got.shape
    tl = tiles(M // 128, Nc // 128, rng)
    rows = sorted({tm for tm, _ in tl})
    Ar = dict(zip(rows, pmap(lambda tm: rows_1x128(a_bits[_sl(tm)], a_fmt), rows)))
    Ba = np.abs(B)
    res = [check_gemm(got[_sl(tm), _sl(tn)], Ar[tm] @ B[_sl(tn)].T, np.abs(Ar[tm]) @ Ba[_sl(tn)].T,
                      K, f"{what} tile {tm},{tn}") for tm, tn in tl]
    return log_margin(what, K, res)


def check_wgrad(got, a_bits, a_fmt, b_bits, b_fmt, what, rng):
    """dW = A^T B over all tokens, both operands quantized 1x128 along the
    tokens (the transposed layouts): sampled tiles from a product set."""
    Mo, Ko = got.shape
    Ntok = a_bits.shape[0]
    rn, ck = tile_grid(Mo // 128, Ko // 128, rng)
    Ac = dict(zip(rn, pmap(lambda t: cols_1x128(a_bits[:, _sl(t)], a_fmt), rn)))
    Bc = dict(zip(ck, pmap(lambda t: cols_1x128(b_bits[:, _sl(t)], b_fmt), ck)))
    Ba = {t: np.abs(v) for t, v in Bc.items()}
    res = []
    for tn in rn:
        A = Ac.pop(tn)
        Aa = np.abs(A)
        for tk in ck:
            res.append(check_gemm(got[_sl(tn), _sl(tk)], A @ Bc[tk].T, Aa @ Ba[tk].T, Ntok,
                                  f"{what} tile {tn},{tk}"))
    return log_margin(what, Ntok, res)
