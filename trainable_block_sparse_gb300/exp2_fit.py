"""Coefficients of the polynomial 2^f on [-1/2, 1/2] used by the kernels'
FMA-pipe exponential (ex2_poly in csrc/sm103_ptx.cuh).

Method: 2^x = 2^n * 2^f with n = round(x) and f = x - n in [-1/2, 1/2]
(range reduction to a half-unit interval); 2^f is approximated by a degree-3
polynomial chosen to minimise the maximum *relative* error on that interval.
The fit is a Remez exchange started from Chebyshev nodes, in float64.

Run `python -m trainable_block_sparse_gb300.exp2_fit` to print the
coefficients and their error bound; tests re-derive them and compare with
the values compiled into the kernels.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3
LO, HI = -0.5, 0.5


def _rel_err(c: np.ndarray, x: np.ndarray) -> np.ndarray:
    return np.polynomial.polynomial.polyval(x, c) / np.exp2(x) - 1.0


def fit(degree: int = DEGREE, iters: int = 30) -> tuple[np.ndarray, float]:
    """Minimax (relative) polynomial for 2^f on [LO, HI]; returns
    (coefficients c0..c_degree, max relative error)."""
    m = degree + 2
    k = np.arange(m)
    x = 0.5 * (LO + HI) + 0.5 * (HI - LO) * np.cos(np.pi * k[::-1] / (m - 1))
    grid = np.linspace(LO, HI, 200001)
    c = np.zeros(degree + 1)
    for _ in range(iters):
        # solve p(x_i) - 2^x_i = (-1)^i E 2^x_i for c and E
        A = np.zeros((m, m))
        A[:, : degree + 1] = x[:, None] ** np.arange(degree + 1)[None, :]
        A[:, -1] = -((-1.0) ** k) * np.exp2(x)
        sol = np.linalg.solve(A, np.exp2(x))
        c = sol[: degree + 1]
        e = _rel_err(c, grid)
        # new reference: the extremum of each sign-alternating segment
        sign = np.sign(e)
        cut = np.flatnonzero(np.diff(sign) != 0) + 1
        segs = np.split(np.arange(grid.size), cut)
        ext = [s[np.argmax(np.abs(e[s]))] for s in segs]
        if len(ext) < m:
            break
        # keep m alternating extrema with the largest errors
        while len(ext) > m:
            drop = 0 if abs(e[ext[0]]) < abs(e[ext[-1]]) else len(ext) - 1
            ext.pop(drop)
        x = grid[ext]
    return c, float(np.max(np.abs(_rel_err(c, grid))))


def float32_coefficients(degree: int = DEGREE) -> list[float]:
    c, _ = fit(degree)
    return [float(np.float32(v)) for v in c]


if __name__ == "__main__":
    c, err = fit()
    for i, v in enumerate(c):
        print(f"c{i} = {np.float32(v)!r}  ({float(np.float32(v)).hex()})")
    print(f"max relative error on [{LO}, {HI}]: {err:.3e} ({np.log2(err):.2f} bits)")
