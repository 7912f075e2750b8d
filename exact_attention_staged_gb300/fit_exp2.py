"""Coefficients of the polynomial 2^f on [-1/2, 1/2] that the kernels use for part of their
exponentials (the FMA-pipe exp2 in csrc/sm100.cuh).

Method: minimax fit of the relative error, solved as a linear program (minimise t subject to
|p(f_i) - 2^f_i| <= t * 2^f_i on a dense grid of f_i), with coefficients rounded to fp32 and
the error re-measured in fp64 on a finer grid.  Usage: ``python -m
exact_attention_staged_gb300.fit_exp2 [degree]``; prints the coefficients (lowest order first)
and the maximal relative error.
"""
from __future__ import annotations

import sys

import numpy as np
from scipy.optimize import linprog


def fit(degree: int = 3, points: int = 4001):
    f = np.linspace(-0.5, 0.5, points)
    y = np.exp2(f)
    # variables: c_0 .. c_degree, t ; minimise t
    V = np.vander(f, degree + 1, increasing=True)
    ones = y[:, None]
    A = np.vstack([np.hstack([V, -ones]), np.hstack([-V, -ones])])
    b = np.concatenate([y, -y])
    cost = np.zeros(degree + 2)
    cost[-1] = 1.0
    res = linprog(cost, A_ub=A, b_ub=b, bounds=[(None, None)] * (degree + 2), method="highs")
    if not res.success:
        raise RuntimeError(res.message)
    c = res.x[:-1].astype(np.float32)
    return c, max_rel_error(c)


def max_rel_error(c, points: int = 200001) -> float:
    f = np.linspace(-0.5, 0.5, points)
    p = np.polyval(np.asarray(c, dtype=np.float64)[::-1], f)
    return float(np.max(np.abs(p / np.exp2(f) - 1.0)))


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    coef, err = fit(deg)
    for i, x in enumerate(coef):
        print(f"c{i} = {float(x)!r}f  ({float(x).hex()})")
    print(f"max relative error {err:.3e}")
