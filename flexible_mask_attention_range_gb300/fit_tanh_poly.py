"""Fit the softcap polynomials used by the kernels (kTanhPoly and kTanhPoly5 in
csrc/ffa_internal.h).

The kernels form the capped logit softcap * tanh(y), y = scale * q.k / softcap, on tiles
whose scores all satisfy |y| <= Y = 0.375 with an odd polynomial y * P(y^2) on the FMA pipe
instead of the exponential and reciprocal a direct evaluation needs: P(t) = c0 + c1 t +
c2 t^2 + c3 t^3 (kTanhPoly, degree 7 in y), or, in the bounded-softcap forward kernel,
P(t) = c0 + c1 t + c2 t^2 (kTanhPoly5, degree 5: one instruction less per pair of scores).
This script finds the coefficients that minimise the largest relative error
|y P(y^2) - tanh(y)| / |tanh(y)| over (0, Y]:

  * start from a least-squares fit of tanh(y)/y on Chebyshev nodes of (0, Y];
  * reweight the nodes by their current error and refit (Lawson's algorithm for the
    minimax fit), until the error equioscillates;
  * report the maximum relative error of the fitted polynomial evaluated by Horner's rule in
    float32 (the kernels' arithmetic) on a dense grid.

Usage: python -m flexible_mask_attention_range_gb300.fit_tanh_poly
"""
from __future__ import annotations

import numpy as np

Y = 0.375
DEGREE = 4  # coefficients of P (in t = y^2) for kTanhPoly; kTanhPoly5 has 3


def fit(nodes: int = 400, iters: int = 2000, degree: int = DEGREE) -> np.ndarray:
    k = np.arange(nodes)
    y = 0.5 * Y * (1.0 - np.cos(np.pi * (k + 0.5) / nodes))  # Chebyshev nodes on (0, Y)
    target = np.tanh(y) / y
    A = np.stack([(y * y) ** i for i in range(degree)], axis=1)
    w = np.full(nodes, 1.0 / nodes)
    c = np.zeros(degree)
    for _ in range(iters):
        sw = np.sqrt(w)
        # relative error of y P(y^2) against tanh(y) equals that of P against tanh(y)/y
        c, *_ = np.linalg.lstsq(A * (sw / target)[:, None], sw, rcond=None)
        err = np.abs(A @ c - target) / target
        w = w * err
        s = w.sum()
        if not (s > 0):
            break
        w /= s
    return c


def max_rel_err_f32(c: np.ndarray, n: int = 200001) -> float:
    y = np.linspace(1e-6, Y, n, dtype=np.float64)
    yf = y.astype(np.float32)
    t = yf * yf
    cf = c.astype(np.float32)
    p = cf[-1]
    for i in range(len(cf) - 2, -1, -1):
        p = p * t + cf[i]
    approx = (yf * p).astype(np.float64)
    return float(np.max(np.abs(approx - np.tanh(y)) / np.tanh(y)))


def main() -> None:
    for name, degree in (("kTanhPoly", DEGREE), ("kTanhPoly5", 3)):
        c = fit(degree=degree)
        print(name + " = {" + ", ".join(f"{x:.9e}" for x in c) + "}")
        print(f"  max relative error (float32 Horner) on (0, {Y}]: {max_rel_err_f32(c):.3e}")


if __name__ == "__main__":
    main()
