"""Derives the coefficients of the cubic used for 2^f, f in [-1/2, 1/2], in the
softmax's FMA-pipe exponential (st_common.cuh: ex2_fma).

Method: weighted least squares on Chebyshev nodes of the interval, weights 1/2^f
so that the relative error is what gets minimised, followed by a few
Lawson-style reweighting passes (each node's weight multiplied by its current
absolute relative error) to move the fit towards the minimax (equi-ripple)
solution. Prints the coefficients (low to high degree) and the maximum
relative error over a dense grid.
"""
import numpy as np


def fit(deg=3, nodes=400, passes=60):
    k = np.arange(nodes)
    f = 0.5 * np.cos((2 * k + 1) * np.pi / (2 * nodes))      # Chebyshev nodes on [-1/2, 1/2]
    y = np.exp2(f)
    V = np.vander(f, deg + 1, increasing=True)
    w = 1.0 / y
    for _ in range(passes):
        c, *_ = np.linalg.lstsq(V * w[:, None], y * w, rcond=None)
        rel = np.abs(V @ c / y - 1.0)
        w = w * (rel / rel.max() + 1e-3)
    return c


def max_rel(c):
    g = np.linspace(-0.5, 0.5, 200001)
    return float(np.max(np.abs(np.polyval(c[::-1], g) / np.exp2(g) - 1.0)))


if __name__ == "__main__":
    c = fit()
    c32 = c.astype(np.float32).astype(np.float64)
    print("coefficients:", ", ".join(f"{x:.9e}" for x in c32))
    print("max relative error (fp32 coefficients): %.3e" % max_rel(c32))
