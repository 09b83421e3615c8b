"""Minimax polynomial for tanh used by the softcap path of the bf16 forward kernel.

The softcap maps a scaled score to ``cap * tanh(y)`` with ``y = scale * s / cap``.
On tiles where every ``|y|`` is small the kernel evaluates tanh as the odd
polynomial ``tanh(y) ~= y * T(y^2)`` with

    T(z) ~= sum_k t_k z^k,   k = 0 .. degree,   z in [0, y_max^2],

on the FMA pipes instead of through the exponential identity (two special-
function operations per score).  Two fits of the same accuracy are used: a
short one for ``|y| <= 0.5`` and a longer one for ``|y| <= 1``; a tile takes the
shortest fit its scores allow.  The coefficients ``t_k`` minimise the largest
relative error ``|T_fit(z) / T(z) - 1|`` with ``T(z) = tanh(sqrt z) / sqrt z``,
which is also the relative error of the approximated tanh.  They are found by
the Remez exchange algorithm (E. Ya. Remez, 1934): solve for the polynomial
whose error equioscillates with height E on DEGREE + 2 reference points, move
the references to the extrema of the new error curve, repeat.

This module is the generator of the constants ``kTanhPolyShort`` and
``kTanhPolyLong`` in ``csrc/attn_fwd_bf16.cu``; ``python -m softmax_attention_attn_gb300.tanh_fit``
prints them, and a CPU test checks that the source holds these values and that
the fp32 Horner evaluation meets ``MAX_REL_ERR``.  Nothing in the library's
run-time path imports it.
"""
from __future__ import annotations

import numpy as np

# (degree in z = y^2, y_max): an odd degree-7 polynomial in y on |y| <= 0.5 and an odd
# degree-11 polynomial on |y| <= 1
FITS = {"short": (3, 0.5), "long": (5, 1.0)}
MAX_REL_ERR = 8e-7    # bound on the relative error of y * T(y^2) evaluated in fp32 (Horner)


def tanh_over_y(z):
    """T(z) = tanh(sqrt z) / sqrt z (T(0) = 1), in float64."""
    z = np.asarray(z, dtype=np.float64)
    y = np.sqrt(z)
    out = np.ones_like(z)
    nz = y > 0
    out[nz] = np.tanh(y[nz]) / y[nz]
    return out


def remez(degree: int, y_max: float, iters: int = 60, grid_points: int = 400001):
    """Coefficients t_0..t_degree (float64) and the minimax relative error on [0, y_max^2]."""
    zmax = y_max * y_max
    n = degree
    j = np.arange(n + 2)
    refs = zmax * (1 - np.cos(np.pi * j / (n + 1))) / 2          # Chebyshev extrema as first references
    grid = np.linspace(0.0, zmax, grid_points)
    tg = tanh_over_y(grid)
    coef, height = None, None
    for _ in range(iters):
        A = np.empty((n + 2, n + 2))
        A[:, :n + 1] = refs[:, None] ** np.arange(n + 1)[None, :]
        A[:, n + 1] = (-1.0) ** j * tanh_over_y(refs)           # P(z_i) - T(z_i) = (-1)^i E T(z_i)
        sol = np.linalg.solve(A, tanh_over_y(refs))
        coef, height = sol[:n + 1], abs(sol[n + 1])
        err = (np.polyval(coef[::-1], grid) - tg) / tg
        # one extremum per run of equal sign
        cuts = np.flatnonzero(np.diff(np.sign(err)) != 0) + 1
        ext = np.array([seg[np.argmax(np.abs(err[seg]))] for seg in np.split(np.arange(grid.size), cuts)])
        while ext.size > n + 2:                                   # drop the smaller end extremum
            ext = ext[1:] if abs(err[ext[0]]) < abs(err[ext[-1]]) else ext[:-1]
        if ext.size < n + 2:
            break
        new = grid[ext]
        if np.allclose(new, refs, rtol=0, atol=zmax * 1e-9):
            break
        refs = new
    err = (np.polyval(coef[::-1], grid) - tg) / tg
    return coef, float(np.abs(err).max())


def fp32_horner_rel_err(coef, y_max: float, points: int = 200001) -> float:
    """Largest relative error of y * T(y^2) against tanh(y) when evaluated in fp32 by Horner's rule."""
    y = np.linspace(-y_max, y_max, points).astype(np.float32)
    z = (y * y).astype(np.float32)
    c = np.asarray(coef, dtype=np.float32)
    p = np.full_like(z, c[-1])
    for ck in c[-2::-1]:
        p = (p * z + ck).astype(np.float32)
    approx = (y.astype(np.float64) * p.astype(np.float64))
    exact = np.tanh(y.astype(np.float64))
    nz = y != 0
    return float(np.max(np.abs(approx[nz] - exact[nz]) / np.abs(exact[nz])))


if __name__ == "__main__":
    for name, (deg, ym) in FITS.items():
        c, e = remez(deg, ym)
        print(f"// {name}: degree {deg} in y^2 on |y| <= {ym}: minimax relative error {e:.3e}, "
              f"fp32 Horner {fp32_horner_rel_err(c, ym):.3e}")
        print(f"constexpr double kTanhPoly{name.capitalize()}[] = {{" + ", ".join(f"{x:.17g}" for x in c) + "};")
