"""Fit the polynomial the prefill kernel uses to evaluate part of its exp2 on
the FMA pipe instead of the special-function unit.

Method. For y = 2^x write x = n + f with n = round(x) (an integer) and
f in [-1/2, 1/2]; then 2^x = 2^n * 2^f. 2^n is applied by adding n to the
IEEE-754 exponent field (an integer add on the result's bits), and 2^f is a
polynomial p(f). The rounding uses the classic magic-number trick: adding
1.5 * 2^23 to x in round-to-nearest mode leaves round(x) in the low mantissa
bits. p is the minimax approximation of 2^f for RELATIVE error on
[-1/2, 1/2], found here with the Remez exchange algorithm (Remez 1934, as
described in e.g. Cheney, "Introduction to Approximation Theory", ch. 3),
with the constant term pinned to 1 so that p(0) = 2^0 exactly.

Run `python -m exact_tiled_attention_03_gb300.exp2_fit [degree]` to print
the coefficients (highest degree first) and the achieved error bound; the
kernel's constants were produced by this script.
"""
from __future__ import annotations

import sys

import numpy as np


def _fit_on_nodes(nodes, degree):
    """Solve for c_1..c_deg and the levelled error E with p(f) = 1 + sum c_k f^k:
    (p(f_i) - 2^f_i) / 2^f_i = (-1)^i E at the degree + 1 nodes."""
    n = len(nodes)
    A = np.zeros((n, degree + 1))
    b = np.zeros(n)
    for i, f in enumerate(nodes):
        t = 2.0 ** f
        for k in range(1, degree + 1):
            A[i, k - 1] = f ** k / t
        A[i, degree] = -((-1) ** i)
        b[i] = 1.0 - 1.0 / t
    sol = np.linalg.solve(A, -b + 0.0)
    # rows say: sum c_k f^k / t - (-1)^i E = 1 - 1/t - ... rearranged below
    return sol[:degree], sol[degree]


def rel_error(coeffs, f):
    p = np.ones_like(f)
    for k, c in enumerate(coeffs, start=1):
        p = p + c * f ** k
    return (p - 2.0 ** f) / 2.0 ** f


def remez(degree: int, iters: int = 60):
    lo, hi = -0.5, 0.5
    m = degree + 1                      # unknowns: degree coefficients + E
    k = np.arange(m)
    nodes = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * (m - 1 - k) / (m - 1))
    grid = np.linspace(lo, hi, 200001)
    coeffs = None
    for _ in range(iters):
        # equioscillation system: (p(f_i) - t_i)/t_i = (-1)^i E
        A = np.zeros((m, m))
        rhs = np.zeros(m)
        for i, f in enumerate(nodes):
            t = 2.0 ** f
            for j in range(1, degree + 1):
                A[i, j - 1] = f ** j / t
            A[i, degree] = -((-1.0) ** i)
            rhs[i] = (t - 1.0) / t
        sol = np.linalg.solve(A, rhs)
        coeffs = sol[:degree]
        err = rel_error(coeffs, grid)
        # new nodes: extrema of the error between sign changes
        sign = np.sign(err)
        sign[sign == 0] = 1
        bounds = np.concatenate(([0], np.nonzero(np.diff(sign))[0] + 1, [len(grid)]))
        ext = [seg_start + np.argmax(np.abs(err[seg_start:seg_end]))
               for seg_start, seg_end in zip(bounds[:-1], bounds[1:])]
        if len(ext) < m:
            break
        # keep m alternating extrema with the largest magnitudes
        while len(ext) > m:
            a0, a1 = abs(err[ext[0]]), abs(err[ext[-1]])
            ext = ext[1:] if a0 < a1 else ext[:-1]
        new_nodes = grid[ext]
        if np.allclose(new_nodes, nodes, atol=1e-12):
            break
        nodes = new_nodes
    return coeffs, float(np.max(np.abs(rel_error(coeffs, grid))))


def as_float32(coeffs):
    return [float(np.float32(c)) for c in coeffs]


def main(argv):
    degree = int(argv[1]) if len(argv) > 1 else 4
    coeffs, bound = remez(degree)
    c32 = as_float32(coeffs)
    grid = np.linspace(-0.5, 0.5, 200001)
    bound32 = float(np.max(np.abs(rel_error(np.array(c32, dtype=np.float64), grid))))
    print(f"degree {degree}: minimax relative error {bound:.3e} (with fp32 coefficients {bound32:.3e})")
    for k in range(degree, 0, -1):
        print(f"  c{k} = {c32[k - 1]!r}f")
    print("  c0 = 1.0f")


if __name__ == "__main__":
    main(sys.argv)
