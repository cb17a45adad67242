"""Fits the polynomial of the forward kernel's FMA-pipe exponential.

The forward kernel computes part of its exponentials 2^x without the special
function unit: x = n + f with n = floor(x) and f in [0, 1), 2^f from a
polynomial p(f), and 2^n applied by adding n to the float's exponent field.

p is fitted here with its constant term fixed at exactly 1 (so that p(0) = 1 and
an input clamped to -127 maps to the float with all bits zero, i.e. +0.0):

    p(f) = 1 + c1 f + c2 f^2 + ... + c_deg f^deg

with c1..c_deg minimising the largest RELATIVE error max |p(f) / 2^f - 1| on
[0, 1].  Method: the Remez exchange algorithm.  At deg + 1 reference points in
(0, 1] the weighted error is forced to alternate with a common magnitude E (a
linear system in c1..c_deg and E); the references then move to the extrema of
the error curve (located on a grid and refined by golden-section search), and
the two steps repeat until the references stop moving.  The coefficients are
rounded to float32, and the error of the rounded polynomial evaluated the way
the kernel does (float32 Horner steps, each a fused multiply-add) is measured
on a dense grid.

    python fit_exp2_poly.py [degree]      (default 3)

prints c1..c_deg as float32 hex literals and decimal values.
"""
from __future__ import annotations

import struct
import sys

import mpmath as mp
import numpy as np

mp.mp.dps = 50


def _rel_err(c, f):
    """p(f) / 2^f - 1 for p = 1 + sum_k c[k-1] f^k."""
    p = mp.mpf(0)
    for a in reversed(c):
        p = (p + a) * f
    return (1 + p) / mp.power(2, f) - 1


def _extremum(c, lo, hi, sign):
    """Golden-section search for the extremum of sign * error on [lo, hi]."""
    g1, g2 = mp.mpf("0.381966011250105151795"), mp.mpf("0.618033988749894848205")
    a, b = lo, hi
    for _ in range(160):
        m1 = a + (b - a) * g1
        m2 = a + (b - a) * g2
        if sign * _rel_err(c, m1) > sign * _rel_err(c, m2):
            b = m2
        else:
            a = m1
    return (a + b) / 2


def remez(deg: int, iters: int = 60, grid_n: int = 4000):
    """c1..c_deg (mp.mpf) of the minimax-relative-error fit of 2^f on [0, 1]
    with p(0) = 1, and the levelled error |E|."""
    n = deg + 1
    ref = [(1 - mp.cos(mp.pi * (i + 1) / n)) / 2 for i in range(n)]  # Chebyshev-like, in (0, 1]
    c, E = None, None
    grid = [mp.mpf(i + 1) / grid_n for i in range(grid_n)]
    for _ in range(iters):
        A = mp.matrix(n, n)
        b = mp.matrix(n, 1)
        for i, x in enumerate(ref):
            for j in range(deg):
                A[i, j] = x ** (j + 1)
            A[i, deg] = -((-1) ** i) * mp.power(2, x)
            b[i] = mp.power(2, x) - 1
        sol = mp.lu_solve(A, b)
        c = [sol[j] for j in range(deg)]
        E = sol[deg]
        errs = [_rel_err(c, x) for x in grid]
        # one extremum per run of equal sign
        ext, start = [], 0
        for i in range(1, grid_n + 1):
            if i == grid_n or (errs[i] > 0) != (errs[start] > 0):
                k = max(range(start, i), key=lambda t: abs(errs[t]))
                if k == grid_n - 1:
                    ext.append(grid[k])  # the end point f = 1
                else:
                    lo = grid[k - 1] if k > 0 else mp.mpf(0)
                    ext.append(_extremum(c, lo, grid[k + 1], 1 if errs[k] > 0 else -1))
                start = i
        if len(ext) != n:
            raise RuntimeError(f"Remez: {len(ext)} extrema for {n} references")
        moved = max(abs(a - b) for a, b in zip(ext, ref))
        ref = ext
        if moved < mp.mpf(10) ** -25:
            break
    return c, abs(E)


def f32(x) -> float:
    return float(np.float32(float(x)))


def f32_hex(x: float) -> str:
    return "0x%08X" % struct.unpack("<I", struct.pack("<f", np.float32(x)))[0]


def horner_f32(c32, f):
    """The kernel's evaluation: p = c_deg; p = p f + c_k (k = deg-1..1); p = p f + 1,
    each step one float32 fused multiply-add (the exact float64 product and sum of
    float32 operands, rounded once)."""
    f = np.asarray(f, dtype=np.float32)
    coef = [1.0] + list(c32)
    p = np.full(f.shape, np.float32(coef[-1]), dtype=np.float32)
    for a in reversed(coef[:-1]):
        p = (p.astype(np.float64) * f.astype(np.float64) + np.float64(np.float32(a))).astype(np.float32)
    return p


def rounded_error(c32, samples: int = 1 << 20) -> float:
    """Largest relative error of horner_f32 against 2^f on a dense grid of [0, 1)."""
    f = np.linspace(0.0, 1.0, samples, endpoint=False).astype(np.float32)
    exact = np.exp2(f.astype(np.float64))
    return float(np.max(np.abs(horner_f32(c32, f).astype(np.float64) / exact - 1.0)))


def fit(deg: int = 3):
    """(float32 c1..c_deg, minimax error of the exact fit, error after rounding)."""
    c, E = remez(deg)
    c32 = [f32(a) for a in c]
    return c32, float(E), rounded_error(c32)


if __name__ == "__main__":
    deg = int(sys.argv[1]) if len(sys.argv) > 1 else 3
    c32, E, err32 = fit(deg)
    print(f"degree {deg}, p(0) = 1: minimax relative error {E:.4e}; float32 Horner/fma error {err32:.4e}")
    for i, a in enumerate(c32):
        print(f"  c{i + 1} = {f32_hex(a)}  ({a:.9g})")
