"""Pins for the FMA-pipe exponential exp2_poly2 of csrc/ptx.cuh (no GPU).

The device function computes 2^x as 2^floor(x) * p(x - floor(x)) with a degree-3
polynomial p whose constant term is 1, after clamping x to >= -127.  Checked
here:
  * the coefficients in ptx.cuh are exactly the float32 values the committed
    Remez fit (csrc/fit_exp2_poly.py) produces;
  * a step-by-step float32 emulation of the device function (clamp, floor by the
    1.5 * 2^23 rounding trick, Horner steps as fused multiply-adds, exponent
    added to the bits) meets the stated bound against the exact 2^x (numpy's
    float64 exp2 on float32 inputs), is exact at integers, gives +0.0 for
    x <= -127 and -inf, and stays below 2^-126 just above -127;
  * planted mistakes in that emulation each fail one of these pins.
"""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_tiled_attention_16_gb300", "csrc")
BOUND = 8.7e-5  # the fit's 8.565e-5 in float32 Horner form plus the final rounding


def kernel_coefficients():
    text = open(os.path.join(CSRC, "ptx.cuh")).read()
    found = dict(re.findall(r"constexpr float kExp2PolyC(\d) = (0x[0-9a-fA-F.]+p[-+]?\d+)f;", text))
    return [float.fromhex(found[k]) for k in ("1", "2", "3")]


def _fma32(a, b, c):
    """float32 fused multiply-add, emulated in float64 (the product of two
    float32s is exact there; the sum is rounded twice only in rare ties, which
    moves a result by at most one float32 step)."""
    return (np.float64(a) * np.float64(b) + np.float64(c)).astype(np.float32)


def exp2_poly_emul(x, c=None, clamp=-127.0, floor_mode="floor", shift=23):
    """Float32 emulation of exp2_poly2, one element at a time."""
    c1, c2, c3 = kernel_coefficients() if c is None else c
    x = np.asarray(x, dtype=np.float32)
    if clamp is not None:
        x = np.where(np.isnan(x), np.float32(clamp), np.maximum(x, np.float32(clamp))).astype(np.float32)
    xd = x.astype(np.float64)
    n = np.floor(xd) if floor_mode == "floor" else np.rint(xd)
    n = np.clip(n, -(2 ** 22), 2 ** 22 - 1)  # the emulation of the bit trick assumes this range
    f = (xd - n).astype(np.float32)                     # exact
    p = _fma32(np.float32(c3), f, np.float32(c2))
    p = _fma32(p, f, np.float32(c1))
    p = _fma32(p, f, np.float32(1.0))
    j_bits = (np.int64(0x4B400000) + n.astype(np.int64)) & 0xFFFFFFFF
    bits = (p.view(np.uint32).astype(np.int64) + ((j_bits << shift) & 0xFFFFFFFF)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def _grid():
    g = np.random.default_rng(3)
    dense = np.linspace(-126.0, 20.0, 400001, dtype=np.float64).astype(np.float32)
    rnd = g.uniform(-126.0, 20.0, 200000).astype(np.float32)
    near_int = (np.arange(-126, 21)[:, None] + np.array([-1e-6, 0.0, 1e-6, 0.5, 0.999999])[None, :]).ravel()
    x = np.concatenate([dense, rnd, near_int.astype(np.float32)])
    return x[(x >= -126.0) & (x <= 20.0)]


def check_bound(fn):
    x = _grid()
    y = fn(x).astype(np.float64)
    exact = np.exp2(x.astype(np.float64))
    rel = np.abs(y / exact - 1.0)
    assert np.all(np.isfinite(y)) and rel.max() <= BOUND, f"max relative error {rel.max():.3e}"


def check_integers_exact(fn):
    n = np.arange(-126, 21, dtype=np.float32)
    assert np.array_equal(fn(n).astype(np.float64), np.exp2(n.astype(np.float64)))


def check_underflow(fn):
    low = np.array([-127.0, -128.0, -300.0, -1e30, -np.inf], dtype=np.float32)
    y = fn(low)
    assert np.all(y.view(np.uint32) == 0), "x <= -127 and -inf must give +0.0"
    mid = np.linspace(-127.0, -126.0, 1001, dtype=np.float32)[1:-1]
    y = fn(mid).astype(np.float64)
    assert np.all((y >= 0.0) & (y < 2.0 ** -126)), "results just above -127 must stay below 2^-126"


CHECKS = [check_bound, check_integers_exact, check_underflow]


def test_coefficients_are_the_committed_fit():
    import importlib.util
    spec = importlib.util.spec_from_file_location("fit_exp2_poly", os.path.join(CSRC, "fit_exp2_poly.py"))
    fit = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(fit)
    c32, err_exact, err32 = fit.fit(3)
    assert kernel_coefficients() == c32
    assert err_exact < 8.6e-5 and err32 < 8.6e-5


@pytest.mark.parametrize("check", CHECKS, ids=[c.__name__ for c in CHECKS])
def test_emulated_device_exponential(check):
    check(exp2_poly_emul)


PLANTED = {
    # f in [-0.5, 0.5) from round-to-nearest, but p was fitted on [0, 1]
    "round_to_nearest": lambda x: exp2_poly_emul(x, floor_mode="nearest"),
    # exponent field one bit off
    "shift_22": lambda x: exp2_poly_emul(x, shift=22),
    # clamp one binade too high: -inf gives 2^-126, not 0
    "clamp_minus_126": lambda x: exp2_poly_emul(x, clamp=-126.0),
    # no clamp: very negative x wraps the exponent into the sign bit
    "no_clamp": lambda x: exp2_poly_emul(x, clamp=None),
    # the quadratic and cubic coefficients exchanged
    "c2_c3_swapped": lambda x: exp2_poly_emul(x, c=[kernel_coefficients()[0], kernel_coefficients()[2],
                                                    kernel_coefficients()[1]]),
    # Taylor coefficients instead of the minimax fit
    "taylor": lambda x: exp2_poly_emul(x, c=[float(np.float32(np.log(2))), float(np.float32(np.log(2) ** 2 / 2)),
                                             float(np.float32(np.log(2) ** 3 / 6))]),
}


@pytest.mark.parametrize("kind", sorted(PLANTED))
def test_planted_mistake_fails_a_pin(kind):
    fn = PLANTED[kind]
    failed = False
    for check in CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(fn)
        except AssertionError:
            failed = True
    assert failed, f"planted mistake {kind} passed every pin"
