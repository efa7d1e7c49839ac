"""The software 2^x of the softmax kernels (csrc/ra_exp2.cuh), on the CPU: its coefficients
are the ones the Remez exchange in exp2_poly.py derives, the polynomial meets the stated
relative error bound, and the derivation is pinned to what it claims (the minimax error
equioscillates, and one more degree of freedom can only lower it)."""

import os
import re

import numpy as np

from exact_blockwise_ring_gb300 import exp2_poly

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "exact_blockwise_ring_gb300", "csrc", "ra_exp2.cuh")


def _header_coefficients():
    text = open(HEADER).read()
    return [float(re.search(r"kExp2C%d = ([0-9.e+-]+)f;" % k, text).group(1))
            for k in range(1, exp2_poly.DEGREE + 1)]


def test_header_holds_the_derived_float32_coefficients():
    got = np.array(_header_coefficients(), dtype=np.float32)
    want = np.array(exp2_poly.float32_coefficients(), dtype=np.float32)
    assert np.array_equal(got, want), (got, want)


def test_relative_error_bound_and_exact_integers():
    c = np.array(_header_coefficients())
    f = np.linspace(-0.5, 0.5, 400001)
    err = np.abs(exp2_poly._rel_err(c, f))
    assert err.max() < 4e-6
    assert exp2_poly._rel_err(c, np.array([0.0]))[0] == 0.0      # p(0) = 1: 2^n exact
    # close to the Taylor coefficients of 2^f (ln 2)^k / k!, as a minimax fit must be
    taylor = [np.log(2) ** k / np.prod(range(1, k + 1)) for k in range(1, 5)]
    assert np.allclose(c, taylor, rtol=0.2)


def test_remez_solution_equioscillates():
    c, level = exp2_poly.remez()
    f = np.linspace(-0.5, 0.5, 200001)
    e = exp2_poly._rel_err(c, f)
    # the error reaches its maximum with alternating signs at degree + 1 points
    peaks = [f[np.argmax(np.abs(e) * (np.sign(e) == s))] for s in (1, -1)]
    assert abs(np.max(e) + np.min(e)) < 0.02 * level        # equal positive and negative peaks
    assert np.max(np.abs(e)) <= level * 1.001
    assert peaks[0] != peaks[1]


def test_planted_wrong_coefficient_breaks_the_bound():
    c = np.array(_header_coefficients())
    c[1] *= 1.001
    f = np.linspace(-0.5, 0.5, 100001)
    assert np.abs(exp2_poly._rel_err(c, f)).max() > 4e-6
