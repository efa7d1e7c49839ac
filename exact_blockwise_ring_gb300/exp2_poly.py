"""Coefficients of the software 2^x the kernels use beside the hardware exponential unit.

Method (Cody and Waite's range reduction, with a minimax polynomial from the Remez
exchange algorithm):

    x = n + f,  n = round(x),  f in [-1/2, 1/2]
    2^x = 2^n * p(f),   p(f) = 1 + f (c1 + f (c2 + f (c3 + f c4)))

p is the polynomial of its form (p(0) = 1 exactly, so an integer x, such as the running
maximum's own score, gives exactly 2^n) that minimises the largest relative error
|p(f) / 2^f - 1| over [-1/2, 1/2].  The Remez exchange algorithm below finds it: it solves
for the polynomial whose relative error alternates in sign with equal size at a reference
set of points, moves the reference to the error's extrema, and repeats until the
extrema are equal.

Run ``python -m exact_blockwise_ring_gb300.exp2_poly`` to print the coefficients rounded to
float32 and the bounds; the CUDA header ``csrc/ra_exp2.cuh`` holds those printed values,
and a CPU test recomputes them.
"""

import numpy as np

DEGREE = 4          # p(f) = 1 + c1 f + ... + c4 f^4
LO, HI = -0.5, 0.5


def _rel_err(c, f):
    q = np.zeros_like(f)
    for cc in c[::-1]:                      # Horner: c1 + f (c2 + f (...))
        q = q * f + cc
    return (1.0 + f * q) / np.exp2(f) - 1.0


def remez(iters=60, grid=200001):
    """Coefficients (c1, ..., c_DEGREE) in float64 and the minimax relative error."""
    n = DEGREE                      # unknowns c1..cn and the level E: n + 1 points
    f = np.linspace(LO, HI, grid)
    # initial reference: Chebyshev points of the interval, avoiding f = 0 where the error
    # of every p of this form vanishes
    k = np.arange(n + 1)
    ref = 0.5 * (LO + HI) + 0.5 * (HI - LO) * np.cos(np.pi * (k + 0.5) / (n + 1))[::-1]
    c = np.zeros(n)
    level = 0.0
    for _ in range(iters):
        # f c1 + f^2 c2 + ... + f^n cn - (-1)^i E 2^f = 2^f - 1 at the reference points
        A = np.zeros((n + 1, n + 1))
        for j in range(n):
            A[:, j] = ref ** (j + 1)
        A[:, n] = -((-1.0) ** np.arange(n + 1)) * np.exp2(ref)
        sol = np.linalg.solve(A, np.exp2(ref) - 1.0)
        c, level = sol[:n], abs(sol[n])
        # new reference: the extremum of the error on each interval between its sign
        # changes, one per alternation
        e = _rel_err(c, f)
        sign = np.sign(e)
        cuts = np.flatnonzero(np.diff(sign) != 0) + 1
        pieces = np.split(np.arange(len(f)), cuts)
        ext = [p[np.argmax(np.abs(e[p]))] for p in pieces if len(p)]
        # keep the n + 1 largest alternating extrema (the zero at f = 0 splits one lobe)
        ext = sorted(ext, key=lambda i: -abs(e[i]))[:n + 1]
        new = np.sort(f[ext])
        if np.allclose(new, ref, atol=1e-12):
            break
        ref = new
    return c, float(np.max(np.abs(_rel_err(c, f))))


def float32_coefficients():
    c, _ = remez()
    return tuple(float(np.float32(x)) for x in c)


def max_rel_error_float32(samples=2000001):
    """Largest relative error of the float32-rounded coefficients over [-1/2, 1/2]
    (evaluated in float64: the polynomial's own error, without the float32 arithmetic)."""
    c = float32_coefficients()
    f = np.linspace(LO, HI, samples)
    return float(np.max(np.abs(_rel_err(np.array(c), f))))


if __name__ == "__main__":
    c64, err = remez()
    c32 = float32_coefficients()
    print("minimax relative error (float64 coefficients): %.3e" % err)
    print("with float32 coefficients: %.3e" % max_rel_error_float32())
    for name, x in zip(["c%d" % (k + 1) for k in range(DEGREE)], c32):
        print("%s = %.9e  (float32 bits 0x%08x)" % (name, x, np.float32(x).view(np.uint32)))
