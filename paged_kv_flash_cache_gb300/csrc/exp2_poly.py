"""Coefficients of the polynomial exp2 used by the prefill softmax on the FMA pipe.

Method: Cody-Waite style range reduction, 2^x = 2^j * 2^f with j = round(x) and
f = x - j in [-1/2, 1/2], and a minimax polynomial p(f) ~ 2^f in the relative-error
sense, computed here with the Remez exchange algorithm (equioscillation of the weighted
error p(f) / 2^f - 1 on degree + 2 reference points). The constant term is pinned to 1 so
that exp2(0) = 1 exactly (a key equal to the running max gets weight 1).

Run `python exp2_poly.py` to print the coefficients and their max relative error; the
values in prefill.cu were produced by this script (rounded to float32).
"""
import numpy as np


def remez_exp2(degree: int, lo: float = -0.5, hi: float = 0.5, iters: int = 40):
    """Minimax p(f) = 1 + c1 f + ... + cn f^n for 2^f on [lo, hi], relative error."""
    n = degree
    # reference points: Chebyshev extrema, n + 1 of them (n unknowns c1..cn plus the level E)
    k = np.arange(n + 1)
    xs = 0.5 * (lo + hi) + 0.5 * (hi - lo) * np.cos(np.pi * k[::-1] / n)
    grid = np.linspace(lo, hi, 200001)
    coef = None
    for _ in range(iters):
        # solve sum_i c_i x^i - E * (-1)^k * 2^x = 2^x - 1   (p(x) - 2^x = E (-1)^k 2^x)
        A = np.zeros((n + 1, n + 1))
        for r, x in enumerate(xs):
            A[r, :n] = [x ** (i + 1) for i in range(n)]
            A[r, n] = -((-1) ** r) * 2.0 ** x
        rhs = 2.0 ** xs - 1.0
        sol = np.linalg.solve(A, rhs)
        coef = np.concatenate([[1.0], sol[:n]])
        err = np.polyval(coef[::-1], grid) / 2.0 ** grid - 1.0
        # new reference: extrema of err between sign changes
        idx = [0]
        for i in range(1, len(grid) - 1):
            if (err[i] - err[i - 1]) * (err[i + 1] - err[i]) <= 0:
                idx.append(i)
        idx.append(len(grid) - 1)
        cand = np.array(idx)
        # keep n + 1 alternating extrema with the largest magnitudes
        pts = []
        for i in cand:
            if pts and np.sign(err[i]) == np.sign(err[pts[-1]]):
                if abs(err[i]) > abs(err[pts[-1]]):
                    pts[-1] = i
            else:
                pts.append(i)
        while len(pts) > n + 1:
            if abs(err[pts[0]]) < abs(err[pts[-1]]):
                pts.pop(0)
            else:
                pts.pop()
        if len(pts) < n + 1:
            break
        xs = grid[pts]
    err = np.polyval(coef[::-1], grid) / 2.0 ** grid - 1.0
    return coef, float(np.abs(err).max())


def emulate_f32(x: np.ndarray, coef32: np.ndarray) -> np.ndarray:
    """The kernel's float32 evaluation order: magic-number rounding, Horner, exponent add."""
    x = x.astype(np.float32)
    magic = np.float32(12582912.0)               # 1.5 * 2^23
    t = (x + magic).astype(np.float32)
    j = (t - magic).astype(np.float32)
    f = (x - j).astype(np.float32)
    p = np.float32(coef32[-1])
    for c in coef32[-2::-1]:
        p = (p * f + np.float32(c)).astype(np.float32)
    jbits = (t.view(np.int32) - magic.view(np.int32)).astype(np.int32)
    return (p.view(np.int32) + (jbits << 23)).astype(np.int32).view(np.float32)


if __name__ == "__main__":
    for deg in (3, 4, 5):
        c, e = remez_exp2(deg)
        c32 = c.astype(np.float32)
        xs = np.linspace(-60, 0, 2000001).astype(np.float32)
        rel = np.abs(emulate_f32(xs, c32).astype(np.float64) / np.exp2(xs.astype(np.float64)) - 1).max()
        print("degree %d: max rel error %.3e (exact coefficients), %.3e (float32 evaluation on [-60, 0])"
              % (deg, e, rel))
        print("  coefficients c0..c%d:" % deg, ", ".join("%.9ef" % v for v in c32))
