"""Coefficients of the polynomial 2^f ~ p(f) on f in [-1/2, 1/2] used by zl_exp2.cuh.

The kernels evaluate 2^x for part of the softmax exponents on the FMA pipe instead of the
special-function unit: x = j + f with j = round(x) (added to the exponent field) and
f in [-1/2, 1/2] (Cody and Waite's range reduction), and 2^f by a polynomial.  This
script fits the polynomial of each degree by iterated weighted least squares towards the
minimax relative error (Lawson's algorithm: the weights of a least-squares fit on a dense
grid are raised where the error is largest), and prints the coefficients and the worst
relative error in exact arithmetic and with the float32 Horner evaluation the kernels use.

    python gen_exp2_poly.py          # prints the table pasted into zl_exp2.cuh
"""
import numpy as np


def fit(degree, iters=400, n=4001):
    f = np.cos(np.linspace(np.pi, 0.0, n)) * 0.5          # Chebyshev-spaced points on [-1/2, 1/2]
    y = np.exp2(f)
    A = np.vander(f, degree + 1, increasing=True) / y[:, None]   # relative error rows
    w = np.full(n, 1.0 / n)
    c = None
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(A * sw[:, None], sw, rcond=None)
        e = np.abs(A @ c - 1.0)
        w = w * e
        w /= w.sum()
    return c


def horner_f32(c, f):
    f = f.astype(np.float32)
    p = np.full_like(f, np.float32(c[-1]))
    for k in range(len(c) - 2, -1, -1):
        p = (p * f + np.float32(c[k])).astype(np.float32)   # separate rounding: a bound for the fused form
    return p


def max_rel_error(c):
    f = np.linspace(-0.5, 0.5, 200001)
    exact = np.abs(np.polyval(c[::-1], f) / np.exp2(f) - 1.0).max()
    f32 = np.abs(horner_f32(c, f).astype(np.float64) / np.exp2(f) - 1.0).max()
    return exact, f32


if __name__ == "__main__":
    for deg in (3, 4, 5):
        c = fit(deg)
        e, e32 = max_rel_error(c)
        print(f"degree {deg}: max rel error {e:.3e} (float32 Horner {e32:.3e})")
        print("  " + ", ".join(f"{float(np.float32(x)).hex()}" for x in c) + "   // " +
              ", ".join(f"{float(np.float32(x)):.9g}" for x in c))
