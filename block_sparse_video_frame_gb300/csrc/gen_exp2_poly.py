"""Coefficients of the polynomial 2^f ~= c0 + c1 f + c2 f^2 + c3 f^3 on f in [-1/2, 1/2]
used by the attention kernel to compute part of its exponentials on the FMA pipe.

Method (written from the mathematics, not from any library's implementation):
  * range reduction: 2^x = 2^r * 2^f with r = round-to-nearest(x), f = x - r in [-1/2, 1/2];
    2^r is applied by adding r to the float's exponent field;
  * 2^f is approximated by a cubic fitted by weighted least squares on 4096 Chebyshev
    nodes of [-1/2, 1/2], weights 1/2^f (so the fit minimises relative error), with
    c0 pinned to 1 so that 2^0 = 1 exactly;
  * the coefficients are rounded to float32 and the float32 Horner evaluation is
    checked on a dense grid against float64 2^f.

The softmax rounds every p to bf16 (relative spacing 2^-8), so a relative error
below 2^-12 is far below the rounding the method already applies.

Run ``python gen_exp2_poly.py`` to print the coefficients and the measured error.
"""
from __future__ import annotations

import numpy as np

DEGREE = 3
MAX_REL_ERR = 2.0 ** -12


def fit():
    k = np.arange(4096)
    f = 0.5 * np.cos(np.pi * (k + 0.5) / 4096)          # Chebyshev nodes on [-1/2, 1/2]
    y = np.exp2(f)
    w = 1.0 / y
    # c0 = 1 fixed: fit (2^f - 1) = c1 f + c2 f^2 + c3 f^3, relative weights
    A = np.stack([f ** d for d in range(1, DEGREE + 1)], axis=1) * w[:, None]
    c, *_ = np.linalg.lstsq(A, (y - 1.0) * w, rcond=None)
    return np.concatenate([[1.0], c]).astype(np.float32)


def horner_f32(c, f):
    f = np.asarray(f, dtype=np.float32)
    acc = np.full_like(f, c[-1], dtype=np.float32)
    for ci in c[-2::-1]:
        acc = (acc * f + np.float32(ci)).astype(np.float32)
    return acc


def max_rel_error(c):
    f = np.linspace(-0.5, 0.5, 200001, dtype=np.float64)
    approx = horner_f32(c, f.astype(np.float32)).astype(np.float64)
    exact = np.exp2(f.astype(np.float32).astype(np.float64))
    return float(np.max(np.abs(approx - exact) / exact))


COEFFS = fit()

if __name__ == "__main__":
    print("coefficients (float32, c0..c3):")
    for i, ci in enumerate(COEFFS):
        print(f"  c{i} = {float(ci):.9e}f   (hex {np.float32(ci).view(np.uint32):#010x})")
    err = max_rel_error(COEFFS)
    print(f"max relative error on [-1/2, 1/2] (float32 Horner): {err:.3e} (bound {MAX_REL_ERR:.3e})")
