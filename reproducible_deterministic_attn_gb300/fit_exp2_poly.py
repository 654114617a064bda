"""Fits the cubic that the head-dim-128 backward kernel uses for 2^f, f in [-1/2, 1/2].

The kernel evaluates part of P = 2^x on the FMA pipe (exp2_fma in csrc/kernels_tc128.cuh):
x = n + f with n = round(x), 2^f from this cubic, 2^n added into the exponent field. The
fit minimises the maximum relative error (Lawson's iteratively reweighted least squares
on a dense grid) and reports it for the fp32 Horner evaluation the kernel performs.

    python -m reproducible_deterministic_attn_gb300.fit_exp2_poly
"""
import numpy as np


def fit(degree=3, points=20001, iters=200):
    f = np.linspace(-0.5, 0.5, points)
    y = np.exp2(f)
    a = np.vstack([f ** k for k in range(degree + 1)]).T
    w = np.ones_like(f)
    c = None
    for _ in range(iters):
        wr = w / y
        c, *_ = np.linalg.lstsq(a * wr[:, None], y * wr, rcond=None)
        err = np.abs(a @ c - y) / y
        w = w * np.sqrt(err / err.max()) + 1e-12
        w /= w.sum()
    return c.astype(np.float32)


def horner_f32(c, f):
    f = np.asarray(f, dtype=np.float32)
    p = np.float32(c[-1])
    for k in range(len(c) - 2, -1, -1):
        p = (p * f + np.float32(c[k])).astype(np.float32)
    return p


if __name__ == "__main__":
    c = fit()
    f = np.linspace(-0.5, 0.5, 20001)
    rel = np.abs(horner_f32(c, f).astype(np.float64) - np.exp2(f)) / np.exp2(f)
    print("c0..c3 =", ", ".join("%.10f" % x for x in c))
    print("max relative error %.3e (bf16 half-ulp %.3e)" % (rel.max(), 2.0 ** -9))
