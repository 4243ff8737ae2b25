"""Fits the polynomial of the FMA-pipe 2^x in rowops of the attention kernels.

2^x for x <= 8 is computed as 2^n * p(f), x = n + f, n = floor(x), f in [0, 1)
(the split is exact in floating point).  p(f) = 1 + f * q(f) with q a polynomial
of degree DEG - 1, so p(0) = 1 exactly (2^n is exact for integer x).  The
coefficients minimise the maximum relative error max |p(f) / 2^f - 1| over
[0, 1], found with the Remez exchange algorithm on the weighted problem

    minimise max_f |w(f) (q(f) - g(f))|,   g(f) = (2^f - 1) / f,   w(f) = f / 2^f,

then rounded to float32.  Run ``python fit_exp2_poly.py`` to print them and the
relative error of the rounded coefficients (float64 evaluation, and float32
Horner evaluation with fused multiply-adds emulated in float64).
"""

from __future__ import annotations

import numpy as np

DEG = 5  # degree of p


def _g(f):
    f = np.asarray(f, dtype=np.float64)
    out = np.empty_like(f)
    small = np.abs(f) < 1e-8
    out[~small] = np.expm1(f[~small] * np.log(2.0)) / f[~small]
    out[small] = np.log(2.0) * (1 + f[small] * np.log(2.0) / 2)
    return out


def _w(f):
    return f / np.exp2(f)


def remez(deg=DEG, iters=60, grid=200001):
    m = deg  # coefficients of q (degree deg - 1)
    x = 0.5 - 0.5 * np.cos(np.pi * (np.arange(m + 1) + 0.5) / (m + 1))  # m + 1 Chebyshev-like points in (0, 1)
    dense = np.linspace(1e-9, 1.0, grid)
    for _ in range(iters):
        # q(x_i) - g(x_i) = (-1)^i E / w(x_i)
        A = np.zeros((m + 1, m + 1))
        for i, xi in enumerate(x):
            A[i, :m] = xi ** np.arange(m)
            A[i, m] = -((-1) ** i) / _w(np.array([xi]))[0]
        sol = np.linalg.solve(A, _g(x))
        a = sol[:m]
        err = _w(dense) * (np.polyval(a[::-1], dense) - _g(dense))
        # new points: the extremum of each sign-alternating run of the error
        sign = np.sign(err)
        runs, start = [], 0
        for k in range(1, len(dense) + 1):
            if k == len(dense) or sign[k] != sign[start]:
                seg = np.abs(err[start:k])
                runs.append(start + int(np.argmax(seg)))
                start = k
        runs = np.array(runs)
        if len(runs) > m + 1:  # keep the m + 1 consecutive extrema with the largest smallest value
            best, bi = -1.0, 0
            for s0 in range(len(runs) - m):
                v = np.abs(err[runs[s0:s0 + m + 1]]).min()
                if v > best:
                    best, bi = v, s0
            runs = runs[bi:bi + m + 1]
        if len(runs) < m + 1:
            break
        x = dense[runs]
    return a


def coefficients():
    """float32 coefficients c_1 .. c_DEG of p(f) = 1 + c_1 f + ... + c_DEG f^DEG."""
    return np.float32(remez())


def rel_error_f64(c):
    f = np.linspace(0.0, 1.0, 1000001)
    p = 1.0 + f * np.polyval(np.asarray(c, np.float64)[::-1], f)
    return float(np.max(np.abs(p / np.exp2(f) - 1.0)))


def _fma32(a, b, c):
    return np.float32(np.float64(a) * np.float64(b) + np.float64(c))


def horner32(c, f):
    """p(f) in float32 as the kernel evaluates it: Horner with fused multiply-adds."""
    f = np.float32(f)
    acc = np.float32(c[-1])
    for ck in c[-2::-1]:
        acc = _fma32(acc, f, ck)
    return _fma32(acc, f, np.float32(1.0))


def rel_error_f32(c, n=200001):
    f = np.linspace(0.0, 1.0, n, dtype=np.float64).astype(np.float32)
    p = horner32(np.asarray(c, np.float32), f).astype(np.float64)
    return float(np.max(np.abs(p / np.exp2(f.astype(np.float64)) - 1.0)))


if __name__ == "__main__":
    c = coefficients()
    for k, ck in enumerate(c, 1):
        print(f"c{k} = {float(ck)!r:>24}  ({np.float32(ck).view(np.uint32):#010x})")
    e64, e32 = rel_error_f64(c), rel_error_f32(c)
    print(f"max relative error: {e64:.3e} (2^{np.log2(e64):.2f}) with float32 coefficients, "
          f"{e32:.3e} (2^{np.log2(e32):.2f}) evaluated in float32")
