"""The FMA-pipe 2^x of the softmax (exp2_poly_pair): its coefficients are the
ones the committed Remez fit produces, its error stays within 2^-22 relative
(the order of the SFU's ex2.approx.f32, which PTX documents at about 2 ulp) on
the whole range the softmax uses, arguments below -126 give exactly 0 as the
flush-to-zero SFU instruction does, and on the GPU its bits are those of the
same operation sequence evaluated exactly on the host."""

import os
import re
from fractions import Fraction

import numpy as np
import pytest
import torch

from tests.helpers import lib_built, need_gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _fit():
    import importlib.util
    path = os.path.join(ROOT, "invariant_dit_attention_gb300", "csrc", "fit_exp2_poly.py")
    spec = importlib.util.spec_from_file_location("fit_exp2_poly", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def kernel_coefficients():
    """c1 .. c5 as written in exp2_poly_pair (hex float literals of the PTX)."""
    text = open(os.path.join(ROOT, "invariant_dit_attention_gb300", "csrc", "common.cuh")).read()
    body = text[text.index("exp2_poly_pair(uint64_t s2"):]
    body = body[:body.index("return r;")]
    found = {name: hx for hx, name in re.findall(r'0f([0-9A-F]{8}), 0f\1\};[^/]*// (c\d)', body)}
    return [np.uint32(int(found[f"c{k}"], 16)).view(np.float32) for k in range(1, 6)]


def test_kernel_coefficients_are_the_remez_fit():
    fit = _fit()
    c = fit.coefficients()
    assert [float(x) for x in kernel_coefficients()] == [float(x) for x in c]
    assert abs(float(c[0]) - np.log(2.0)) < 1e-4  # p'(0) ~ ln 2


def _emulate(x):
    """The kernel's sequence in float32 (fused multiply-adds in float64, exact
    for these operands up to one rounding)."""
    fit = _fit()
    c = np.asarray(kernel_coefficients(), np.float32)
    x = np.maximum(np.asarray(x, np.float32), np.float32(-127.0))
    n = np.floor(x.astype(np.float64))
    f = (x.astype(np.float64) - n).astype(np.float32)
    p = fit.horner32(c, f).astype(np.float64)
    e = np.where(n + 127 > 0, np.exp2(n), 0.0)
    return (p * e).astype(np.float32)


def test_relative_error_within_two_to_the_minus_22_on_the_softmax_range():
    x = np.concatenate([np.linspace(-126.0, 8.0, 2_000_001, dtype=np.float32),
                        np.float32(-126.0) + np.arange(4096, dtype=np.float32) * np.float32(2.0 ** -12),
                        np.arange(-126, 9, dtype=np.float32)])
    y = _emulate(x).astype(np.float64)
    rel = np.abs(y / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() <= 2.0 ** -22, f"max relative error 2^{np.log2(rel.max()):.2f}"


def test_integers_are_exact_and_small_arguments_flush_to_zero():
    k = np.arange(-126, 9, dtype=np.float32)
    assert np.array_equal(_emulate(k), np.exp2(k.astype(np.float64)).astype(np.float32))
    tiny = np.array([-126.5, -127.0, -200.0, -1e30, -np.inf], np.float32)
    assert np.array_equal(_emulate(tiny), np.zeros(5, np.float32))


# ---- on the GPU: exact host evaluation of the same operation sequence

def _round_f32(fr: Fraction) -> np.float32:
    """Correct (nearest-even) rounding of an exact rational to float32."""
    v = float(fr)  # correctly rounded to float64
    f = np.float32(v)
    if Fraction(float(f)) == fr:
        return f
    lo = f if Fraction(float(f)) < fr else np.nextafter(f, np.float32(-np.inf))
    hi = np.nextafter(lo, np.float32(np.inf))
    mid = (Fraction(float(lo)) + Fraction(float(hi))) / 2
    if fr < mid:
        return lo
    if fr > mid:
        return hi
    return lo if (lo.view(np.uint32) & 1) == 0 else hi


def _exact_poly(x: np.float32) -> np.float32:
    c = [Fraction(float(ck)) for ck in kernel_coefficients()]
    xs = max(float(x), -127.0)
    n = np.floor(xs)
    f = Fraction(float(_round_f32(Fraction(xs) - Fraction(n))))  # x - n, rounded once as the kernel does
    acc = _round_f32(c[4])
    for ck in (c[3], c[2], c[1], c[0], Fraction(1)):
        acc = _round_f32(Fraction(float(acc)) * f + ck)
    if n + 127 <= 0:
        return np.float32(0.0)
    return _round_f32(Fraction(float(acc)) * Fraction(2) ** int(n))


@pytest.mark.gpu
def test_device_polynomial_bits_and_agreement_with_the_sfu():
    need_gpu()
    lib_built()
    from invariant_dit_attention_gb300.h3attn import debug_exp2
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.uniform(-126, 8, 3000).astype(np.float32), np.arange(-126, 9, dtype=np.float32),
                        np.array([-126.5, -127, -300, -np.inf, 0.0, -0.0, 1e-30, 7.999999], np.float32)])
    xd = torch.from_numpy(x).cuda()
    poly = debug_exp2(xd, "poly").cpu().numpy()
    sfu = debug_exp2(xd, "sfu").cpu().numpy()
    ref = np.array([_exact_poly(v) for v in x], np.float32)
    assert np.array_equal(poly.view(np.uint32), ref.view(np.uint32))
    normal = x >= -126
    rel = np.abs(poly[normal].astype(np.float64) / sfu[normal].astype(np.float64) - 1.0)
    assert rel.max() <= 2.0 ** -21
    assert np.all(poly[~normal] == 0) and np.all(sfu[~normal] == 0)
