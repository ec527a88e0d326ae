"""The softmax+sigmoid epilogue evaluates sigmoid(t), t in (0, 1], as
1/2 + tanh(t/2)/2 with tanh's Maclaurin series truncated after u^13.

Pins: the coefficients in the kernel source equal 2^2n (2^2n - 1) B_2n / (2n)!
(B_2n the Bernoulli numbers), and the fp32 Horner evaluation the kernel performs
stays within 1e-7 of the exact sigmoid on a dense grid of (0, 1].
"""
import os
import re
from fractions import Fraction
from math import factorial

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "transposed_convolution_convt3d_gb300", "csrc", "tc.cu")


def bernoulli(n):
    B = [Fraction(0)] * (n + 1)
    B[0] = Fraction(1)
    for m in range(1, n + 1):
        B[m] = -sum(Fraction(factorial(m + 1), factorial(k) * factorial(m + 1 - k)) * B[k] for k in range(m)) / (m + 1)
    return B


def tanh_series(nterms):
    B = bernoulli(2 * nterms + 2)
    return [Fraction(2 ** (2 * n + 2) * (2 ** (2 * n + 2) - 1)) * B[2 * n + 2] / factorial(2 * n + 2)
            for n in range(nterms)]


def kernel_coefficients():
    body = open(SRC).read()
    fn = body[body.index("float sigmoid_unit(float t)"):]
    fn = fn[:fn.index("}")]
    fracs = re.findall(r"(-?\d+)\.0f\s*/\s*(\d+)\.0f", fn)
    coefs = [Fraction(int(a), int(b)) for a, b in fracs]
    assert "fmaf(p, u2, 1.0f)" in fn
    return list(reversed(coefs)) if coefs else []


def test_coefficients_are_the_maclaurin_series_of_tanh():
    k = kernel_coefficients()  # u^3 ... u^13 terms, highest first in the source
    series = tanh_series(7)
    assert series[0] == 1
    assert k == series[1:]


def test_fp32_horner_error_bound():
    c = [np.float32(float(x)) for x in tanh_series(7)]
    t = np.linspace(0.0, 1.0, 400001, dtype=np.float64)[1:]
    tf = t.astype(np.float32)
    u = np.float32(0.5) * tf
    u2 = u * u
    p = c[6]
    for cc in (c[5], c[4], c[3], c[2], c[1], c[0]):
        p = (p * u2 + cc).astype(np.float32)
    sig = (np.float32(0.5) * u * p + np.float32(0.5)).astype(np.float32)
    exact = 1.0 / (1.0 + np.exp(-t))
    assert np.max(np.abs(sig - exact)) < 1e-7
    # the truncation bound quoted in the kernel comment: next term at u = 1/2
    nxt = abs(tanh_series(8)[7]) * 0.5 ** 15
    assert nxt < 5e-8
