"""The kernels' FMA-pipe exponential (ex2_poly in csrc/common.cuh), emulated step
by step in float32 on the host: its coefficients, read from the source, must
keep the relative error of 2^x below 8e-5 over the range the kernels use, and
inputs below -126 (masked scores, -inf) must give exactly 0.  The GPU parity
tests then check the kernels that use it end to end."""
import os
import re

import numpy as np

from conftest import ROOT

SRC = os.path.join(ROOT, "blockwise_online_softmax_cpattn_gb300", "csrc", "common.cuh")


def _coeffs():
    body = open(SRC).read().split("float ex2_poly(float x)")[1].split("}")[0]
    c = [float(v) for v in re.findall(r"(-?\d+\.\d+)f", body)]
    assert len(c) == 4          # c3, c2, c1, c0 in Horner order
    return tuple(np.float32(v) for v in c)


def _fma(a, b, c):
    return np.float32(np.float64(a) * np.float64(b) + np.float64(c))


def _ex2_poly(x, c3, c2, c1, c0):
    x = np.float32(x)
    with np.errstate(invalid="ignore"):
        t = np.float32(x + np.float32(12582912.0))
        n = np.float32(t - np.float32(12582912.0))
        f = np.float32(x - n)
    q = _fma(_fma(_fma(c3, f, c2), f, c1), f, c0)
    qb = np.array([q], dtype=np.float32).view(np.int32)[0]
    tb = np.array([t], dtype=np.float32).view(np.int32)[0]
    r = np.array([np.int32(qb + np.int32(np.int64(tb) << 23 & 0xFFFFFFFF).astype(np.int32))],
                 dtype=np.int32).view(np.float32)[0]
    return np.float32(0.0) if x < -126 else r


def test_ex2_poly_error_bound():
    c = _coeffs()
    assert abs(float(c[3]) - 1.0) < 1e-3 and abs(float(c[2]) - np.log(2)) < 1e-2
    xs = np.concatenate([np.linspace(-125, 8, 40001), -np.logspace(-7, 1, 801),
                         np.logspace(-7, 0.9, 801)]).astype(np.float32)
    worst = max(abs(float(_ex2_poly(x, *c)) - 2.0 ** float(x)) / 2.0 ** float(x) for x in xs)
    assert worst < 8e-5, worst


def test_ex2_poly_masked_inputs_are_zero():
    c = _coeffs()
    for x in (-np.inf, -1e30, -200.0, -126.5):
        assert _ex2_poly(x, *c) == 0.0
    assert _ex2_poly(0.0, *c) == np.float32(c[3])
