"""The CUDA kernels evaluate the exact (erf-form) GELU with erf taken from
Abramowitz & Stegun, Handbook of Mathematical Functions, formula 7.1.26,
whose absolute error is at most 1.5e-7.  This CPU test reads the constants
from the CUDA header itself and checks that the formula they define meets
that bound against the C library's erf, so a mistyped constant fails here
without a GPU.  (The GPU parity tests check the fp32 kernels end to end.)
"""
import math
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "convolution_normalization_gb300", "csrc", "cn_common.cuh")


def constants():
    src = open(HDR).read()
    vals = {}
    for name in ("P", "A1", "A2", "A3", "A4", "A5"):
        m = re.search(r"#define CN_AS_%s (-?[0-9.]+)f" % name, src)
        assert m, name
        vals[name] = float(m.group(1))
    return vals


def erf_as(x, c):
    ax = np.abs(x)
    t = 1.0 / (1.0 + c["P"] * ax)
    poly = t * (c["A1"] + t * (c["A2"] + t * (c["A3"] + t * (c["A4"] + t * c["A5"]))))
    return np.sign(x) * (1.0 - poly * np.exp(-ax * ax))


def test_formula_meets_published_bound():
    c = constants()
    x = np.linspace(-8.0, 8.0, 200001)
    ref = np.array([math.erf(v) for v in x])
    err = np.abs(erf_as(x, c) - ref)
    assert err.max() <= 1.5e-7, err.max()


def test_gelu_from_formula_is_within_tolerance_of_exact():
    c = constants()
    x = np.linspace(-10.0, 10.0, 100001)
    exact = np.array([0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in x])
    approx = 0.5 * x * (1.0 + erf_as(x / math.sqrt(2.0), c))
    # |x| * 0.5 * 1.5e-7 at most: far inside the 1e-4 parity tolerance
    assert np.max(np.abs(approx - exact)) <= 0.5 * 10.0 * 1.5e-7 + 1e-15
