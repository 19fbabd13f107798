"""The CUDA kernels evaluate the exact (erf-form) GELU with erf taken from
Abramowitz & Stegun, Handbook of Mathematical Functions, formula 7.1.26,
whose absolute error is at most 1.5e-7.  This CPU test reads the constants
from the CUDA header itself and checks that the formula they define meets
that bound against the C library's erf, and that the rearranged GELU the
kernels evaluate (max(v, 0) - |v| g with the constants folded) equals
0.5 v (1 + erf(v / sqrt 2)) within the bound it inherits, so a mistyped
constant or a wrong rearrangement fails here without a GPU.  (The GPU
parity tests check the fp32 kernels end to end.)
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


def gelu_folded(v, c):
    """The GELU of the CUDA header in exact arithmetic: t = 1 / (1 + (p / sqrt 2)
    |v|), y = 0.5 (a1 t + ... + a5 t^5), g = y exp(-v^2 / 2),
    GELU = max(v, 0) - |v| g."""
    av = np.abs(v)
    t = 1.0 / (1.0 + c["P"] / math.sqrt(2.0) * av)
    y = 0.5 * t * (c["A1"] + t * (c["A2"] + t * (c["A3"] + t * (c["A4"] + t * c["A5"]))))
    g = y * np.exp(-0.5 * v * v)
    return np.maximum(v, 0.0) - av * g


def test_folded_gelu_matches_exact_gelu():
    c = constants()
    x = np.linspace(-12.0, 12.0, 240001)
    exact = np.array([0.5 * v * (1.0 + math.erf(v / math.sqrt(2.0))) for v in x])
    err = np.abs(gelu_folded(x, c) - exact)
    # the erf bound scaled by 0.5 |v|
    assert np.all(err <= 0.5 * np.abs(x) * 1.5e-7 + 1e-15), float(np.max(err))


def test_folded_gelu_special_values():
    c = constants()
    v = np.array([0.0, 1e-30, -1e-30, 30.0, -30.0])
    out = gelu_folded(v, c)
    assert out[0] == 0.0
    assert abs(out[1] - 0.5e-30) < 1e-36 and abs(out[2] + 0.5e-30) < 1e-36
    assert out[3] == 30.0 and abs(out[4]) < 1e-150
