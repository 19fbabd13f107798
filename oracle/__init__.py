"""fp64 CPU oracle for the fused convolution + normalization forward, and
for its backward pass (the gradients of a loss through the same layers).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package; the library itself never does.
It shares no code with the CUDA path (it does not import the product
package); inputs come from the seeded generator module, passed in as arrays.

The C routines in ``oracle.c`` hold every arithmetic step as a plain loop
in double precision; this file only composes them in the order the
transcripts state the models:

  conv (Conv3d / Conv2d / ConvTranspose2d)  ->  activation  ->  normalization
  ->  post scale  ->  spatial reduction

Pins against independent facts (worked example, closed forms, invariants,
library routines) live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (-O2, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i, L, d = ctypes.c_int, ctypes.c_long, ctypes.c_double
        lib.ocn_conv3d.argtypes = [_dp, i, i, i, i, i, _dp, i, i, i, i, i, _dp, _dp]
        lib.ocn_conv_transpose2d.argtypes = [_dp, i, i, i, i, _dp, i, i, i, _dp, _dp]
        lib.ocn_hardswish.argtypes = [_dp, L]
        lib.ocn_gelu_erf.argtypes = [_dp, L]
        lib.ocn_softmax_channels.argtypes = [_dp, i, i, L]
        lib.ocn_group_norm.argtypes = [_dp, i, i, L, i, d, _dp, _dp, _dp]
        lib.ocn_scale.argtypes = [_dp, L, d]
        lib.ocn_mean_spatial.argtypes = [_dp, i, i, L, _dp]
        lib.ocn_maxpool3d_2.argtypes = [_dp, i, i, i, i, i, _dp]
        lib.ocn_conv3d_grad_input.argtypes = [_dp, i, i, i, i, i, _dp, i, i, i, i, i, _dp]
        lib.ocn_conv3d_grad_weight.argtypes = [_dp, i, i, i, i, i, _dp, i, i, i, i, i, _dp, _dp]
        lib.ocn_conv_transpose2d_grad_input.argtypes = [_dp, i, i, i, i, _dp, i, i, i, _dp]
        lib.ocn_conv_transpose2d_grad_weight.argtypes = [_dp, i, i, i, i, _dp, i, i, i, _dp, _dp]
        lib.ocn_hardswish_grad.argtypes = [_dp, _dp, L]
        lib.ocn_gelu_erf_grad.argtypes = [_dp, _dp, L]
        lib.ocn_group_norm_grad.argtypes = [_dp, i, i, L, i, d, _dp, _dp, _dp, _dp, _dp]
        lib.ocn_num_threads.restype = i
        lib.ocn_set_num_threads.argtypes = [i]
        _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_dp)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def num_threads() -> int:
    return _load().ocn_num_threads()


def set_num_threads(n: int) -> None:
    _load().ocn_set_num_threads(int(n))


# ---- primitives (numpy in, numpy out, all fp64) ---------------------------

def conv3d(x, w, b=None, groups=1):
    x, w, b = _f64(x), _f64(w), _f64(b)
    N, Ci, D, H, W = x.shape
    Co, _, kd, kh, kw = w.shape
    y = np.empty((N, Co, D - kd + 1, H - kh + 1, W - kw + 1))
    _load().ocn_conv3d(_p(x), N, Ci, D, H, W, _p(w), Co, kd, kh, kw, groups, _p(b), _p(y))
    return y


def conv2d(x, w, b=None, groups=1):
    N, Ci, H, W = x.shape
    Co, Cig, kh, kw = w.shape
    y = conv3d(np.asarray(x).reshape(N, Ci, 1, H, W),
               np.asarray(w).reshape(Co, Cig, 1, kh, kw), b, groups)
    return y.reshape(N, Co, H - kh + 1, W - kw + 1)


def conv_transpose2d(x, w, b=None, groups=1):
    x, w, b = _f64(x), _f64(w), _f64(b)
    N, Ci, H, W = x.shape
    _, Cog, k, k2 = w.shape
    assert k == k2
    Co = Cog * groups
    y = np.empty((N, Co, H + k - 1, W + k - 1))
    _load().ocn_conv_transpose2d(_p(x), N, Ci, H, W, _p(w), Co, k, groups, _p(b), _p(y))
    return y


def hardswish(v):
    v = np.array(v, dtype=np.float64, order="C", copy=True)
    _load().ocn_hardswish(_p(v), v.size)
    return v


def gelu_erf(v):
    v = np.array(v, dtype=np.float64, order="C", copy=True)
    _load().ocn_gelu_erf(_p(v), v.size)
    return v


def softmax_channels(v):
    v = np.array(v, dtype=np.float64, order="C", copy=True)
    N, C = v.shape[:2]
    _load().ocn_softmax_channels(_p(v), N, C, int(np.prod(v.shape[2:])))
    return v


def group_norm(y, G, eps=1e-5, gamma=None, beta=None):
    y = _f64(y)
    N, C = y.shape[:2]
    S = int(np.prod(y.shape[2:]))
    out = np.empty_like(y)
    _load().ocn_group_norm(_p(y), N, C, S, G, eps, _p(_f64(gamma)), _p(_f64(beta)), _p(out))
    return out


def scale(v, s):
    v = np.array(v, dtype=np.float64, order="C", copy=True)
    _load().ocn_scale(_p(v), v.size, float(s))
    return v


def mean_spatial(v):
    v = _f64(v)
    N, C = v.shape[:2]
    out = np.empty((N, C))
    _load().ocn_mean_spatial(_p(v), N, C, int(np.prod(v.shape[2:])), _p(out))
    return out


def maxpool3d_2(v):
    v = _f64(v)
    N, C, D, H, W = v.shape
    out = np.empty((N, C, D // 2, H // 2, W // 2))
    _load().ocn_maxpool3d_2(_p(v), N, C, D, H, W, _p(out))
    return out


# ---- the whole forward ------------------------------------------------------

def conv_stage(s, inputs, samples=None):
    """Convolution output (before activation) for workload dict ``s``."""
    x = inputs["x"] if samples is None else inputs["x"][list(samples)]
    w, b, G = inputs["w"], inputs.get("b"), s["groups"]
    if s["conv"] == "conv3d":
        return conv3d(x, w, b, G)
    if s["conv"] == "conv2d":
        return conv2d(x, w, b, G)
    return conv_transpose2d(x, w, b, G)


def forward(s, inputs, samples=None):
    """fp64 result of the whole fused forward for workload dict ``s``.

    ``samples`` optionally restricts the batch to a list of sample indices;
    every step is per sample, so the rows returned equal those rows of the
    full result.
    """
    y = conv_stage(s, inputs, samples)
    act = s["act"]
    if act == "hardswish":
        y = hardswish(y)
    elif act == "gelu_erf":
        y = gelu_erf(y)
    elif act == "softmax_c":
        y = softmax_channels(y)
    norm = s["norm"]
    if norm != "none":
        G = s["num_groups"] if norm == "group" else y.shape[1]
        aff = bool(s["affine"])
        y = group_norm(y, G, s["eps"], inputs["gamma"] if aff else None,
                       inputs["beta"] if aff else None)
    if s["post_scale"] != 1.0:
        y = scale(y, s["post_scale"])
    red = s["red"]
    if red == "mean_spatial":
        y = mean_spatial(y)
    elif red == "maxpool2_x2":
        y = maxpool3d_2(maxpool3d_2(y))
    return y


# ---- the backward pass ------------------------------------------------------
# Gradients of a loss L through the forward above, given dout = dL/d(output).
# Each primitive is the derivative of the forward primitive of the same name.

def conv3d_grad_input(dy, w, groups=1):
    dy, w = _f64(dy), _f64(w)
    N, Co, Do, Ho, Wo = dy.shape
    _, Cig, kd, kh, kw = w.shape
    Ci = Cig * groups
    dx = np.empty((N, Ci, Do + kd - 1, Ho + kh - 1, Wo + kw - 1))
    _load().ocn_conv3d_grad_input(_p(dy), N, Co, Do, Ho, Wo, _p(w), Ci, kd, kh, kw, groups, _p(dx))
    return dx


def conv3d_grad_weight(x, dy, w_shape, groups=1):
    x, dy = _f64(x), _f64(dy)
    N, Ci, D, H, W = x.shape
    Co, Cig, kd, kh, kw = w_shape
    dw = np.empty(w_shape)
    db = np.empty(Co)
    _load().ocn_conv3d_grad_weight(_p(x), N, Ci, D, H, W, _p(dy), Co, kd, kh, kw, groups, _p(dw), _p(db))
    return dw, db


def conv2d_grad_input(dy, w, groups=1):
    N, Co, Ho, Wo = dy.shape
    Co_, Cig, kh, kw = w.shape
    dx = conv3d_grad_input(np.asarray(dy).reshape(N, Co, 1, Ho, Wo),
                           np.asarray(w).reshape(Co_, Cig, 1, kh, kw), groups)
    return dx.reshape(N, Cig * groups, Ho + kh - 1, Wo + kw - 1)


def conv2d_grad_weight(x, dy, w_shape, groups=1):
    N, Ci, H, W = x.shape
    Co, Cig, kh, kw = w_shape
    dw, db = conv3d_grad_weight(np.asarray(x).reshape(N, Ci, 1, H, W),
                                np.asarray(dy).reshape(dy.shape[0], dy.shape[1], 1, *dy.shape[2:]),
                                (Co, Cig, 1, kh, kw), groups)
    return dw.reshape(w_shape), db


def conv_transpose2d_grad_input(dy, w, groups=1):
    dy, w = _f64(dy), _f64(w)
    N, Co, Ho, Wo = dy.shape
    Ci, _, k, _ = w.shape
    H, W = Ho - k + 1, Wo - k + 1
    dx = np.empty((N, Ci, H, W))
    _load().ocn_conv_transpose2d_grad_input(_p(dy), N, Co, H, W, _p(w), Ci, k, groups, _p(dx))
    return dx


def conv_transpose2d_grad_weight(x, dy, w_shape, groups=1):
    x, dy = _f64(x), _f64(dy)
    N, Ci, H, W = x.shape
    _, Cog, k, _ = w_shape
    Co = Cog * groups
    dw = np.empty(w_shape)
    db = np.empty(Co)
    _load().ocn_conv_transpose2d_grad_weight(_p(x), N, Ci, H, W, _p(dy), Co, k, groups, _p(dw), _p(db))
    return dw, db


def hardswish_grad(v, g):
    g = np.array(g, dtype=np.float64, order="C", copy=True)
    _load().ocn_hardswish_grad(_p(_f64(v)), _p(g), g.size)
    return g


def gelu_erf_grad(v, g):
    g = np.array(g, dtype=np.float64, order="C", copy=True)
    _load().ocn_gelu_erf_grad(_p(_f64(v)), _p(g), g.size)
    return g


def group_norm_grad(y, dout, G, eps=1e-5, gamma=None):
    """(dy, dgamma, dbeta) of group_norm(y, G, eps, gamma, beta) for dout."""
    y, dout = _f64(y), _f64(dout)
    N, C = y.shape[:2]
    S = int(np.prod(y.shape[2:]))
    dy = np.empty_like(y)
    dgamma, dbeta = np.empty(C), np.empty(C)
    _load().ocn_group_norm_grad(_p(y), N, C, S, G, eps, _p(_f64(gamma)), _p(dout), _p(dy),
                                _p(dgamma), _p(dbeta))
    return dy, dgamma, dbeta


def backward(s, inputs, dout, intermediates=False):
    """Gradients of the whole fused block for workload dict ``s`` (spatial
    reductions none or the spatial mean; activations none, HardSwish or
    GELU): dict with dx, dw, db (None without bias), dgamma and dbeta (None
    without an affine norm).  The forward's intermediates are recomputed;
    with ``intermediates`` the dict also holds dA, the gradient with respect
    to the conv output."""
    act, norm, red = s["act"], s["norm"], s["red"]
    assert red in ("none", "mean_spatial") and act in ("none", "hardswish", "gelu_erf")
    x, w, G = inputs["x"], inputs["w"], s["groups"]
    a = conv_stage(s, inputs)                       # pre-activation
    y = a if act == "none" else (hardswish(a) if act == "hardswish" else gelu_erf(a))
    g = np.asarray(dout, dtype=np.float64)
    if red == "mean_spatial":                       # d(mean)/dv = 1/S for every position
        S = int(np.prod(a.shape[2:]))
        g = np.broadcast_to((g / S).reshape(g.shape + (1,) * (a.ndim - 2)), a.shape).copy()
    if s["post_scale"] != 1.0:
        g = scale(g, s["post_scale"])
    dgamma = dbeta = None
    aff = bool(s["affine"]) and norm != "none"
    if norm != "none":
        Gn = s["num_groups"] if norm == "group" else a.shape[1]
        g, dgamma, dbeta = group_norm_grad(y, g, Gn, s["eps"], inputs["gamma"] if aff else None)
        if not aff:
            dgamma = dbeta = None
    if act == "hardswish":
        g = hardswish_grad(a, g)
    elif act == "gelu_erf":
        g = gelu_erf_grad(a, g)
    if s["conv"] == "conv3d":
        dx = conv3d_grad_input(g, w, G)
        dw, db = conv3d_grad_weight(x, g, w.shape, G)
    elif s["conv"] == "conv2d":
        dx = conv2d_grad_input(g, w, G)
        dw, db = conv2d_grad_weight(x, g, w.shape, G)
    else:
        dx = conv_transpose2d_grad_input(g, w, G)
        dw, db = conv_transpose2d_grad_weight(x, g, w.shape, G)
    res = {"dx": dx, "dw": dw, "db": db if s["has_bias"] else None, "dgamma": dgamma, "dbeta": dbeta}
    if intermediates:
        res["dA"] = g
    return res
