"""Pins for the fp64 oracle against facts that do not come from the oracle.

Each check is chosen so that a plausible slip in the oracle (a dropped
term, a wrong sign or index, a transposed operand, a flipped kernel, a
sample instead of population variance, eps outside the root) fails at least
one of them.  Independent sources used here:

* the values printed in l2_p19's hand-worked transposed-convolution example
  (tests/golden/convt2d_worked_example.json);
* closed forms and identities (impulse response, adjoint identity, sums,
  the mean-after-GroupNorm closed form of l2_p27, pool composition of l2_p6);
* invariants (normalized groups have mean 0 and variance var/(var+eps),
  softmax sums to 1);
* independent library routines (PyTorch CPU ops in float64, numpy
  sliding-window im2col products) on small shapes.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from convolution_normalization_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


def t64(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))


# ---------------------------------------------------------------- conv ----

@pytest.mark.parametrize("shape", [
    # N, Ci, Co, D, H, W, k, groups
    (2, 3, 4, 5, 6, 7, 3, 1),
    (1, 4, 6, 4, 5, 5, 2, 2),
    (2, 2, 2, 3, 4, 6, 1, 1),
    (1, 3, 5, 6, 6, 6, 4, 1),
])
def test_conv3d_matches_torch(shape):
    N, Ci, Co, D, H, W, k, G = shape
    x = rng.standard_normal((N, Ci, D, H, W))
    w = rng.standard_normal((Co, Ci // G, k, k, k))
    b = rng.standard_normal(Co)
    y = oracle.conv3d(x, w, b, G)
    assert y.shape == (N, Co, D - k + 1, H - k + 1, W - k + 1)  # L - k + 1
    ref = F.conv3d(t64(x), t64(w), t64(b), groups=G).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_conv3d_im2col_independent():
    # Second formulation: sliding windows (im2col) times the flattened filter.
    x = rng.standard_normal((2, 3, 6, 7, 8))
    w = rng.standard_normal((5, 3, 3, 3, 3))
    win = np.lib.stride_tricks.sliding_window_view(x, (3, 3, 3), axis=(2, 3, 4))
    ref = np.einsum("ncdhwapq,ocapq->nodhw", win, w)
    np.testing.assert_allclose(oracle.conv3d(x, w), ref, rtol=1e-12, atol=1e-12)


def test_conv3d_impulse_reproduces_filter():
    # A one-hot input at an interior point P gives y[P - (a,p,q)] = w[a,p,q]
    # (cross-correlation: the filter appears reversed around P).
    k = 3
    x = np.zeros((1, 1, 7, 7, 7))
    x[0, 0, 3, 3, 3] = 1.0
    w = rng.standard_normal((1, 1, k, k, k))
    y = oracle.conv3d(x, w)
    for a in range(k):
        for p in range(k):
            for q in range(k):
                assert y[0, 0, 3 - a, 3 - p, 3 - q] == w[0, 0, a, p, q]
    assert np.count_nonzero(y) == k ** 3


def test_conv3d_k1_is_channel_matmul():
    x = rng.standard_normal((2, 4, 3, 5, 6))
    w = rng.standard_normal((3, 4, 1, 1, 1))
    ref = np.einsum("oc,ncdhw->nodhw", w[:, :, 0, 0, 0], x)
    np.testing.assert_allclose(oracle.conv3d(x, w), ref, rtol=1e-13, atol=1e-13)


def test_conv2d_matches_torch():
    x = rng.standard_normal((2, 6, 9, 11))
    w = rng.standard_normal((4, 6, 3, 3))
    b = rng.standard_normal(4)
    ref = F.conv2d(t64(x), t64(w), t64(b)).numpy()
    np.testing.assert_allclose(oracle.conv2d(x, w, b), ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------- transposed conv --

def test_convt2d_page_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "convt2d_worked_example.json")))
    x = np.array(g["x"], dtype=np.float64)[None, None]
    w = np.array(g["w"], dtype=np.float64)[None, None]
    y = oracle.conv_transpose2d(x, w)[0, 0]
    assert list(y.shape) == g["out_shape"]  # (L - 1) * s + k = 4
    for e in g["printed_values"]:
        assert y[e["i"], e["j"]] == e["value"]
    # The page's printed out[0,3] = 0 is garbled; its own formula gives 1.
    gb = g["garbled"]
    assert y[gb["i"], gb["j"]] == gb["reading"]


@pytest.mark.parametrize("shape", [
    # N, Ci, Co, H, W, k, groups
    (2, 4, 4, 5, 6, 3, 1),
    (1, 8, 16, 6, 5, 3, 4),
    (2, 6, 6, 4, 4, 2, 6),
    (1, 2, 3, 3, 7, 4, 1),
])
def test_convt2d_matches_torch(shape):
    N, Ci, Co, H, W, k, G = shape
    x = rng.standard_normal((N, Ci, H, W))
    w = rng.standard_normal((Ci, Co // G, k, k))
    b = rng.standard_normal(Co)
    y = oracle.conv_transpose2d(x, w, b, G)
    assert y.shape == (N, Co, H + k - 1, W + k - 1)
    ref = F.conv_transpose2d(t64(x), t64(w), t64(b), stride=1, padding=0, groups=G).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_convt2d_is_adjoint_of_conv2d():
    # <conv(x; w), u> = <x, convT(u; w')> with w' the same stored numbers
    # read in the transposed layer's (C_in, C_out/groups, k, k) order:
    # for groups G the conv maps Ci -> Co with w (Co, Ci/G, k, k) and its
    # adjoint maps Co -> Ci with the same array seen as (Co, Ci/G, k, k).
    G, Ci, Co, k = 2, 4, 6, 3
    x = rng.standard_normal((1, Ci, 8, 7))
    w = rng.standard_normal((Co, Ci // G, k, k))
    y = oracle.conv2d(x, w, None, G)
    u = rng.standard_normal(y.shape)
    lhs = float(np.sum(y * u))
    rhs = float(np.sum(x * oracle.conv_transpose2d(u, w, None, G)))
    assert math.isclose(lhs, rhs, rel_tol=1e-12, abs_tol=1e-12)


def test_convt2d_total_sum_and_depthwise():
    # One channel, no bias: every x value meets every filter tap exactly once
    # inside the (H+k-1) x (W+k-1) output, so sum(out) = sum(x) * sum(w).
    x = rng.standard_normal((1, 1, 5, 6))
    w = rng.standard_normal((1, 1, 3, 3))
    y = oracle.conv_transpose2d(x, w)
    assert math.isclose(y.sum(), x.sum() * w.sum(), rel_tol=1e-12, abs_tol=1e-12)
    # groups = C (depthwise): each channel is an independent 2-D full
    # convolution, equal to a zero-padded correlation with the flipped kernel.
    C = 3
    x = rng.standard_normal((1, C, 4, 5))
    w = rng.standard_normal((C, 1, 3, 3))
    y = oracle.conv_transpose2d(x, w, None, C)
    for c in range(C):
        xp = np.pad(x[0, c], 2)
        ref = oracle.conv2d(xp[None, None], w[c, 0, ::-1, ::-1].copy()[None, None])[0, 0]
        np.testing.assert_allclose(y[0, c], ref, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------- activations --

def test_hardswish_special_values():
    v = np.array([-10.0, -3.0, -1.5, 0.0, 1.0, 3.0, 7.5])
    h = oracle.hardswish(v)
    assert h[0] == 0.0 and h[1] == 0.0 and h[3] == 0.0  # x <= -3 -> 0
    assert h[5] == 3.0 and h[6] == 7.5                  # x >= 3 -> x
    assert math.isclose(h[2], -1.5 * 1.5 / 6.0) and math.isclose(h[4], 4.0 / 6.0)
    np.testing.assert_allclose(h, F.hardswish(t64(v)).numpy(), rtol=1e-15, atol=0)


def test_gelu_erf_properties():
    v = np.linspace(-8, 8, 161)
    g = oracle.gelu_erf(v)
    assert g[80] == 0.0
    # gelu(-x) = gelu(x) - x  (Phi(-x) = 1 - Phi(x))
    np.testing.assert_allclose(g[::-1], g - v, rtol=0, atol=1e-14)
    assert abs(g[-1] - 8.0) < 1e-14
    np.testing.assert_allclose(g, F.gelu(t64(v), approximate="none").numpy(), rtol=1e-14, atol=1e-15)
    # The tanh approximation differs by more than the tolerance somewhere.
    assert np.max(np.abs(g - F.gelu(t64(v), approximate="tanh").numpy())) > 1e-4


def test_softmax_channels():
    v = rng.standard_normal((2, 16, 3, 4, 5)) * 5
    s = oracle.softmax_channels(v)
    np.testing.assert_allclose(s.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.all(s > 0) and np.all(s < 1)
    np.testing.assert_allclose(s, torch.softmax(t64(v), dim=1).numpy(), rtol=1e-13, atol=1e-16)
    # Shift invariance along channels (the max subtraction changes nothing).
    np.testing.assert_allclose(oracle.softmax_channels(v + 100.0), s, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- norms --

@pytest.mark.parametrize("G", [1, 2, 4, 16])
def test_group_norm_invariants_and_torch(G):
    y = rng.standard_normal((3, 16, 2, 3, 5)) * 2.0 + 0.7
    eps = 1e-5
    z = oracle.group_norm(y, G, eps)
    zg = z.reshape(3, G, -1)
    yg = y.reshape(3, G, -1)
    var = yg.var(axis=2)  # population variance of the input groups
    np.testing.assert_allclose(zg.mean(axis=2), 0.0, atol=1e-13)
    np.testing.assert_allclose(zg.var(axis=2), var / (var + eps), rtol=1e-12)
    gamma = rng.standard_normal(16)
    beta = rng.standard_normal(16)
    za = oracle.group_norm(y, G, eps, gamma, beta)
    ref = F.group_norm(t64(y), G, t64(gamma), t64(beta), eps).numpy()
    np.testing.assert_allclose(za, ref, rtol=1e-11, atol=1e-12)
    # gamma = 1, beta = 0 is the identity on the normalized values.
    np.testing.assert_allclose(oracle.group_norm(y, G, eps, np.ones(16), np.zeros(16)), z, rtol=0, atol=0)


def test_instance_norm_is_group_norm_with_g_equal_c():
    y = rng.standard_normal((2, 5, 7, 9)) + 3.0
    z = oracle.group_norm(y, 5, 1e-5)
    ref = F.instance_norm(t64(y), eps=1e-5).numpy()
    np.testing.assert_allclose(z, ref, rtol=1e-11, atol=1e-12)


def test_eps_inside_root_and_population_variance():
    # A group with two values a, b: var = ((a-b)/2)^2 exactly.
    y = np.array([1.0, 3.0]).reshape(1, 1, 2)
    z = oracle.group_norm(y, 1, 0.25)
    assert math.isclose(z[0, 0, 1], 1.0 / math.sqrt(1.0 + 0.25), rel_tol=1e-15)


# ------------------------------------------------------------ reductions --

def test_mean_after_groupnorm_closed_form():
    # l2_p27: the spatial mean of GroupNorm's output needs only per-channel
    # spatial means m_c and group statistics:
    #   out_c = gamma_c * (m_c - mu_g) / sqrt(var_g + eps) + beta_c,
    #   mu_g = mean_c m_c,  var_g = mean_c E_s[y^2] - mu_g^2.
    y = rng.standard_normal((2, 16, 3, 4, 5)) * 1.3 + 0.2
    G, eps = 4, 1e-5
    gamma, beta = rng.standard_normal(16), rng.standard_normal(16)
    lit = oracle.mean_spatial(oracle.group_norm(y, G, eps, gamma, beta))
    m = y.reshape(2, 16, -1).mean(axis=2)
    q = (y.reshape(2, 16, -1) ** 2).mean(axis=2)
    mu = m.reshape(2, G, -1).mean(axis=2)
    var = q.reshape(2, G, -1).mean(axis=2) - mu ** 2
    cf = gamma * (m - np.repeat(mu, 4, axis=1)) / np.sqrt(np.repeat(var, 4, axis=1) + eps) + beta
    np.testing.assert_allclose(lit, cf, rtol=1e-11, atol=1e-12)
    # Invariant: sum over a group's channels of (out_c - beta_c)/gamma_c = 0.
    r = ((lit - beta) / gamma).reshape(2, G, -1).sum(axis=2)
    np.testing.assert_allclose(r, 0.0, atol=1e-12)


def test_maxpool_twice_is_one_stride4_pool():
    # l2_p6: floor(floor(L/2)/2) = floor(L/4) and max is associative, so two
    # 2x2x2 pools equal one 4x4x4 stride-4 pool; the tail is dropped.
    v = rng.standard_normal((2, 3, 14, 30, 29))
    p2 = oracle.maxpool3d_2(oracle.maxpool3d_2(v))
    assert p2.shape == (2, 3, 3, 7, 7)
    ref = F.max_pool3d(t64(v), 4, 4).numpy()
    np.testing.assert_array_equal(p2, ref)
    np.testing.assert_array_equal(oracle.maxpool3d_2(v), F.max_pool3d(t64(v), 2, 2).numpy())


def test_mean_spatial():
    v = rng.standard_normal((2, 3, 4, 5, 6))
    np.testing.assert_allclose(oracle.mean_spatial(v), v.mean(axis=(2, 3, 4)), rtol=1e-13)


# ------------------------------------------------------------ forward ----

def _torch_forward(s, inp):
    """The same model stated with PyTorch fp64 CPU ops (an independent
    implementation of every step)."""
    x = t64(inp["x"])
    w = t64(inp["w"])
    b = t64(inp["b"]) if inp["b"] is not None else None
    if s["conv"] == "conv3d":
        y = F.conv3d(x, w, b, groups=s["groups"])
    elif s["conv"] == "conv2d":
        y = F.conv2d(x, w, b, groups=s["groups"])
    else:
        y = F.conv_transpose2d(x, w, b, groups=s["groups"])
    if s["act"] == "hardswish":
        y = F.hardswish(y)
    elif s["act"] == "gelu_erf":
        y = F.gelu(y)
    elif s["act"] == "softmax_c":
        y = torch.softmax(y, dim=1)
    if s["norm"] != "none":
        G = s["num_groups"] if s["norm"] == "group" else y.shape[1]
        ga = t64(inp["gamma"]) if s["affine"] else None
        be = t64(inp["beta"]) if s["affine"] else None
        y = F.group_norm(y, G, ga, be, s["eps"])
    y = y * s["post_scale"]
    if s["red"] == "mean_spatial":
        y = y.mean(dim=tuple(range(2, y.dim())))
    elif s["red"] == "maxpool2_x2":
        y = F.max_pool3d(F.max_pool3d(y, 2, 2), 2, 2)
    return y.numpy()


SMALL = [
    wl.WORKLOADS[0],
    wl.with_overrides(wl.WORKLOADS[1], N=2, D=7, H=9, W=10),
    wl.with_overrides(wl.WORKLOADS[2], N=2, C_in=8, C_out=6, H=11, W=13),
    wl.with_overrides(wl.WORKLOADS[3], N=2, D=9, H=12, W=11),
    wl.with_overrides(wl.WORKLOADS[4], N=2, C_in=16, C_out=16, H=9, W=7),
    # a post scale before the pool and before the mean (the other cases use 1)
    wl.with_overrides(wl.WORKLOADS[3], N=2, D=8, H=9, W=12, post_scale=0.5,
                      name="pool_scaled"),
    wl.with_overrides(wl.WORKLOADS[1], N=2, D=6, H=8, W=9, post_scale=0.25,
                      name="mean_scaled"),
]


@pytest.mark.parametrize("s", SMALL, ids=[s["name"] for s in SMALL])
def test_forward_matches_torch_model(s):
    inp = wl.make_inputs(s)
    out = oracle.forward(s, inp)
    ref = _torch_forward(s, inp)
    assert out.shape == ref.shape
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-11)


def test_forward_samples_subset_equals_rows():
    s = SMALL[1]
    inp = wl.make_inputs(s)
    full = oracle.forward(s, inp)
    np.testing.assert_array_equal(oracle.forward(s, inp, samples=[1]), full[1:2])


def test_oracle_threads_do_not_change_results():
    s = SMALL[2]
    inp = wl.make_inputs(s)
    n0 = oracle.num_threads()
    a = oracle.forward(s, inp)
    oracle.set_num_threads(1)
    try:
        c = oracle.forward(s, inp)
    finally:
        oracle.set_num_threads(n0)
    np.testing.assert_array_equal(a, c)


def test_workload_shapes():
    # Output-size formulas for the five workloads.
    shapes = []
    for s in wl.WORKLOADS:
        k = s["k"]
        if s["conv"] == "conv3d":
            sp = [s["D"] - k + 1, s["H"] - k + 1, s["W"] - k + 1]
        elif s["conv"] == "conv2d":
            sp = [s["H"] - k + 1, s["W"] - k + 1]
        else:
            sp = [s["H"] + k - 1, s["W"] + k - 1]
        if s["red"] == "mean_spatial":
            shapes.append((s["N"], s["C_out"]))
        elif s["red"] == "maxpool2_x2":
            shapes.append((s["N"], s["C_out"], *[(L // 2) // 2 for L in sp]))
        else:
            shapes.append((s["N"], s["C_out"], *sp))
    assert shapes == [(2, 16), (512, 16), (32, 128, 126, 126), (128, 16, 3, 7, 7),
                      (32, 64, 258, 258)]
