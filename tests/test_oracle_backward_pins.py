"""Pins of the oracle's backward pass (``oracle.backward``) against facts
that do not come from its own formulas:

* PyTorch float64 autograd through the same model stated with torch.nn.functional
  ops (an independent implementation of every derivative);
* central finite differences of the oracle's forward, L = sum(out * dout),
  at random coordinates of every input (brute force, no derivative formula);
* the adjoint identities of the convolutions: <grad_input(dy), x> = <dy, conv(x)>
  and <grad_weight(x, dy), w> = <dy, conv(x; w)> with no bias;
* GroupNorm's gradient sums to zero over each group (its output does not
  change when the group's inputs shift together);
* HardSwish and GELU derivatives at special points and against finite
  differences of the forward primitives.

These run on the CPU (-m "not gpu").
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from convolution_normalization_gb300 import workloads as wl

W = wl.WORKLOAD_BY_NAME


def t64(a, grad=False):
    t = torch.tensor(np.asarray(a, dtype=np.float64))
    if grad:
        t.requires_grad_(True)
    return t


def torch_grads(s, inp, dout):
    x, w = t64(inp["x"], True), t64(inp["w"], True)
    b = t64(inp["b"], True) if s["has_bias"] else None
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
    ga = be = None
    if s["norm"] != "none":
        G = s["num_groups"] if s["norm"] == "group" else y.shape[1]
        if s["affine"]:
            ga, be = t64(inp["gamma"], True), t64(inp["beta"], True)
        y = F.group_norm(y, G, ga, be, s["eps"])
    y = y * s["post_scale"]
    if s["red"] == "mean_spatial":
        y = y.mean(dim=tuple(range(2, y.dim())))
    (y * t64(dout)).sum().backward()
    g = lambda t: None if t is None else t.grad.numpy()
    return {"dx": g(x), "dw": g(w), "db": g(b), "dgamma": g(ga), "dbeta": g(be)}


CASES = [
    wl.with_overrides(W["conv2d_in_half_n32"], N=2, C_in=8, C_out=6, H=9, W=11, seed=50),
    wl.with_overrides(W["conv2d_in_half_n32"], N=2, C_in=8, C_out=8, H=7, W=8, groups=2,
                      norm="group", num_groups=4, affine=1, act="hardswish", seed=51),
    wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=2, C_in=16, C_out=16, H=6, W=7, seed=52),
    wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=2, C_in=8, C_out=8, H=5, W=6, groups=1,
                      num_groups=2, has_bias=0, post_scale=0.5, seed=53),
    wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=1, C_in=8, C_out=8, H=5, W=5, norm="none",
                      affine=0, act="none", seed=54),
    wl.with_overrides(W["conv3d_hswish_gn4_mean_n2"], N=2, D=6, H=7, W=8, seed=55),
    wl.with_overrides(W["conv3d_hswish_gn4_mean_n2"], N=2, D=6, H=7, W=8, red="none",
                      act="gelu_erf", seed=56),
]


def dout_for(s, inp, seed):
    out = oracle.forward(s, inp)
    return np.random.default_rng(seed).standard_normal(out.shape)


@pytest.mark.parametrize("s", CASES, ids=[str(i) for i in range(len(CASES))])
def test_backward_matches_torch_autograd(s):
    inp = wl.make_inputs(s)
    dout = dout_for(s, inp, 7)
    got = oracle.backward(s, inp, dout)
    ref = torch_grads(s, inp, dout)
    for k in ("dx", "dw", "db", "dgamma", "dbeta"):
        if ref[k] is None:
            assert got[k] is None, k
            continue
        np.testing.assert_allclose(got[k], ref[k], rtol=1e-9, atol=1e-11, err_msg=k)


@pytest.mark.parametrize("s", [CASES[1], CASES[3], CASES[5]], ids=["conv2d_gn", "convt_g1", "conv3d_mean"])
def test_backward_matches_finite_differences(s):
    inp = {k: (None if v is None else np.asarray(v, dtype=np.float64)) for k, v in wl.make_inputs(s).items()}
    dout = dout_for(s, inp, 8)
    got = oracle.backward(s, inp, dout)
    rng = np.random.default_rng(9)

    def loss(inp2):
        return float(np.sum(oracle.forward(s, inp2) * dout))

    names = ["x", "w"] + (["b"] if s["has_bias"] else []) + (
        ["gamma", "beta"] if s["affine"] and s["norm"] != "none" else [])
    for name in names:
        g = got["d" + name]
        for _ in range(4):
            idx = tuple(int(rng.integers(0, n)) for n in inp[name].shape)
            h = 1e-5 * max(1.0, abs(float(inp[name][idx])))
            up = dict(inp)
            dn = dict(inp)
            up[name] = inp[name].copy()
            dn[name] = inp[name].copy()
            up[name][idx] += h
            dn[name][idx] -= h
            fd = (loss(up) - loss(dn)) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


@pytest.mark.parametrize("conv", ["conv3d", "conv2d", "convt2d"])
def test_conv_gradients_are_adjoints(conv):
    rng = np.random.default_rng(10)
    G = 2
    if conv == "conv3d":
        x = rng.standard_normal((2, 4, 5, 6, 7))
        w = rng.standard_normal((6, 2, 2, 3, 2))
        y = oracle.conv3d(x, w, None, G)
        dy = rng.standard_normal(y.shape)
        gi = oracle.conv3d_grad_input(dy, w, G)
        gw, gb = oracle.conv3d_grad_weight(x, dy, w.shape, G)
    elif conv == "conv2d":
        x = rng.standard_normal((2, 4, 6, 7))
        w = rng.standard_normal((6, 2, 3, 2))
        y = oracle.conv2d(x, w, None, G)
        dy = rng.standard_normal(y.shape)
        gi = oracle.conv2d_grad_input(dy, w, G)
        gw, gb = oracle.conv2d_grad_weight(x, dy, w.shape, G)
    else:
        x = rng.standard_normal((2, 4, 5, 6))
        w = rng.standard_normal((4, 3, 3, 3))
        y = oracle.conv_transpose2d(x, w, None, G)
        dy = rng.standard_normal(y.shape)
        gi = oracle.conv_transpose2d_grad_input(dy, w, G)
        gw, gb = oracle.conv_transpose2d_grad_weight(x, dy, w.shape, G)
    lhs = float(np.sum(dy * y))
    assert abs(float(np.sum(gi * x)) - lhs) <= 1e-10 * abs(lhs)  # linear in x
    assert abs(float(np.sum(gw * w)) - lhs) <= 1e-10 * abs(lhs)  # linear in w
    np.testing.assert_allclose(gb, dy.sum(axis=tuple(i for i in range(dy.ndim) if i != 1)), rtol=1e-12)


def test_group_norm_gradient_sums_to_zero_per_group():
    rng = np.random.default_rng(11)
    y = rng.standard_normal((3, 8, 50)) * 2.0 + 5.0
    dout = rng.standard_normal(y.shape)
    gamma = rng.standard_normal(8)
    dy, dgamma, dbeta = oracle.group_norm_grad(y, dout, 4, 1e-5, gamma)
    sums = dy.reshape(3, 4, 2 * 50).sum(axis=2)
    assert np.max(np.abs(sums)) < 1e-10
    np.testing.assert_allclose(dbeta, dout.sum(axis=(0, 2)), rtol=1e-12)


def test_activation_derivatives():
    v = np.array([-5.0, -3.5, -3.0, -1.0, 0.0, 1.0, 3.0, 3.5, 5.0])
    one = np.ones_like(v)
    hs = oracle.hardswish_grad(v, one)
    np.testing.assert_allclose(hs, [0, 0, -0.5, 1 / 6, 0.5, 5 / 6, 1.5, 1, 1], atol=1e-15)
    ge = oracle.gelu_erf_grad(np.array([0.0]), np.array([1.0]))
    assert abs(ge[0] - 0.5) < 1e-15  # Phi(0) + 0
    # both against central differences of the forward primitives (away from the kinks)
    u = np.linspace(-6, 6, 97) + 0.013
    h = 1e-6
    for fwd, grad in ((oracle.hardswish, oracle.hardswish_grad), (oracle.gelu_erf, oracle.gelu_erf_grad)):
        fd = (fwd(u + h) - fwd(u - h)) / (2 * h)
        np.testing.assert_allclose(grad(u, np.ones_like(u)), fd, atol=1e-7)
