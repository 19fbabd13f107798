"""GPU parity on the method's numerical edge cases, for every kernel family.

The statistics of GroupNorm / InstanceNorm are where an fp32 implementation
can lose accuracy without any bug in the conv: a one-pass variance E[y^2] -
E[y]^2 (or sums about a shift far from the data) cancels when a plane's
mean is many standard deviations from zero; near-constant planes make eps
dominate the variance; the channel softmax must survive large logits; and
the 4x4x4 max must return the right value when a window holds exact ties.

Cases (each on the tensor-core kernel and on the CUDA-core kernel of the
same problem, the plan's kernel list is checked first):
  * inputs with a large DC offset, x * s + o: the conv output of channel c
    then sits at about o * sum(w_c) with a spread of s * |w_c|, i.e. mean /
    std ratios of 30 to several thousand;
  * near-constant planes (x * 1e-3: variance far below eps) and exactly
    constant ones (x = 0: every plane is its bias);
  * softmax logits x 50 (channel spreads of ~100: exp underflows for all but
    the largest channels);
  * pooling windows full of exact ties (constant x; x and w quantised so
    that many conv outputs are bitwise equal);
  * (spatial mean) groups whose channels share one large DC level, so the
    group statistics must resolve a small spread under a large mean.

Tolerance: |gpu - ref| <= 1e-4 + 1e-4 |ref| per element, the bound of the
fused forward, with the fp64 oracle on the same inputs as reference.

An input offset also makes the conv itself ill-conditioned: an fp32 conv
output carries an absolute rounding error of about 2^-24 * o * sum|w| times
a growth factor of up to sqrt(C_in k^2), which normalization divides by the
plane's standard deviation.  For InstanceNorm of the 64 -> 128 Conv2d at
x + 100, an fp32 conv that accumulates its 576 products in order, followed
by exact (fp64) statistics, already reaches 1.9x the bound (max error
2.0e-4; 0.58x at x + 30), and at x * 0.01 + 50 even PyTorch's fp32 CPU conv
is 30x over it.  So the InstanceNorm cases use x + 30 and x * 0.1 + 5
(mean / std of about 50); GroupNorm, whose groups mix channels with
different offsets, is also tested at x + 100 and x * 0.01 + 50.
"""
import numpy as np
import pytest

import oracle
from convolution_normalization_gb300 import binding as B
from convolution_normalization_gb300 import workloads as wl

from _gpu_common import assert_parity, run_gpu

pytestmark = pytest.mark.gpu

W = wl.WORKLOAD_BY_NAME


def kernels(spec):
    with B.Plan(spec) as p:
        return p.info()["kernel_names"]


def affine_input(inp, scale, offset):
    out = dict(inp)
    out["x"] = (inp["x"] * np.float32(scale) + np.float32(offset)).astype(np.float32)
    return out


def check(spec, inp, kernel, what, monkeypatch=None, cuda_cores=False):
    if cuda_cores:
        monkeypatch.setenv("CN_NO_TC", "1")
    names = kernels(spec)
    assert kernel in names, (kernel, names)
    assert_parity(run_gpu(spec, inp), oracle.forward(spec, inp), what)


# ---- problems and the kernel each path runs ----------------------------------

MEAN = wl.with_overrides(W["conv3d_hswish_gn4_mean_n512"], N=4, seed=900)
MEAN_IN = wl.with_overrides(MEAN, norm="instance", act="gelu_erf", seed=901)
CONV2D = wl.with_overrides(W["conv2d_in_half_n32"], N=2, seed=902)
CONV2D_GN = wl.with_overrides(W["conv2d_in_half_n32"], N=2, C_in=16, C_out=32, H=40, W=44,
                              norm="group", num_groups=4, affine=1, act="hardswish", seed=903)
CONVT = wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=2, H=64, W=64, seed=904)
CONVT_G1 = wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=2, C_in=16, C_out=16, H=40,
                             W=40, groups=1, num_groups=2, seed=905)
CONV3D_FULL = wl.with_overrides(W["conv3d_hswish_gn4_mean_n2"], N=2, D=10, H=20, W=24,
                                red="none", seed=906)
POOL = wl.with_overrides(W["conv3d_softmax_pool2x2_n128"], N=2, seed=907)
POOL_CC = wl.with_overrides(W["conv3d_softmax_pool2x2_n128"], N=3, D=11, H=13, W=14, seed=908)

# (spec, kernel on the default path, kernel with CN_NO_TC=1)
NORM_PATHS = {
    "mean_gn": (MEAN, "k_conv3d_tc_mean", "k_conv3d_act_mean"),
    "mean_in": (MEAN_IN, "k_conv3d_tc_mean", "k_conv3d_act_mean"),
    "conv2d_in": (CONV2D, "k_conv2d_tc", "k_conv2d_act_stats"),
    "conv2d_gn": (CONV2D_GN, "k_conv2d_act_stats", "k_conv2d_act_stats"),
    "convt_g8": (CONVT, "k_convt2d_tc", "k_conv2d_act_stats"),
    "convt_g1": (CONVT_G1, "k_conv2d_act_stats", "k_conv2d_act_stats"),
    "conv3d_full": (CONV3D_FULL, "k_conv2d_act_stats", "k_conv2d_act_stats"),
}

# (path, x scale, x offset).  InstanceNorm paths: offsets an fp32 conv can
# meet the bound on (module docstring); GroupNorm paths: x + 100 and
# x * 0.01 + 50 as well.
OFFSET_CASES = [
    ("mean_gn", 1.0, 100.0), ("mean_gn", 0.01, 50.0), ("mean_in", 1.0, 100.0),
    ("mean_in", 0.01, 50.0),
    ("conv2d_in", 1.0, 30.0), ("conv2d_in", 0.1, 5.0),
    ("conv2d_gn", 1.0, 100.0), ("conv2d_gn", 0.01, 50.0),
    ("convt_g8", 1.0, 100.0), ("convt_g8", 0.01, 50.0),
    ("convt_g1", 1.0, 100.0), ("convt_g1", 0.01, 50.0),
    ("conv3d_full", 1.0, 30.0), ("conv3d_full", 0.01, 50.0),
]


@pytest.mark.parametrize("cuda_cores", [False, True], ids=["default", "cuda_cores"])
@pytest.mark.parametrize("path,scale,offset", OFFSET_CASES,
                         ids=[f"{p}_x{s:g}+{o:g}" for p, s, o in OFFSET_CASES])
def test_norm_large_dc_offset(path, scale, offset, cuda_cores, monkeypatch):
    spec, k_tc, k_cc = NORM_PATHS[path]
    inp = affine_input(wl.make_inputs(spec), scale, offset)
    check(spec, inp, k_cc if cuda_cores else k_tc, f"{path} x*{scale}+{offset}",
          monkeypatch, cuda_cores)


# Channels of a group that share one large DC level and differ by little:
# filters equal within each group up to +-1e-3 perturbations, x + offset.
# The group's variance is then mostly within-channel and (m_c - mu_g) * rstd
# is O(1), so the statistics must resolve a spread some 300x below the
# channels' common mean: sums about a fixed shift far from the data (such as
# act(bias)) lose that to cancellation, sums about a value of the data do
# not.  The spatial-mean kernels, GroupNorm(4) of 16 channels, no activation
# (so no group is clipped to a constant).
SHARED_DC = wl.with_overrides(MEAN, act="none", seed=910)
SHARED_DC_SMALL = wl.with_overrides(W["conv3d_hswish_gn4_mean_n2"], act="none", seed=911)


def shared_dc_input(spec, offset):
    inp = dict(wl.make_inputs(spec))
    w = inp["w"]
    cpg = spec["C_out"] // spec["num_groups"]
    rng = np.random.default_rng(912)
    base = np.repeat(w[::cpg], cpg, axis=0)
    inp["w"] = (base + rng.uniform(-1e-3, 1e-3, size=w.shape)).astype(np.float32)
    inp["x"] = (inp["x"] + np.float32(offset)).astype(np.float32)
    return inp


@pytest.mark.parametrize("offset", [100.0, 300.0])
@pytest.mark.parametrize("kernel", ["k_conv3d_tc_mean", "k_conv3d_act_mean", "k_conv3d_mean_small"])
def test_mean_group_with_shared_dc_level(kernel, offset, monkeypatch):
    spec = SHARED_DC_SMALL if kernel == "k_conv3d_mean_small" else SHARED_DC
    if kernel == "k_conv3d_act_mean":
        monkeypatch.setenv("CN_NO_TC", "1")
    inp = shared_dc_input(spec, offset)
    ref = oracle.forward(spec, inp)
    # the case is the intended one: outputs of order one, not all beta
    assert float(np.max(np.abs(ref - np.repeat(inp["beta"][None, :], spec["N"], axis=0)))) > 0.3
    check(spec, inp, kernel, f"{kernel} shared DC x+{offset:g}")


@pytest.mark.parametrize("cuda_cores", [False, True], ids=["default", "cuda_cores"])
@pytest.mark.parametrize("path", sorted(NORM_PATHS))
def test_norm_near_constant_planes(path, cuda_cores, monkeypatch):
    # x * 1e-3: each plane's variance (~3e-7 before the activation) is far
    # below eps = 1e-5, so eps sets the scale of the normalized output
    spec, k_tc, k_cc = NORM_PATHS[path]
    inp = affine_input(wl.make_inputs(spec), 1e-3, 0.0)
    check(spec, inp, k_cc if cuda_cores else k_tc, f"{path} x*1e-3", monkeypatch, cuda_cores)


@pytest.mark.parametrize("cuda_cores", [False, True], ids=["default", "cuda_cores"])
@pytest.mark.parametrize("path", sorted(NORM_PATHS))
def test_norm_constant_planes(path, cuda_cores, monkeypatch):
    # x = 0: every conv output plane equals its bias, variance exactly 0
    # per channel (InstanceNorm gives beta, GroupNorm the bias spread of the
    # group's channels)
    spec, k_tc, k_cc = NORM_PATHS[path]
    inp = affine_input(wl.make_inputs(spec), 0.0, 0.0)
    check(spec, inp, k_cc if cuda_cores else k_tc, f"{path} x=0", monkeypatch, cuda_cores)


POOL_PATHS = {"tc": (POOL, "k_conv3d_tc_pool"), "cuda_cores": (POOL_CC, "k_conv3d_softmax_pool4")}


@pytest.mark.parametrize("path", sorted(POOL_PATHS))
def test_softmax_large_logits(path):
    # conv outputs x 50: channel logits spread over ~100, so exp(v - max)
    # underflows to 0 for most channels and the max channel's value is ~1
    spec, kern = POOL_PATHS[path]
    inp = affine_input(wl.make_inputs(spec), 50.0, 0.0)
    check(spec, inp, kern, f"pool {path} x*50")


@pytest.mark.parametrize("path", sorted(POOL_PATHS))
def test_pool_windows_of_constant_input(path):
    # constant x: every position of a channel has the same softmax value,
    # so every pooling window is 64 exact ties
    spec, kern = POOL_PATHS[path]
    inp = affine_input(wl.make_inputs(spec), 0.0, 0.5)
    check(spec, inp, kern, f"pool {path} constant x")


@pytest.mark.parametrize("path", sorted(POOL_PATHS))
def test_pool_windows_with_quantised_ties(path):
    # x in {-1, 0, 1} and w, b multiples of 1/8: conv outputs are exact
    # small multiples of 1/8, so many positions of a window tie bit for bit
    spec, kern = POOL_PATHS[path]
    inp = dict(wl.make_inputs(spec))
    rng = np.random.default_rng(909)
    inp["x"] = rng.integers(-1, 2, size=inp["x"].shape).astype(np.float32)
    inp["w"] = (rng.integers(-2, 3, size=inp["w"].shape) / 8.0).astype(np.float32)
    inp["b"] = (rng.integers(-2, 3, size=inp["b"].shape) / 8.0).astype(np.float32)
    check(spec, inp, kern, f"pool {path} quantised ties")
