"""GPU parity of the tensor-core Conv3d -> activation -> norm -> mean path
(k_conv3d_tc_mean: split-TF32 implicit GEMM on tcgen05, positions x (channel,
kx tap)) against the fp64 oracle.

The shapes cover what its planner and epilogue vary: both filter sizes
(k = 3: a zero-padded hi*hi pair; k = 4), 1 to 4 input channels (the unused
channels of the 4-channel operand are zero), 16 and 32 output channels (4
or 2 output planes per MMA group), rows that divide a 32-lane quadrant and
rows that cross one (the shared kx halo), 1 to 21 row bands per plane,
partial plane groups, one group per sample and several (the per-sample
ticket merge), every norm and activation, no bias.  Each case first checks
that the plan really runs the tensor-core kernel.  Tolerance: |gpu - ref| <=
1e-4 + 1e-4 |ref|, the fp32 bound of the fused forward.
"""
import numpy as np
import pytest

import oracle
from convolution_normalization_gb300 import workloads as wl
from convolution_normalization_gb300 import binding as B

from _gpu_common import assert_parity, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def no_small_kernel(monkeypatch):
    # these shapes are small enough for the one-CTA-per-group kernel; keep
    # them on the tensor-core kernel this file tests
    monkeypatch.setenv("CN_NO_SMALL", "1")

BASE = wl.WORKLOAD_BY_NAME["conv3d_hswish_gn4_mean_n2"]

TC_MEAN_CASES = [
    dict(N=2, D=8, H=16, W=16, k=3),                                    # the n2 workload shape
    dict(N=3, D=16, H=32, W=32, k=4),                                   # the n512 geometry
    dict(N=2, D=6, H=20, W=20, k=4, C_in=1),                            # quadrant halo, 3 bands
    dict(N=2, D=5, H=9, W=12, k=3, C_in=2, act="gelu_erf"),            # partial plane group
    dict(N=1, D=7, H=40, W=36, k=3, C_in=4, norm="instance", affine=1),  # 13 bands
    dict(N=2, D=4, H=4, W=4, k=4),                                      # 1x1x1 output
    dict(N=1, D=3, H=44, W=44, k=3, C_in=1, norm="none", affine=0, act="none"),  # 21 bands
    dict(N=5, D=11, H=12, W=8, k=3, num_groups=1, post_scale=0.25),      # 3 plane groups
    dict(N=2, D=6, H=10, W=28, k=4, has_bias=0, num_groups=2),
    dict(N=1, D=5, H=8, W=64, k=3, act="hardswish", num_groups=16),     # rows wider than a quadrant
    dict(N=2, D=7, H=12, W=16, k=4, C_out=32, num_groups=8),            # 32 channels, 2 planes a group
    dict(N=2, D=6, H=10, W=32, k=3, C_in=2, C_out=32, norm="instance", affine=1),
]


def uses_tc(spec):
    with B.Plan(spec) as p:
        return "k_conv3d_tc_mean" in p.info()["kernel_names"]


@pytest.mark.parametrize("kw", TC_MEAN_CASES, ids=[str(i) for i in range(len(TC_MEAN_CASES))])
def test_tc_mean_shapes(kw):
    s = wl.with_overrides(BASE, seed=700, **kw)
    assert uses_tc(s), s
    inp = wl.make_inputs(s)
    assert_parity(run_gpu(s, inp), oracle.forward(s, inp), s["name"])


def test_tc_mean_large_magnitude_inputs():
    # No activation or norm: the output is the spatial mean of the conv,
    # linear in x.  With x scaled by 1e3 the mean is a sum of terms far
    # larger than itself, so the fp32 bound is relative to the product
    # magnitudes (the same forward on |x| and |w|): 2^-16 of it holds for a
    # correct fp32 conv over K = 81 terms, not for plain TF32 (~2^-11).
    s = wl.with_overrides(BASE, N=2, D=6, H=12, W=16, act="none", norm="none", affine=0,
                          seed=701)
    assert uses_tc(s)
    inp = wl.make_inputs(s)
    inp["x"] = (inp["x"] * np.float32(1000.0)).astype(np.float32)
    ref = oracle.forward(s, inp)
    mag_in = dict(inp, x=np.abs(inp["x"]), w=np.abs(inp["w"]), b=np.zeros_like(inp["b"]))
    mag = oracle.forward(s, mag_in)
    gpu = run_gpu(s, inp).astype(np.float64)
    err = np.abs(gpu - ref)
    bound = 1e-4 + 1e-4 * np.abs(ref) + 2.0 ** -16 * mag
    assert np.all(err <= bound), float(np.max(err / bound))
    assert float(np.median(mag)) > 1e3


def test_tc_mean_and_cuda_core_paths_agree_with_oracle(monkeypatch):
    s = wl.with_overrides(BASE, N=3, D=12, H=32, W=32, k=4, seed=702)
    inp = wl.make_inputs(s)
    ref = oracle.forward(s, inp)
    assert uses_tc(s)
    assert_parity(run_gpu(s, inp), ref, "tensor cores")
    monkeypatch.setenv("CN_NO_TC", "1")
    assert not uses_tc(s)
    assert_parity(run_gpu(s, inp), ref, "CUDA cores")


def test_tc_mean_repeat_is_bitwise_deterministic():
    # fixed-order sums everywhere: two forwards give identical bits, also
    # with more items than CTAs (the work counter and tickets reset)
    s = wl.with_overrides(BASE, N=100, D=10, H=16, W=16, k=3, seed=703)  # 200 items
    assert uses_tc(s)
    inp = wl.make_inputs(s)
    with B.Plan(s) as p:
        a = run_gpu(s, inp, plan=p)
        b = run_gpu(s, inp, plan=p)
    assert np.array_equal(a, b)
    assert_parity(a, oracle.forward(s, inp), s["name"])
