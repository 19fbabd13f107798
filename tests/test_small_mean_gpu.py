"""GPU parity of the small-problem Conv3d -> activation -> norm -> mean kernel
(k_conv3d_mean_small: one CTA per (sample, normalization group), the sample
staged in shared memory) against the fp64 oracle.

The cases cover what it varies: every filter size, 1 to 5 input channels,
normalization groups of 1 (InstanceNorm, no norm), 2, 4 and 8 channels,
every activation, post scale, no bias, inputs whose size is not a multiple of
four floats (scalar staging), 1x1x1 outputs, and the l2_p27 workload itself
(2 samples, 8x16x16, k = 3).  Each case checks that the plan runs this
kernel; the edge cases of the statistics (large offsets, near-constant and
constant planes) run on it as well.  Tolerance: |gpu - ref| <= 1e-4 +
1e-4 |ref|.
"""
import numpy as np
import pytest

import oracle
from convolution_normalization_gb300 import binding as B
from convolution_normalization_gb300 import workloads as wl

from _gpu_common import assert_parity, run_gpu

pytestmark = pytest.mark.gpu

BASE = wl.WORKLOAD_BY_NAME["conv3d_hswish_gn4_mean_n2"]


def kernel_of(spec):
    with B.Plan(spec) as p:
        return p.info()["kernel_names"]


SMALL_CASES = [
    dict(),                                                       # the workload
    dict(N=3, D=7, H=9, W=10, k=3, C_in=5),                       # 3150 floats: scalar staging
    dict(N=2, D=5, H=6, W=7, k=1, C_out=8, num_groups=1),         # 8 channels a group
    dict(N=4, D=6, H=8, W=8, k=2, C_in=1, C_out=16, num_groups=8),  # 2 channels a group
    dict(N=2, D=9, H=10, W=12, k=4, C_in=2),
    dict(N=3, D=4, H=4, W=4, k=4),                                # 1x1x1 output
    dict(N=2, D=8, H=10, W=12, k=3, norm="instance"),
    dict(N=2, D=8, H=10, W=12, k=3, norm="none", affine=0, act="none", post_scale=0.5),
    dict(N=2, D=8, H=10, W=12, k=3, act="gelu_erf", has_bias=0),
    dict(N=8, D=8, H=16, W=16, k=3),                              # 32 groups
]


@pytest.mark.parametrize("kw", SMALL_CASES, ids=[str(i) for i in range(len(SMALL_CASES))])
def test_small_mean_shapes(kw):
    s = wl.with_overrides(BASE, seed=1200, **kw) if kw else BASE
    assert kernel_of(s).startswith("k_conv3d_mean_small"), kernel_of(s)
    inp = wl.make_inputs(s)
    assert_parity(run_gpu(s, inp), oracle.forward(s, inp), s["name"])


@pytest.mark.parametrize("scale,offset", [(1.0, 100.0), (0.01, 50.0), (1e-3, 0.0), (0.0, 0.0)])
def test_small_mean_statistics_edge_cases(scale, offset):
    s = wl.with_overrides(BASE, N=2, seed=1201)
    inp = dict(wl.make_inputs(s))
    inp["x"] = (inp["x"] * np.float32(scale) + np.float32(offset)).astype(np.float32)
    assert kernel_of(s).startswith("k_conv3d_mean_small")
    assert_parity(run_gpu(s, inp), oracle.forward(s, inp), f"x*{scale}+{offset}")


def test_small_and_tensor_core_kernels_agree(monkeypatch):
    s = wl.with_overrides(BASE, N=4, seed=1202)
    inp = wl.make_inputs(s)
    ref = oracle.forward(s, inp)
    small = run_gpu(s, inp)
    monkeypatch.setenv("CN_NO_SMALL", "1")
    assert kernel_of(s).startswith("k_conv3d_tc_mean")
    assert_parity(small, ref, "small kernel")
    assert_parity(run_gpu(s, inp), ref, "tensor cores")


def test_small_mean_is_bitwise_deterministic():
    s = wl.with_overrides(BASE, N=8, seed=1203)
    inp = wl.make_inputs(s)
    with B.Plan(s) as p:
        a = run_gpu(s, inp, plan=p)
        b = run_gpu(s, inp, plan=p)
    assert np.array_equal(a, b)
