"""GPU parity of the Conv3d problems with a full output (l2_p27's block
without the spatial mean: Conv3d -> activation -> GroupNorm / InstanceNorm /
none), which run on the 2-D kernel as samples (n, output depth) over
depth-stacked input channels (ci, kd), staged with one 5-D TMA box per stage
(or bulk / cp.async row copies when W is not a multiple of 4).  The oracle
computes the plain 3-D definition.  Tolerance: |gpu - ref| <= 1e-4 +
1e-4 |ref|."""
import pytest

import oracle
from convolution_normalization_gb300 import workloads as wl
from convolution_normalization_gb300 import binding as B

from _gpu_common import assert_parity, run_gpu

pytestmark = pytest.mark.gpu

BASE = wl.WORKLOAD_BY_NAME["conv3d_hswish_gn4_mean_n2"]

CASES = [
    dict(),                                                      # l2_p27 shape, GroupNorm(4)
    dict(N=3, D=10, H=20, W=24, k=4),                            # k = 4
    dict(N=2, D=6, H=12, W=12, k=2, norm="instance", affine=0),
    dict(N=2, D=5, H=9, W=13, act="gelu_erf"),                   # W % 4 != 0: row copies
    dict(N=2, C_in=8, C_out=32, D=7, H=16, W=16, num_groups=8, act="none"),
    dict(N=1, D=4, H=8, W=8, k=1, norm="none", post_scale=0.5),
    dict(N=2, C_in=5, C_out=16, D=6, H=10, W=20, norm="group", num_groups=1),
]


@pytest.mark.parametrize("kw", CASES, ids=[str(i) for i in range(len(CASES))])
def test_conv3d_full_output(kw):
    s = wl.with_overrides(BASE, red="none", seed=800, **kw)
    with B.Plan(s) as p:
        assert "k_conv2d_act_stats" in p.info()["kernel_names"]
    inp = wl.make_inputs(s)
    assert_parity(run_gpu(s, inp), oracle.forward(s, inp), s["name"])


def test_conv3d_full_output_larger_batch_sampled():
    # the n512 shape without the mean, on 16 samples, every output element
    s = wl.with_overrides(wl.WORKLOAD_BY_NAME["conv3d_hswish_gn4_mean_n512"], red="none", N=16,
                          seed=801)
    inp = wl.make_inputs(s)
    assert_parity(run_gpu(s, inp), oracle.forward(s, inp), s["name"])
