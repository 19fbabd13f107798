"""GPU parity of the tensor-core Conv3d -> channel softmax -> 4x4x4 max pool
path (k_conv3d_tc_pool: the split-TF32 implicit GEMM of k_conv3d_tc with
four output planes per MMA, softmax in registers, the window max by shuffles
and shared-memory atomic max) against the fp64 oracle.

The shapes cover what its epilogue varies: rows of 32, 16 and 8 positions
(one, two and four rows per 32-lane quadrant, so the window's rows come from
other quadrants, from both, or from the same warp), both filter sizes, 1 to
4 input channels, extents that are not multiples of 4 (the pool's floor
drops the tail), one pooled voxel per sample, no bias and a post scale.
Each case first checks that the plan really runs the tensor-core kernel.
Tolerance: |gpu - ref| <= 1e-4 + 1e-4 |ref|.
"""
import pytest

import oracle
from convolution_normalization_gb300 import workloads as wl
from convolution_normalization_gb300 import binding as B

from _gpu_common import assert_parity, run_gpu

pytestmark = pytest.mark.gpu

BASE = wl.WORKLOAD_BY_NAME["conv3d_softmax_pool2x2_n128"]

TC_POOL_CASES = [
    dict(N=3, D=16, H=32, W=32, k=3),                                # the n128 geometry
    dict(N=2, D=9, H=12, W=16, k=3, C_in=1),                         # two rows per quadrant
    dict(N=2, D=12, H=14, W=8, k=4, C_in=2),                         # four rows per quadrant
    dict(N=2, D=11, H=19, W=32, k=4, has_bias=0, post_scale=0.5),
    dict(N=5, D=7, H=7, W=8, k=3, C_in=4),                           # 1x1x1 pooled per sample
    dict(N=2, D=8, H=12, W=16, k=3, post_scale=2.0),
]


def uses_tc(spec):
    with B.Plan(spec) as p:
        return "k_conv3d_tc_pool" in p.info()["kernel_names"]


@pytest.mark.parametrize("kw", TC_POOL_CASES, ids=[str(i) for i in range(len(TC_POOL_CASES))])
def test_tc_pool_shapes(kw):
    s = wl.with_overrides(BASE, seed=800, **kw)
    assert uses_tc(s), s
    inp = wl.make_inputs(s)
    assert_parity(run_gpu(s, inp), oracle.forward(s, inp), s["name"])


def test_tc_pool_and_cuda_core_paths_agree_with_oracle(monkeypatch):
    s = wl.with_overrides(BASE, N=4, seed=801)
    inp = wl.make_inputs(s)
    ref = oracle.forward(s, inp)
    assert uses_tc(s)
    assert_parity(run_gpu(s, inp), ref, "tensor cores")
    monkeypatch.setenv("CN_NO_TC", "1")
    assert not uses_tc(s)
    assert_parity(run_gpu(s, inp), ref, "CUDA cores")
