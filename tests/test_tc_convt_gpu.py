"""GPU parity of the tensor-core grouped transposed conv (k_convt2d_tc:
split-TF32 implicit GEMM on tcgen05, 8 input and 8 output channels per
group, k = 3) against the fp64 oracle.

The shapes cover what the kernel's tiling varies: units of 6 output rows x
30 output columns (ragged last bands and segments, outputs narrower than one
unit), tiles of four units that cross sample boundaries and a last tile with
1-3 units, 1 to 16 groups (CTAs split over the groups; several groups per
CTA count when the groups outnumber the SMs' share), every activation and
normalization epilogue (GroupNorm groups equal to, finer or coarser than
the conv groups, InstanceNorm, none with a post scale), no bias, and the
l2_p19 workload itself.  Each case first checks that the plan runs the
tensor-core kernel.  Tolerance: |gpu - ref| <= 1e-4 + 1e-4 |ref|, the fp32
bound of the fused forward.
"""
import numpy as np
import pytest

import oracle
from convolution_normalization_gb300 import binding as B
from convolution_normalization_gb300 import workloads as wl

from _gpu_common import assert_parity, run_gpu

pytestmark = pytest.mark.gpu

BASE = wl.WORKLOAD_BY_NAME["convt2d_g8_gelu_gn8_n32"]


def uses_tct(spec):
    with B.Plan(spec) as p:
        return "k_convt2d_tc" in p.info()["kernel_names"]


TCT_CASES = [
    dict(N=2, H=64, W=64),                                    # 11 bands x 3 segments, GN(8)
    dict(N=1, H=4, W=4),                                      # 6x6 output: one unit per (n, g)
    dict(N=3, H=1, W=4),                                      # 3x6 output: a partial band
    dict(N=2, H=10, W=28),                                    # 12x30: one whole unit
    dict(N=2, H=11, W=32),                                    # 13x34: ragged band and segment
    dict(N=5, H=7, W=60),                                     # 9x62, 10 units a sample (tiles cross n)
    dict(N=1, H=30, W=256),                                   # 258-wide rows: 9 segments
    dict(N=2, H=16, W=40, C_in=16, C_out=16, groups=2, num_groups=2),
    dict(N=2, H=12, W=20, C_in=128, C_out=128, groups=16, num_groups=16),  # 16 groups
    dict(N=2, H=12, W=20, C_in=8, C_out=8, groups=1, num_groups=1),
    dict(N=2, H=20, W=24, act="hardswish", num_groups=4),     # GN coarser than the conv groups
    dict(N=2, H=20, W=24, act="none", norm="instance", affine=0, post_scale=0.5),
    dict(N=2, H=20, W=24, norm="group", num_groups=32),       # GN finer than the conv groups
    dict(N=2, H=14, W=36, norm="none", affine=0, post_scale=2.0),
    dict(N=2, H=14, W=36, norm="none", affine=0),             # conv + GELU only
    dict(N=2, H=14, W=36, has_bias=0),
]


@pytest.mark.parametrize("kw", TCT_CASES, ids=[str(i) for i in range(len(TCT_CASES))])
def test_tct_shapes(kw):
    s = wl.with_overrides(BASE, seed=1000, **kw)
    assert uses_tct(s), s
    inp = wl.make_inputs(s)
    assert_parity(run_gpu(s, inp), oracle.forward(s, inp), s["name"])


def test_tct_large_magnitude_inputs():
    # x scaled by 1e3, no normalization or activation: outputs arise from
    # sums of terms far larger than themselves, so the fp32 bound is
    # relative to the product magnitudes sum |w||x| (the oracle's transposed
    # conv of |x| with |w|); a correct fp32 conv over K = 72 terms stays well
    # inside 2^-16 of it, plain TF32 (~2^-11) does not.
    s = wl.with_overrides(BASE, N=2, H=24, W=32, act="none", norm="none", affine=0, seed=1001)
    assert uses_tct(s)
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


def test_tct_and_cuda_core_paths_agree_with_oracle(monkeypatch):
    s = wl.with_overrides(BASE, N=3, H=40, W=44, seed=1002)
    inp = wl.make_inputs(s)
    ref = oracle.forward(s, inp)
    assert uses_tct(s)
    assert_parity(run_gpu(s, inp), ref, "tensor cores")
    monkeypatch.setenv("CN_NO_TC", "1")
    assert not uses_tct(s)
    assert_parity(run_gpu(s, inp), ref, "CUDA cores")


def test_tct_repeat_is_bitwise_deterministic():
    # fixed-order sums: two forwards on one plan give identical bits, with
    # far more tiles than CTAs (the per-group work counters reset)
    s = wl.with_overrides(BASE, N=6, H=96, W=96, seed=1003)
    assert uses_tct(s)
    inp = wl.make_inputs(s)
    with B.Plan(s) as p:
        a = run_gpu(s, inp, plan=p)
        b = run_gpu(s, inp, plan=p)
    assert np.array_equal(a, b)
    assert_parity(a, oracle.forward(s, inp), s["name"])


def test_tct_plan_reports_three_launches():
    with B.Plan(BASE) as p:
        info = p.info()
    assert info["kernel_names"].startswith("k_convt2d_tc<2>")
    assert info["launches_per_forward"] == 3
    assert info["grid_ctas"] % 8 == 0  # the same CTA count for every group
