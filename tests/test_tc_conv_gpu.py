"""GPU parity of the tensor-core conv path (k_conv2d_tc: split-TF32 implicit
GEMM on tcgen05) against the fp64 oracle.

The shapes cover what the tile planner varies: output rows per tile
(1, 2, 4, 6, 8), MMA widths below 256 positions, every filter size the path
takes (1, 2, 3: one padded, two paired and mixed tap layouts), two output
channel blocks, ragged last row tiles, the widest row (W = 256), and each
activation / normalization epilogue.  Each case first checks that the plan
really runs the tensor-core kernel.  Tolerance: |gpu - ref| <= 1e-4 +
1e-4 |ref|, the fp32 bound of the fused forward.
"""
import os

import numpy as np
import pytest

import oracle
from convolution_normalization_gb300 import workloads as wl
from convolution_normalization_gb300 import binding as B

from _gpu_common import assert_parity, run_gpu

pytestmark = pytest.mark.gpu

BASE = wl.WORKLOAD_BY_NAME["conv2d_in_half_n32"]

TC_CASES = [
    dict(N=2, C_in=64, C_out=128, H=40, W=128),                       # 2 rows per tile
    dict(N=2, C_in=8, C_out=128, H=33, W=64),                         # 4 rows, ragged last tile
    dict(N=3, C_in=4, C_out=256, H=10, W=32, act="hardswish", norm="group", num_groups=8,
         affine=1),                                                   # 8 rows, 2 channel blocks
    dict(N=2, C_in=12, C_out=128, H=9, W=8, act="gelu_erf", norm="none", post_scale=1.0),
    dict(N=2, C_in=16, C_out=128, H=20, W=128, k=1),                  # 1 tap (padded pair)
    dict(N=2, C_in=8, C_out=128, H=17, W=96, k=2),                    # 4 taps, N = 192
    dict(N=1, C_in=4, C_out=128, H=6, W=256, act="gelu_erf"),          # 1 row per tile
    dict(N=2, C_in=32, C_out=128, H=35, W=36, norm="group", num_groups=1, affine=1,
         post_scale=2.0),
]


def uses_tc(spec):
    with B.Plan(spec) as p:
        return "k_conv2d_tc" in p.info()["kernel_names"]


@pytest.mark.parametrize("kw", TC_CASES, ids=[str(i) for i in range(len(TC_CASES))])
def test_tc_shapes(kw):
    s = wl.with_overrides(BASE, seed=500, **kw)
    assert uses_tc(s), s
    inp = wl.make_inputs(s)
    gpu = run_gpu(s, inp)
    assert_parity(gpu, oracle.forward(s, inp), s["name"])


def test_tc_large_magnitude_inputs():
    # x scaled by 1e3, no normalization: outputs of order 1 arise from sums of
    # terms of order 1e3, so no fp32 conv meets 1e-4 relative to the output.
    # The fp32 bound is relative to the product magnitudes, sum |w||x|
    # (computed by the oracle as the conv of |x| with |w|): a correct fp32
    # conv over K = 576 terms stays well inside 2^-16 of it, while dropping a
    # split term (plain TF32, error ~2^-11 of it) does not.
    s = wl.with_overrides(BASE, N=2, H=20, W=64, norm="none", post_scale=1.0, seed=501)
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
    # and the scale of the check: plain TF32 would be ~2^-11 * mag off
    assert float(np.median(mag)) > 1e3


def test_tc_and_cuda_core_paths_agree_with_oracle(monkeypatch):
    s = wl.with_overrides(BASE, N=2, H=24, seed=502)
    inp = wl.make_inputs(s)
    ref = oracle.forward(s, inp)
    assert uses_tc(s)
    assert_parity(run_gpu(s, inp), ref, "tensor cores")
    monkeypatch.setenv("CN_NO_TC", "1")
    assert not uses_tc(s)
    assert_parity(run_gpu(s, inp), ref, "CUDA cores")


@pytest.mark.parametrize("order", ["larger_first", "smaller_first"])
def test_plans_of_one_kernel_with_different_shared_memory_coexist(order):
    # Two live plans of k_conv2d_tc whose launches need different dynamic
    # shared memory: creating the second must not lower the kernel's limit
    # below what the first plan's launches need.
    a = wl.with_overrides(BASE, N=1, C_in=64, C_out=128, H=24, W=128, seed=740)   # 2 rows a tile
    b = wl.with_overrides(BASE, N=1, C_in=128, C_out=128, H=12, W=132, seed=741)  # 1 row a tile
    smem = {}
    for s in (a, b):
        with B.Plan(s) as p:
            info = p.info()
            assert "k_conv2d_tc" in info["kernel_names"]
            smem[s["name"]] = info["smem_bytes_per_cta"]
    assert smem[a["name"]] != smem[b["name"]]
    big, small = (a, b) if smem[a["name"]] > smem[b["name"]] else (b, a)
    first, second = (big, small) if order == "larger_first" else (small, big)
    with B.Plan(first) as p1, B.Plan(second) as p2:
        for s, p in ((first, p1), (second, p2), (first, p1)):
            inp = wl.make_inputs(s)
            assert_parity(run_gpu(s, inp, plan=p), oracle.forward(s, inp), s["name"])
