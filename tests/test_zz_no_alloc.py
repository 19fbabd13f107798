"""GPU test of conv_norm_forward_noalloc, the forward for callers that cannot
allocate device memory (engine plugins or real-time loops whose memory is
reserved up front by another allocator, where cudaMalloc may fail or
synchronize the device).

The entry point keeps its scratch in a fixed array in the library's device
globals instead of a plan workspace.  Its output must match the regular
plan-based conv_norm_forward within the tolerance the parity tests use,
on two calls in a row (the second call finds the first call's leftovers in
the shared array).  This file is collected last so that a run stopping at
the first failure has already run every other test; it also passes alone
in a fresh process.
"""
import numpy as np
import pytest
import torch

from convolution_normalization_gb300 import binding as B
from convolution_normalization_gb300 import workloads as wl

from _gpu_common import assert_parity, to_dev

pytestmark = pytest.mark.gpu

W = {s["name"]: s for s in wl.WORKLOADS}

CASES = [
    W["conv3d_hswish_gn4_mean_n2"],
    W["conv3d_hswish_gn4_mean_n512"],
    wl.with_overrides(W["conv3d_hswish_gn4_mean_n2"], N=5, D=7, H=9, W=10, seed=11),
    wl.with_overrides(W["conv3d_hswish_gn4_mean_n2"], N=3, D=9, H=17, W=16, norm="instance",
                      act="gelu_erf", seed=12),
]


def _plan_forward(spec, dev):
    with B.Plan(spec) as p:
        out = torch.empty(p.out_shape, dtype=torch.float32, device="cuda")
        p.forward(dev["x"], dev["w"], dev["b"], dev["gamma"], dev["beta"], out)
        torch.cuda.synchronize()
        assert p.check_device() == B.CN_OK
        return out.cpu().numpy()


@pytest.mark.parametrize("spec", CASES, ids=[s["name"] for s in CASES])
def test_noalloc_matches_plan_forward_twice(spec):
    inp = wl.make_inputs(spec)
    dev = {k: to_dev(v) for k, v in inp.items()}
    ref = _plan_forward(spec, dev).astype(np.float64)
    desc = B.make_desc(spec)
    for call in range(2):
        out = torch.full(B.conv_norm_output_shape(desc), float("nan"), dtype=torch.float32,
                         device="cuda")
        B.conv_norm_forward_noalloc(desc, dev["x"], dev["w"], dev["b"], dev["gamma"],
                                    dev["beta"], out)
        torch.cuda.synchronize()
        # no bounded wait gave up (the calls' flag, read with a NULL plan)
        assert B.lib.conv_norm_plan_check_device(None, None) == B.CN_OK
        assert_parity(out.cpu().numpy(), ref, f"{spec['name']} no-alloc call {call + 1}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 4096 samples of the 16x32x32 k=4 problem need about 8.4 MB of scratch (4 MiB is the limit)
    spec = wl.with_overrides(W["conv3d_hswish_gn4_mean_n512"], N=4096)
    desc = B.make_desc(spec)
    dummy = torch.zeros(16, device="cuda")
    st = B.lib.conv_norm_forward_noalloc(B.ctypes.byref(desc), dummy.data_ptr(), dummy.data_ptr(),
                                         dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
                                         dummy.data_ptr(), None)
    assert st == B.CN_ERR_UNSUPPORTED


def test_noalloc_rejects_other_problem_kinds():
    desc = B.make_desc(W["conv2d_in_half_n32"])
    dummy = torch.zeros(16, device="cuda")
    st = B.lib.conv_norm_forward_noalloc(B.ctypes.byref(desc), dummy.data_ptr(), dummy.data_ptr(),
                                         dummy.data_ptr(), None, None, dummy.data_ptr(), None)
    assert st == B.CN_ERR_UNSUPPORTED
