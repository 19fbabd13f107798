"""GPU tests of the failure path of the tensor-core kernels, in the form that
faults, traps and hangs nothing: a wait on a barrier phase that nothing
completes runs out.

conv_norm_plan_inject_stall makes the plan's next forward leave the first
input copy of CTA 0 unissued.  Every wait of that CTA is bounded, so with a
short wait limit (conv_norm_plan_set_wait_limit, 2 ms here) the CTA gives
up: it records CN_ERR_TIMEOUT, stops all its roles, waits for its own
copies and MMAs in flight, frees its tensor memory and exits, while the
other CTAs finish their work.  conv_norm_plan_check_device then reports the
timeout and clears the plan's tickets and counters, and the next forward on
the same plan must match the oracle again.  One case per tensor-core kernel
family (Conv3d -> mean, Conv3d -> softmax -> pool, Conv2d, grouped
ConvTranspose2d).
"""
import numpy as np
import pytest
import torch

import oracle
from convolution_normalization_gb300 import binding as B
from convolution_normalization_gb300 import workloads as wl

from _gpu_common import assert_parity, to_dev

pytestmark = pytest.mark.gpu

W = wl.WORKLOAD_BY_NAME
CASES = {
    "k_conv3d_tc_mean": wl.with_overrides(W["conv3d_hswish_gn4_mean_n512"], N=64, seed=1100),
    "k_conv3d_tc_pool": wl.with_overrides(W["conv3d_softmax_pool2x2_n128"], N=32, seed=1101),
    "k_conv2d_tc": wl.with_overrides(W["conv2d_in_half_n32"], N=2, seed=1102),
    "k_convt2d_tc": wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=2, H=128, W=128, seed=1103),
}
DEFAULT_LIMIT_NS = 200_000_000


@pytest.mark.parametrize("kernel", sorted(CASES))
def test_stalled_cta_times_out_and_the_plan_recovers(kernel):
    spec = CASES[kernel]
    inp = wl.make_inputs(spec)
    dev = {k: to_dev(v) for k, v in inp.items()}
    ref = oracle.forward(spec, inp)
    with B.Plan(spec) as p:
        assert kernel in p.info()["kernel_names"]
        out = torch.full(p.out_shape, float("nan"), dtype=torch.float32, device="cuda")

        def forward():
            out.fill_(float("nan"))
            p.forward(dev["x"], dev["w"], dev["b"], dev["gamma"], dev["beta"], out)
            torch.cuda.synchronize()

        assert p.set_wait_limit(2_000_000) == B.CN_OK
        assert p.inject_stall() == B.CN_OK
        forward()  # returns: the stalled CTA gave up, nothing hangs
        assert p.check_device() == B.CN_ERR_TIMEOUT
        assert p.check_device() == B.CN_OK  # the flag was cleared
        # the same plan, default limit: a normal forward again
        assert p.set_wait_limit(DEFAULT_LIMIT_NS) == B.CN_OK
        forward()
        assert p.check_device() == B.CN_OK
        assert_parity(out.cpu().numpy(), ref, f"{kernel} after a timeout")
        # the stall is one-shot, and a limit far below the default (20 ms)
        # does not trip a normal forward of this size
        assert p.set_wait_limit(20_000_000) == B.CN_OK
        forward()
        assert p.check_device() == B.CN_OK
        assert_parity(out.cpu().numpy(), ref, f"{kernel} with a 20 ms limit")


def test_hooks_reject_plans_without_a_tensor_core_kernel(monkeypatch):
    monkeypatch.setenv("CN_NO_TC", "1")
    with B.Plan(CASES["k_conv2d_tc"]) as p:
        assert "k_conv2d_tc" not in p.info()["kernel_names"]
        assert p.set_wait_limit(1000) == B.CN_ERR_UNSUPPORTED
        assert p.inject_stall() == B.CN_ERR_UNSUPPORTED
    with B.Plan(CASES["k_convt2d_tc"]) as p:
        assert B.lib.conv_norm_plan_set_wait_limit(p.handle, 0) == B.CN_ERR_INVALID_ARG
    assert B.lib.conv_norm_plan_inject_stall(None) == B.CN_ERR_INVALID_ARG
