"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare with the fp64 oracle element by element.

Tolerance (fp32 arithmetic vs an fp64 reference): |gpu - ref| <= 1e-4 +
1e-4 * |ref| per element, the bound the fused forward is specified to meet.
"""
import numpy as np
import torch

from convolution_normalization_gb300 import binding as B

ATOL = 1e-4
RTOL = 1e-4


def to_dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_gpu(spec, inp, stream=None, plan=None, out=None):
    own = plan is None
    if own:
        plan = B.Plan(spec)
    dev = {k: to_dev(v) for k, v in inp.items()}
    if out is None:
        out = torch.full(plan.out_shape, float("nan"), dtype=torch.float32, device="cuda")
    plan.forward(dev["x"], dev["w"], dev["b"], dev["gamma"], dev["beta"], out, stream)
    torch.cuda.synchronize()
    assert plan.check_device() == B.CN_OK
    res = out.cpu().numpy()
    if own:
        plan.close()
    return res


def assert_parity(gpu, ref, what=""):
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    gpu64 = gpu.astype(np.float64)
    err = np.abs(gpu64 - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = ~(err <= bound)  # also catches NaN
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} outside |err| <= {ATOL} + {RTOL}|ref|; "
            f"worst at {idx}: gpu={gpu64[idx]!r} ref={ref[idx]!r} err={err[idx]:.3e}; "
            f"max err {np.nanmax(err):.3e}")
    return float(err.max()) if err.size else 0.0
