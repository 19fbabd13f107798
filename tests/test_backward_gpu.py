"""GPU parity of the backward pass (conv_norm_backward: Conv2d or grouped
ConvTranspose2d -> activation -> GroupNorm / InstanceNorm / none -> post
scale) against the fp64 oracle's backward, through the C ABI.

Cases: the l2_p17 block (Conv2d 64 -> 128, InstanceNorm, x0.5) and the l2_p19
block (ConvTranspose2d 64 -> 64, groups 8, GELU, GroupNorm(8)) at their full
spatial sizes with two samples, and small shapes over every activation and
norm, grouped and plain convs, affine or not, bias or not.  dout is a seeded
N(0, 1) tensor.

Tolerance, per gradient tensor g against the oracle's r:
  |g - r| <= 1e-4 (|r| + rms(r)) + 1e-6 m,
the forward's relative bound with, added, a floor at the tensor's own scale
and one at the magnitude m of the sum each element is: every gradient sums
many products of both signs (dw over every sample and position), so elements
near zero carry the rounding error of terms far larger than themselves (db
under InstanceNorm without an activation is exactly zero).  m is the same
gradient taken from absolute values: the adjoint conv of |dA| with |w| for
dx, the correlation of |dA| with |x| for dw, sum |dA| for db (dA the
oracle's gradient at the conv output); 0 for dgamma and dbeta.
"""
import numpy as np
import pytest
import torch

import oracle
from convolution_normalization_gb300 import binding as B
from convolution_normalization_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

W = wl.WORKLOAD_BY_NAME


def run_backward(spec, inp, dout, plan=None):
    dev = {k: (None if v is None else torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).cuda())
           for k, v in inp.items()}
    g = torch.from_numpy(np.ascontiguousarray(dout, dtype=np.float32)).cuda()
    aff = bool(spec["affine"]) and spec["norm"] != "none"
    dx = torch.empty_like(dev["x"])
    dw = torch.empty_like(dev["w"])
    db = torch.empty_like(dev["b"]) if spec["has_bias"] else None
    dgamma = torch.empty(spec["C_out"], device="cuda") if aff else None
    dbeta = torch.empty(spec["C_out"], device="cuda") if aff else None
    own = plan is None
    p = plan or B.BwdPlan(spec)
    try:
        p.backward(dev["x"], dev["w"], dev["b"], dev["gamma"] if aff else None,
                   dev["beta"] if aff else None, g, dx, dw, db, dgamma, dbeta)
        torch.cuda.synchronize()
        assert p.check_device() == B.CN_OK
    finally:
        if own:
            p.close()
    c = lambda t: None if t is None else t.cpu().numpy().astype(np.float64)
    return {"dx": c(dx), "dw": c(dw), "db": c(db), "dgamma": c(dgamma), "dbeta": c(dbeta)}


def magnitudes(spec, inp, dA):
    a, x, w, G = np.abs(dA), np.abs(inp["x"]).astype(np.float64), np.abs(inp["w"]).astype(np.float64), spec["groups"]
    if spec["conv"] == "conv2d":
        mx, (mw, _) = oracle.conv2d_grad_input(a, w, G), oracle.conv2d_grad_weight(x, a, w.shape, G)
    else:
        mx, (mw, _) = oracle.conv_transpose2d_grad_input(a, w, G), oracle.conv_transpose2d_grad_weight(x, a, w.shape, G)
    return {"dx": mx, "dw": mw, "db": a.sum(axis=(0, 2, 3)), "dgamma": 0.0, "dbeta": 0.0}


def reference(spec, inp, dout):
    ref = oracle.backward(spec, inp, dout, intermediates=True)
    ref["mag"] = magnitudes(spec, inp, ref.pop("dA"))
    return ref


def assert_grads(got, ref, what):
    for k in ("dx", "dw", "db", "dgamma", "dbeta"):
        if ref[k] is None:
            assert got[k] is None, (what, k)
            continue
        r, g = ref[k], got[k]
        assert g.shape == r.shape, (what, k)
        rms = float(np.sqrt(np.mean(r * r)))
        err = np.abs(g - r)
        bound = 1e-4 * (np.abs(r) + rms) + 1e-6 * ref["mag"][k]
        bad = int(np.sum(~(err <= bound)))
        assert bad == 0, f"{what} {k}: {bad} of {r.size} outside; max err/bound {float(np.max(err / bound)):.3g}"


def case(spec, seed=0):
    inp = wl.make_inputs(spec)
    out_shape = B.conv_norm_output_shape(B.make_desc(spec))
    dout = np.random.default_rng(1000 + seed).standard_normal(out_shape).astype(np.float32)
    return inp, dout


BWD_CASES = [
    wl.with_overrides(W["conv2d_in_half_n32"], N=2, C_in=8, C_out=8, H=12, W=14, seed=1200),
    wl.with_overrides(W["conv2d_in_half_n32"], N=2, C_in=16, C_out=8, H=10, W=9, groups=2,
                      norm="group", num_groups=4, affine=1, act="hardswish", seed=1201),
    wl.with_overrides(W["conv2d_in_half_n32"], N=3, C_in=8, C_out=16, H=9, W=13, act="gelu_erf",
                      norm="none", affine=0, has_bias=0, post_scale=1.5, seed=1202),
    wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=2, H=20, W=24, seed=1203),
    wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=2, C_in=16, C_out=16, H=10, W=11, groups=1,
                      num_groups=2, act="hardswish", seed=1204),
    wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=2, C_in=16, C_out=16, H=9, W=9, groups=2,
                      norm="instance", affine=0, post_scale=0.5, seed=1205),
    wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=1, C_in=8, C_out=8, H=7, W=7, groups=1,
                      norm="none", affine=0, act="none", seed=1206),
    # dense Conv2d with 128 output channels and 16 k input channels: dw and dx on the tensor cores
    wl.with_overrides(W["conv2d_in_half_n32"], N=2, C_in=16, C_out=128, H=10, W=12, act="gelu_erf",
                      seed=1210),
    wl.with_overrides(W["conv2d_in_half_n32"], N=3, C_in=32, C_out=256, H=7, W=40, k=2, norm="group",
                      num_groups=8, affine=1, seed=1211),
    wl.with_overrides(W["conv2d_in_half_n32"], N=1, C_in=16, C_out=128, H=5, W=36, k=1, has_bias=0,
                      seed=1212),
    # 8 channels a group on both sides with k = 2 and k = 1: the sliding-window dw and dx kernels
    wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=2, C_in=32, C_out=32, H=13, W=16, groups=4, k=2,
                      num_groups=4, seed=1208),
    wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=1, C_in=16, C_out=16, H=9, W=36, groups=2, k=1,
                      act="hardswish", seed=1209),
]


@pytest.mark.parametrize("spec", BWD_CASES, ids=[str(i) for i in range(len(BWD_CASES))])
def test_backward_shapes(spec):
    inp, dout = case(spec)
    assert_grads(run_backward(spec, inp, dout), reference(spec, inp, dout), spec["name"])


@pytest.mark.parametrize("name", ["conv2d_in_half_n32", "convt2d_g8_gelu_gn8_n32"])
def test_backward_page_blocks_full_spatial_size(name):
    spec = wl.with_overrides(W[name], N=2)
    inp, dout = case(spec, 1)
    assert_grads(run_backward(spec, inp, dout), reference(spec, inp, dout), name)


def test_backward_large_dc_offset():
    # GroupNorm of outputs whose mean is far from zero: the statistics and
    # the dy coefficients use shifts taken from the data
    spec = wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=2, H=16, W=16, seed=1207)
    inp, dout = case(spec, 2)
    inp = dict(inp, x=(inp["x"] + np.float32(30.0)).astype(np.float32))
    assert_grads(run_backward(spec, inp, dout), reference(spec, inp, dout), "x + 30")


@pytest.mark.parametrize("idx", [1, 7], ids=["sliding_window", "tensor_cores"])
def test_backward_repeat_is_bitwise_deterministic(idx):
    spec = BWD_CASES[idx]
    inp, dout = case(spec, 3)
    with B.BwdPlan(spec) as p:
        a = run_backward(spec, inp, dout, plan=p)
        b = run_backward(spec, inp, dout, plan=p)
    for k in a:
        if a[k] is not None:
            assert np.array_equal(a[k], b[k]), k


def test_backward_conv2d_tensor_cores_large_dc_offset():
    # the Conv2d block's dx and dw on the tensor cores with inputs far from
    # zero mean: the split-TF32 products keep fp32 accuracy on x + 30
    spec = wl.with_overrides(W["conv2d_in_half_n32"], N=2, C_in=16, C_out=128, H=12, W=16, seed=1213)
    inp, dout = case(spec, 4)
    inp = dict(inp, x=(inp["x"] + np.float32(30.0)).astype(np.float32))
    assert_grads(run_backward(spec, inp, dout), reference(spec, inp, dout), "conv2d x + 30")


def test_backward_argument_checks():
    spec = BWD_CASES[0]  # has bias, no affine
    with B.BwdPlan(spec) as p:
        x = torch.zeros(spec["N"], spec["C_in"], spec["H"], spec["W"], device="cuda")
        w = torch.zeros(spec["C_out"], spec["C_in"], 3, 3, device="cuda")
        b = torch.zeros(spec["C_out"], device="cuda")
        out_shape = B.conv_norm_output_shape(p.desc)
        g = torch.zeros(out_shape, device="cuda")
        dx, dw, db = torch.empty_like(x), torch.empty_like(w), torch.empty_like(b)
        st = B.lib.conv_norm_backward(p.handle, x.data_ptr(), w.data_ptr(), b.data_ptr(), None, None,
                                      g.data_ptr(), dx.data_ptr(), dw.data_ptr(), None, None, None, None)
        assert st == B.CN_ERR_INVALID_ARG  # db missing although the conv has a bias
        st = B.lib.conv_norm_backward(p.handle, x.data_ptr(), w.data_ptr(), b.data_ptr(), None, None,
                                      g.data_ptr(), dx.data_ptr(), dw.data_ptr(), db.data_ptr(),
                                      db.data_ptr(), None, None)
        assert st == B.CN_ERR_INVALID_ARG  # dgamma given without an affine norm
    with pytest.raises(B.ConvNormError) as e:  # spatial-mean blocks have no backward here
        B.BwdPlan(W["conv3d_hswish_gn4_mean_n2"])
    assert e.value.status == B.CN_ERR_UNSUPPORTED
