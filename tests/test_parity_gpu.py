"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Cases: the five workloads at full size (every sample), smaller shapes that
span several tiles with ragged tails, every kernel extent, grouped and plain
transposed convs, activation and normalization variants, and edge cases
(empty batch, empty pooled output, minimal spatial extents).  Tolerance: |gpu - ref| <= 1e-4 + 1e-4 |ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from convolution_normalization_gb300 import workloads as wl
from convolution_normalization_gb300 import binding as B

from _gpu_common import assert_parity, run_gpu, to_dev

pytestmark = pytest.mark.gpu

W = {s["name"]: s for s in wl.WORKLOADS}


def check(spec, samples=None):
    inp = wl.make_inputs(spec)
    gpu = run_gpu(spec, inp)
    ref = oracle.forward(spec, inp, samples=samples)
    if samples is not None:
        gpu = gpu[list(samples)]
    return assert_parity(gpu, ref, spec["name"])


# ---- the five workloads at their full sizes ---------------------------------

def test_w1_conv3d_hswish_gn_mean_n2_full():
    check(W["conv3d_hswish_gn4_mean_n2"])


def test_w2_conv3d_hswish_gn_mean_n512_full():
    check(W["conv3d_hswish_gn4_mean_n512"])


def test_w3_conv2d_instnorm_half_n32_full():
    check(W["conv2d_in_half_n32"])


def test_w4_conv3d_softmax_pool_n128_full():
    check(W["conv3d_softmax_pool2x2_n128"])


def test_w5_convt2d_gelu_gn_n32_full():
    check(W["convt2d_g8_gelu_gn8_n32"])


# ---- smaller shapes: several tiles, ragged tails, other extents -----------------

MEAN_CASES = [
    dict(N=3, D=7, H=9, W=10, k=3),                # segmented rows, ragged chunks
    dict(N=2, D=6, H=12, W=33, k=4),               # Wo = 30 -> RW 16 segments
    dict(N=5, D=5, H=5, W=5, k=1),                 # k = 1
    dict(N=2, D=4, H=11, W=13, k=2, C_in=5),
    dict(N=2, D=16, H=32, W=32, k=4),              # the n512 geometry, 2 samples
    dict(N=3, D=4, H=4, W=4, k=4),                 # 1x1x1 output
    dict(N=2, D=9, H=17, W=16, k=3, C_out=32, num_groups=8),
    dict(N=2, D=9, H=17, W=16, k=3, norm="instance", affine=1),
    dict(N=2, D=9, H=17, W=16, k=3, norm="none", affine=0),
    dict(N=2, D=8, H=10, W=12, k=3, act="gelu_erf"),
    dict(N=2, D=8, H=10, W=12, k=3, act="none", post_scale=0.5),
    dict(N=2, D=8, H=10, W=12, k=3, has_bias=0),
]


@pytest.mark.parametrize("small", [True, False], ids=["small_kernel", "persistent_kernels"])
@pytest.mark.parametrize("kw", MEAN_CASES, ids=[str(i) for i in range(len(MEAN_CASES))])
def test_mean_variant_shapes(kw, small, monkeypatch):
    # these batches fit the one-CTA-per-group kernel; CN_NO_SMALL=1 runs them
    # on the persistent (tensor-core or CUDA-core) kernels instead
    if not small:
        monkeypatch.setenv("CN_NO_SMALL", "1")
    check(wl.with_overrides(W["conv3d_hswish_gn4_mean_n2"], seed=100, **kw))


POOL_CASES = [
    dict(N=3, D=9, H=12, W=11, k=3),
    dict(N=2, D=16, H=32, W=32, k=3),
    dict(N=2, D=12, H=14, W=15, k=4, C_in=2),
    dict(N=3, D=8, H=9, W=10, k=1, C_in=4),
    dict(N=2, D=10, H=10, W=10, k=2),
    dict(N=17, D=7, H=7, W=7, k=3),                # 1x1x1 pooled per sample, many CTAs
    dict(N=2, D=9, H=12, W=11, k=3, has_bias=0),
    dict(N=2, D=9, H=12, W=11, k=3, post_scale=0.5),   # the scale applies before the max
]


@pytest.mark.parametrize("kw", POOL_CASES, ids=[str(i) for i in range(len(POOL_CASES))])
def test_pool_variant_shapes(kw):
    check(wl.with_overrides(W["conv3d_softmax_pool2x2_n128"], seed=200, **kw))


FULL_CASES = [
    # conv2d + instance norm
    dict(base="conv2d_in_half_n32", N=2, C_in=16, C_out=32, H=21, W=35),
    dict(base="conv2d_in_half_n32", N=2, C_in=64, C_out=128, H=40, W=128),
    dict(base="conv2d_in_half_n32", N=2, C_in=5, C_out=16, H=9, W=9, k=1),
    dict(base="conv2d_in_half_n32", N=3, C_in=8, C_out=8, H=7, W=20, k=2),
    dict(base="conv2d_in_half_n32", N=2, C_in=6, C_out=16, H=12, W=19, k=4),
    dict(base="conv2d_in_half_n32", N=2, C_in=16, C_out=16, H=20, W=20, post_scale=1.0),
    dict(base="conv2d_in_half_n32", N=2, C_in=16, C_out=32, H=20, W=20, groups=2),
    dict(base="conv2d_in_half_n32", N=2, C_in=16, C_out=16, H=20, W=20, norm="group",
         num_groups=4, affine=1, act="hardswish"),
    dict(base="conv2d_in_half_n32", N=2, C_in=8, C_out=16, H=13, W=14, norm="none"),
    # transposed conv + GroupNorm
    dict(base="convt2d_g8_gelu_gn8_n32", N=2, C_in=64, C_out=64, H=30, W=41),
    dict(base="convt2d_g8_gelu_gn8_n32", N=2, C_in=64, C_out=64, H=64, W=64),
    dict(base="convt2d_g8_gelu_gn8_n32", N=2, C_in=16, C_out=16, H=12, W=20, groups=1,
         num_groups=2),
    dict(base="convt2d_g8_gelu_gn8_n32", N=2, C_in=16, C_out=32, H=9, W=11, groups=2,
         num_groups=4, k=2),
    dict(base="convt2d_g8_gelu_gn8_n32", N=2, C_in=8, C_out=8, H=5, W=6, groups=1,
         num_groups=1, k=4),
    dict(base="convt2d_g8_gelu_gn8_n32", N=2, C_in=8, C_out=16, H=7, W=7, groups=1,
         num_groups=16, k=1),
    dict(base="convt2d_g8_gelu_gn8_n32", N=2, C_in=16, C_out=16, H=10, W=10, groups=2,
         norm="instance", affine=0, act="none"),
    dict(base="convt2d_g8_gelu_gn8_n32", N=1, C_in=8, C_out=8, H=1, W=1, groups=1,
         num_groups=2),  # 1x1 input -> 3x3 output
]


@pytest.mark.parametrize("kw", FULL_CASES, ids=[str(i) for i in range(len(FULL_CASES))])
def test_full_variant_shapes(kw):
    kw = dict(kw)
    base = W[kw.pop("base")]
    check(wl.with_overrides(base, seed=300, **kw))


def test_groups1_convt_full_n4():
    # The l2_p19 page's literal layer passes no groups argument.
    s = wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=2, groups=1, H=64, W=64)
    check(s)


# ---- edge cases --------------------------------------------------------------

def test_empty_batch_writes_nothing():
    s = wl.with_overrides(W["conv3d_hswish_gn4_mean_n2"], N=0)
    with B.Plan(s) as p:
        x = torch.empty((0, 3, 8, 16, 16), device="cuda")
        w = torch.zeros((16, 3, 3, 3, 3), device="cuda")
        v = torch.zeros(16, device="cuda")
        out = torch.empty((0, 16), device="cuda")
        # a zero-size tensor may have a null data pointer: pass a valid one
        dummy = torch.zeros(4, device="cuda")
        assert p.forward(dummy, w, v, v, v, dummy) == 0
        torch.cuda.synchronize()
        assert p.info()["launches_per_forward"] == 0


def test_empty_pooled_output():
    s = wl.with_overrides(W["conv3d_softmax_pool2x2_n128"], N=2, D=5, H=12, W=12)
    inp = wl.make_inputs(s)
    gpu = run_gpu(s, inp)
    assert gpu.shape == (2, 16, 0, 2, 2)


def test_deterministic_bitwise():
    for name in ("conv3d_hswish_gn4_mean_n2", "conv2d_in_half_n32"):
        s = W[name]
        if name == "conv2d_in_half_n32":
            s = wl.with_overrides(s, N=2, H=40, W=50)
        inp = wl.make_inputs(s)
        a = run_gpu(s, inp)
        b = run_gpu(s, inp)
        np.testing.assert_array_equal(a, b)


def test_reused_plan_and_side_stream():
    s = wl.with_overrides(W["convt2d_g8_gelu_gn8_n32"], N=2, H=20, W=20)
    inp = wl.make_inputs(s)
    ref = oracle.forward(s, inp)
    with B.Plan(s) as p:
        st = torch.cuda.Stream()
        for _ in range(3):  # tickets reset between launches
            with torch.cuda.stream(st):
                out = run_gpu(s, inp, stream=st, plan=p)
            assert_parity(out, ref, "side stream")


def test_forward_host_matches():
    s = W["conv3d_hswish_gn4_mean_n2"]
    inp = wl.make_inputs(s)
    ref = oracle.forward(s, inp)
    with B.Plan(s) as p:
        hp = {k: (torch.from_numpy(v).pin_memory() if v is not None else None) for k, v in inp.items()}
        out = torch.empty(p.out_shape, dtype=torch.float32).pin_memory()
        p.forward_host(hp["x"], hp["w"], hp["b"], hp["gamma"], hp["beta"], out)
        assert_parity(out.numpy(), ref, "forward_host")
        # pageable host memory works too
        out2 = np.empty(p.out_shape, dtype=np.float32)
        p.forward_host(inp["x"], inp["w"], inp["b"], inp["gamma"], inp["beta"], out2)
        np.testing.assert_array_equal(out2, out.numpy())


@pytest.mark.parametrize("name,N,chunks", [("conv3d_hswish_gn4_mean_n512", 203, None),
                                           ("conv3d_hswish_gn4_mean_n512", 203, 3),
                                           ("conv3d_hswish_gn4_mean_n512", 203, 8),
                                           ("conv3d_hswish_gn4_mean_n512", 203, 16),
                                           ("convt2d_g8_gelu_gn8_n32", 5, None)])
def test_forward_host_chunked_matches_device_forward(name, N, chunks, monkeypatch):
    # more than 16 MB of input: the host entry point pipelines chunks of whole
    # samples, alternating between two compute streams (203 samples: by
    # default 6 chunks, five of 34 and one of 33; in 3 chunks: 68, 68, 67;
    # in 8: seven of 26 and one of 21; in 16, the most: fifteen of 13 and one
    # of 8; 5 large samples: one per chunk)
    if chunks is not None:
        monkeypatch.setenv("CN_HOST_CHUNKS", str(chunks))
    s = wl.with_overrides(W[name], N=N)
    inp = wl.make_inputs(s)
    dev = {k: to_dev(v) for k, v in inp.items()}
    with B.Plan(s) as p:
        ref = torch.empty(p.out_shape, dtype=torch.float32, device="cuda")
        p.forward(dev["x"], dev["w"], dev["b"], dev["gamma"], dev["beta"], ref)
        torch.cuda.synchronize()
        hp = {k: (torch.from_numpy(v).pin_memory() if v is not None else None) for k, v in inp.items()}
        for _ in range(2):  # the second call reuses the staging set up by the first
            out = torch.full(p.out_shape, float("nan"), dtype=torch.float32).pin_memory()
            p.forward_host(hp["x"], hp["w"], hp["b"], hp["gamma"], hp["beta"], out)
            np.testing.assert_array_equal(out.numpy(), ref.cpu().numpy())
        assert p.check_device() == B.CN_OK  # the chunk plans' error flags too
    last = [0, N - 1]
    assert_parity(out.numpy()[last], oracle.forward(s, inp, samples=last), name + " chunked")


def test_bad_pointers_rejected():
    s = W["conv3d_hswish_gn4_mean_n2"]
    inp = wl.make_inputs(s)
    dev = {k: to_dev(v) for k, v in inp.items()}
    with B.Plan(s) as p:
        out = torch.empty(p.out_shape, device="cuda")
        h = p.handle
        L = B.lib
        args = [dev["x"].data_ptr(), dev["w"].data_ptr(), dev["b"].data_ptr(),
                dev["gamma"].data_ptr(), dev["beta"].data_ptr(), out.data_ptr()]
        assert L.conv_norm_forward(h, *args, None) == B.CN_OK
        bad = list(args)
        bad[0] = None
        assert L.conv_norm_forward(h, *bad, None) == B.CN_ERR_INVALID_ARG
        bad = list(args)
        bad[0] += 4  # misaligned x
        assert L.conv_norm_forward(h, *bad, None) == B.CN_ERR_INVALID_ARG
        bad = list(args)
        bad[2] = None  # has_bias = 1 but no bias
        assert L.conv_norm_forward(h, *bad, None) == B.CN_ERR_INVALID_ARG
        bad = list(args)
        bad[3] = None  # affine but no gamma
        assert L.conv_norm_forward(h, *bad, None) == B.CN_ERR_INVALID_ARG
        torch.cuda.synchronize()


def test_plan_info_reports_kernels():
    for s in wl.WORKLOADS:
        with B.Plan(s) as p:
            info = p.info()
            assert info["launches_per_forward"] >= 1
            assert info["kernel_names"]
            assert info["grid_ctas"] > 0


def test_launch_events_time_each_kernel():
    s = wl.with_overrides(W["conv2d_in_half_n32"], N=2, H=24)
    inp = wl.make_inputs(s)
    dev = {k: to_dev(v) for k, v in inp.items()}
    with B.Plan(s) as p:
        L = p.info()["launches_per_forward"]
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(L + 1)]
        for e in evs:
            e.record()
        torch.cuda.synchronize()
        with pytest.raises(B.ConvNormError):
            p.set_launch_events(evs[:-1])
        p.set_launch_events(evs)
        out = torch.empty(p.out_shape, dtype=torch.float32, device="cuda")
        p.forward(dev["x"], dev["w"], dev["b"], dev["gamma"], dev["beta"], out, None)
        torch.cuda.synchronize()
        d = [evs[i].elapsed_time(evs[i + 1]) for i in range(L)]
        assert all(v > 0 for v in d), d
        p.set_launch_events(None)
        assert_parity(out.cpu().numpy(), oracle.forward(s, inp), s["name"])
