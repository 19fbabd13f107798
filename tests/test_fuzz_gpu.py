"""Seeded random problems across the whole supported descriptor space, each
compared element by element with the fp64 oracle.

The fixed-shape suites pin each kernel's geometry; this one draws problems
the way a user might: every conv kind and reduction, random kernel extents,
channel counts, conv groups, normalization groups, activations, affine and
bias choices, eps and post scale, and spatial extents that are rarely
multiples of any tile.  Plan selection then picks whatever kernel fits
(tensor-core, small-batch or CUDA-core), so the cases also cover the
boundaries between kernels.  The draws are seeded: a failure names a case
that reruns identically.

On the CPU: every drawn descriptor is valid and supported (a host-only
query of the library), and the draws cover every conv kind, reduction,
activation and normalization.  On the GPU: each case matches the oracle
within |gpu - ref| <= 1e-4 + 1e-4 |ref|, and the kernels' error flags stay
clear.  A second set of random 2-D blocks goes through the backward, against
the oracle's backward at the backward suite's tolerance.
"""
import numpy as np
import pytest

import oracle
from convolution_normalization_gb300 import binding as B
from convolution_normalization_gb300 import workloads as wl

NCASES = 320
SEED = 20261203


def _divisors(n):
    return [d for d in range(1, n + 1) if n % d == 0]


def draw(rng, i):
    """One random supported problem (a workloads.spec dict).  Every other
    case of a kind takes the shape class of that kind's tensor-core kernel
    (which the plan may still decline for other reasons)."""
    kind = ["mean", "pool", "full3d", "conv2d", "convt2d"][i % 5]
    tc = (i // 5) % 2 == 1
    k = int(rng.integers(1, 5))
    N = int(rng.integers(1, 4))
    has_bias = int(rng.integers(0, 2))
    eps = float(rng.choice([1e-5, 1e-3]))
    post_scale = float(rng.choice([1.0, 0.5, 2.0]))
    acts = ["none", "hardswish", "gelu_erf"]
    if kind == "pool":
        D, H, W = (int(v) for v in rng.integers(k + 3, k + 24, 3))
        if tc:
            k = int(rng.integers(3, 5))
            W = int(rng.choice([8, 16, 32]))
        return wl.spec("conv3d", N, int(rng.integers(1, 5)), 16, max(D, k), max(H, k), max(W, k), k,
                       has_bias=has_bias, act="softmax_c", post_scale=post_scale, red="maxpool2_x2",
                       seed=SEED + i, name=f"fuzz{i}_pool")
    norm = str(rng.choice(["group", "instance", "none"]))
    affine = int(rng.integers(0, 2)) if norm != "none" else 0
    act = str(rng.choice(acts))
    if kind in ("mean", "full3d"):
        C_in = int(rng.integers(1, 6))
        C_out = int(rng.choice([4, 8, 12, 16, 32]))
        lim = 20 if kind == "mean" else 12
        D, H, W = (int(v) for v in rng.integers(k, k + lim, 3))
        if kind == "mean" and tc:
            k = int(rng.integers(3, 5))
            C_in = int(rng.integers(1, 5))
            C_out = int(rng.choice([16, 32]))
            W = int(rng.choice([8, 12, 16, 20, 32, 36, 64]))
            D, H = max(D, k), max(H, k)
        G = int(rng.choice(_divisors(C_out)))
        return wl.spec("conv3d", N, C_in, C_out, D, H, W, k, has_bias=has_bias, act=act, norm=norm,
                       num_groups=G, affine=affine, eps=eps, post_scale=post_scale,
                       red="mean_spatial" if kind == "mean" else "none", seed=SEED + i,
                       name=f"fuzz{i}_{kind}")
    groups = int(rng.choice([1, 2, 4, 8]))
    cin_g = int(rng.choice([1, 2, 3, 4, 8]))
    cout_g = int(rng.choice([4, 8, 12]))
    H, W = (int(v) for v in rng.integers(k, k + 60, 2))
    if rng.integers(0, 2):
        W = int(4 * rng.integers(max(1, (k + 3) // 4), 17))  # 16-byte rows
    if tc and kind == "conv2d":  # the dense tensor-core Conv2d
        k = int(rng.integers(1, 4))
        groups, cin_g, cout_g = 1, int(4 * rng.integers(1, 9)), 128
        H, W = max(H, k), max(W, k)
    if tc and kind == "convt2d":  # the grouped tensor-core transposed conv
        k, cin_g, cout_g = 3, 8, 8
        W = int(4 * rng.integers(1, 17))
    C_in, C_out = groups * cin_g, groups * cout_g
    G = int(rng.choice(_divisors(C_out)))
    return wl.spec(kind, N, C_in, C_out, 1, H, W, k, groups=groups, has_bias=has_bias, act=act,
                   norm=norm, num_groups=G, affine=affine, eps=eps, post_scale=post_scale,
                   seed=SEED + i, name=f"fuzz{i}_{kind}")


CASES = [draw(np.random.default_rng(SEED + i), i) for i in range(NCASES)]


def test_draws_are_supported_and_cover_the_space():
    for s in CASES:
        st = B.conv_norm_desc_validate(B.make_desc(s))
        assert st == B.CN_OK, (s["name"], B.conv_norm_status_string(st))
    seen = lambda f: {s[f] for s in CASES}
    assert seen("conv") == set(wl.CONV_KINDS)
    assert seen("red") == set(wl.REDS)
    assert seen("act") == set(wl.ACTS)
    assert seen("norm") == set(wl.NORMS)
    assert seen("k") == {1, 2, 3, 4}
    assert {s["groups"] for s in CASES if s["conv"] != "conv3d"} >= {1, 2, 4, 8}


@pytest.mark.gpu
@pytest.mark.parametrize("s", CASES, ids=[s["name"] for s in CASES])
def test_fuzz_case_matches_oracle(s):
    from _gpu_common import assert_parity, run_gpu
    inp = wl.make_inputs(s)
    gpu = run_gpu(s, inp)
    ref = oracle.forward(s, inp)
    assert_parity(gpu, ref, s["name"])


# ---- the backward: seeded random 2-D blocks ----------------------------------

NBWD = 80


def draw_bwd(rng, i):
    """One random block the backward takes: Conv2d or grouped ConvTranspose2d
    (input and output channels a group multiples of 4), any activation but
    softmax, any norm.  Every other block is in the shape class of the
    tensor-core gradient kernels (dense Conv2d to 128 output channels from a
    multiple of 16 input channels; 8 channels a group on both sides of a
    transposed conv)."""
    kind = ["conv2d", "convt2d"][i % 2]
    tc = (i // 2) % 2 == 1
    k = int(rng.integers(1, 5))
    groups = int(rng.choice([1, 2, 4, 8]))
    cin_g, cout_g = int(rng.choice([4, 8, 12, 16])), int(rng.choice([4, 8, 12]))
    if tc and kind == "conv2d":
        k, groups, cin_g, cout_g = int(rng.integers(1, 4)), 1, int(16 * rng.integers(1, 3)), 128
    if tc and kind == "convt2d":
        k, cin_g, cout_g = int(rng.integers(1, 4)), 8, 8
    H, W = (int(v) for v in rng.integers(k, k + 24, 2))
    norm = str(rng.choice(["group", "instance", "none"]))
    C_out = groups * cout_g
    return wl.spec(kind, int(rng.integers(1, 4)), groups * cin_g, C_out, 1, H, W, k, groups=groups,
                   has_bias=int(rng.integers(0, 2)), act=str(rng.choice(["none", "hardswish", "gelu_erf"])),
                   norm=norm, num_groups=int(rng.choice(_divisors(C_out))),
                   affine=int(rng.integers(0, 2)) if norm != "none" else 0,
                   eps=float(rng.choice([1e-5, 1e-3])), post_scale=float(rng.choice([1.0, 0.5, 2.0])),
                   seed=SEED + 1000 + i, name=f"fuzz_bwd{i}_{kind}")


BWD = [draw_bwd(np.random.default_rng(SEED + 1000 + i), i) for i in range(NBWD)]


def test_backward_draws_are_supported_forwards_with_supported_adjoints():
    for s in BWD:
        assert B.conv_norm_desc_validate(B.make_desc(s)) == B.CN_OK, s["name"]
        assert (s["C_in"] // s["groups"]) % 4 == 0, s["name"]
    assert {s["k"] for s in BWD} == {1, 2, 3, 4}
    assert {s["act"] for s in BWD} == {"none", "hardswish", "gelu_erf"}
    assert {s["norm"] for s in BWD} == set(wl.NORMS)


@pytest.mark.gpu
@pytest.mark.parametrize("s", BWD, ids=[s["name"] for s in BWD])
def test_fuzz_backward_matches_oracle(s):
    from test_backward_gpu import assert_grads, case, reference, run_backward
    inp, dout = case(s, 7)
    assert_grads(run_backward(s, inp, dout), reference(s, inp, dout), s["name"])
