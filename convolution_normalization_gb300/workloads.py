"""Seeded synthetic workloads for the fused conv + norm forward.

This module only describes problem shapes and draws seeded random inputs.
It holds none of the method's arithmetic, so both the CUDA path and the
fp64 oracle can take their inputs from it without sharing any computation.

Each workload is a plain dict whose string-valued fields name the
convolution, activation, normalization and reduction.  Shapes follow the
four problem statements in the source transcripts:

* l2_p27 "Conv3d -> HardSwish -> GroupNorm -> mean": Conv3d(3->16) with
  GroupNorm(4 groups) and a mean over D, H, W.
* l2_p17 "Conv2d -> InstanceNorm2d -> divide": Conv2d(64->128, k=3) with
  InstanceNorm (no affine) and a division by 2 (stated here as x0.5).
* l2_p6 "Conv3d -> Softmax -> MaxPool3d -> MaxPool3d": Conv3d(3->16, k=3),
  channel softmax and two 2x2x2 max pools.
* l2_p19 "ConvTranspose2d -> GELU -> GroupNorm": transposed conv 64->64,
  k=3, stride 1, groups=8, exact GELU and GroupNorm(8).

Batch sizes and spatial sizes are the five benchmark configurations; the
transcripts' own batch sizes (1024/128/128/128) are larger.

Input recipe (same for every workload): one numpy PCG64 generator seeded
with the workload seed draws, in this order, x ~ N(0,1); the conv weight
and then the bias ~ U(-a, a) with a = 1/sqrt(fan_in); gamma = 1 + 0.1*N(0,1);
beta = 0.1*N(0,1).  gamma/beta are drawn only when the norm is affine.
fan_in follows PyTorch's default initialisation: weight.size(1) * prod(k),
i.e. (C_in/groups)*k^d for a convolution and (C_out/groups)*k^2 for a
transposed convolution.
"""
from __future__ import annotations

import math

import numpy as np

# Field names match the C descriptor in include/conv_norm.h; enum-like
# fields are strings here.
CONV_KINDS = ("conv3d", "conv2d", "convt2d")
ACTS = ("none", "hardswish", "gelu_erf", "softmax_c")
NORMS = ("none", "group", "instance")
REDS = ("none", "mean_spatial", "maxpool2_x2")


def spec(conv, N, C_in, C_out, D, H, W, k, groups=1, has_bias=1, act="none",
         norm="none", num_groups=0, affine=0, eps=1e-5, post_scale=1.0,
         red="none", seed=0, name=None):
    assert conv in CONV_KINDS and act in ACTS and norm in NORMS and red in REDS
    if conv != "conv3d":
        D = 1
    return dict(conv=conv, N=N, C_in=C_in, C_out=C_out, D=D, H=H, W=W, k=k,
                groups=groups, has_bias=has_bias, act=act, norm=norm,
                num_groups=num_groups, affine=affine, eps=eps,
                post_scale=post_scale, red=red, seed=seed,
                name=name or f"{conv}_{act}_{norm}_{red}")


# The five benchmark workloads, in order.
WORKLOADS = [
    spec("conv3d", 2, 3, 16, 8, 16, 16, 3, act="hardswish", norm="group",
         num_groups=4, affine=1, red="mean_spatial", seed=0,
         name="conv3d_hswish_gn4_mean_n2"),
    spec("conv3d", 512, 3, 16, 16, 32, 32, 4, act="hardswish", norm="group",
         num_groups=4, affine=1, red="mean_spatial", seed=1,
         name="conv3d_hswish_gn4_mean_n512"),
    spec("conv2d", 32, 64, 128, 1, 128, 128, 3, norm="instance", affine=0,
         post_scale=0.5, seed=2, name="conv2d_in_half_n32"),
    spec("conv3d", 128, 3, 16, 16, 32, 32, 3, act="softmax_c",
         red="maxpool2_x2", seed=3, name="conv3d_softmax_pool2x2_n128"),
    spec("convt2d", 32, 64, 64, 1, 256, 256, 3, groups=8, act="gelu_erf",
         norm="group", num_groups=8, affine=1, seed=4,
         name="convt2d_g8_gelu_gn8_n32"),
]
WORKLOAD_BY_NAME = {w["name"]: w for w in WORKLOADS}


def with_overrides(base, **kw):
    """Copy of a workload dict with some fields replaced (e.g. a smaller N)."""
    out = dict(base)
    out.update(kw)
    if "name" not in kw:
        out["name"] = base["name"] + "_" + "_".join(f"{k}{v}" for k, v in kw.items())
    return out


def input_shapes(s):
    """Shapes of x, w, b, gamma, beta (None where the tensor is not used)."""
    k, G = s["k"], s["groups"]
    if s["conv"] == "conv3d":
        x = (s["N"], s["C_in"], s["D"], s["H"], s["W"])
        w = (s["C_out"], s["C_in"] // G, k, k, k)
    elif s["conv"] == "conv2d":
        x = (s["N"], s["C_in"], s["H"], s["W"])
        w = (s["C_out"], s["C_in"] // G, k, k)
    else:  # transposed: PyTorch stores (C_in, C_out/groups, kH, kW)
        x = (s["N"], s["C_in"], s["H"], s["W"])
        w = (s["C_in"], s["C_out"] // G, k, k)
    b = (s["C_out"],) if s["has_bias"] else None
    aff = s["norm"] != "none" and s["affine"]
    g = (s["C_out"],) if aff else None
    return dict(x=x, w=w, b=b, gamma=g, beta=g)


def make_inputs(s, seed=None):
    """Draw the seeded fp32 inputs of one workload (host numpy arrays)."""
    rng = np.random.Generator(np.random.PCG64(s["seed"] if seed is None else seed))
    shp = input_shapes(s)
    fan_in = shp["w"][1] * int(np.prod(shp["w"][2:]))
    a = 1.0 / math.sqrt(fan_in)
    out = {}
    out["x"] = rng.standard_normal(shp["x"], dtype=np.float32)
    out["w"] = rng.uniform(-a, a, size=shp["w"]).astype(np.float32)
    out["b"] = (rng.uniform(-a, a, size=shp["b"]).astype(np.float32)
                if shp["b"] else None)
    if shp["gamma"]:
        out["gamma"] = (1.0 + 0.1 * rng.standard_normal(shp["gamma"])).astype(np.float32)
        out["beta"] = (0.1 * rng.standard_normal(shp["beta"])).astype(np.float32)
    else:
        out["gamma"] = None
        out["beta"] = None
    return out
