"""Host-side checks of the C ABI (no GPU needed): the shared library loads,
exports every function include/conv_norm.h declares, and the host-only
queries validate descriptors and compute output shapes."""
import ctypes
import os
import re

import pytest

from convolution_normalization_gb300 import build as cn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    cn_build.build()
    from convolution_normalization_gb300 import binding
    return binding


def header_functions():
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(conv_norm_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(B):
    declared = header_functions()
    assert "conv_norm_forward" in declared and "conv_norm_plan_create" in declared
    lib = ctypes.CDLL(B.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(B.EXPORTED) >= declared


def test_struct_layout_matches_header(B):
    # 15 ints + 2 floats, no padding
    assert ctypes.sizeof(B.conv_norm_desc) == 17 * 4


WORKLOAD_SHAPES = [(2, 16), (512, 16), (32, 128, 126, 126), (128, 16, 3, 7, 7), (32, 64, 258, 258)]


def test_workloads_validate_and_shapes(B):
    from convolution_normalization_gb300 import workloads as wl
    for s, shp in zip(wl.WORKLOADS, WORKLOAD_SHAPES):
        d = B.make_desc(s)
        assert B.conv_norm_desc_validate(d) == B.CN_OK, s["name"]
        assert B.conv_norm_output_shape(d) == shp


def _base(**kw):
    f = dict(conv="conv2d", N=2, C_in=8, C_out=16, D=1, H=10, W=12, k=3, groups=1, has_bias=1,
             act="none", norm="instance", num_groups=0, affine=0, eps=1e-5, post_scale=1.0,
             red="none")
    f.update(kw)
    return f


@pytest.mark.parametrize("kw,status", [
    (dict(), 0),
    (dict(C_in=7, groups=2), -1),            # C_in % groups
    (dict(H=2), -1),                          # kernel larger than input
    (dict(norm="group", num_groups=3), -1),   # C_out % num_groups
    (dict(eps=0.0), -1),
    (dict(eps=float("nan")), -1),
    (dict(D=3), -1),                          # 2-D conv needs D = 1
    (dict(red="maxpool2_x2"), -1),            # pooling is 3-D only
    (dict(N=-1), -1),
    (dict(k=0), -1),
    (dict(act="softmax_c"), -2),              # no full-output softmax kernel
    (dict(C_out=10), -2),                     # channel slices of 4 or 8
    (dict(conv="conv3d", D=6, red="mean_spatial", groups=2, C_in=8), -2),
    (dict(conv="conv3d", D=6), 0),            # Conv3d with the full output
    (dict(conv="conv3d", D=6, groups=2, C_in=8), -2),
    (dict(conv="conv3d", D=6, act="softmax_c"), -2),
    (dict(N=0), 0),                           # empty batch is valid
    (dict(conv="conv3d", D=9, act="softmax_c", norm="none", red="maxpool2_x2"), 0),
    (dict(conv="conv3d", D=9, act="softmax_c", norm="none", red="maxpool2_x2", post_scale=0.5), 0),
    # a post scale <= 0 does not commute with the max: no kernel
    (dict(conv="conv3d", D=9, act="softmax_c", norm="none", red="maxpool2_x2", post_scale=-1.0), -2),
    (dict(conv="conv3d", D=9, act="softmax_c", norm="none", red="maxpool2_x2", post_scale=0.0), -2),
])
def test_descriptor_validation(B, kw, status):
    d = B.make_desc(_base(**kw))
    assert B.conv_norm_desc_validate(d) == status


def test_output_shapes(B):
    assert B.conv_norm_output_shape(B.make_desc(_base())) == (2, 16, 8, 10)
    assert B.conv_norm_output_shape(B.make_desc(_base(conv="convt2d"))) == (2, 16, 12, 14)
    d = B.make_desc(_base(conv="conv3d", D=9, act="softmax_c", norm="none", red="maxpool2_x2"))
    assert B.conv_norm_output_shape(d) == (2, 16, 1, 2, 2)  # floor(floor(L/2)/2)
    assert B.conv_norm_output_shape(B.make_desc(_base(conv="conv3d", D=6))) == (2, 16, 4, 8, 10)
    d = B.make_desc(_base(conv="conv3d", D=5, act="softmax_c", norm="none", red="maxpool2_x2"))
    assert B.conv_norm_output_shape(d) == (2, 16, 0, 2, 2)


def test_status_strings(B):
    for s in range(-6, 1):
        assert B.conv_norm_status_string(s)
    assert B.conv_norm_status_string(-99) == "unknown status"


def test_null_arguments_rejected(B):
    assert B.lib.conv_norm_desc_validate(None) == B.CN_ERR_INVALID_ARG
    assert B.lib.conv_norm_plan_create(None, None) == B.CN_ERR_INVALID_ARG
    assert B.lib.conv_norm_forward(None, None, None, None, None, None, None, None) == B.CN_ERR_INVALID_ARG
    assert B.lib.conv_norm_plan_info(None, None) == B.CN_ERR_INVALID_ARG
    assert B.lib.conv_norm_workspace_bytes(None) == 0
    B.lib.conv_norm_plan_destroy(None)


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "convolution_normalization_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "liboracle" not in src, f


def _declarations_with_comments():
    """(function name, the comment block right before its declaration)."""
    out = {}
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        for m in re.finditer(r"/\*((?:(?!\*/).)*)\*/\s*(?:[\w\s\*]+?)\b(conv_norm_\w+)\s*\(",
                             src, flags=re.S):
            out[m.group(2)] = m.group(1)
    return out


def test_boundary_calls_cite_their_passage():
    # the four calls of the boundary each say which passage of the problem
    # pages they follow (or that none does); every other call is documented
    docs = _declarations_with_comments()
    assert set(docs) == header_functions()
    for name in ("conv_norm_plan_create", "conv_norm_forward", "conv_norm_workspace_bytes",
                 "conv_norm_plan_destroy"):
        assert "Cites:" in docs[name], name
        assert re.search(r"l2_p\d+|no page passage", docs[name]), name
    for name, doc in docs.items():
        assert len(doc.split()) >= 8, name
