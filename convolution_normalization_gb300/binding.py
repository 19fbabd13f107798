"""Thin ctypes binding of the conv_norm C ABI (include/conv_norm.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libconv_norm.so``.  Function names match the C entry points.
Tensors are passed as raw pointers; PyTorch tensors (``.data_ptr()``) or
plain integers are accepted, and streams as ``torch.cuda.Stream`` objects,
raw ``cudaStream_t`` integers or None (legacy default stream).

If the shared library has not been built, importing this module raises
ImportError: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# CONV_NORM_LIB=checked loads the bounds-checked build (libconv_norm_checked.so,
# ``build(checked=True)``) instead of the normal one
LIB_PATH = os.path.join(_HERE, "libconv_norm_checked.so"
                        if os.environ.get("CONV_NORM_LIB") == "checked" else "libconv_norm.so")

CN_OK = 0
CN_ERR_INVALID_ARG = -1
CN_ERR_UNSUPPORTED = -2
CN_ERR_CUDA = -3
CN_ERR_TIMEOUT = -4
CN_ERR_DEVICE_CHECK = -5
CN_ERR_ALLOC = -6

CN_CONV3D, CN_CONV2D, CN_CONVT2D = 0, 1, 2
CN_ACT_NONE, CN_ACT_HARDSWISH, CN_ACT_GELU_ERF, CN_ACT_SOFTMAX_C = 0, 1, 2, 3
CN_NORM_NONE, CN_NORM_GROUP, CN_NORM_INSTANCE = 0, 1, 2
CN_RED_NONE, CN_RED_MEAN_SPATIAL, CN_RED_MAXPOOL2_X2 = 0, 1, 2

_CONV = {"conv3d": CN_CONV3D, "conv2d": CN_CONV2D, "convt2d": CN_CONVT2D}
_ACT = {"none": CN_ACT_NONE, "hardswish": CN_ACT_HARDSWISH, "gelu_erf": CN_ACT_GELU_ERF,
        "softmax_c": CN_ACT_SOFTMAX_C}
_NORM = {"none": CN_NORM_NONE, "group": CN_NORM_GROUP, "instance": CN_NORM_INSTANCE}
_RED = {"none": CN_RED_NONE, "mean_spatial": CN_RED_MEAN_SPATIAL,
        "maxpool2_x2": CN_RED_MAXPOOL2_X2}


class conv_norm_desc(ctypes.Structure):
    _fields_ = [("conv", ctypes.c_int), ("N", ctypes.c_int), ("C_in", ctypes.c_int),
                ("C_out", ctypes.c_int), ("D", ctypes.c_int), ("H", ctypes.c_int),
                ("W", ctypes.c_int), ("k", ctypes.c_int), ("groups", ctypes.c_int),
                ("has_bias", ctypes.c_int), ("act", ctypes.c_int), ("norm", ctypes.c_int),
                ("num_groups", ctypes.c_int), ("affine", ctypes.c_int),
                ("eps", ctypes.c_float), ("post_scale", ctypes.c_float), ("red", ctypes.c_int)]


class conv_norm_info(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("launches_per_forward", ctypes.c_int),
                ("kernel_names", ctypes.c_char_p), ("out_numel", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_size_t), ("grid_ctas", ctypes.c_int),
                ("threads_per_cta", ctypes.c_int), ("smem_bytes_per_cta", ctypes.c_int)]


# Every symbol include/conv_norm.h declares (checked by the ABI test).
EXPORTED = ("conv_norm_desc_validate", "conv_norm_output_shape", "conv_norm_status_string",
            "conv_norm_plan_create", "conv_norm_plan_destroy", "conv_norm_workspace_bytes",
            "conv_norm_plan_info", "conv_norm_forward", "conv_norm_forward_host",
            "conv_norm_plan_check_device", "conv_norm_forward_noalloc",
            "conv_norm_plan_set_launch_events", "conv_norm_plan_set_wait_limit",
            "conv_norm_plan_inject_stall", "conv_norm_bwd_plan_create", "conv_norm_backward",
            "conv_norm_bwd_workspace_bytes", "conv_norm_bwd_check_device",
            "conv_norm_bwd_plan_destroy")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"conv_norm CUDA library not built ({LIB_PATH} missing); run "
            "`python -m convolution_normalization_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, pd = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(conv_norm_desc)
    lib.conv_norm_desc_validate.argtypes = [pd]
    lib.conv_norm_desc_validate.restype = i
    lib.conv_norm_output_shape.argtypes = [pd, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(i)]
    lib.conv_norm_output_shape.restype = i
    lib.conv_norm_status_string.argtypes = [i]
    lib.conv_norm_status_string.restype = ctypes.c_char_p
    lib.conv_norm_plan_create.argtypes = [pd, ctypes.POINTER(vp)]
    lib.conv_norm_plan_create.restype = i
    lib.conv_norm_plan_destroy.argtypes = [vp]
    lib.conv_norm_plan_destroy.restype = None
    lib.conv_norm_workspace_bytes.argtypes = [vp]
    lib.conv_norm_workspace_bytes.restype = ctypes.c_size_t
    lib.conv_norm_plan_info.argtypes = [vp, ctypes.POINTER(conv_norm_info)]
    lib.conv_norm_plan_info.restype = i
    fwd = [vp, vp, vp, vp, vp, vp, vp, vp]
    lib.conv_norm_forward.argtypes = fwd
    lib.conv_norm_forward.restype = i
    lib.conv_norm_forward_host.argtypes = fwd
    lib.conv_norm_forward_host.restype = i
    lib.conv_norm_plan_check_device.argtypes = [vp, vp]
    lib.conv_norm_plan_check_device.restype = i
    lib.conv_norm_forward_noalloc.argtypes = [pd] + fwd[1:]
    lib.conv_norm_forward_noalloc.restype = i
    lib.conv_norm_plan_set_launch_events.argtypes = [vp, ctypes.POINTER(vp), i]
    lib.conv_norm_plan_set_launch_events.restype = i
    lib.conv_norm_plan_set_wait_limit.argtypes = [vp, ctypes.c_uint64]
    lib.conv_norm_plan_set_wait_limit.restype = i
    lib.conv_norm_plan_inject_stall.argtypes = [vp]
    lib.conv_norm_plan_inject_stall.restype = i
    lib.conv_norm_bwd_plan_create.argtypes = [pd, ctypes.POINTER(vp)]
    lib.conv_norm_bwd_plan_create.restype = i
    lib.conv_norm_backward.argtypes = [vp] * 13
    lib.conv_norm_backward.restype = i
    lib.conv_norm_bwd_workspace_bytes.argtypes = [vp]
    lib.conv_norm_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.conv_norm_bwd_check_device.argtypes = [vp, vp]
    lib.conv_norm_bwd_check_device.restype = i
    lib.conv_norm_bwd_plan_destroy.argtypes = [vp]
    lib.conv_norm_bwd_plan_destroy.restype = None
    return lib


lib = _load()


class ConvNormError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {conv_norm_status_string(status)} ({status})")


def _check(status, what):
    if status != CN_OK:
        raise ConvNormError(status, what)
    return status


def make_desc(spec=None, **kw) -> conv_norm_desc:
    """Builds a descriptor from a workload dict (string enums) and/or fields."""
    f = dict(spec or {})
    f.update(kw)
    d = conv_norm_desc()
    d.conv = _CONV[f["conv"]] if isinstance(f["conv"], str) else int(f["conv"])
    for k in ("N", "C_in", "C_out", "H", "W", "k"):
        setattr(d, k, int(f[k]))
    d.D = int(f.get("D", 1))
    d.groups = int(f.get("groups", 1))
    d.has_bias = int(f.get("has_bias", 1))
    a = f.get("act", "none")
    d.act = _ACT[a] if isinstance(a, str) else int(a)
    n = f.get("norm", "none")
    d.norm = _NORM[n] if isinstance(n, str) else int(n)
    d.num_groups = int(f.get("num_groups", 0))
    d.affine = int(f.get("affine", 0))
    d.eps = float(f.get("eps", 1e-5))
    d.post_scale = float(f.get("post_scale", 1.0))
    r = f.get("red", "none")
    d.red = _RED[r] if isinstance(r, str) else int(r)
    return d


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    if hasattr(t, "ctypes"):  # numpy
        return t.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(t)}")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ---- C entry points ----------------------------------------------------------

def conv_norm_status_string(status: int) -> str:
    return lib.conv_norm_status_string(int(status)).decode()


def conv_norm_desc_validate(desc: conv_norm_desc) -> int:
    return lib.conv_norm_desc_validate(ctypes.byref(desc))


def conv_norm_output_shape(desc: conv_norm_desc):
    dims = (ctypes.c_int64 * 5)()
    nd = ctypes.c_int(0)
    _check(lib.conv_norm_output_shape(ctypes.byref(desc), dims, ctypes.byref(nd)),
           "conv_norm_output_shape")
    return tuple(int(dims[i]) for i in range(nd.value))


def conv_norm_plan_create(desc: conv_norm_desc) -> int:
    h = ctypes.c_void_p()
    _check(lib.conv_norm_plan_create(ctypes.byref(desc), ctypes.byref(h)), "conv_norm_plan_create")
    return h.value


def conv_norm_plan_destroy(plan: int) -> None:
    lib.conv_norm_plan_destroy(plan)


def conv_norm_workspace_bytes(plan: int) -> int:
    return int(lib.conv_norm_workspace_bytes(plan))


def conv_norm_plan_info(plan: int) -> dict:
    info = conv_norm_info()
    _check(lib.conv_norm_plan_info(plan, ctypes.byref(info)), "conv_norm_plan_info")
    return {k: (getattr(info, k).decode() if k == "kernel_names" and getattr(info, k) else
                getattr(info, k)) for k, _ in info._fields_}


def conv_norm_forward(plan, x, w, b, gamma, beta, out, stream=None) -> int:
    return _check(lib.conv_norm_forward(plan, _ptr(x), _ptr(w), _ptr(b), _ptr(gamma), _ptr(beta),
                                        _ptr(out), _stream(stream)), "conv_norm_forward")


def conv_norm_forward_host(plan, x, w, b, gamma, beta, out, stream=None) -> int:
    return _check(lib.conv_norm_forward_host(plan, _ptr(x), _ptr(w), _ptr(b), _ptr(gamma),
                                             _ptr(beta), _ptr(out), _stream(stream)),
                  "conv_norm_forward_host")


def conv_norm_forward_noalloc(desc, x, w, b, gamma, beta, out, stream=None) -> int:
    """Forward without a plan or any allocation (spatial-mean problems only):
    for callers that cannot call cudaMalloc; see include/conv_norm.h."""
    return _check(lib.conv_norm_forward_noalloc(ctypes.byref(desc), _ptr(x), _ptr(w), _ptr(b),
                                                _ptr(gamma), _ptr(beta), _ptr(out),
                                                _stream(stream)), "conv_norm_forward_noalloc")


def conv_norm_plan_check_device(plan, stream=None) -> int:
    return lib.conv_norm_plan_check_device(plan, _stream(stream))


def conv_norm_plan_set_wait_limit(plan, ns) -> int:
    """Status of setting the tensor-core kernel's progress-wait limit (ns)."""
    return lib.conv_norm_plan_set_wait_limit(plan, int(ns))


def conv_norm_plan_inject_stall(plan) -> int:
    """Status of arming the one-shot stall of the plan's next forward."""
    return lib.conv_norm_plan_inject_stall(plan)


def conv_norm_plan_set_launch_events(plan, events) -> int:
    """events: launches_per_forward + 1 torch.cuda.Event objects (already
    recorded once, so the CUDA events exist), or None/[] to stop."""
    if not events:
        return _check(lib.conv_norm_plan_set_launch_events(plan, None, 0),
                      "conv_norm_plan_set_launch_events")
    arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    return _check(lib.conv_norm_plan_set_launch_events(plan, arr, len(events)),
                  "conv_norm_plan_set_launch_events")


def conv_norm_bwd_plan_create(desc: conv_norm_desc) -> int:
    h = ctypes.c_void_p()
    _check(lib.conv_norm_bwd_plan_create(ctypes.byref(desc), ctypes.byref(h)), "conv_norm_bwd_plan_create")
    return h.value


def conv_norm_bwd_plan_destroy(plan: int) -> None:
    lib.conv_norm_bwd_plan_destroy(plan)


def conv_norm_bwd_workspace_bytes(plan: int) -> int:
    return int(lib.conv_norm_bwd_workspace_bytes(plan))


def conv_norm_backward(plan, x, w, b, gamma, beta, dout, dx, dw, db, dgamma, dbeta, stream=None) -> int:
    return _check(lib.conv_norm_backward(plan, _ptr(x), _ptr(w), _ptr(b), _ptr(gamma), _ptr(beta),
                                         _ptr(dout), _ptr(dx), _ptr(dw), _ptr(db), _ptr(dgamma),
                                         _ptr(dbeta), _stream(stream)), "conv_norm_backward")


def conv_norm_bwd_check_device(plan, stream=None) -> int:
    return lib.conv_norm_bwd_check_device(plan, _stream(stream))


class Plan:
    """Owns one conv_norm plan; a convenience wrapper over the C calls."""

    def __init__(self, spec=None, **kw):
        self.desc = make_desc(spec, **kw)
        self.handle = conv_norm_plan_create(self.desc)
        self.out_shape = conv_norm_output_shape(self.desc)

    def info(self):
        return conv_norm_plan_info(self.handle)

    def forward(self, x, w, b, gamma, beta, out, stream=None):
        return conv_norm_forward(self.handle, x, w, b, gamma, beta, out, stream)

    def forward_host(self, x, w, b, gamma, beta, out, stream=None):
        return conv_norm_forward_host(self.handle, x, w, b, gamma, beta, out, stream)

    def check_device(self, stream=None):
        return conv_norm_plan_check_device(self.handle, stream)

    def set_launch_events(self, events):
        return conv_norm_plan_set_launch_events(self.handle, events)

    def set_wait_limit(self, ns):
        """Limit (ns) of the tensor-core kernel's progress waits; returns the status."""
        return conv_norm_plan_set_wait_limit(self.handle, ns)

    def inject_stall(self):
        """The next forward stalls one CTA on purpose (failure-path test hook)."""
        return conv_norm_plan_inject_stall(self.handle)

    def close(self):
        if self.handle:
            conv_norm_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


class BwdPlan:
    """Owns one backward plan (full-output 2-D blocks); a convenience wrapper."""

    def __init__(self, spec=None, **kw):
        self.desc = make_desc(spec, **kw)
        self.handle = conv_norm_bwd_plan_create(self.desc)

    def backward(self, x, w, b, gamma, beta, dout, dx, dw, db, dgamma, dbeta, stream=None):
        return conv_norm_backward(self.handle, x, w, b, gamma, beta, dout, dx, dw, db, dgamma, dbeta, stream)

    def check_device(self, stream=None):
        return conv_norm_bwd_check_device(self.handle, stream)

    def workspace_bytes(self):
        return conv_norm_bwd_workspace_bytes(self.handle)

    def close(self):
        if self.handle:
            conv_norm_bwd_plan_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
