"""The bounds-checked build (-DCN_CHECKS, a stand-in for a memory checker).

Its kernels test the index of every main global store and shared-memory
operand write against the buffer it goes to; a failed test records
CN_ERR_DEVICE_CHECK in the plan's flag and the access is skipped.  On the
CPU: the checked library builds and exports the whole ABI.  On the GPU: the
parity suites pass when they run on it, and since every parity run ends with
conv_norm_plan_check_device == CN_OK, no check tripped on any of their
shapes.
"""
import ctypes
import os
import re
import subprocess
import sys

import pytest

from convolution_normalization_gb300 import build as cn_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PARITY_FILES = ["tests/test_parity_gpu.py", "tests/test_tc_conv_gpu.py", "tests/test_tc_mean_gpu.py",
                "tests/test_tc_pool_gpu.py", "tests/test_tc_convt_gpu.py",
                "tests/test_conv3d_full_gpu.py", "tests/test_numerics_edges_gpu.py",
                "tests/test_backward_gpu.py", "tests/test_fuzz_gpu.py"]


def test_checked_library_builds_and_exports_the_abi():
    path = cn_build.build(checked=True)
    assert path.endswith("libconv_norm_checked.so")
    src = open(os.path.join(ROOT, "include", "conv_norm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    lib = ctypes.CDLL(path)
    for name in set(re.findall(r"\b(conv_norm_\w+)\s*\(", src)):
        assert hasattr(lib, name), name


@pytest.mark.gpu
def test_parity_suites_pass_on_the_checked_build():
    cn_build.build(checked=True)
    env = dict(os.environ, CONV_NORM_LIB="checked")
    probe = subprocess.run([sys.executable, "-c",
                            "from convolution_normalization_gb300 import binding as B; print(B.LIB_PATH)"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0 and probe.stdout.strip().endswith("libconv_norm_checked.so"), probe
    r = subprocess.run([sys.executable, "-m", "pytest", *PARITY_FILES, "-m", "gpu", "-q", "-x",
                        "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
