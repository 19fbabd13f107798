"""Host-side arithmetic and the CPU reference arm of bench.py (no GPU).

The expected FLOP counts below are worked out by hand from each workload's
definition: outputs of the computed region x 2 x (C_in / groups) x k^d
multiply-adds.  The double max pool (floor mode) needs only the
4*floor(L/4) region; the grouped ConvTranspose2d has 64 / 8 = 8 input
channels per output.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from convolution_normalization_gb300 import workloads as wl  # noqa: E402

EXPECTED_FLOPS = {
    # 2 samples x 16 ch x (6 x 14 x 14) outputs x 2 x 3 x 27
    "conv3d_hswish_gn4_mean_n2": 6_096_384,
    # 512 x 16 x (13 x 29 x 29) x 2 x 3 x 64
    "conv3d_hswish_gn4_mean_n512": 34_392_244_224,
    # 32 x 128 x (126 x 126) x 2 x 64 x 9
    "conv2d_in_half_n32": 74_912_366_592,
    # 128 x 16 x (12 x 28 x 28: the kept part of 14 x 30 x 30) x 2 x 3 x 27
    "conv3d_softmax_pool2x2_n128": 3_121_348_608,
    # 32 x 64 x (258 x 258) x 2 x 8 x 9
    "convt2d_g8_gelu_gn8_n32": 19_630_522_368,
}

EXPECTED_OUT = {
    "conv3d_hswish_gn4_mean_n2": (2, 16),
    "conv3d_hswish_gn4_mean_n512": (512, 16),
    "conv2d_in_half_n32": (32, 128, 126, 126),
    "conv3d_softmax_pool2x2_n128": (128, 16, 3, 7, 7),
    "convt2d_g8_gelu_gn8_n32": (32, 64, 258, 258),
}


@pytest.mark.parametrize("name", sorted(EXPECTED_FLOPS))
def test_algorithmic_flops_and_output_shapes(name):
    s = wl.WORKLOAD_BY_NAME[name]
    assert bench.algorithmic_flops(s) == EXPECTED_FLOPS[name]
    assert tuple(bench.out_shape(s)) == EXPECTED_OUT[name]


def test_step_roofline_picks_the_larger_bound():
    pk = {"fp32_tflops": 80.0, "hbm_gbs": 8000.0}
    s = wl.WORKLOAD_BY_NAME["conv3d_hswish_gn4_mean_n512"]
    ms, bound = bench.roofline_ms(s, pk)
    assert bound == "alu" and ms == pytest.approx(34_392_244_224 / 80e12 * 1e3)
    # the same problem against a very slow memory is bandwidth bound
    ms, bound = bench.roofline_ms(s, {"fp32_tflops": 80.0, "hbm_gbs": 1.0})
    assert bound == "hbm" and ms == pytest.approx(bench.compulsory_bytes(s) / 1e9 * 1e3)
    # x alone is 512 x 3 x 16 x 32 x 32 floats
    assert bench.compulsory_bytes(s) > 4 * 512 * 3 * 16 * 32 * 32


def test_kernel_roofline_units():
    pk = {"fp32_tflops": 80.0, "hbm_gbs": 8000.0, "bf16_tflops": 2250.0, "sm_max_mhz": 2070.0,
          "source": "test", "sms": 152, "sms_source": "test"}
    s = wl.WORKLOAD_BY_NAME["conv3d_hswish_gn4_mean_n512"]
    r = bench.kernel_roofline(s, "k_conv3d_tc_mean<4,16>", 1.0, pk)
    # the method's own work (2 x MACs) against the tf32 peak 2250 x 1.1 / 2.25
    # = 1100; what the split runs on the tensor pipe (three tf32 products per
    # fp32 product) is reported beside it
    assert r["bound"] == "tensor" and r["peak"] == pytest.approx(1100.0)
    assert r["achieved"] == pytest.approx(34_392_244_224 / 1e-3 / 1e12)
    assert r["split_tf32"]["achieved"] == pytest.approx(3 * r["achieved"])
    assert r["frac_of_fp32_peak"] == pytest.approx(r["achieved"] / 80.0)
    s2 = wl.WORKLOAD_BY_NAME["convt2d_g8_gelu_gn8_n32"]
    r = bench.kernel_roofline(s2, "k_norm_apply", 1.0, pk)
    # read + write of the 32 x 64 x 258 x 258 output
    assert r["bound"] == "hbm" and r["achieved"] == pytest.approx(8.0 * 32 * 64 * 258 * 258 / 1e-3 / 1e9)
    r = bench.kernel_roofline(s2, "k_conv2d_act_stats<3,12,4,4,1,2,2>", 1.0, pk)
    assert r["bound"] == "alu" and r["peak"] == 80.0


def test_reference_arm_prints_one_json_line():
    # the fp64 oracle on the host cores, on the smallest workload
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "conv3d_hswish_gn4_mean_n2", "--steps", "2", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "GFLOP/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["steps"] == 2 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["config"] == bench.config_of(wl.WORKLOAD_BY_NAME["conv3d_hswish_gn4_mean_n2"])
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_fp32_peak_follows_the_device_sm_count():
    assert bench.peaks(148)["fp32_tflops"] == pytest.approx(
        148 / 152 * bench.peaks(152)["fp32_tflops"])
    assert bench.peaks(148)["sms_source"] == "device"
    assert bench.peaks()["sms"] == bench.DEFAULT_SMS
