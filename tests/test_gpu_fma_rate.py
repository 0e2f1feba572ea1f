"""The FP32 FMA-rate program that `build()` compiles beside the library runs on the device and
prints one JSON line whose rates are positive and no higher than the lane count allows: 128 FP32
lanes per SM, two FLOPs per FMA, at the device's maximum SM clock (5 % margin for clock reads)."""
import json
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu


def test_fma_rate_program_reports_rates_within_the_lane_count(cuda_device):
    from gated_deltanet_linear_step_gb300 import _build

    assert os.path.exists(_build.FMA_RATE_EXE), "the FMA-rate program is missing: run build() first"
    r = subprocess.run([_build.FMA_RATE_EXE, "64", "3"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["metric"] == "fp32_fma_rate" and d["unit"] == "TFLOP/s"
    assert d["sms"] > 0 and d["max_sm_mhz"] > 0
    lanes = d["sms"] * 128 * 2 * d["max_sm_mhz"] * 1e6 / 1e12
    assert abs(d["derived_tflops"] - lanes) < 0.01 * lanes
    for form in ("scalar", "packed"):
        assert 0 < d[form]["best_ms"] <= d[form]["median_ms"]
        assert 0 < d[form]["tflops_median"] <= d[form]["tflops_best"] <= 1.05 * lanes


def test_fma_rate_program_rejects_bad_arguments(cuda_device):
    from gated_deltanet_linear_step_gb300 import _build

    r = subprocess.run([_build.FMA_RATE_EXE, "0", "3"], capture_output=True, text=True, timeout=60)
    assert r.returncode == 2 and "usage" in r.stderr
