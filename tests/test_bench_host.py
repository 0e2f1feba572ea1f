"""Host-side logic of bench.py on the CPU: both arms print the same config, the
reference arm's line has the contract's keys, traffic figures are only used on
the kernel source they were taken on, and the clock summary keeps the samples
of the timed region."""
import json
import os
import subprocess
import sys

import numpy as np

import bench
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_gpu_arms_config():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1", "--workload", "decode_b1_l1_t1"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    w = W.WORKLOADS["decode_b1_l1_t1"]
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["config"] == bench.step_config(w, w, 1)
    assert line["metric"] == bench.METRIC and line["unit"] == bench.UNIT and line["higher_is_better"] is True
    assert line["value"] > 0 and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_step_config_names_the_l2_treatment():
    big = W.WORKLOADS["decode_b128_l36_t1_beta_hi_decay_hi"]
    small = W.WORKLOADS["decode_b1_l1_t1"]
    assert bench.step_config(big, big, 1)["l2"] == bench.L2_NOTE_LARGE
    assert bench.step_config(small, small, 1)["l2"] == bench.L2_NOTE_FLUSH
    assert bench.DEFAULT_WORKLOAD == big.name  # the largest single-GPU workload is the headline


def test_traffic_is_used_only_on_the_kernel_source_it_was_taken_on(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    import hashlib

    h = hashlib.sha256()
    for p in bench.kernel_sources(1):
        h.update(open(p, "rb").read())
    good = f"workload: decode_b64_l36_t1\ntraffic_bytes_per_launch: 123\nkernel_source_sha256: {h.hexdigest()}\n"
    (tmp_path / "k_traffic_a.txt").write_text(good)
    (tmp_path / "k_traffic_b.txt").write_text(good.replace("decode_b64_l36_t1", "decode_b1_l1_t1")
                                              .replace(h.hexdigest(), "0" * 64))
    assert bench.committed_traffic("decode_b64_l36_t1", 1) == 123.0
    assert bench.committed_traffic("decode_b1_l1_t1", 1) is None  # taken on another source
    assert bench.committed_traffic("decode_b64_l36_t1", 8) is None  # another kernel's source


def test_clock_summary_keeps_the_timed_region():
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.source = "test"
    c.t0, c.t1 = 10.0, 10.1
    c.samples = [(9.9, 1500.0, 2070.0, 300.0, []), (10.02, 2070.0, 2070.0, 900.0, ["sw_power_cap"]),
                 (10.05, 2060.0, 2070.0, 950.0, []), (10.3, 1000.0, 2070.0, 200.0, ["hw_slowdown"])]
    s = c.summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 2065.0 and s["reasons"] == ["sw_power_cap"]
    assert "note" not in s
    c.samples = [(9.9, 1500.0, 2070.0, 300.0, [])]
    assert "note" in c.summary()


def test_kernel_sources_follow_the_library_dispatch():
    """Each window length maps to the source of the kernel the library runs for it (the traffic
    records are keyed to those sources)."""
    import bench

    names = lambda T: [os.path.basename(p) for p in bench.kernel_sources(T)]
    names_small = lambda units, sms: [os.path.basename(p) for p in bench.kernel_sources(1, units, sms)]
    assert names(1)[0] == "gdn_decode_t1.cu"
    assert names(2)[0] == names(bench.CHUNK_MAX_T)[0] == "gdn_chunk.cu"
    assert names(bench.TC_MIN_T)[0] == names(1024)[0] == "gdn_window_tc.cu"
    # with the default thresholds no window runs the register kernel; with others it takes the gap
    assert bench.CHUNK_MAX_T + 1 == bench.TC_MIN_T
    saved = bench.CHUNK_MAX_T, bench.TC_MIN_T
    try:
        bench.CHUNK_MAX_T, bench.TC_MIN_T = 8, 20
        assert names(9)[0] == names(19)[0] == "gdn_step.cu" and bench.kernel_name(12) == "gdn_window_kernel"
    finally:
        bench.CHUNK_MAX_T, bench.TC_MIN_T = saved
    # the kernel names the configs block reports, one per source
    assert [bench.kernel_name(T) for T in (1, 2, bench.CHUNK_MAX_T, bench.TC_MIN_T)] == [
        "gdn_decode_t1_kernel", "gdn_chunk_kernel", "gdn_chunk_kernel", "gdn_window_tc_kernel"]
    for T in (1, 2, bench.TC_MIN_T):
        kernel_src = open(bench.kernel_sources(T)[0]).read()
        assert "void __launch_bounds__" in kernel_src and bench.kernel_name(T) in kernel_src
    # single-token launches: the register kernel's 3-CTA clusters where their rounds (101 units on 152 SMs
    # when the occupancy count is not given: 2 SMs / 3) cost no more than the single-token kernel's (152
    # units), at 7.1 against 10.7 us a round
    on_clusters = {16: True, 96: True, 101: True, 102: False, 112: False, 128: False, 152: False, 160: True,
                   256: True, 384: True, 576: True, 768: True, 909: True, 912: False, 1024: False, 36864: False}
    for units, want in on_clusters.items():
        assert bench.small_single_token(units, 152) == want, units
        assert bench.kernel_name(1, units, 152) == ("gdn_window_kernel" if want else "gdn_decode_t1_kernel")
    assert names_small(16, 152)[0] == "gdn_step.cu" and names_small(128, 152)[0] == "gdn_decode_t1.cu"
    # with the 97 clusters the occupancy query gives on a 152-SM GB300, 400 units need a fifth round
    assert bench.small_single_token(400, 152) and not bench.small_single_token(400, 152, clusters=97)
    assert bench.small_window(97, 152, clusters=97) and not bench.small_window(98, 152, clusters=97)
    # windows of 2-23 tokens: the clusters when all units fit one round of them (101 on 152 SMs by default)
    assert bench.kernel_name(2, 16, 152) == bench.kernel_name(23, 101, 152) == "gdn_window_kernel"
    assert bench.kernel_name(8, 102, 152) == bench.kernel_name(8, 9216, 152) == "gdn_chunk_kernel"
    assert bench.kernel_name(24, 16, 152) == "gdn_window_tc_kernel"
    assert os.path.basename(bench.kernel_sources(8, 64, 152)[0]) == "gdn_step.cu"
    # given the library's own answer, the sources follow it
    for k, first in [("gdn_decode_t1_kernel", "gdn_decode_t1.cu"), ("gdn_window_kernel", "gdn_step.cu"),
                     ("gdn_chunk_kernel", "gdn_chunk.cu"), ("gdn_window_tc_kernel", "gdn_window_tc.cu")]:
        assert os.path.basename(bench.kernel_sources(1, kernel=k)[0]) == first
        assert "void __launch_bounds__" in open(bench.kernel_sources(1, kernel=k)[0]).read()
    # the thresholds are the library's defaults
    src = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "gated_deltanet_linear_step_gb300", "csrc", "gdn_step.cu")).read()
    assert f"#define GDN_CHUNK_MAX_T {bench.CHUNK_MAX_T}" in src
    assert f"#define GDN_TC_MIN_T {bench.TC_MIN_T}" in src
    assert "return single_token_on_clusters(units, sms, clusters) ? DecodeKernel::kClusters : DecodeKernel::kSingleToken;" in src
    assert "if (units > 6LL * sms || clusters <= 0) return false;" in src
    assert "return 2 * ((units + c - 1) / c) <= 3 * ((units + sms - 1) / sms);" in src
    assert "return window_on_clusters(units, clusters) ? DecodeKernel::kClusters : DecodeKernel::kChunked;" in src
    assert "static bool window_on_clusters(long long units, int clusters) { return units <= clusters; }" in src
    assert "return 2 * ((units + c - 1) / c) <= 3 * ((units + sms - 1) / sms);" in src


def test_tensor_core_flop_count():
    """Per 64-token chunk: a Gram product per k head (three per v head past one chunk) and four
    products per v head, each as three BF16 MMAs; sequences with no valid token cost nothing."""
    import bench
    import workloads as W

    gram = 3 * 2 * 128 ** 3
    per_v = 3 * 2 * (128 ** 3 + 2 * 128 * 64 * 64 + 128 * 128 * 64)
    w = W.WORKLOADS["decode_b64_l36_t1"].scaled(B=3, L=2, T=130)
    lens = np.array([0, 64, 130], np.int32)
    expect = (1 * (gram + 3 * per_v) + 3 * (3 * gram + 3 * per_v)) * 2 * 16
    assert bench.tc_mma_flops(w, lens) == expect
    assert bench.tc_mma_flops(w.scaled(T=64), None) == 3 * (gram + 3 * per_v) * 2 * 16
