"""Benchmark of the fused GDN decode step on GB300.

One step is one call of the whole decode path (conv, SiLU, norms, gates, the
gated delta rule, the gated RMSNorm) over one batch of synthetic input: by
default the large-batch decode workload of 128 sequences x 36 layers x 1 token
(beta and decay near 1, state ~N(0, 0.05)), the largest of the five workloads.
The metric is GDN state updates per second (sequence x layer x valid token)
together with the achieved HBM bandwidth against the measured GB300 copy peak.
The same run also measures the other four workloads, each on its own, and
reports them in the line's ``configs`` object.

Timed regions use CUDA events on the launching stream, bracketed by a barrier
and a device synchronise. The state (14.5 GB at the default workload) is far
larger than the 129 MB L2, so no step finds its inputs in L2; the one workload
that fits in L2 is timed call by call with L2 flushed before each call.

``--impl reference`` times the fp64 CPU oracle instead, on a bounded sample of
the same workload, on this machine's host cores.

Multi-GPU: ``torchrun --nproc-per-node N bench.py --gpus N`` runs one process
per GPU; each rank takes its own 64 sequences of a 64*N-sequence batch (weak
scaling, no collective on the data path) and the slowest rank's time counts.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

# The oracle legs run single-threaded numpy: pin BLAS pools to one thread before numpy loads.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

DEFAULT_WORKLOAD = "decode_b128_l36_t1_beta_hi_decay_hi"
METRIC = "GDN state-updates/sec (seq*layer*token) and achieved HBM GB/s vs GB300 peak"
UNIT = "state-updates/s"
PROFILES = os.path.join(ROOT, "profiles")
L2_BYTES = 129e6
L2_NOTE_LARGE = "inputs larger than L2: the working set is far larger than the 129 MB L2; state updated in place"
L2_NOTE_FLUSH = "working set fits in L2: L2 flushed (512 MB written) before each timed call"


# ------------------------------------------------------------------ args --
def parse():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--op", default="step", choices=["step", "ab_gates", "in_proj", "step_inputs", "mixer", "verify"],
                    help="step: the decode step (the default bench line); ab_gates: the fused alpha/beta projection; "
                         "in_proj: the qkv and z input projections on the tensor cores; step_inputs: qkv, z and "
                         "the alpha/beta gates in one tensor-core pass; mixer: step_inputs then the decode step "
                         "on its outputs, from the layer input x to y; verify: a two-phase verify window "
                         "(gdn_verify_window over every sequence's draft tokens, then gdn_verify_commit of a "
                         "seeded number of accepted tokens)")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(W.WORKLOADS))
    ap.add_argument("--batch", type=int, default=None,
                    help="sequences per GPU (default: the workload's B); smaller values are for profiling")
    ap.add_argument("--layers", type=int, default=None,
                    help="layers (default: the workload's L); smaller values are for profiling")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--timing", default="graph", choices=["graph", "direct"],
                    help="graph: the K timed steps are one captured CUDA graph (no host gaps between launches); "
                         "direct: K calls from Python")
    ap.add_argument("--packed", action="store_true",
                    help="in_proj, step_inputs and mixer: weights packed once by gdn_pack_proj_weights before the "
                         "timed region, the calls on the packed weights timed")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (the line's configs object), e.g. for profiling")
    return ap.parse_args()


# --------------------------------------------------------- distributed ----
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def shard_rows(rank: int, per_rank: int) -> tuple:
    """Rank r owns sequences [r * per_rank, (r + 1) * per_rank) of the global batch."""
    return rank * per_rank, (rank + 1) * per_rank


# ------------------------------------------------------------- counting --
def valid_tokens(w: W.Workload, lens) -> int:
    """Valid (sequence, layer, token) updates of one step."""
    if lens is None:
        return w.B * w.L * w.T
    return int(np.sum(lens)) * w.L


def algorithmic_bytes(w: W.Workload, lens) -> dict:
    """Bytes one step must move at least: each state tile and conv history read and
    written once, each valid token's inputs read and its y written once, each layer's
    weights read once."""
    B, L, T = w.B, w.L, w.T
    tok = valid_tokens(w, lens)  # sequence x layer x valid token
    state = B * L * 48 * 128 * 128 * 4 * 2
    conv = B * L * 10240 * 3 * 4 * 2
    per_token = (10240 + 6144 + 48 + 48 + 6144) * 4
    weights = L * (10240 * 4 + 48 + 48 + 128) * 4
    if lens is not None:  # untouched sequences (length 0) move no state; lengths here are >= 1
        pass
    return {"state": state, "total": state + conv + tok * per_token + weights}


ALU_PEAK_TFLOPS = 152 * 128 * 2 * 2070e6 / 1e12  # FP32 lanes x FMA x the maximum SM clock
ALU_PEAK_KIND = "derived: 152 SMs x 128 FP32 lanes x 2 x 2070 MHz"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# The library's dispatch: one token runs the single-token kernel, or the register kernel's 3-CTA
# clusters for launches of up to 6 units (sequence, layer, k head) per SM whose rounds of one unit per
# cluster cost no more (measured rounds: 7.1 us against 10.7 us); windows of 2-23 tokens run the
# kernel with the tiles in shared memory, or the clusters when all units fit one round of them;
# 24 tokens or more the tensor-core chunk kernel (the register kernel takes larger windows only in
# builds with other thresholds). The library counts the clusters that can run at once by the
# occupancy query (97 on a 152-SM GB300); without it the functions below assume 2 SMs / 3.
CHUNK_MAX_T, TC_MIN_T, TC_CHUNK = 23, 24, 64


def clusters_at_once(sms: int, clusters: int | None = None) -> int:
    """3-CTA clusters that run at once: the occupancy query's count when known, else 2 sms // 3."""
    return clusters if clusters is not None else 2 * sms // 3


def small_single_token(units: int | None, sms: int | None, clusters: int | None = None) -> bool:
    """A single-token launch of `units` units that runs the register kernel on a GPU of `sms` SMs:
    at most 6 units per SM, and 2 ceil(units / C) <= 3 ceil(units / sms), C clusters at once."""
    if units is None or sms is None or units > 6 * sms:
        return False
    c = clusters_at_once(sms, clusters)
    return 2 * -(-units // c) <= 3 * -(-units // sms)


def small_window(units: int | None, sms: int | None, clusters: int | None = None) -> bool:
    """A window of 2 to CHUNK_MAX_T tokens over `units` units that runs on the 3-CTA clusters: all
    its units fit one round of them."""
    return units is not None and sms is not None and units <= clusters_at_once(sms, clusters)


def kernel_name(T: int, units: int | None = None, sms: int | None = None, clusters: int | None = None) -> str:
    """The kernel a call with T tokens over `units` units runs on `sms` SMs (the library's dispatch;
    without the counts, a launch larger than the GPU)."""
    if T == 1:
        return "gdn_window_kernel" if small_single_token(units, sms, clusters) else "gdn_decode_t1_kernel"
    if T <= CHUNK_MAX_T:
        return "gdn_window_kernel" if small_window(units, sms, clusters) else "gdn_chunk_kernel"
    if T < TC_MIN_T:
        return "gdn_window_kernel"
    return "gdn_window_tc_kernel"


SOURCES_OF = {"gdn_decode_t1_kernel": ("gdn_decode_t1.cu", "gdn_device.cuh"),
              "gdn_window_kernel": ("gdn_step.cu", "gdn_device.cuh"),
              "gdn_chunk_kernel": ("gdn_chunk.cu", "gdn_device.cuh"),
              "gdn_window_tc_kernel": ("gdn_window_tc.cu", "gdn_tc.cuh", "gdn_device.cuh")}


def kernel_sources(T: int, units: int | None = None, sms: int | None = None, kernel: str | None = None) -> list:
    """The sources of the kernel a call with T tokens runs (arguments as for `kernel_name`; `kernel`,
    the library's own answer, decides when given)."""
    if kernel is not None:
        return [os.path.join(ROOT, "gated_deltanet_linear_step_gb300", "csrc", f) for f in SOURCES_OF[kernel]]
    if T == 1 and small_single_token(units, sms):
        names = ("gdn_step.cu", "gdn_device.cuh")
    elif T == 1:
        names = ("gdn_decode_t1.cu", "gdn_device.cuh")
    elif T <= CHUNK_MAX_T and small_window(units, sms):
        names = ("gdn_step.cu", "gdn_device.cuh")
    elif T <= CHUNK_MAX_T:
        names = ("gdn_chunk.cu", "gdn_device.cuh")
    elif T < TC_MIN_T:
        names = ("gdn_step.cu", "gdn_device.cuh")
    else:
        names = ("gdn_window_tc.cu", "gdn_tc.cuh", "gdn_device.cuh")
    return [os.path.join(ROOT, "gated_deltanet_linear_step_gb300", "csrc", f) for f in names]


def tc_mma_flops(w: W.Workload, lens) -> float:
    """Tensor-core flops of one call on the chunk kernel: per 64-token chunk and k head the Gram
    matrix (128x128x128), per chunk and v head the state, solve, output and update products
    (128x128x128, 128x64x64 twice, 128x128x64), each as three BF16 MMAs. A window longer than
    one chunk recomputes the Gram matrix for each v head."""
    gram = 3 * 2 * 128 * 128 * 128
    per_v = 3 * 2 * (128 * 128 * 128 + 2 * 128 * 64 * 64 + 128 * 128 * 64)
    ns = [w.T] * w.B if lens is None else [int(n) for n in lens]
    total = 0.0
    for n in ns:
        if n <= 0:
            continue
        chunks = -(-n // TC_CHUNK)
        total += chunks * (gram * (3 if n > TC_CHUNK else 1) + 3 * per_v)
    return total * w.L * 16


def committed_traffic(workload: str, T: int, units: int | None = None, sms: int | None = None,
                      kernel: str | None = None):
    """Per-launch DRAM bytes from a committed ncu summary (``profiles/*traffic*.txt``) taken on this
    workload and on the kernel source as it stands (its sha256 must match), else None."""
    digest = hashlib.sha256()
    for path in kernel_sources(T, units, sms, kernel):
        digest.update(open(path, "rb").read())
    want = digest.hexdigest()
    if not os.path.isdir(PROFILES):
        return None
    for fn in sorted(os.listdir(PROFILES)):
        if "traffic" not in fn or not fn.endswith(".txt"):
            continue
        text = open(os.path.join(PROFILES, fn)).read()
        wm = re.search(r"^workload:\s*(\S+)", text, re.M)
        m = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
        h = re.search(r"^kernel_source_sha256:\s*([0-9a-f]{64})", text, re.M)
        if wm and m and h and wm.group(1) == workload and h.group(1) == want:
            return float(m.group(1))
    return None


# --------------------------------------------------------------- clocks --
class ClockSampler:
    """Samples the SM clock, power and clock-event (throttle) reasons during the timed region.

    NVML is read directly (ctypes on libnvidia-ml, read-only queries) every 5 ms by a
    thread, so even a timed region of a few tens of milliseconds gets samples of its
    own; without NVML, ``nvidia-smi -lms 50`` is used. ``summary`` keeps the samples
    that fall inside [mark_start, mark_end].
    """

    # NVML clock-event reason bits (nvml.h: nvmlClocksEventReason*)
    REASON_BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}
    SMI_QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap")
    SMI_NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    PERIOD_S = 0.005

    def __init__(self, device):
        self.device = device
        self.samples = []  # (host time, sm MHz, max sm MHz, power W, [reason names])
        self.t0 = self.t1 = None
        self.source = None
        self._stop = False
        self.proc = None
        self.thread = None

    def _gpu_id(self):
        try:
            uuid = str(torch.cuda.get_device_properties(self.device).uuid)
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:  # noqa: BLE001 - older torch: fall back to the visible index
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            ids = [v for v in vis.split(",") if v.strip()]
            return ids[self.device.index] if self.device.index < len(ids) else str(self.device.index)

    def _start_nvml(self):
        import ctypes
        import threading

        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return False
        handle = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByUUID(self._gpu_id().encode(), ctypes.byref(handle)) != 0:
            return False
        reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        clk, mx, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if nv.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) != 0:  # 1 = NVML_CLOCK_SM
            return False

        def reader():
            while not self._stop:
                ok = nv.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(clk)) == 0
                ok = ok and nv.nvmlDeviceGetPowerUsage(handle, ctypes.byref(pw)) == 0
                ok = ok and reasons_fn(handle, ctypes.byref(rs)) == 0
                if ok:
                    names = [n for bit, n in self.REASON_BITS.items() if rs.value & bit]
                    self.samples.append((time.time(), float(clk.value), float(mx.value), pw.value / 1000.0, names))
                time.sleep(self.PERIOD_S)
            nv.nvmlShutdown()

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        self.source = "nvml, every 5 ms"
        return True

    def _start_smi(self):
        import threading

        self.proc = subprocess.Popen(["nvidia-smi", f"--id={self._gpu_id()}", f"--query-gpu={self.SMI_QUERY}",
                                      "--format=csv,noheader,nounits", "-lms", "50"],
                                     stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)

        def reader():
            for line in self.proc.stdout:
                parts = [q.strip() for q in line.split(",")]
                try:
                    names = [self.SMI_NAMES[i] for i, v in enumerate(parts[3:7]) if v.lower() == "active"]
                    self.samples.append((time.time(), float(parts[0]), float(parts[1]), float(parts[2]), names))
                except (ValueError, IndexError):
                    continue

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        self.source = "nvidia-smi -lms 50"

    def __enter__(self):
        try:
            started = self._start_nvml()
        except (OSError, AttributeError):
            started = False
        if not started:
            try:
                self._start_smi()
            except (OSError, FileNotFoundError):
                self.source = None
        time.sleep(0.2)
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        time.sleep(0.02)
        self._stop = True
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        rows = list(self.samples)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= self.t1]
        note = None
        if not inside:  # timed region shorter than the sampling period: nearest samples
            inside = sorted(rows, key=lambda r: abs(r[0] - (self.t0 or r[0])))[:2]
            note = "timed region shorter than the sampling period; nearest samples"
        reasons = sorted({n for r in inside for n in r[4]})
        out = {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
               "power_w_max": max(r[3] for r in inside), "samples": len(inside), "reasons": reasons,
               "source": self.source}
        if note:
            out["note"] = note
        return out


# ----------------------------------------------------------- cpu legs ----
def oracle_sample(w: W.Workload, seconds: float, max_slices: int | None = None, wall_seconds: float | None = None):
    """Times the oracle on (sequence, layer) slices of the workload until `seconds` of oracle time
    have passed (or `wall_seconds` of wall time, input generation included). Returns (updates done,
    oracle seconds, slices)."""
    import oracle

    lens = W.seq_lens(w)
    done, spent, slices = 0, 0.0, 0
    order = [(b, l) for l in range(w.L) for b in range(w.B)]
    rng = np.random.default_rng(7)
    rng.shuffle(order)
    wall0 = time.perf_counter()
    for b, l in order:
        if spent >= seconds or (max_slices is not None and slices >= max_slices):
            break
        if slices > 0 and wall_seconds is not None and time.perf_counter() - wall0 >= wall_seconds:
            break
        sl = W.sequence_slice(w, b, l)
        wt = W.layer_weights(w, l)
        n = w.T if lens is None else int(lens[b])
        t0 = time.perf_counter()
        oracle.gdn_decode_slice(sl, wt, n)
        spent += time.perf_counter() - t0
        done += n
        slices += 1
    return done, spent, slices


def step_config(w_global: W.Workload, per_rank: W.Workload, world: int) -> dict:
    """The workload description printed in `config` by both arms (the same keys and values)."""
    working = algorithmic_bytes(per_rank, W.seq_lens(per_rank))["total"]
    return {"workload": w_global.name, "B": w_global.B, "L": w_global.L, "T": w_global.T, "B_per_gpu": per_rank.B,
            "head_dim": 128, "k_heads": 16, "v_heads": 48, "conv_channels": 10240,
            "l2": L2_NOTE_LARGE if working > 2 * L2_BYTES else L2_NOTE_FLUSH,
            "parallelism": f"dp{world} (sequences sharded, no collective)"}


def run_reference(args, w_global, per_rank, world, rank):
    if rank != 0:
        return
    # Bounded by wall time (input generation included) so the whole run stays near two minutes.
    wall_per_step = min(6.0, max(1.0, 100.0 / max(1, args.steps)))
    for _ in range(args.warmup):
        oracle_sample(per_rank, 0.2, wall_seconds=0.5)
    done_total, spent_total, slices_total = 0, 0.0, 0
    for _ in range(args.steps):
        d, s_, n = oracle_sample(per_rank, wall_per_step, wall_seconds=wall_per_step)
        done_total += d
        spent_total += s_
        slices_total += n
    value = done_total / spent_total
    sample = (f"{slices_total} random (sequence, layer) slices of {per_rank.name} over {args.steps} steps "
              f"(at most {wall_per_step:.1f} s of wall time each, input generation not timed), fp64 numpy, one thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * spent_total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(w_global, per_rank, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def make_step(g, t, y):
    """One decode call on the device tensors `t` (state and conv_state updated in place)."""
    def step():
        if t["seq_len"] is None:
            g.gdn_decode_step(t["qkv"], t["z"], t["alpha"], t["beta"], t["dt"], t["ssm_a"], t["conv_w"],
                              t["ssm_norm"], t["conv_state"], t["state"], y)
        else:
            g.gdn_decode_step_varlen(t["qkv"], t["z"], t["alpha"], t["beta"], t["dt"], t["ssm_a"], t["conv_w"],
                                     t["ssm_norm"], t["conv_state"], t["state"], y, t["seq_len"])
    return step


def roofline_of(w: W.Workload, lens, mean_launch_s: float, traffic) -> dict:
    """Roofline of one decode call: HBM against the measured copy peak, or the FP32 ALUs when the
    recurrence's arithmetic (7 flops per state element per token, FMA = 2) bounds the call more
    tightly than its bytes."""
    bytes_alg = algorithmic_bytes(w, lens)
    peak, peak_kind = measured_peaks()
    achieved = bytes_alg["total"] / mean_launch_s / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "peak_kind": peak_kind, "state_only_gbs": bytes_alg["state"] / mean_launch_s / 1e9,
            "state_only_frac": bytes_alg["state"] / mean_launch_s / 1e9 / peak,
            "algorithmic_bytes_per_launch": bytes_alg["total"]}
    flops = 7.0 * 128 * 128 * 48 * valid_tokens(w, lens)
    if flops / (ALU_PEAK_TFLOPS * 1e12) > bytes_alg["total"] / (peak * 1e9):
        tf = flops / mean_launch_s / 1e12
        roof.update({"bound": "alu", "achieved": tf, "peak": ALU_PEAK_TFLOPS, "unit": "TFLOP/s",
                     "frac": tf / ALU_PEAK_TFLOPS, "peak_kind": ALU_PEAK_KIND, "hbm_gbs": achieved,
                     "hbm_frac": achieved / peak, "flops_per_launch": flops})
    if w.T >= TC_MIN_T:
        # the chunk kernel runs the definition's contractions on the tensor cores: their rate, for context
        tflops = tc_mma_flops(w, lens) / mean_launch_s / 1e12
        bf16 = measured_bf16_tflops()
        roof.update({"tensor_tflops": tflops, "tensor_peak": bf16, "tensor_frac": tflops / bf16,
                     "tensor_note": "BF16 MMA flops (three per product) of the chunk kernel, against the "
                                    "measured dense BF16 peak (burst)"})
    return roof


def measured_bf16_tflops() -> float:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    return 1900.0


def measure_workload(g, name: str, steps: int, warmup: int, dev) -> dict:
    """One workload on its own: device-timed decode calls, with the roofline of its kernel.
    Working sets larger than L2 run `steps` calls from one captured CUDA graph; the one that fits
    in L2 runs call by call, each after a write of 512 MB that evicts L2, each timed alone."""
    w = W.WORKLOADS[name]
    t = W.device_inputs(w, dev, threads=16)
    lens = W.seq_lens(w)
    y = torch.empty(t["z"].shape, device=dev)
    step = make_step(g, t, y)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize(dev)
    working = algorithmic_bytes(w, lens)["total"]
    if working > 2 * L2_BYTES:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(steps):
                step()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms = a.elapsed_time(b) / steps
        l2 = L2_NOTE_LARGE
        del graph
    else:
        flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        times = []
        for _ in range(steps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step()
            b.record(stream)
            times.append((a, b))
        torch.cuda.synchronize(dev)
        ms = float(np.mean([a.elapsed_time(b) for a, b in times]))
        l2 = L2_NOTE_FLUSH
        del flush
        # the same calls back to back from one captured graph, the working set left in L2 (reported
        # beside, not the value; issued one by one from the host they would wait on the launches)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(steps):
                step()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        warm_ms = a.elapsed_time(b) / steps
        del graph
    # A window of T > 1 tokens (all valid) is also timed as T single-token calls over the same
    # inputs, the alternative a caller without the window kernels has (same graph timing).
    singles = None
    if w.T > 1 and t["seq_len"] is None and working > 2 * L2_BYTES:
        y1 = torch.empty(t["z"][:, :, :1].shape, device=dev)
        calls = []
        for tt in range(w.T):
            one = dict(t)
            for k in ("qkv", "z", "alpha", "beta"):
                one[k] = t[k][:, :, tt:tt + 1].contiguous()
            calls.append(make_step(g, one, y1))
        for call in calls:
            call()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(steps):
                for call in calls:
                    call()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms1 = a.elapsed_time(b) / steps
        singles = {"calls_per_step": w.T, "ms_per_step": ms1, "value": valid_tokens(w, lens) / (ms1 / 1e3),
                   "kernel": g.gdn_dispatch_kernel(w.B, w.L, 1, device=dev)}
        del graph, calls, y1
    assert g.gdn_read_device_error(device=dev) == 0, f"a kernel reported a device error on {name}"
    updates = valid_tokens(w, lens)
    kernel = g.gdn_dispatch_kernel(w.B, w.L, w.T, device=dev)  # the library's own choice
    roof = roofline_of(w, lens, ms / 1e3, committed_traffic(name, w.T, kernel=kernel))
    out = {"workload": name, "B": w.B, "L": w.L, "T": w.T, "steps": steps, "ms_per_step": ms,
           "value": updates / (ms / 1e3), "unit": UNIT,
           "kernel": kernel, "l2": l2, "roofline": roof}
    if singles is not None:
        out["as_single_token_calls"] = singles
    if working <= 2 * L2_BYTES:
        out["warm_l2_ms_per_step"] = warm_ms
    del t, y, step
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------- gpu arm ----
def run_gdn(args, w_global, world, rank, local):
    import gated_deltanet_linear_step_gb300 as g

    g.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    per_rank = args.batch if args.batch is not None else W.WORKLOADS[args.workload].B
    rows = shard_rows(rank, per_rank)
    w = w_global.scaled(B=per_rank) if world > 1 else w_global
    t = W.device_inputs(w_global, dev, threads=16, batch_rows=rows)
    lens_all = W.seq_lens(w_global)
    lens = None if lens_all is None else lens_all[rows[0]:rows[1]]
    y = torch.empty(t["z"].shape, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = make_step(g, t, y)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)

    graph = None
    if args.timing == "graph":
        # K steps captured once; one replay runs them back to back on the device.
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(args.steps):
                step()
        torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev) as clocks:
        clocks.mark_start()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        if graph is not None:
            graph.replay()
        else:
            for s_, e_ in ev:
                s_.record(stream)
                step()
                e_.record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark_end()
    barrier(world)
    elapsed_ms = t_start.elapsed_time(t_end)
    launch_ms = [elapsed_ms / args.steps] if graph is not None else [s_.elapsed_time(e_) for s_, e_ in ev]
    assert g.gdn_read_device_error(device=dev) == 0, "the kernel reported a device error"
    del graph

    updates_rank = valid_tokens(w, lens) * args.steps
    total_updates = sum_over_ranks(updates_rank, world, dev)
    max_ms = max_over_ranks(elapsed_ms, world, dev)
    value = total_updates / (max_ms / 1000.0)

    # end to end through the C ABI with host buffers: every step's activations come from
    # pinned host memory and its y goes back to it (gdn_host_pipeline_*); the copies of
    # neighbouring steps overlap the step's kernel on separate streams.
    e2e = None
    if not args.no_e2e:
        from gated_deltanet_linear_step_gb300.host_pipeline import HostDecodePipeline

        host = {k: torch.empty(t[k].shape, dtype=t[k].dtype, pin_memory=True) for k in ("qkv", "z", "alpha", "beta")}
        for k in host:
            host[k].copy_(t[k])
        y_host = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for _ in range(2)]
        weights = {k: t[k] for k in ("dt", "ssm_a", "conv_w", "ssm_norm")}
        pipe = HostDecodePipeline(weights, t["conv_state"], t["state"], (w.B, w.L, w.T), seq_len=t["seq_len"],
                                  device=dev)
        for k in range(3):
            pipe.submit(host, y_host[k % 2])
        pipe.synchronize()
        barrier(world)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for k in range(args.steps):
            pipe.submit(host, y_host[k % 2])
        pipe.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1000.0, world, dev)
        e2e = {"value": total_updates / (e2e_ms / 1000.0), "unit": UNIT, "h2d_bytes_per_step": pipe.in_bytes,
               "d2h_bytes_per_step": pipe.out_bytes,
               "method": "wall clock over K steps through the C-ABI host pipeline (gdn_host_pipeline_submit with "
                         "pinned host buffers); copies of neighbouring steps overlap the kernel on separate streams"}
        del pipe, host, y_host

    mean_launch_s = float(np.mean(launch_ms)) / 1000.0
    kernel = g.gdn_dispatch_kernel(w.B, w.L, w.T, device=dev)
    traffic = committed_traffic(w_global.name, w.T, kernel=kernel) if world == 1 else None
    roofline = roofline_of(w, lens, mean_launch_s, traffic)
    del t, y, step
    torch.cuda.empty_cache()

    # The other workloads, each measured on its own in this run (rank 0 of a one-GPU run).
    configs = None
    if rank == 0 and world == 1 and not args.no_configs:
        configs = {}
        for name in W.WORKLOADS:
            if name != w_global.name:
                configs[name] = measure_workload(g, name, args.steps, args.warmup, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        done, spent, slices = oracle_sample(w, args.cpu_seconds, wall_seconds=2.5 * args.cpu_seconds)
        cpu = {"value": done / spent, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{slices} random (sequence, layer) slices of {w.name}, {done} updates, "
                         f"{spent:.1f} s of oracle time (input generation not timed), fp64 numpy on one host thread"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": step_config(w_global, w, world),
            "timing": f"{args.timing}: {args.steps} steps" + (" in one captured CUDA graph" if args.timing == "graph" else ""),
            "clocks": clocks.summary(), "e2e": e2e, "gpu_launches": args.steps, "roofline": roofline,
            "cpu_baseline": cpu,
            "launch_ms": {"mean": float(np.mean(launch_ms)), "min": float(np.min(launch_ms)),
                          "max": float(np.max(launch_ms))},
            "configs": configs,
        }
        print(json.dumps(line), flush=True)


def run_ab_gates(args, w):
    """Times the fused alpha/beta projection with its gate epilogue on the workload's shape."""
    import gated_deltanet_linear_step_gb300 as g

    g.load_library()
    dev = torch.device("cuda", 0)
    h = W.host_ab_inputs(w)
    x = torch.from_numpy(h["x"]).to(dev)
    wa = torch.from_numpy(h["w_alpha"].view(np.int16)).to(dev).view(torch.bfloat16)
    wb = torch.from_numpy(h["w_beta"].view(np.int16)).to(dev).view(torch.bfloat16)
    dt = torch.from_numpy(h["dt"]).to(dev)
    sa = torch.from_numpy(h["ssm_a"]).to(dev)
    gate = torch.empty((w.B, w.L, w.T, 48), device=dev)
    beta = torch.empty_like(gate)

    def step():
        g.gdn_ab_gates(x, wa, wb, dt, sa, gate, beta)

    for _ in range(max(3, args.warmup)):
        step()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            step()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev) as clocks:
        clocks.mark_start()
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize(dev)
        clocks.mark_end()
    assert g.gdn_read_device_error(device=dev) == 0, "the kernel reported a device error"
    ms = a.elapsed_time(b) / args.steps
    rows = w.B * w.L * w.T
    flops = 2.0 * rows * 96 * W.N_EMBD
    byts = rows * W.N_EMBD * 4 + w.L * 96 * W.N_EMBD * 2 + rows * 96 * 4
    peak, peak_kind = measured_peaks()
    achieved = byts / (ms / 1e3) / 1e9
    print(json.dumps({
        "metric": "alpha/beta projection + gate epilogue, rows (seq*layer*token) per second", "op": "ab_gates",
        "value": rows / (ms / 1e3), "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16 x (bf16 hi + lo of f32), f32 accumulate", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "L": w.L, "T": w.T, "n_embd": W.N_EMBD, "outputs": 96,
                   "timing": f"{args.steps} launches in one captured CUDA graph"},
        "clocks": clocks.summary(), "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "algorithmic_bytes_per_launch": byts,
                     "tensor_tflops": flops / (ms / 1e3) / 1e12},
    }), flush=True)


def run_in_proj(args, w, with_ab=False):
    """Times the qkv and z input projections (x split + tensor-core GEMM) on the workload's shape;
    with_ab: also the alpha/beta projections with the gate epilogue (gdn_step_inputs)."""
    from concurrent.futures import ThreadPoolExecutor

    import gated_deltanet_linear_step_gb300 as g

    g.load_library()
    dev = torch.device("cuda", 0)
    E = W.N_EMBD
    B, L, T = w.B, w.L, w.T
    x = torch.from_numpy(np.stack([np.stack([W.ab_x(w, b, l, E) for l in range(L)]) for b in range(B)])).to(dev)
    wq = torch.empty((L, W.CONV_CHANNELS, E), dtype=torch.bfloat16, device=dev)
    wg = torch.empty((L, W.VALUE_DIM, E), dtype=torch.bfloat16, device=dev)

    def fill(l):
        d = W.proj_weights(w, l, E)
        return l, d

    with ThreadPoolExecutor(16) as ex:
        for l, d in ex.map(fill, range(L)):
            wq[l] = torch.from_numpy(d["w_qkv"].view(np.int16)).view(torch.bfloat16).to(dev)
            wg[l] = torch.from_numpy(d["w_gate"].view(np.int16)).view(torch.bfloat16).to(dev)
    qkv = torch.empty((B, L, T, W.CONV_CHANNELS), device=dev)
    z = torch.empty((B, L, T, W.VALUE_DIM), device=dev)
    ws = torch.empty(g.gdn_in_proj_workspace_size(B, L, T, E), dtype=torch.uint8, device=dev)
    if with_ab:
        h = W.host_ab_inputs(w, E)
        wa = torch.from_numpy(h["w_alpha"].view(np.int16)).to(dev).view(torch.bfloat16)
        wb = torch.from_numpy(h["w_beta"].view(np.int16)).to(dev).view(torch.bfloat16)
        dt = torch.from_numpy(h["dt"]).to(dev)
        sa = torch.from_numpy(h["ssm_a"]).to(dev)
        gate = torch.empty((B, L, T, 48), device=dev)
        beta = torch.empty_like(gate)
    packed = None
    if args.packed:
        packed = torch.empty(g.gdn_proj_pack_bytes(L, E), dtype=torch.uint8, device=dev)
        g.gdn_pack_proj_weights(wq, wg, packed, wa if with_ab else None, wb if with_ab else None)

    def step():
        if with_ab and packed is not None:
            g.gdn_step_inputs_packed(x, packed, dt, sa, qkv, z, gate, beta, ws)
        elif with_ab:
            g.gdn_step_inputs(x, wq, wg, wa, wb, dt, sa, qkv, z, gate, beta, ws)
        elif packed is not None:
            g.gdn_in_proj_packed(x, packed, qkv, z, ws)
        else:
            g.gdn_in_proj(x, wq, wg, qkv, z, ws)

    for _ in range(max(3, args.warmup)):
        step()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            step()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev) as clocks:
        clocks.mark_start()
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize(dev)
        clocks.mark_end()
    assert g.gdn_read_device_error(device=dev) == 0, "the kernel reported a device error"
    ms = a.elapsed_time(b) / args.steps
    rows = B * L * T
    n_out = W.CONV_CHANNELS + W.VALUE_DIM + (2 * 48 if with_ab else 0)
    byts = L * n_out * E * 2 + rows * E * 4 + rows * n_out * 4 + (L * 2 * 48 * 4 if with_ab else 0)
    flops = 2.0 * rows * n_out * E
    peak, peak_kind = measured_peaks()
    achieved = byts / (ms / 1e3) / 1e9
    print(json.dumps({
        "metric": ("qkv + z + alpha/beta gate projections" if with_ab else "qkv + z input projections")
                  + ", rows (seq*layer*token) per second", "op": "step_inputs" if with_ab else "in_proj",
        "value": rows / (ms / 1e3), "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16 x (bf16 hi + lo of f32), f32 accumulate",
        "data": "synthetic",
        "config": {"workload": w.name, "B": B, "L": L, "T": T, "n_embd": E, "outputs": n_out,
                   "weights_bytes": L * n_out * E * 2, "weights": "packed" if args.packed else "row-major",
                   "l2": "weights far larger than the 129 MB L2, streamed once per step",
                   "timing": f"{args.steps} calls (2 launches each) in one captured CUDA graph"},
        "clocks": clocks.summary(), "gpu_launches": 2 * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "algorithmic_bytes_per_launch": byts,
                     "tensor_tflops": flops / (ms / 1e3) / 1e12},
    }), flush=True)


def run_mixer(args, w):
    """Times the mixer from the layer input to y: gdn_step_inputs (qkv, z and the gates on the
    tensor cores) then gdn_decode_step_ex with GDN_FLAG_GATES_READY, K steps in one graph."""
    from concurrent.futures import ThreadPoolExecutor

    import gated_deltanet_linear_step_gb300 as g

    g.load_library()
    dev = torch.device("cuda", 0)
    E = W.N_EMBD
    B, L, T = w.B, w.L, w.T
    t = W.device_inputs(w, dev, threads=16)
    h = W.host_ab_inputs(w, E)
    x = torch.from_numpy(h["x"]).to(dev)
    wa = torch.from_numpy(h["w_alpha"].view(np.int16)).to(dev).view(torch.bfloat16)
    wb = torch.from_numpy(h["w_beta"].view(np.int16)).to(dev).view(torch.bfloat16)
    wq = torch.empty((L, W.CONV_CHANNELS, E), dtype=torch.bfloat16, device=dev)
    wg = torch.empty((L, W.VALUE_DIM, E), dtype=torch.bfloat16, device=dev)
    with ThreadPoolExecutor(16) as ex:
        for l, d in ex.map(lambda l: (l, W.proj_weights(w, l, E)), range(L)):
            wq[l] = torch.from_numpy(d["w_qkv"].view(np.int16)).view(torch.bfloat16).to(dev)
            wg[l] = torch.from_numpy(d["w_gate"].view(np.int16)).view(torch.bfloat16).to(dev)
    ws = torch.empty(g.gdn_in_proj_workspace_size(B, L, T, E), dtype=torch.uint8, device=dev)
    gate = torch.empty(t["alpha"].shape, device=dev)
    beta = torch.empty(t["beta"].shape, device=dev)
    y = torch.empty(t["z"].shape, device=dev)
    packed = None
    if args.packed:
        packed = torch.empty(g.gdn_proj_pack_bytes(L, E), dtype=torch.uint8, device=dev)
        g.gdn_pack_proj_weights(wq, wg, packed, wa, wb)

    def step():
        if packed is not None:
            g.gdn_step_inputs_packed(x, packed, t["dt"], t["ssm_a"], t["qkv"], t["z"], gate, beta, ws)
        else:
            g.gdn_step_inputs(x, wq, wg, wa, wb, t["dt"], t["ssm_a"], t["qkv"], t["z"], gate, beta, ws)
        g.gdn_decode_step_ex(t["qkv"], t["z"], gate, beta, t["dt"], t["ssm_a"], t["conv_w"], t["ssm_norm"],
                             t["conv_state"], t["state"], y, seq_len=t["seq_len"], flags=g.FLAG_GATES_READY)

    for _ in range(max(3, args.warmup)):
        step()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            step()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev) as clocks:
        clocks.mark_start()
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize(dev)
        clocks.mark_end()
    assert g.gdn_read_device_error(device=dev) == 0, "a kernel reported a device error"
    ms = a.elapsed_time(b) / args.steps
    lens = W.seq_lens(w)
    updates = valid_tokens(w, lens)
    rows = B * L * T
    n_out = W.CONV_CHANNELS + W.VALUE_DIM + 2 * W.V_HEADS
    proj_bytes = L * n_out * E * 2 + rows * E * 4 + rows * n_out * 4
    step_bytes = algorithmic_bytes(w, lens)["total"]
    peak, peak_kind = measured_peaks()
    gbs = (proj_bytes + step_bytes) / (ms / 1e3) / 1e9
    print(json.dumps({
        "metric": "mixer steps from the layer input x to y (projections + decode step), state-updates/s",
        "op": "mixer", "value": updates / (ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "f32 (bf16 weights)",
        "data": "synthetic",
        "config": {"workload": w.name, "B": B, "L": L, "T": T, "n_embd": E,
                   "weights": "packed" if args.packed else "row-major",
                   "timing": f"{args.steps} x (gdn_step_inputs + gdn_decode_step_ex) in one captured CUDA graph"},
        "clocks": clocks.summary(), "gpu_launches": 3 * args.steps,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "peak_kind": peak_kind, "bytes_per_step": proj_bytes + step_bytes,
                     "note": "the projections' bytes (weights, x, qkv/z/gate/beta written) plus the decode "
                             "step's algorithmic bytes; qkv and z cross HBM twice between the two calls"},
    }), flush=True)


def run_verify(args, w):
    """Times the two-phase verify window: gdn_verify_window (y for every sequence's draft tokens,
    the state read only) then gdn_verify_commit (the state advanced by n_keep[b] accepted tokens,
    drawn per sequence from U{0..len[b]} with a fixed seed), K pairs in one captured graph."""
    import gated_deltanet_linear_step_gb300 as g

    g.load_library()
    dev = torch.device("cuda", 0)
    B, L, T = w.B, w.L, w.T
    t = W.device_inputs(w, dev, threads=16)
    lens = W.seq_lens(w)
    lens = np.full(B, T, np.int32) if lens is None else lens
    keep = np.random.default_rng(w.seed + 1).integers(0, lens + 1).astype(np.int32)
    seq_len = torch.from_numpy(lens).to(dev)
    n_keep = torch.from_numpy(keep).to(dev)
    y = torch.empty(t["z"].shape, device=dev)

    def window():
        g.gdn_verify_window(t["qkv"], t["z"], t["alpha"], t["beta"], t["dt"], t["ssm_a"], t["conv_w"], t["ssm_norm"],
                            t["conv_state"], t["state"], y, seq_len=seq_len)

    def commit():
        g.gdn_verify_commit(t["qkv"], t["alpha"], t["beta"], t["dt"], t["ssm_a"], t["conv_w"], t["conv_state"],
                            t["state"], n_keep)

    def step():
        window()
        commit()

    def alone_ms(fn):
        # one call kind on its own, the same number of calls in a captured graph (the commit repeated
        # on the state it advanced: the bytes and the work do not depend on the values)
        for _ in range(3):
            fn()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for _ in range(args.steps):
                fn()
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record()
        gr.replay()
        eb.record()
        torch.cuda.synchronize(dev)
        return ea.elapsed_time(eb) / args.steps

    for _ in range(max(3, args.warmup)):
        step()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            step()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev) as clocks:
        clocks.mark_start()
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize(dev)
        clocks.mark_end()
    ms = a.elapsed_time(b) / args.steps
    window_ms, commit_ms = alone_ms(window), alone_ms(commit)
    assert g.gdn_read_device_error(device=dev) == 0, "a kernel reported a device error"
    drafted = int(lens.sum()) * L
    kept = int(keep.sum()) * L
    tile = 48 * 128 * 128 * 4
    conv = 10240 * 3 * 4
    weights = L * (10240 * 4 + 48 + 48 + 128) * 4
    # window: every tile and conv history read, the drafted tokens' inputs read and their y written;
    # commit: the tiles and histories of sequences that keep a token read and written, the kept
    # tokens' qkv, alpha and beta read.
    advanced = int((keep > 0).sum()) * L
    window_bytes = B * L * (tile + conv) + drafted * (10240 + 6144 + 48 + 48 + 6144) * 4 + weights
    commit_bytes = advanced * 2 * (tile + conv) + kept * (10240 + 48 + 48) * 4 + weights
    peak, peak_kind = measured_peaks()
    gbs = (window_bytes + commit_bytes) / (ms / 1e3) / 1e9
    print(json.dumps({
        "metric": "verified draft tokens (seq*layer*token) per second, window + commit",
        "op": "verify", "value": drafted / (ms / 1e3), "unit": "draft-tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": B, "L": L, "T": T, "drafted_per_layer": int(lens.sum()),
                   "kept_per_layer": int(keep.sum()),
                   "n_keep": "per sequence from U{0..len[b]}, numpy default_rng(seed + 1)",
                   "timing": f"{args.steps} x (gdn_verify_window + gdn_verify_commit) in one captured CUDA graph; "
                             "then each call alone, the same number of times in its own graph"},
        "clocks": clocks.summary(), "gpu_launches": 2 * args.steps,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "peak_kind": peak_kind, "bytes_per_step": window_bytes + commit_bytes,
                     "window_bytes": window_bytes, "commit_bytes": commit_bytes,
                     "window_ms_alone": window_ms, "window_frac": window_bytes / (window_ms / 1e3) / 1e9 / peak,
                     "commit_ms_alone": commit_ms, "commit_frac": commit_bytes / (commit_ms / 1e3) / 1e9 / peak},
    }), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.gpus != world and world > 1:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    base = W.WORKLOADS[args.workload]
    if args.batch is not None:
        base = base.scaled(B=args.batch, name=f"{base.name}_b{args.batch}")
    if args.layers is not None:
        base = base.scaled(L=args.layers, name=f"{base.name}_l{args.layers}")
    w_global = base.scaled(B=base.B * world) if world > 1 else base
    if args.op == "ab_gates":
        if rank == 0:
            run_ab_gates(args, base)
    elif args.op in ("in_proj", "step_inputs"):
        if rank == 0:
            run_in_proj(args, base, with_ab=args.op == "step_inputs")
    elif args.op == "verify":
        if rank == 0:
            run_verify(args, base)
    elif args.op == "mixer":
        if rank == 0:
            run_mixer(args, base)
    elif args.impl == "reference":
        run_reference(args, w_global, base, world, rank)
    else:
        run_gdn(args, w_global, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
