"""Benchmark of gemm_tn_f16 on GB300: one JSON line on stdout (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c1..c9] [--impl reference]

A step is one gemm_tn_f16 call (the whole path: one persistent kernel) on
seeded synthetic fp16 inputs already resident in HBM.  The K timed steps run
back to back between one pair of CUDA events on the launching stream, and
cycle through R copies of A, B and D whose total exceeds 3 x L2, so each
launch reads operands evicted from L2 by the launches in between (inputs
larger than L2); ms_per_step = elapsed / K.  Default workload: 8192 x 8192 x
8192, U[-1, 1] operands.

Extra keys:
  roofline         the GEMM kernel against the measured peak that binds: HBM
                   copy bandwidth when the arithmetic intensity is under the
                   measured ridge point, else the dense bf16 tensor rate (fp16
                   runs at the same nominal rate) -- the burst figure when the
                   timed region lasts under a second, the sustained (power-
                   capped) figure when it lasts longer;
  tensor_nominal   the same rate against SMs x 8192 flop/clk x SM clock, at the
                   maximum clock and at the clock sampled in the timed region;
  sustained        the same launches back to back for --sustained-s seconds:
                   the power-capped rate, with its own clock record;
  configs          (default workload) the other configurations -- 256^3,
                   1024^3 {-1,0,1}, 4096^3, the skinny 128 x 14336 x 4096 and the
                   tall 81920 x 256 x 256 -- each timed back to back with its
                   roofline, its D checked against the oracle (max |err|, ulps,
                   exact fraction) and the oracle's CPU rate on that check;
  launch_ms_isolated, cpu_baseline, e2e, clocks (NVML sampled every 5 ms
  during the timed region), gpu_launches.

--impl reference times the CPU oracle itself (the only other implementation
of this computation here) on the same workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from multistage_smem_pipeline_gb300 import synthetic  # noqa: E402

METRIC = "fp16 GEMM TFLOP/s at 8192³ and % of dense FP16 tensor peak (1 GB300)"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# The sources that decide the GEMM kernel's code and its launch plan: the
# recorded DRAM traffic stays valid while these are unchanged.
KERNEL_SOURCES = ("ptx.cuh", "pipeline.cuh", "gemm_kernel.cuh", "gemm_pair_kernel.cuh",
                  "gemm_skinny_kernel.cuh", "gemm_splitk_kernel.cuh", "gemm_tn_f16.cu")


def code_tokens(text: str) -> str:
    """C/C++ source with comments removed and whitespace runs collapsed, so
    that an edit to comments or layout alone keeps the recorded traffic."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":                       # string or character literal, kept whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "multistage_smem_pipeline_gb300", "csrc", name),
                  encoding="utf-8") as fh:
            h.update(code_tokens(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the kernel sources as they are now; otherwise None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("source_hash") != source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
CLOCK_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]
# NVML clock-event reason bits (nvmlClocksEventReason*), the ones a run is judged by
REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}
NVML_CLOCK_SM = 1


def reasons_from_mask(mask: int) -> list:
    return sorted(n for n, bit in REASON_BITS.items() if mask & bit)


class _Nvml:
    """The few NVML queries the sampler needs, through ctypes (read-only:
    current and maximum SM clock, power draw, clock-event reasons)."""

    def __init__(self, bus_id: str):
        import ctypes
        self.c = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), ctypes.byref(self.h)) != 0:
            raise OSError(f"no NVML device at {bus_id}")
        self._reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(self.h, NVML_CLOCK_SM, ctypes.byref(mx))
        self.max_mhz = float(mx.value)

    def sample(self):
        c = self.c
        clk, pw, rs = c.c_uint(0), c.c_uint(0), c.c_ulonglong(0)
        if self.lib.nvmlDeviceGetClockInfo(self.h, NVML_CLOCK_SM, c.byref(clk)) != 0:
            return None
        self.lib.nvmlDeviceGetPowerUsage(self.h, c.byref(pw))
        self._reasons(self.h, c.byref(rs))
        return float(clk.value), pw.value / 1000.0, int(rs.value)


class ClockSampler:
    """SM clock, power draw and clock-event reasons of one GPU, sampled every
    `period_s` on a background thread, each sample stamped with the host's
    perf_counter so a region's samples can be picked out afterwards.  NVML
    through ctypes (5 ms period by default); nvidia-smi -lms where NVML
    cannot be loaded.  The GPU is named by its PCI bus id, so the samples
    describe the device this process computes on whatever
    CUDA_VISIBLE_DEVICES says."""

    def __init__(self, bus_id: str, period_s: float = 0.005):
        self.bus_id = bus_id
        self.period_s = period_s
        self.samples = []          # (t, sm_mhz, power_w, reason mask)
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()
        self._t = None
        self.proc = None

    def start(self):
        try:
            nv = _Nvml(self.bus_id)
            self.max_mhz = nv.max_mhz
            self.source = f"NVML every {self.period_s * 1e3:.0f} ms"
            self._t = threading.Thread(target=self._poll, args=(nv,), daemon=True)
        except (OSError, AttributeError):
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", self.bus_id, "--query-gpu=" + ",".join(CLOCK_FIELDS),
                     "--format=csv,noheader,nounits", "-lms", "10"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                return
            self.source = "nvidia-smi -lms 10"
            self._t = threading.Thread(target=self._read_smi, daemon=True)
        self._t.start()
        time.sleep(0.05)

    def _poll(self, nv):
        while not self._stop.is_set():
            s = nv.sample()
            if s is not None:
                self.samples.append((time.perf_counter(),) + s)
            time.sleep(self.period_s)

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(CLOCK_FIELDS):
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
                pw = float(parts[2])
            except ValueError:
                continue
            self.max_mhz = mx
            mask = sum(REASON_BITS[n] for n, v in zip(names, parts[4:])
                       if v.lower().startswith("active"))
            self.samples.append((time.perf_counter(), sm, pw, mask))

    def stop(self):
        self._stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self._t:
            self._t.join(timeout=5)

    def region(self, t0: float, t1: float):
        """Summary of the samples taken between host times t0 and t1; when
        none fell inside (a region shorter than the period), the nearest one."""
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside and self.samples:
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda s: abs(s[0] - mid))]
        if not inside:
            return None
        sm = [s[1] for s in inside]
        mask = 0
        for s in inside:
            mask |= s[3]
        return {"sm_mhz": statistics.median(sm), "sm_mhz_min": min(sm),
                "sm_max_mhz": self.max_mhz, "power_w_max": max(s[2] for s in inside),
                "samples": len(inside), "reasons": reasons_from_mask(mask),
                "source": self.source}


def pci_bus_id(torch, dev) -> str:
    p = torch.cuda.get_device_properties(dev)
    return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"


# The dense fp16 rate of one SM's tensor pipe: a 128 x 256 x 16 kind::f16
# MMA (1,048,576 flops) every 128 cycles; the MMA latency probe of this
# library measures 513 cycles for four of them (8176 flop/clk).
TENSOR_FLOP_PER_CLK_PER_SM = 8192


def tensor_nominal(tflops: float, sms: int, max_mhz, sm_mhz) -> dict:
    """The fraction of the nominal dense tensor rate (SMs x flop/clk x clock),
    at the maximum SM clock and at the clock sampled under load."""
    out = {"flop_per_clk_per_sm": TENSOR_FLOP_PER_CLK_PER_SM, "sms": sms}
    for key, mhz in (("max_clock", max_mhz), ("sampled_clock", sm_mhz)):
        if mhz:
            peak = sms * TENSOR_FLOP_PER_CLK_PER_SM * mhz * 1e6 / 1e12
            out[key] = {"sm_mhz": mhz, "peak_tflops": peak, "frac": tflops / peak}
    return out


# ------------------------------------------------------------------ CPU oracle
def oracle_block(tag, a_bits, b_bits, rows, cols, threads):
    """The oracle function that matches workload `tag`, on the block of D made
    of its first `rows` rows and `cols` columns (B sliced to those columns in
    either layout; C to that block in the scaled form)."""
    import oracle
    spec = synthetic.WORKLOADS[tag]
    a = np.ascontiguousarray(a_bits[:rows])
    if spec.get("b_kn"):
        b = np.ascontiguousarray(b_bits[:, :cols])
    else:
        b = np.ascontiguousarray(b_bits[:cols])
    if "alpha" in spec:
        c = np.ascontiguousarray(synthetic.workload_c(tag)[:rows, :cols]) if spec["beta"] else None
        return lambda: oracle.gemm_scaled(a, b, c, spec["alpha"], spec["beta"],
                                          bool(spec.get("b_kn")), threads=threads)
    if spec.get("acc_f16"):
        return lambda: oracle.gemm_tn_f16acc(a, b, threads=threads)
    return lambda: oracle.gemm_tn(a, b, threads=threads)


def oracle_rate(tag, a_bits, b_bits, target_s: float):
    """Time the workload's oracle on a slice of rows of D sized to about
    target_s seconds of wall time on this host.
    Returns (flop/s, rows, threads, seconds)."""
    import oracle
    spec = synthetic.WORKLOADS[tag]
    threads = oracle.default_threads()
    K, N = spec["K"], spec["N"]
    t0 = time.perf_counter()
    oracle_block(tag, a_bits, b_bits, 1, N, 1)()
    one_row = max(time.perf_counter() - t0, 1e-6)             # seconds for one row, 1 thread
    rows = int(max(1, min(spec["M"], round(target_s / one_row) * threads)))
    rows = max(threads, (rows // threads) * threads) if rows >= threads else rows
    rows = min(rows, spec["M"])
    step = oracle_block(tag, a_bits, b_bits, rows, N, threads)
    t0 = time.perf_counter()
    step()
    dt = time.perf_counter() - t0
    return 2.0 * rows * N * K / dt, rows, min(threads, rows), dt


def oracle_rate_one_thread(tag, a_bits, b_bits, target_s: float):
    """The same oracle on one thread, over as many rows as fit in about
    target_s seconds.  Returns (flop/s, rows, seconds)."""
    spec = synthetic.WORKLOADS[tag]
    K, N = spec["K"], spec["N"]
    t0 = time.perf_counter()
    oracle_block(tag, a_bits, b_bits, 1, N, 1)()
    one_row = max(time.perf_counter() - t0, 1e-6)
    rows = int(max(1, min(spec["M"], round(target_s / one_row))))
    step = oracle_block(tag, a_bits, b_bits, rows, N, 1)
    t0 = time.perf_counter()
    step()
    dt = time.perf_counter() - t0
    return 2.0 * rows * N * K / dt, rows, dt


def fp16_order(bits: np.ndarray) -> np.ndarray:
    """fp16 bit patterns as integers in the order of their values (+0 == -0),
    so that the difference of two is their distance in fp16 ulps."""
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def parity_stats(got: np.ndarray, ref: np.ndarray, K: int, amax: float, bmax: float) -> dict:
    """Element-wise agreement of the GPU's D with the oracle's on the same
    elements, against the bound |d - ref| <= 2e-3 sqrt(K) max|A| max|B| +
    ulp(ref) (fp32 accumulation against exact accumulation, both rounded to
    fp16 once)."""
    g = got.view(np.float16).astype(np.float64)
    r = ref.view(np.float16).astype(np.float64)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -14))) - 10)
    tol = 2e-3 * np.sqrt(max(K, 1)) * amax * bmax + ulp
    err = np.abs(g - r)
    err = np.where(np.isnan(g) & np.isnan(r), 0.0, err)
    err = np.where(np.isnan(err), np.inf, err)
    ulps = np.abs(fp16_order(got) - fp16_order(ref))
    return {"elements": int(got.size), "out_of_bound": int(np.count_nonzero(err > tol)),
            "max_abs_err": float(err.max()), "max_ulps": int(ulps.max()),
            "exact_frac": float(np.mean(got == ref)), "bit_exact": bool(np.array_equal(got, ref)),
            "bound": "2e-3*sqrt(K)*max|A|*max|B| + 1 ulp"}


def oracle_kind(spec) -> str:
    if spec.get("acc_f16"):
        return "oracle with an fp16 accumulator rounded after every 16-deep K slice"
    if "alpha" in spec:
        return "full oracle of alpha A op(B) + beta C (double arithmetic, one fp16 rounding)"
    return "full oracle (double accumulation, one fp16 rounding)"


def run_reference(args, tag):
    rank = _env_int("RANK", 0)
    if rank != 0:
        return 0
    import oracle
    spec = synthetic.WORKLOADS[tag]
    a_bits, b_bits, _ = synthetic.workload(tag)
    threads = oracle.default_threads()
    K = spec["K"]
    # size one step (a block of D: `threads` rows x `cols` columns) so that the
    # whole run stays near args.reference_budget seconds of wall time
    probe_cols = min(256, spec["N"])
    t0 = time.perf_counter()
    oracle_block(tag, a_bits, b_bits, 1, probe_cols, 1)()
    per_elem = max(time.perf_counter() - t0, 1e-9) / probe_cols
    budget = max(0.05, args.reference_budget / max(1, args.steps + args.warmup))
    rows = min(spec["M"], threads)
    cols = int(min(spec["N"], max(8, budget * min(threads, rows) / per_elem / rows)))
    step = oracle_block(tag, a_bits, b_bits, rows, cols, threads)
    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    flops = 2.0 * rows * cols * K
    ms = statistics.mean(times) * 1e3
    value = flops / (ms * 1e-3) / 1e12
    sample = (f"a {rows} x {cols} block of D (of {spec['M']} x {spec['N']}, K={K}) per step, "
              f"{oracle_kind(spec)}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(tag, spec),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(threads, rows),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def slowest_rank_ms(ms: float, world: int) -> float:
    """The step time every rank agrees on: the maximum over ranks (gloo,
    host tensors; the GEMM itself exchanges nothing between GPUs)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / (ms * 1e-3)


def workload_config(tag, spec, extra=None):
    c = {"workload": synthetic.WORKLOAD_NAMES[tag], "M": spec["M"], "N": spec["N"],
         "K": spec["K"], "layout": "TN: A MxK, B NxK row-major, D MxN row-major",
         "accumulate": "fp32", "output": "fp16", "parallelism": "replicas (one GEMM per GPU)"}
    if extra:
        c.update(extra)
    return c


# ------------------------------------------------------------------ GPU arm
def launches_per_step(spec) -> int:
    """Kernels one call launches: the GEMM, plus for the padded entry one
    repack per operand it reads whose rows are not 16-byte aligned (A and B
    when K % 8, a K x N B when N % 8).  A D whose rows are not aligned is
    stored by the GEMM itself when C is not read (the padded workloads)."""
    if not spec.get("padded"):
        return 1
    M, N, K = spec["M"], spec["N"], spec["K"]
    n = 1
    n += K % 8 != 0                                       # A
    n += (N % 8 != 0) if spec.get("b_kn") else (K % 8 != 0)  # B
    return n


def padded_gemm_kernel_ms(args, binding, torch, dev, stream, spec, a, b, l2):
    """The GEMM launch of a padded call, timed alone: the padded call itself on
    A and B already repacked to rows of a multiple of 8 (M x Kp and N x Kp,
    +0 in the pad), so it launches only its GEMM -- with D's rows still
    unaligned, so the same kernel, storing D directly (checked: no workspace
    needed, same plan).  Back-to-back launches over copies spanning > 3 x L2,
    replayed from a CUDA graph, one event pair."""
    M, N, K = spec["M"], spec["N"], spec["K"]
    Kp = -(-K // 8) * 8
    per = 2 * (M * Kp + N * Kp + M * N)
    R = max(2, -(-3 * l2 // per))
    ap = torch.zeros((R, M, Kp), dtype=torch.float16, device=dev)
    bp = torch.zeros((R, N, Kp), dtype=torch.float16, device=dev)
    dp = torch.empty((R, M, N), dtype=torch.float16, device=dev)
    ap[:, :, :K] = a
    bp[:, :, :K] = b
    ws = torch.empty(16, dtype=torch.uint8, device=dev)
    for i in range(R):
        if binding.padded_workspace_bytes(ap[i], bp[i], None, dp[i], 0.0, "nk") != 0:
            raise SystemExit("the stand-alone GEMM timing would also time repacks")

    def call(i, st):
        binding.gemm_f16_padded(ap[i], bp[i], None, 1.0, 0.0, "nk", out=dp[i], workspace=ws,
                                stream=st)

    for i in range(max(3, args.warmup)):
        call(i % R, stream)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        cap = torch.cuda.current_stream(dev)
        for i in range(R):
            call(i, cap)
    stream.wait_stream(side)
    g.replay()
    torch.cuda.synchronize(dev)
    reps = max(1, args.steps // R)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(reps):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    ms = t0.elapsed_time(t1) / (reps * R)
    note = (f"the GEMM launch of gemm_f16_padded timed alone: the padded call on A and B "
            f"already repacked ({M} x {Kp}, {N} x {Kp}), which launches only its GEMM (D stored "
            f"directly), {reps * R} back-to-back launches over {R} copies (> 3 x L2) from a "
            f"CUDA graph")
    del ap, bp, dp
    return ms, note


# The other configurations of the headline metric's set, measured in the same
# run: launches timed back to back, and the oracle's check of the result.
CONFIG_TAGS = ("c1", "c2", "c3", "c5", "c6")
CONFIG_LAUNCHES = {"c1": 400, "c2": 400, "c3": 100, "c5": 400, "c6": 400}
FULL_ORACLE = ("c1", "c2")          # checked on every element; the rest on seeded samples


def roofline_of(flops, alg_bytes, ms, peaks, peak_src, region_s):
    """The roofline that binds (arithmetic intensity against the measured
    ridge point) with the achieved rate against its measured peak.  A
    tensor-bound region shorter than a second runs before the power cap
    settles: the burst peak applies; a longer one takes the sustained peak."""
    ridge = float(peaks["bf16_tflops"]) * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
    if flops / alg_bytes < ridge:
        achieved = alg_bytes / (ms * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_source": f"{peak_src} hbm_gbs (copy bandwidth)"}
    achieved = flops / (ms * 1e-3) / 1e12
    burst = float(peaks["bf16_tflops"])
    sust = float(peaks.get("bf16_tflops_sustained", burst))
    long_region = region_s >= 1.0
    peak = sust if long_region else burst
    key = "bf16_tflops_sustained" if long_region else "bf16_tflops"
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": achieved / peak, "frac_of_burst_peak": achieved / burst,
            "frac_of_sustained_peak": achieved / sust,
            "peak_source": (f"{peak_src} {key}: the timed region lasted {region_s * 1e3:.1f} ms, "
                            + ("at least 1 s, long enough to reach the power cap"
                               if long_region else "under 1 s, before the power cap settles")
                            + "; fp16 runs at the bf16 nominal rate (1:1)")}


def time_graph_replays(torch, dev, stream, graph, launches_per_replay, reps, clocks):
    """Replays `graph` `reps` times back to back between one event pair on
    `stream`; returns (ms per launch, host window t0, t1, clock summary)."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    w0 = time.perf_counter()
    e0.record(stream)
    for _ in range(reps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    w1 = time.perf_counter()
    ms = e0.elapsed_time(e1) / (reps * launches_per_replay)
    return ms, w0, w1, (clocks.region(w0, w1) if clocks else None)


def bench_config(tag, binding, torch, dev, stream, l2, peaks, peak_src, clocks):
    """One configuration: ms per launch over back-to-back launches replayed
    from a CUDA graph and cycling through operand copies that span > 3 x L2,
    its roofline, and its D checked against the oracle (every element for
    the small cubes, seeded samples plus tile seams for the rest), the
    oracle's own time on that check giving its CPU rate."""
    import oracle
    spec = synthetic.WORKLOADS[tag]
    M, N, K = spec["M"], spec["N"], spec["K"]
    flops = 2.0 * M * N * K
    alg_bytes = 2.0 * (M * K + N * K + M * N)
    a_bits, b_bits, _ = synthetic.workload(tag)
    R = max(2, -(-3 * l2 // int(alg_bytes)))
    a = torch.from_numpy(a_bits.view(np.float16)).to(dev)
    b = torch.from_numpy(b_bits.view(np.float16)).to(dev)
    a_all = a.unsqueeze(0).expand(R, M, K).contiguous()
    b_all = b.unsqueeze(0).expand(R, N, K).contiguous()
    d_all = torch.empty((R, M, N), dtype=torch.float16, device=dev)
    del a, b
    for i in range(3 * R):
        binding.gemm_tn_f16(a_all[i % R], b_all[i % R], out=d_all[i % R], stream=stream)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        cap = torch.cuda.current_stream(dev)
        for i in range(R):
            binding.gemm_tn_f16(a_all[i], b_all[i], out=d_all[i], stream=cap)
    stream.wait_stream(side)
    g.replay()
    reps = max(1, CONFIG_LAUNCHES[tag] // R)
    ms, w0, w1, clk = time_graph_replays(torch, dev, stream, g, R, reps, clocks)
    status, raw = binding.get_device_error(stream)
    if status != 0:
        raise SystemExit(f"device error in the {tag} timing: {raw:#x}")
    d = d_all[0].cpu().numpy().view(np.uint16)
    del a_all, b_all, d_all, g
    cfg = binding.query_config(M, N, K)
    entry = {"workload": synthetic.WORKLOAD_NAMES[tag], "M": M, "N": N, "K": K,
             "ms_per_launch": ms, "launches": reps * R,
             "tflops": flops / (ms * 1e-3) / 1e12, "gbs": alg_bytes / (ms * 1e-3) / 1e9,
             "roofline": roofline_of(flops, alg_bytes, ms, peaks, peak_src, ms * reps * R / 1e3),
             "roofline_ms": max(flops / (float(peaks["bf16_tflops"]) * 1e12),
                                alg_bytes / (float(peaks["hbm_gbs"]) * 1e9)) * 1e3,
             "plan": {k: cfg[k] for k in ("path", "bn", "kstage", "katoms", "ctas", "epi_warps",
                                          "b_resident", "wide", "small_m", "split_k",
                                          "cluster")},
             "l2": f"{R} operand copies ({R * int(alg_bytes) >> 20} MiB > 3 x L2) cycled",
             "clocks": clk}
    entry["roofline_frac"] = entry["roofline_ms"] / ms
    # the oracle's check of D, timed: the CPU baseline of this configuration
    t0 = time.perf_counter()
    if tag in FULL_ORACLE:
        threads = oracle.default_threads()
        ref = oracle.gemm_tn(a_bits, b_bits, threads=threads)
        got = d
        sample = f"every element of D ({M} x {N})"
        o_flops, cores = flops, threads
    else:
        rows, cols = synthetic.sample_coords(synthetic.seeds(tag)[2], M, N)
        ref = oracle.gemm_tn_sampled(a_bits, b_bits, rows, cols)
        got = d[rows, cols]
        sample = f"{rows.size} seeded elements of D plus tile seams and corners"
        o_flops, cores = 2.0 * K * rows.size, 1
    dt = time.perf_counter() - t0
    amax = float(np.abs(a_bits.view(np.float16).astype(np.float64)).max())
    bmax = float(np.abs(b_bits.view(np.float16).astype(np.float64)).max())
    entry["parity"] = parity_stats(got, ref, K, amax, bmax)
    entry["parity"]["checked"] = sample
    entry["parity"]["ok"] = (entry["parity"]["out_of_bound"] == 0 and
                             (entry["parity"]["bit_exact"] or tag != "c2"))
    entry["cpu_baseline"] = {"value": o_flops / dt / 1e12, "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": f"{sample} in {dt:.2f} s"}
    return entry


def run_gpu(args, tag):
    import torch
    import torch.distributed as dist

    from multistage_smem_pipeline_gb300 import binding

    rank, world, local = _env_int("RANK", 0), _env_int("WORLD_SIZE", 1), _env_int("LOCAL_RANK", 0)
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    spec = synthetic.WORKLOADS[tag]
    M, N, K = spec["M"], spec["N"], spec["K"]
    flops = 2.0 * M * N * K
    alg_bytes = 2.0 * (M * K + N * K + M * N)

    a_bits, b_bits, _ = synthetic.workload(tag)
    a_host = torch.from_numpy(a_bits.view(np.float16)).pin_memory()
    b_host = torch.from_numpy(b_bits.view(np.float16)).pin_memory()
    a = a_host.to(dev)
    b = b_host.to(dev)
    # the scaled form D = alpha A op(B) + beta C also reads C (M x N) each step
    scaled = "alpha" in spec
    b_kn = bool(spec.get("b_kn"))
    # the general-shape entry: rows not 16-byte aligned are repacked around the GEMM
    padded = bool(spec.get("padded"))
    if scaled:
        c_host = torch.from_numpy(synthetic.workload_c(tag).view(np.float16)).pin_memory()
        if spec["beta"] != 0:
            alg_bytes += 2.0 * M * N
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = torch.cuda.current_stream(dev)
    opts = {"path": ["auto", "square", "skinny", "pair"].index(args.path), "bn": args.bn,
            "kstage": args.kstage, "katoms": args.katoms, "group_m": args.group_m,
            "epi_warps": args.epi_warps, "b_resident": args.b_resident, "pdl": args.pdl,
            "wide": args.wide, "small_m": args.small_m, "split_k": args.split_k}
    forced = any(opts.values())
    cfg = binding.query_config(M, N, K, b_layout=1 if spec.get("b_kn") else 0,
                               acc_f16=1 if spec.get("acc_f16") else 0, **opts)

    # Operand copies for the timed launches: launch i uses copy i % R, and the R
    # copies together span at least 3 x L2, so every launch reads operands that
    # the launches in between have evicted from L2 (inputs larger than L2).
    per_copy = int(alg_bytes)
    R = max(2, -(-3 * l2 // per_copy)) if args.timing == "rotate" else 1
    b_shape = (K, N) if b_kn else (N, K)
    a_all = torch.empty((R, M, K), dtype=torch.float16, device=dev)
    b_all = torch.empty((R,) + b_shape, dtype=torch.float16, device=dev)
    d_all = torch.empty((R, M, N), dtype=torch.float16, device=dev)
    a_all.copy_(a.unsqueeze(0).expand(R, M, K))
    b_all.copy_(b.unsqueeze(0).expand((R,) + b_shape))
    c_all = None
    if scaled:
        c_all = torch.empty((R, M, N), dtype=torch.float16, device=dev)
        c_all.copy_(c_host.to(dev).unsqueeze(0).expand(R, M, N))
    del a, b
    ws = None
    if padded:
        need = max(binding.padded_workspace_bytes(a_all[r], b_all[r], None, d_all[r], 0.0, "nk")
                   for r in range(R))
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)

    def gemm(a_, b_, d_, c_=None, stream_=None, ws_=None):
        st = stream_ if stream_ is not None else stream
        if padded:
            return binding.gemm_f16_padded(a_, b_, None, 1.0, 0.0, "nk", out=d_,
                                           workspace=ws if ws_ is None else ws_, stream=st,
                                           **opts)
        if scaled:
            return binding.gemm_f16_scaled(a_, b_, c_, spec["alpha"], spec["beta"],
                                           "kn" if b_kn else "nk", out=d_, stream=st, **opts)
        if forced or spec.get("acc_f16"):
            return binding.gemm_tn_f16_ex(a_, b_, out=d_, stream=st,
                                          acc_f16=1 if spec.get("acc_f16") else 0, **opts)
        return binding.gemm_tn_f16(a_, b_, out=d_, stream=st)

    def launch(i):
        r = i % R
        gemm(a_all[r], b_all[r], d_all[r], c_all[r] if c_all is not None else None)

    for i in range(args.warmup):
        launch(i)
    torch.cuda.synchronize(dev)
    status, raw = binding.get_device_error(stream)
    if status != 0:
        raise SystemExit(f"device error after warm-up: {raw:#x}")

    # The rotated launches are replayed from CUDA graphs (one graph of R
    # launches, one of the K mod R remainder), so the host's per-call Python
    # and ctypes overhead does not starve the GPU on small shapes.
    graphs = None
    if args.timing == "rotate" and not args.no_graphs:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)

        def capture(n):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                cap = torch.cuda.current_stream(dev)
                for i in range(n):
                    r = i % R
                    gemm(a_all[r], b_all[r], d_all[r], c_all[r] if c_all is not None else None,
                         stream_=cap)
            return g

        graphs = (capture(R), capture(args.steps % R) if args.steps % R else None)
        stream.wait_stream(side)
        graphs[0].replay()                      # one untimed replay
        torch.cuda.synchronize(dev)

    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    clean = torch.zeros(2 * l2 // 4, dtype=torch.int32, device=dev)
    sleep_cycles = int(args.launch_slack_us * 2.0e3)   # ~2 GHz SM clock

    def isolated_launches(n, read_clean):
        """Per-launch event pairs, each after an L2 flush (2 x L2 bytes
        written, then optionally a clean buffer read) and a device sleep so the
        launch is enqueued before its start event.  Each launch then also
        carries the ~4-5 us event-to-kernel latency of an isolated launch."""
        st = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        en = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(n):
            flush.zero_()
            if read_clean:
                clean.sum()
            if sleep_cycles:
                torch.cuda._sleep(sleep_cycles)
            st[i].record(stream)
            gemm(a_all[0], b_all[0], d_all[0], c_all[0] if c_all is not None else None)
            en[i].record(stream)
        torch.cuda.synchronize(dev)
        return [x.elapsed_time(y) for x, y in zip(st, en)]

    clocks = ClockSampler(pci_bus_id(torch, dev), args.clock_period_ms / 1e3)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    if args.timing == "rotate":
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        if graphs is not None:
            g_full, g_rem = graphs
            t_start.record(stream)
            for _ in range(args.steps // R):
                g_full.replay()
            if g_rem is not None:
                g_rem.replay()
            t_end.record(stream)
        else:
            t_start.record(stream)
            for i in range(args.steps):
                launch(i)
            t_end.record(stream)
        torch.cuda.synchronize(dev)
        ms = t_start.elapsed_time(t_end) / args.steps
        launches_ms = None
    else:
        launches_ms = isolated_launches(args.steps, True)
        ms = statistics.mean(launches_ms)
    wall1 = time.perf_counter()
    wall = wall1 - wall0
    if world > 1:
        dist.barrier()
    clk = clocks.region(wall0, wall1)

    # The same launches for at least --sustained-s seconds back to back: the
    # power-capped steady state, with its own clock record (the last half of
    # the window, once the clock has settled).
    sustained = None
    if graphs is not None and args.sustained_s > 0:
        reps = max(1, int(np.ceil(args.sustained_s / (ms * R * 1e-3))))
        s_ms, w0, w1, _ = time_graph_replays(torch, dev, stream, graphs[0], R, reps, clocks)
        sustained = {"seconds": s_ms * reps * R / 1e3, "launches": reps * R,
                     "ms_per_launch": s_ms,
                     "clocks_whole": clocks.region(w0, w1),
                     "clocks_steady": clocks.region(w0 + 0.5 * (w1 - w0), w1)}
    iso = None
    if args.alt_steps > 0:
        n_iso = min(args.steps, args.alt_steps)
        iso_clean = isolated_launches(n_iso, True)
        iso_dirty = isolated_launches(n_iso, False)
        iso = {"steps": n_iso, "mean_ms_clean_flush": statistics.mean(iso_clean),
               "median_ms_clean_flush": statistics.median(iso_clean),
               "p10_ms_clean_flush": float(np.percentile(iso_clean, 10)),
               "p90_ms_clean_flush": float(np.percentile(iso_clean, 90)),
               "mean_ms_write_only_flush": statistics.mean(iso_dirty),
               "note": "per-launch event pairs after an L2 flush; includes the isolated "
                       "launch latency (an empty kernel measures ~4.5 us this way)"}
    kernel_ms = None
    if padded:
        kernel_ms, kernel_note = padded_gemm_kernel_ms(args, binding, torch, dev, stream, spec,
                                                       a_all[0], b_all[0], l2)
    ms = slowest_rank_ms(ms, world)
    status, raw = binding.get_device_error(stream)
    if status != 0:
        raise SystemExit(f"device error in timed region: {raw:#x}")
    d = d_all[0]

    # End to end from pinned host buffers through the public API.  Each step
    # copies its A and B (and C) host -> device, runs the GEMM and copies D
    # device -> host.  Steps alternate over `lanes` streams, each with its own
    # device buffers, so a step's copies overlap the neighbouring steps' GEMMs
    # (the copy engines and the SMs work at once), as a caller streaming
    # batches would run them; stream order keeps each lane's buffers safe.
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    lanes = max(1, args.e2e_lanes)
    lane_streams = [torch.cuda.Stream(dev) for _ in range(lanes)]
    d_hosts = [torch.empty((M, N), dtype=torch.float16, pin_memory=True) for _ in range(lanes)]
    lane_bufs, lane_ws = [], []
    for _ in range(lanes):
        lane_bufs.append((torch.empty((M, K), dtype=torch.float16, device=dev),
                          torch.empty(b_shape, dtype=torch.float16, device=dev),
                          torch.empty((M, N), dtype=torch.float16, device=dev) if scaled else None,
                          torch.empty((M, N), dtype=torch.float16, device=dev)))
        if padded:  # calls in flight at once need their own workspaces
            la, lb, _, ld = lane_bufs[-1]
            need = binding.padded_workspace_bytes(la, lb, None, ld, 0.0, "nk")
            lane_ws.append(torch.empty(max(need, 16), dtype=torch.uint8, device=dev))
        else:
            lane_ws.append(None)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)

    def e2e_step(i):
        ls = lane_streams[i % lanes]
        a_e, b_e, c_e, d_e = lane_bufs[i % lanes]
        with torch.cuda.stream(ls):
            a_e.copy_(a_host, non_blocking=True)
            b_e.copy_(b_host, non_blocking=True)
            if scaled:
                c_e.copy_(c_host, non_blocking=True)
            gemm(a_e, b_e, d_e, c_e, stream_=ls, ws_=lane_ws[i % lanes])
            d_hosts[i % lanes].copy_(d_e, non_blocking=True)

    for ls in lane_streams:           # one untimed step per lane: first use of its buffers
        ls.wait_stream(stream)
    for i in range(lanes):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e_start.record(stream)
    for ls in lane_streams:
        ls.wait_stream(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    for ls in lane_streams:
        stream.wait_stream(ls)
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e_start.elapsed_time(e_end) / e2e_steps
    # the result that came back is the one the timed region computed
    if not torch.equal(d_hosts[(e2e_steps - 1) % lanes].to(dev).view(torch.int16),
                       d_all[0].view(torch.int16)):
        raise SystemExit("end-to-end result differs from the device-resident result")
    e2e_ms = slowest_rank_ms(e2e_ms, world)

    if rank != 0:
        clocks.stop()
        return 0

    peaks, peak_src = load_peaks()
    # the dominant kernel's own launch time: the step itself, or for the padded
    # entry the GEMM launch inside it (timed alone on the repacked operands)
    k_ms = kernel_ms if kernel_ms is not None else ms
    roof = roofline_of(flops, alg_bytes, k_ms, peaks, peak_src, ms * args.steps / 1e3)
    nominal = None
    if roof["bound"] == "tensor":
        nominal = tensor_nominal(roof["achieved"], sms, clk["sm_max_mhz"] if clk else None,
                                 clk["sm_mhz"] if clk else None)
        if iso:
            iso["tflops_clean_flush"] = flops / (iso["mean_ms_clean_flush"] * 1e-3) / 1e12
            iso["frac_of_burst_peak"] = iso["tflops_clean_flush"] / float(peaks["bf16_tflops"])
    if sustained is not None:
        s_roof = roofline_of(flops, alg_bytes, sustained["ms_per_launch"], peaks, peak_src,
                             sustained["seconds"])
        sustained["achieved"] = s_roof["achieved"]
        sustained["unit"] = s_roof["unit"]
        sustained["frac"] = s_roof["frac"]
        sustained["peak"] = s_roof["peak"]
        sustained["peak_source"] = s_roof["peak_source"]
        st_clk = sustained["clocks_steady"] or sustained["clocks_whole"]
        if s_roof["bound"] == "tensor" and st_clk:
            sustained["tensor_nominal"] = tensor_nominal(s_roof["achieved"], sms,
                                                         st_clk["sm_max_mhz"], st_clk["sm_mhz"])
    direct_d = padded and spec["N"] % 8 != 0     # a padded call with unaligned D rows, C not read
    flag = lambda x: "true" if x else "false"
    roof["kernel"] = ("gemm_tn_f16_pair<%d, %s, %d, %s>" % (cfg["epi_warps"], flag(direct_d),
                                                            2 if cfg["wide"] else 1,
                                                            flag(scaled))
                      if cfg["path"] == 3 else
                      ("gemm_tn_f16_splitk (cluster of %d)" % cfg["cluster"]) if cfg["split_k"] else
                      "gemm_tn_f16_skinny<%s>" % flag(direct_d) if cfg["small_m"] else
                      "gemm_tn_f16_persistent<%d, %s, %s>" % (cfg["epi_warps"],
                                                              flag(cfg["b_resident"]),
                                                              flag(direct_d)))
    if kernel_ms is not None:
        roof["kernel_ms"] = kernel_ms
        roof["kernel_timing"] = kernel_note
    roof["traffic"] = recorded_traffic(tag)
    roof["alg_bytes_per_launch"] = alg_bytes
    roof["flops_per_launch"] = flops

    line = {"metric": METRIC, "value": job_throughput(flops, world, ms) / 1e12, "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16 (fp16 accumulator)" if spec.get("acc_f16") else "f16",
            "entry": ("gemm_f16_padded" if padded else "gemm_f16_scaled" if scaled else
                      "gemm_tn_f16_ex" if (forced or spec.get("acc_f16")) else "gemm_tn_f16"),
            "data": "synthetic (seeded splitmix64, fp16-rounded)",
            "config": workload_config(tag, spec, {
                "l2": (f"inputs larger than L2: {R} copies of A, B, D ({R * per_copy >> 20} MiB "
                       f"> 3 x L2) cycled, launch i using copy i % {R}; one event pair around "
                       f"the {args.steps} back-to-back launches" +
                       (" (replayed from CUDA graphs)" if graphs is not None else "")
                       if args.timing == "rotate" else
                       "flushed before every timed launch: 2 x L2 bytes written, then 2 x L2 "
                       "bytes of a clean buffer read, outside the launch's event pair"),
                "timing": args.timing,
                "path": ["auto", "square", "skinny", "pair"][cfg["path"]], "bm": cfg["bm"],
                "bn": cfg["bn"], "bk": cfg["bk"], "kstage": cfg["kstage"], "ctas": cfg["ctas"],
                "tiles": cfg["tiles"], "katoms": cfg["katoms"], "epi_warps": cfg["epi_warps"],
                "b_resident": cfg["b_resident"], "pdl": cfg["pdl"], "wide": cfg["wide"],
                "small_m": cfg["small_m"], "split_k": cfg["split_k"], "forced": forced}),
            "launch_ms": ({"mean": ms, "median": statistics.median(launches_ms),
                           "p10": float(np.percentile(launches_ms, 10)),
                           "p90": float(np.percentile(launches_ms, 90))}
                          if launches_ms else {"mean": ms}),
            "launch_ms_isolated": iso,
            "roofline": roof,
            "tensor_nominal": nominal,
            "sustained": sustained,
            "e2e": {"value": job_throughput(flops, world, e2e_ms) / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": 2 * (M * K + N * K + (M * N if scaled else 0)),
                    "d2h_bytes_per_step": 2 * M * N,
                    "ms_per_step": e2e_ms, "steps": e2e_steps, "lanes": lanes,
                    "note": "pinned host A, B (C) -> device, the GEMM, D -> pinned host every "
                            "step; steps alternate over the lanes' streams so copies overlap "
                            "the neighbouring steps' GEMMs"},
            "gpu_launches": args.steps * launches_per_step(spec),
            "clocks": clk,
            "wall_s_timed_region": wall}
    run_configs = args.configs == "on" or (args.configs == "auto" and tag == "c4")
    if world == 1 and run_configs:
        line["configs"] = {t: bench_config(t, binding, torch, dev, stream, l2, peaks, peak_src,
                                           clocks)
                           for t in CONFIG_TAGS if t != tag}
    clocks.stop()
    if world == 1 and not args.no_cpu:
        rate, rows, cores, dt = oracle_rate(tag, a_bits, b_bits, args.cpu_seconds)
        rate1, rows1, dt1 = oracle_rate_one_thread(tag, a_bits, b_bits,
                                                   min(2.0, args.cpu_seconds / 4))
        line["cpu_baseline"] = {"value": rate / 1e12, "unit": UNIT, "cores": cores,
                                "kind": "oracle",
                                "sample": f"{rows} rows of D ({rows}x{N}, K={K}) in {dt:.1f} s; "
                                          f"{oracle_kind(spec)}",
                                "one_thread": {"value": rate1 / 1e12, "unit": UNIT, "cores": 1,
                                               "sample": f"{rows1} rows of D in {dt1:.2f} s"},
                                "full_problem_s_extrapolated": flops / rate}
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(synthetic.WORKLOADS), default="c4")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--e2e-lanes", type=int, default=2,
                    help="streams the end-to-end steps alternate over (1 = strictly serial)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-budget", type=float, default=90.0,
                    help="target wall seconds for the whole --impl reference run")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--timing", choices=["rotate", "flush"], default="rotate",
                    help="rotate: back-to-back launches over operand copies spanning > 3 x L2 "
                         "(one event pair); flush: per-launch event pairs after an L2 flush")
    ap.add_argument("--alt-steps", type=int, default=100,
                    help="extra isolated launches (flush + per-launch events), reported beside "
                         "the value")
    ap.add_argument("--sustained-s", type=float, default=2.0,
                    help="seconds of back-to-back launches for the power-capped 'sustained' "
                         "figure (0 = skip)")
    ap.add_argument("--configs", choices=["auto", "on", "off"], default="auto",
                    help="also measure and check the other configurations (auto: with the "
                         "default 8192^3 workload on one GPU)")
    ap.add_argument("--clock-period-ms", type=float, default=5.0,
                    help="clock sampling period during the timed regions")
    ap.add_argument("--katoms", type=int, default=0, help="diagnostics: force K slices per stage")
    ap.add_argument("--group-m", type=int, default=0, help="diagnostics: rasterisation group")
    ap.add_argument("--epi-warps", type=int, default=0, help="diagnostics: epilogue warps (4, 8)")
    ap.add_argument("--no-graphs", action="store_true",
                    help="launch the rotated steps one by one instead of replaying CUDA graphs")
    ap.add_argument("--launch-slack-us", type=float, default=100.0,
                    help="device-side sleep before each start event (outside the timed pair)")
    ap.add_argument("--path", choices=["auto", "square", "skinny", "pair"], default="auto",
                    help="diagnostics: force a kernel path (default: the library's choice)")
    ap.add_argument("--bn", type=int, default=0, help="diagnostics: force the tile width")
    ap.add_argument("--kstage", type=int, default=0, help="diagnostics: force the ring depth")
    ap.add_argument("--b-resident", type=int, default=0, choices=[0, 1, 2],
                    help="diagnostics: resident B (0 choose, 1 never, 2 always)")
    ap.add_argument("--pdl", type=int, default=0, choices=[0, 1],
                    help="diagnostics: 1 = launch without programmatic dependent launch")
    ap.add_argument("--wide", type=int, default=0, choices=[0, 1, 2],
                    help="diagnostics: pair units of two n-tiles (0 choose, 1 never, 2 always)")
    ap.add_argument("--split-k", type=int, default=0, choices=[0, 1, 2],
                    help="diagnostics: k split over a CTA pair (0 choose, 1 never, 2 always)")
    ap.add_argument("--small-m", type=int, default=0, choices=[0, 1, 2],
                    help="diagnostics: the small-M kernel, one tile per CTA (0 choose, 1 never, "
                         "2 always)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args, args.workload)
    return run_gpu(args, args.workload)


if __name__ == "__main__":
    sys.exit(main())
