"""Benchmark of the tiled-contraction hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input
(inputs resident in HBM):
  * gemm_bf16              8192^3, bf16 in, f32 D, CTA pairs (cta_group::2)
  * gemm_mxfp8_blockscaled 8192^3, E4M3 x E8M0/32 in, bf16 D, CTA pairs
                           (its scale-image rearrangement kernel included)
  * tile_transpose_b16     8192 x 8192 16-bit patterns
value = GEMM FLOPs of the step (2*M*N*K for each GEMM) / device time of the
step, in TFLOP/s.  The inputs of one step (516 MB) exceed the 129 MB L2 and
every kernel's operands are evicted by the other kernels' traffic before
they are used again, so no separate L2 flush is inserted.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (float64, the machine's host cores) on
a bounded sample of the same workload per step and prints the same JSON
line with "impl": "reference".

The library is single-GPU code (one process drives one GPU; its short-K and
opt-in kernels use TMA multicast within that GPU's clusters).  ``--gpus N``
with N > 1, or a launch with WORLD_SIZE > 1, does no GPU work: rank 0 prints
one line saying so and every rank exits 0.

The line also carries what checks the timed work: the oracle's values on the
CPU-baseline sample compared with the last timed step's outputs
("parity"), the SM clock sampled while each kernel ran (NVML) and the one
the GEMM kernels' own cycle counters saw (tg_kernel_clock_read), and the
fraction of the tensor pipe's own rate (SMs x FLOP per SM per clock from the
rate probe x a clock: the probe's own, and the kernel's).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from blackwell_tile_gemm_gb300 import synth  # noqa: E402

METRIC = "GEMM TFLOP/s at 1 GB300 (bf16, MXFP8) and % of dense tensor-pipe peak"
UNIT = "TFLOP/s"
SIZE = 8192
def workload() -> str:
    return (f"bf16 GEMM {SIZE}^3 fp32 D (CTA pairs) + MXFP8 GEMM {SIZE}^3 bf16 D (CTA pairs) "
            f"+ b16 transpose {SIZE}^2")


# Per-launch DRAM traffic of each kernel comes from a committed ncu summary
# under profiles/, valid only while the kernel sources still hash to the
# value recorded next to the counters (otherwise the traffic is reported as
# null: the counters describe an older kernel).
_CSRC = "blackwell_tile_gemm_gb300/csrc/"
KERNEL_SOURCES = {
    "gemm": [_CSRC + f for f in ("gemm_kernel.cuh", "tg_ptx.cuh", "gemm_launch.cuh",
                                 "gemm_kinds.h", "epilogue.cuh", "gemm_bf16.cu",
                                 "gemm_blockscaled.cu", "gemm_fp4.cu")],
    "transpose": [_CSRC + f for f in ("transpose.cu", "tg_ptx.cuh")],
}
PROFILES = {
    "gemm_bf16": ("profiles/gemm_bf16_8192_pair.md", "gemm"),
    "gemm_mxfp8_blockscaled": ("profiles/gemm_mxfp8_8192_pair.md", "gemm"),
    "tile_transpose_b16": ("profiles/transpose_b16_8192.md", "transpose"),
    "gemm_mxfp4_blockscaled": ("profiles/gemm_mxfp4_8192_pair.md", "gemm"),
    "gemm_nvfp4_blockscaled": ("profiles/gemm_nvfp4_8192_pair.md", "gemm"),
}


def sources_sha256(group: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[group]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the kernel's ncu summary, or None if stale/absent."""
    path, group = PROFILES[kernel]
    try:
        with open(os.path.join(ROOT, path)) as fh:
            fields = dict(line.split(": ", 1) for line in fh.read().splitlines() if ": " in line)
    except OSError:
        return None
    if fields.get("kernel_sources_sha256", "").strip() != sources_sha256(group):
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def gpu_ids(torch, dev_index):
    """(uuid string "GPU-...", or None) of the CUDA device, for NVML / nvidia-smi."""
    try:
        u = getattr(torch.cuda.get_device_properties(dev_index), "uuid", None)
    except Exception:               # noqa: BLE001
        u = None
    if u is None:
        return None
    u = str(u)
    return u if u.startswith("GPU-") else "GPU-" + u


class ClockSampler:
    """SM clock and throttle reasons sampled during the timed region, with host
    timestamps (time.perf_counter), so that each sample can be attributed to
    the kernel that was running.  NVML (read-only queries through the
    driver's libnvidia-ml) every ~1 ms; else nvidia-smi every 100 ms."""

    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown"}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid, index: int, period_ms: float = 1.0):
        self.uuid = uuid
        self.index = index
        self.period = period_ms
        self.samples = []          # (host time, sm MHz, max sm MHz, set of reasons)
        self.source = None
        self._stop = threading.Event()
        self._t = None
        self._proc = None

    def _nvml(self):
        import ctypes
        try:
            L = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return None
        if L.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        ok = False
        if self.uuid:
            ok = L.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) == 0
        if not ok:
            ok = L.nvmlDeviceGetHandleByIndex_v2(self.index, ctypes.byref(h)) == 0
        if not ok:
            return None
        reasons = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(L, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        return L, h, reasons

    def __enter__(self):
        import ctypes
        nv = self._nvml()
        if nv is not None:
            L, h, reasons_fn = nv
            self.source = "nvml"
            smax = ctypes.c_uint(0)
            L.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(smax))

            def loop():
                c = ctypes.c_uint(0)
                m = ctypes.c_ulonglong(0)
                while not self._stop.is_set():
                    t = time.perf_counter()
                    if L.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(c)) == 0:
                        rs = set()
                        if reasons_fn is not None and reasons_fn(h, ctypes.byref(m)) == 0:
                            rs = {n for b, n in self.REASON_BITS.items() if m.value & b}
                        self.samples.append((t, float(c.value), float(smax.value), rs))
                    time.sleep(self.period * 1e-3)
            self._t = threading.Thread(target=loop, daemon=True)
            self._t.start()
            return self
        try:
            ident = self.uuid or str(self.index)
            self._proc = subprocess.Popen(
                ["nvidia-smi", f"--id={ident}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms=100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"

            def read():
                names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                         "sw_power_cap"]
                for line in self._proc.stdout:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) < 9:
                        continue
                    try:
                        sm, smax = float(parts[1]), float(parts[2])
                    except ValueError:
                        continue
                    rs = {n for n, v in zip(names, parts[5:9]) if v.lower() == "active"}
                    self.samples.append((time.perf_counter(), sm, smax, rs))
            self._t = threading.Thread(target=read, daemon=True)
            self._t.start()
        except (OSError, ValueError):
            self._proc = None
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
        if self._t is not None:
            self._t.join(timeout=5)

    @staticmethod
    def _summary(samples):
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        for x in samples:
            reasons |= x[3]
        return {"sm_mhz": statistics.median(x[1] for x in samples),
                "sm_max_mhz": max(x[2] for x in samples), "reasons": sorted(reasons),
                "samples": len(samples)}

    def summary(self):
        d = self._summary(self.samples)
        d["source"] = self.source
        return d

    def per_interval(self, t0_host: float, intervals):
        """Median clock of the samples that fall in each named interval.

        intervals: {name: [(start_ms, end_ms), ...]} on the device timeline,
        relative to an event recorded on an idle stream at host time t0_host."""
        out = {}
        for name, ivs in intervals.items():
            got = []
            for x in self.samples:
                g = (x[0] - t0_host) * 1e3
                if any(a <= g < b for a, b in ivs):
                    got.append(x)
            out[name] = self._summary(got)
        return out


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def make_step_inputs(torch, dev):
    def bf16(bits):
        return torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)

    def u8(bits):
        return torch.from_numpy(bits).to(dev)

    host = {
        "bf16": synth.make_inputs("sq8k", M=SIZE, N=SIZE, K=SIZE),
        "mx": synth.make_inputs("mx8k", M=SIZE, N=SIZE, K=SIZE),
        "tr": synth.make_inputs("tr8k", M=SIZE, N=SIZE),
    }
    d = {
        "A": bf16(host["bf16"]["A"]), "B": bf16(host["bf16"]["B"]),
        "mA": u8(host["mx"]["A"]), "mB": u8(host["mx"]["B"]),
        "SFA": u8(host["mx"]["SFA"]), "SFB": u8(host["mx"]["SFB"]),
        "X": torch.from_numpy(host["tr"]["X"].view(np.int16)).to(dev),
        "D": torch.empty((SIZE, SIZE), dtype=torch.float32, device=dev),
        "mD": torch.empty((SIZE, SIZE), dtype=torch.bfloat16, device=dev),
        "XT": torch.empty((SIZE, SIZE), dtype=torch.int16, device=dev),
    }
    return host, d


def probe_rates(torch, dev):
    """The tensor pipe's own rate, measured live by the library's rate probe
    (back-to-back MMAs on every SM, no memory traffic) for bf16 kind::f16 and
    E4M3 block-scaled kind::mxf8f6f4: dense FLOP per SM per clock, the SM
    clock the probe itself ran at (its cycle counter over its elapsed
    nanoseconds) and the resulting chip rate.  Run right after the timed
    region, at a similar length (~0.6 ms), so that it sees the same power
    state; the SM cycle counter, not NVML's clock reading, gives the clock
    under tensor load."""
    from blackwell_tile_gemm_gb300 import probes
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {}
    for name, kind, k, iters in (("bf16", 0, 16, 2048), ("mxfp8", 1, 32, 1024)):
        cyc = torch.zeros(2 * sms, dtype=torch.int64, device=dev)
        probes.mma_rate(kind, iters, sms, cyc)
        torch.cuda.synchronize()
        v = cyc.view(sms, 2).double()
        c = v[:, 0].median().item()
        ns = v[:, 1].median().item()
        rate = 2 * 128 * 256 * k * 4 * iters / c
        out[name] = {"flop_per_clk_per_sm": rate, "mhz": 1e3 * c / ns,
                     "tflops": sms * rate * (c / ns) * 1e9 / 1e12}
    return sms, out


def run_ours(args):
    import torch

    import blackwell_tile_gemm_gb300 as tg
    from blackwell_tile_gemm_gb300 import build as tgbuild

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the library has no CPU path)")
    tgbuild.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    host, d = make_step_inputs(torch, dev)
    flops_gemm = 2 * SIZE ** 3

    run_bf16 = args.kernel in ("all", "gemm_bf16")
    run_mx = args.kernel in ("all", "gemm_mxfp8")
    run_tr = args.kernel in ("all", "transpose")
    # FP4 GEMMs are not part of the step; --kernel times one of them alone.
    run_f4 = args.kernel in ("gemm_mxfp4", "gemm_nvfp4")
    if run_f4:
        x4 = synth.make_inputs("mxf4_8k" if args.kernel == "gemm_mxfp4" else "nvf4_8k",
                               M=SIZE, N=SIZE, K=SIZE)
        f4 = {k: torch.from_numpy(x4[k]).to(dev) for k in ("A", "B", "SFA", "SFB")}
        f4_call = tg.gemm_mxfp4_blockscaled if args.kernel == "gemm_mxfp4" \
            else tg.gemm_nvfp4_blockscaled
    flops_step = flops_gemm * (int(run_bf16) + int(run_mx) + int(run_f4))

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        if run_bf16:
            tg.gemm_bf16(d["A"], d["B"], d["D"], cta_pair=True, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        if run_mx:
            tg.gemm_mxfp8_blockscaled(d["mA"], d["mB"], d["SFA"], d["SFB"], d["mD"],
                                      cta_pair=True, stream=stream)
        if run_f4:
            f4_call(f4["A"], f4["B"], f4["SFA"], f4["SFB"], d["mD"], cta_pair=True, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        if run_tr:
            tg.tile_transpose_b16(d["X"], d["XT"], stream=stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    code, site = tg.tg_device_status()
    if code != tg.TG_OK:
        raise SystemExit(f"device status {code} (site {site}) during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    # The GEMM kernels' own SM clock over the timed launches (their cycle
    # counter against the global timer), beside NVML's samples.
    tg.kernel_clock_record(True)
    with ClockSampler(gpu_ids(torch, 0), 0) as clk:
        time.sleep(0.005)                 # a few idle samples before the region
        h0 = time.perf_counter()          # the stream is idle: t_start runs at once
        t_start.record(stream)
        for k in range(args.steps):
            step(evs[k])
        t_end.record(stream)
        torch.cuda.synchronize()
        time.sleep(0.002)
    kclk = {"bf16": tg.kernel_clock_read(tg.TG_CLOCK_BF16),
            "mxfp8": tg.kernel_clock_read(tg.TG_CLOCK_MXFP8)}
    tg.kernel_clock_record(False)
    sms, probe = probe_rates(torch, dev)
    total_ms = t_start.elapsed_time(t_end)
    code, site = tg.tg_device_status()
    if code != tg.TG_OK:
        raise SystemExit(f"device status {code} (site {site}) in the timed region")
    per = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]), e[2].elapsed_time(e[3])]
                    for e in evs])
    # Each kernel's intervals on the device timeline (ms after t_start), to
    # attribute the clock samples.
    starts = np.array([[t_start.elapsed_time(e[i]) for i in range(4)] for e in evs])
    ms_step = total_ms / args.steps
    if flops_step:
        value = flops_step / (ms_step * 1e-3) / 1e12
    else:   # transpose alone: report its bandwidth instead
        value = 2 * 2 * SIZE * SIZE / (ms_step * 1e-3) / 1e9

    peaks, peak_src = measured_peaks()
    bf16_ms, mx_ms, tr_ms = (float(per[:, i].mean()) for i in range(3))
    peak_bf16 = float(peaks["bf16_tflops"])
    names = ["gemm_bf16", f"{args.kernel}_blockscaled" if run_f4 else "gemm_mxfp8_blockscaled",
             "tile_transpose_b16"]
    clk_by_kernel = clk.per_interval(h0, {
        n: [(float(starts[k, i]), float(starts[k, i + 1])) for k in range(args.steps)]
        for i, n in enumerate(names)})

    def theoretical(tflops, kind):
        return tflops / probe[kind]["tflops"]

    def at_kernel_clock(entry, tflops, kind):
        # the pipe's peak at the clock the kernel itself ran at
        mhz, units = kclk[kind]
        if mhz > 0:
            peak = sms * probe[kind]["flop_per_clk_per_sm"] * mhz * 1e6 / 1e12
            entry.update(sm_mhz_in_kernel=mhz, frac_theoretical_at_kernel_clock=tflops / peak)

    kern = {}
    if run_bf16:
        t = flops_gemm / (bf16_ms * 1e-3) / 1e12
        c = clk_by_kernel["gemm_bf16"]
        kern["gemm_bf16"] = {"ms": bf16_ms, "tflops": t, "frac_of_bf16_peak": t / peak_bf16,
                             "sm_mhz": c["sm_mhz"], "clock_samples": c["samples"],
                             "frac_theoretical": theoretical(t, "bf16")}
        at_kernel_clock(kern["gemm_bf16"], t, "bf16")
    if run_mx:
        t = flops_gemm / (mx_ms * 1e-3) / 1e12
        c = clk_by_kernel["gemm_mxfp8_blockscaled"]
        kern["gemm_mxfp8_blockscaled"] = {
            "ms": mx_ms, "tflops": t, "frac_of_2x_bf16_peak": t / (2 * peak_bf16),
            "sm_mhz": c["sm_mhz"], "clock_samples": c["samples"],
            "frac_theoretical": theoretical(t, "mxfp8")}
        at_kernel_clock(kern["gemm_mxfp8_blockscaled"], t, "mxfp8")
    if run_f4:
        t = flops_gemm / (mx_ms * 1e-3) / 1e12
        c = clk_by_kernel[names[1]]
        kern[names[1]] = {"ms": mx_ms, "tflops": t, "frac_of_6x_bf16_peak": t / (6 * peak_bf16),
                          "sm_mhz": c["sm_mhz"], "clock_samples": c["samples"]}
    if run_tr:
        g = 2 * 2 * SIZE * SIZE / (tr_ms * 1e-3) / 1e9
        c = clk_by_kernel["tile_transpose_b16"]
        kern["tile_transpose_b16"] = {"ms": tr_ms, "gbs": g,
                                      "frac_of_hbm_peak": g / float(peaks["hbm_gbs"]),
                                      "sm_mhz": c["sm_mhz"], "clock_samples": c["samples"]}
    dominant = max(kern, key=lambda n: kern[n]["ms"])
    if dominant == "tile_transpose_b16":
        achieved, peak = kern[dominant]["gbs"], float(peaks["hbm_gbs"])
        peak_note = f"HBM copy, {peak_src}"
    elif dominant == "gemm_bf16":
        achieved, peak = kern["gemm_bf16"]["tflops"], peak_bf16
        peak_note = f"bf16 cuBLAS burst, {peak_src}"
    elif dominant == "gemm_mxfp8_blockscaled":
        achieved, peak = kern[dominant]["tflops"], 2 * peak_bf16
        peak_note = f"2 x bf16 cuBLAS burst (fp8/bf16 nominal ratio), {peak_src}"
    else:
        achieved, peak = kern[dominant]["tflops"], 6 * peak_bf16
        peak_note = f"6 x bf16 cuBLAS burst (fp4/bf16 nominal ratio), {peak_src}"
    roofline = {"bound": "hbm" if dominant == "tile_transpose_b16" else "tensor",
                "kernel": dominant, "achieved": achieved, "peak": peak,
                "unit": "GB/s" if dominant == "tile_transpose_b16" else "TFLOP/s",
                "frac": achieved / peak,
                "traffic": profiled_traffic(dominant) if SIZE == 8192 else None,
                "peak_source": peak_note}
    if dominant in ("gemm_bf16", "gemm_mxfp8_blockscaled"):
        kind = "bf16" if dominant == "gemm_bf16" else "mxfp8"
        pr = probe[kind]
        max_mhz = clk.summary()["sm_max_mhz"] or 2070.0
        at_max = sms * pr["flop_per_clk_per_sm"] * max_mhz * 1e6 / 1e12
        roofline.update({
            "frac_theoretical": achieved / pr["tflops"],
            "theoretical_peak": pr["tflops"],
            "frac_theoretical_at_kernel_clock": kern[dominant].get("frac_theoretical_at_kernel_clock"),
            "kernel_sm_mhz": kern[dominant].get("sm_mhz_in_kernel"),
            "frac_theoretical_at_max_clock": achieved / at_max,
            "theoretical_basis": (
                f"{sms} SMs x {pr['flop_per_clk_per_sm']:.0f} FLOP/clk/SM x {pr['mhz']:.0f} MHz: "
                f"the rate probe's back-to-back tcgen05.mma on every SM, at the SM clock its "
                f"cycle counter showed (NVML reports {max_mhz:.0f} MHz meanwhile; the SM cycle "
                f"counter runs slower under tensor load); at {max_mhz:.0f} MHz the peak would "
                f"be {at_max:.0f} TFLOP/s; frac_theoretical_at_kernel_clock takes the clock "
                f"the kernel's own cycle counter showed over the timed launches "
                f"(kernel_sm_mhz)")})

    # Check the timed work: the last step's outputs against the oracle on the
    # CPU-baseline sample (and the transpose against a host transpose).
    # (The end-to-end loop runs first: the oracle's host threads and buffers
    # would otherwise share the host's memory system with its copies.)
    e2e = measure_e2e(torch, tg, host, dev, stream, args.e2e_steps if args.kernel == "all" else 0,
                      flops_step)
    parity = None
    cpu = None
    if args.kernel == "all":
        cpu, samples = cpu_baseline(args.cpu_seconds)
        parity = step_parity(torch, d, host, samples)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT if flops_step else "GB/s", "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e2m1 (f32 accumulate)" if run_f4 else "bf16+e4m3 (f32 accumulate)",
        "data": "synthetic (seeded numpy; recipes in blackwell_tile_gemm_gb300/synth.py)",
        "config": {"workload": workload() if args.kernel == "all" else f"{args.kernel} only",
                   "M": SIZE, "N": SIZE, "K": SIZE,
                   "tiles": "256x256 per CTA pair, 128-byte K stages",
                   "parallelism": "single GPU",
                   "l2": "not flushed: 516 MB of step inputs > 129 MB L2"},
        "roofline": roofline, "kernels": kern, "e2e": e2e,
        "gpu_launches": (int(run_bf16) + 2 * int(run_mx) + 2 * int(run_f4) + int(run_tr))
        * args.steps,
        "clocks": clk.summary(),
        "tensor_pipe_probe": {"sms": sms, **probe},
    }
    if parity is not None:
        line["parity"] = parity
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


def step_parity(torch, d, host, samples):
    """Worst |D - ref| / tol of the timed step's GEMM outputs on the oracle's
    sample, and whether the transpose equals the host transpose bit for bit."""
    rows, cols, ref_b, mag_b, ref_m, mag_m = samples
    r_t = torch.from_numpy(rows).to(d["D"].device)
    got_b = d["D"].index_select(0, r_t).cpu().numpy().astype(np.float64)[:, cols]
    bits = d["mD"].view(torch.int16).index_select(0, r_t).cpu().numpy().view(np.uint16)[:, cols]
    got_m = synth.bf16_bits_to_f32(bits).astype(np.float64)
    # |D - ref| <= rtol * sum_k |a_k b_k| + atol: f32 D (bf16 GEMM), bf16 D (MXFP8)
    rb = float(np.max(np.abs(got_b - ref_b) / (1e-5 * mag_b + 1e-6)))
    rm = float(np.max(np.abs(got_m - ref_m) / (8e-3 * mag_m + 1e-3)))
    if not (np.all(np.isfinite(got_b)) and np.all(np.isfinite(got_m))):
        rb = rm = float("inf")
    xt = d["XT"].cpu().numpy().view(np.uint16)
    tr_ok = bool(np.array_equal(xt, host["tr"]["X"].T))
    return {"max_err_over_tol": max(rb, rm), "gemm_bf16": rb, "gemm_mxfp8_blockscaled": rm,
            "transpose_bit_exact": tr_ok,
            "sample": f"{rows.size} rows x {cols.size} columns of each GEMM's D from the last "
                      f"timed step vs the float64 oracle; transpose: every element"}


def measure_e2e(torch, tg, host, dev, stream, steps, flops_step):
    """Same step through the public API with pinned host buffers, every step:
    H2D of the step's inputs, the three calls, D2H of the three results.

    Steps are pipelined the way a caller would use the C ABI: copies in,
    compute and copies out run on three streams with two device buffer sets,
    so step i's compute overlaps step i+1's inputs and step i-1's results.
    """
    if steps <= 0:
        return None
    pin = {}
    for k, arr in (("A", host["bf16"]["A"]), ("B", host["bf16"]["B"]),
                   ("mA", host["mx"]["A"]), ("mB", host["mx"]["B"]),
                   ("SFA", host["mx"]["SFA"]), ("SFB", host["mx"]["SFB"]),
                   ("X", host["tr"]["X"])):
        t = torch.from_numpy(arr.view(np.int16) if arr.dtype == np.uint16 else arr)
        pin[k] = t.pin_memory()
    nb = 2
    out_h = [{"D": torch.empty((SIZE, SIZE), dtype=torch.float32).pin_memory(),
              "mD": torch.empty((SIZE, SIZE), dtype=torch.int16).pin_memory(),
              "XT": torch.empty((SIZE, SIZE), dtype=torch.int16).pin_memory()} for _ in range(nb)]
    ins = [{k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in pin.items()}
           for _ in range(nb)]
    outs = [{"D": torch.empty((SIZE, SIZE), dtype=torch.float32, device=dev),
             "mD": torch.empty((SIZE, SIZE), dtype=torch.bfloat16, device=dev),
             "XT": torch.empty((SIZE, SIZE), dtype=torch.int16, device=dev)} for _ in range(nb)]
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = sum(v.numel() * v.element_size() for v in out_h[0].values())
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()                                      # noqa: E731
    in_done = [ev() for _ in range(nb)]
    comp_done = [ev() for _ in range(nb)]
    out_done = [ev() for _ in range(nb)]
    for b in range(nb):                 # all buffers start free
        comp_done[b].record(s_comp)
        out_done[b].record(s_out)

    def one(i):
        b = i % nb
        d, o, oh = ins[b], outs[b], out_h[b]
        with torch.cuda.stream(s_in):
            s_in.wait_event(comp_done[b])          # inputs b no longer read
            for k in pin:
                d[k].copy_(pin[k], non_blocking=True)
            in_done[b].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_done[b])
            s_comp.wait_event(out_done[b])         # results b already copied out
            tg.gemm_bf16(d["A"].view(torch.bfloat16), d["B"].view(torch.bfloat16), o["D"],
                         cta_pair=True, stream=s_comp)
            tg.gemm_mxfp8_blockscaled(d["mA"], d["mB"], d["SFA"], d["SFB"], o["mD"],
                                      cta_pair=True, stream=s_comp)
            tg.tile_transpose_b16(d["X"], o["XT"], stream=s_comp)
            comp_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            oh["D"].copy_(o["D"], non_blocking=True)
            oh["mD"].copy_(o["mD"].view(torch.int16), non_blocking=True)
            oh["XT"].copy_(o["XT"], non_blocking=True)
            out_done[b].record(s_out)

    for i in range(nb):
        one(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    s_comp.wait_event(t0)
    s_out.wait_event(t0)
    for i in range(steps):
        one(i)
    s_in.wait_stream(s_comp)
    s_in.wait_stream(s_out)
    t1.record(s_in)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    code, site = tg.tg_device_status()
    if code != tg.TG_OK:
        raise SystemExit(f"device status {code} (site {site}) in the end-to-end loop")
    return {"value": flops_step / (ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "pipelining": "3 streams (H2D / compute / D2H), 2 device buffer sets"}


# ---------------------------------------------------------------------------
# per-workload table (--configs): one JSON line per workload, not the contract line
# ---------------------------------------------------------------------------

def run_configs(args):
    import torch

    import blackwell_tile_gemm_gb300 as tg
    from blackwell_tile_gemm_gb300 import build as tgbuild

    tgbuild.build()
    dev = torch.device("cuda", 0)
    peaks, _ = measured_peaks()
    def median_ms(fn):
        # median over 5 rounds of 10 back-to-back calls (per call), after warm-up
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        times = []
        for _ in range(5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(10):
                fn()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) / 10)
        return statistics.median(times)

    side = torch.cuda.Stream()

    def graph_ms(fn):
        # device time per call without host overhead: a CUDA graph of 10
        # calls captured on a side stream (warmed up there first, so that its
        # workspace exists before capture), median of 5 replays
        with torch.cuda.stream(side):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for _ in range(10):
                    fn()
            g.replay()
            torch.cuda.synchronize()
            times = []
            for _ in range(5):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(side)
                g.replay()
                e1.record(side)
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1) / 10)
        del g
        return statistics.median(times)

    # Fused-epilogue rows: the same 8192^3 products with each non-trivial op.
    bias = torch.linspace(-2.0, 2.0, SIZE, device=dev, dtype=torch.float32)
    epilogue_rows = {"silu_affine": dict(silu_affine=(1.5, -0.25)), "bias": dict(bias=bias),
                     "bias_silu": dict(bias=bias, bias_silu=True)}
    rows = [(name, w, {}) for name, w in synth.WORKLOADS.items()]
    rows += [(f"{base}+{op}", synth.WORKLOADS[base], kw) for base in ("sq8k", "mx8k")
             for op, kw in epilogue_rows.items()]
    # the gathered-row product with the rows loaded inside the GEMM by gather4
    rows += [("moe_8k+gather_tma", synth.WORKLOADS["moe_8k"], {"gather_tma": True})]
    if args.only:
        keep = set(args.only.split(","))
        rows = [r for r in rows if r[0] in keep]
    for name, w, epi in rows:
        x = synth.make_inputs(w)
        if w.kind == "transpose":
            X = torch.from_numpy(x["X"].view(np.int16)).to(dev)
            out = torch.empty((w.N, w.M), dtype=torch.int16, device=dev)
            fn = lambda: tg.tile_transpose_b16(X, out)           # noqa: E731
        elif w.kind in ("mxfp8", "mxfp4", "nvfp4"):
            A, B, SFA, SFB = (torch.from_numpy(x[k]).to(dev) for k in ("A", "B", "SFA", "SFB"))
            D = torch.empty((w.M, w.N), device=dev,
                            dtype=torch.bfloat16 if w.d_dtype == "bf16" else torch.float32)
            call = {"mxfp8": tg.gemm_mxfp8_blockscaled, "mxfp4": tg.gemm_mxfp4_blockscaled,
                    "nvfp4": tg.gemm_nvfp4_blockscaled}[w.kind]
            fn = lambda: call(A, B, SFA, SFB, D, cta_pair=w.cta_pair, **epi)  # noqa: E731
        else:
            A = torch.from_numpy(x["A"].view(np.int16)).to(dev).view(torch.bfloat16)
            B = torch.from_numpy(x["B"].view(np.int16)).to(dev).view(torch.bfloat16)
            D = torch.empty((w.M, w.N), device=dev,
                            dtype=torch.bfloat16 if w.d_dtype == "bf16" else torch.float32)
            if not epi and w.epi_add:
                epi = dict(epilogue_add=w.epi_add)
            if w.kind == "gather":
                idx = torch.from_numpy(x["idx"]).to(dev)
                fn = lambda: tg.gemm_bf16_gather(A, idx, B, D, cta_pair=w.cta_pair, **epi)  # noqa
                # the dense product of the same shape (A rows in place), for comparison
                ms_tile = None if epi else median_ms(
                    lambda: tg.gemm_bf16(A[:w.M], B, D, cta_pair=w.cta_pair))
            elif w.kind == "skinny":
                fn = lambda: tg.gemm_bf16_skinny(A, B, D, **epi)  # noqa: E731
                # the same product through the 128 x 256 tile kernel, for comparison
                ms_tile = median_ms(lambda: tg.gemm_bf16(A, B, D))
            else:
                fn = lambda: tg.gemm_bf16(A, B, D, cta_pair=w.cta_pair,  # noqa: E731
                                          multicast=w.multicast, **epi)
        ms = median_ms(fn)
        ms_g = graph_ms(fn)
        code, _ = tg.tg_device_status()
        line = {"workload": name, "describe": w.describe, "status": code, "ms_median": ms,
                "timing": "median of 5 rounds of 10 back-to-back calls",
                "ms_graph": ms_g,
                "timing_graph": "CUDA graph of 10 calls, median of 5 replays (no host overhead)"}
        if epi:
            line["epilogue"] = sorted(epi)
        if w.kind == "transpose":
            gbs = 2 * 2 * w.M * w.N / (ms * 1e-3) / 1e9
            line.update(gbs=gbs, frac_of_hbm=gbs / float(peaks["hbm_gbs"]),
                        gbs_graph=2 * 2 * w.M * w.N / (ms_g * 1e-3) / 1e9)
        elif w.kind == "skinny":
            # algorithmic bytes: B and A read once, D written once (bf16)
            nbytes = 2 * w.N * w.K + 2 * w.M * w.K + 2 * w.M * w.N
            gbs = nbytes / (ms * 1e-3) / 1e9
            line.update(gbs=gbs, frac_of_hbm=gbs / float(peaks["hbm_gbs"]),
                        gbs_graph=nbytes / (ms_g * 1e-3) / 1e9,
                        tflops=w.flops / (ms * 1e-3) / 1e12,
                        splits=tg.skinny_split_count(w.N, w.K, 0),
                        tile_kernel_ms=ms_tile)
        elif w.kind == "gather":
            tf = w.flops / (ms * 1e-3) / 1e12
            line.update(tflops=tf, frac_of_cublas_bf16_burst_scaled=tf / float(peaks["bf16_tflops"]),
                        tflops_graph=w.flops / (ms_g * 1e-3) / 1e12, dense_same_shape_ms=ms_tile)
        else:
            tf = w.flops / (ms * 1e-3) / 1e12
            # nominal dense ratios to bf16 (2.25 / 4.5 / 13.5 PFLOP/s per GPU)
            ratio = {"mxfp8": 2, "mxfp4": 6, "nvfp4": 6}.get(w.kind, 1)
            pk = float(peaks["bf16_tflops"]) * ratio
            line.update(tflops=tf, frac_of_cublas_bf16_burst_scaled=tf / pk,
                        tflops_graph=w.flops / (ms_g * 1e-3) / 1e12)
            if w.kind in ("mxfp4", "nvfp4"):
                # the tensor-pipe rate the FP4 rate probe measures: 4x bf16 per clock
                line["frac_of_probe_rate_4x_bf16"] = tf / (float(peaks["bf16_tflops"]) * 4)
        print(json.dumps(line), flush=True)
        del fn
        torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------

_SAMPLE = {}


def _oracle_sample_inputs():
    if not _SAMPLE:
        _SAMPLE["bf16"] = synth.make_inputs("sq8k", M=SIZE, N=SIZE, K=SIZE)
        _SAMPLE["mx"] = synth.make_inputs("mx8k", M=SIZE, N=SIZE, K=SIZE)
    return _SAMPLE


def oracle_sample(rows_per_gemm: int, cols: int, offset: int):
    """Oracle on `rows_per_gemm` full-K rows x `cols` columns of each 8192^3
    GEMM; returns (flops, seconds, (rows, cols, ref, mag of bf16, ref, mag of
    MXFP8))."""
    import oracle
    x = _oracle_sample_inputs()
    rows = np.unique((np.arange(rows_per_gemm) * 61 + offset) % SIZE)
    cs = np.unique((np.arange(cols) * 37 + offset) % SIZE)
    t0 = time.perf_counter()
    rb, mb = oracle.gemm_bf16(x["bf16"]["A"], x["bf16"]["B"], rows=rows, cols=cs)
    rm, mm = oracle.gemm_mxfp8(x["mx"]["A"], x["mx"]["B"], x["mx"]["SFA"], x["mx"]["SFB"],
                               rows=rows, cols=cs)
    dt = time.perf_counter() - t0
    return 2 * 2 * rows.size * cs.size * SIZE, dt, (rows, cs, rb, mb, rm, mm)


def single_thread_tiny():
    """The oracle on one thread for the 128 x 128 x 256 bf16 product (f32 D):
    median seconds of 5 runs."""
    import oracle
    x = synth.make_inputs("tiny")
    n = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        times = []
        for _ in range(5):
            t0 = time.perf_counter()
            oracle.gemm_bf16(x["A"], x["B"])
            times.append(time.perf_counter() - t0)
    finally:
        oracle.set_num_threads(n)
    return statistics.median(times)


def cpu_baseline(target_seconds: float):
    """The oracle on a growing sample until one run takes about target_seconds;
    returns (the cpu_baseline object, the last sample's oracle values)."""
    import oracle
    oracle.build()
    _oracle_sample_inputs()
    cores = oracle.num_threads()
    cols = min(1024, SIZE)
    rows = max(cores, 16)
    flops, dt, samples = oracle_sample(rows, cols, 0)
    while dt < 0.6 * target_seconds and rows < SIZE:
        rows = min(SIZE, rows * 2)
        flops, dt, samples = oracle_sample(rows, cols, rows)
    t1 = single_thread_tiny()
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "seconds": dt, "cpu_model": cpu_model(),
            "single_thread": {"workload": "bf16 128x128x256, f32 D (the tiny workload)",
                              "seconds": t1, "gflops": 2 * 128 * 128 * 256 / t1 / 1e9},
            "sample": (f"float64 oracle on {samples[0].size} rows x {samples[1].size} columns "
                       f"(all K = {SIZE}) of each {SIZE}^3 GEMM (bf16 and MXFP8), operands "
                       f"decoded per call")}, samples


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    _oracle_sample_inputs()
    cores = oracle.num_threads()
    rows, cols = min(4 * cores, SIZE), min(512, SIZE)
    for _ in range(args.warmup):
        oracle_sample(rows, cols, 0)
    flops = 0.0
    secs = 0.0
    for k in range(args.steps):
        f, dt, _ = oracle_sample(rows, cols, k + 1)
        flops += f
        secs += dt
    value = flops / secs / 1e12
    sample = (f"per step: float64 oracle on {rows} rows x {cols} columns (all K = {SIZE}) of "
              f"each {SIZE}^3 GEMM (bf16 and MXFP8)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded numpy; recipes in blackwell_tile_gemm_gb300/synth.py)",
        "config": {"workload": workload() if args.kernel == "all" else f"{args.kernel} only",
                   "M": SIZE, "N": SIZE, "K": SIZE,
                   "parallelism": "host cores (OpenMP over output rows)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--configs", action="store_true",
                    help="time every workload of the table (one JSON line each) and exit")
    ap.add_argument("--size", type=int, default=8192,
                    help="M = N = K of the GEMMs and the transpose side (default 8192)")
    ap.add_argument("--only", default="",
                    help="with --configs: comma-separated workload rows to run (default all)")
    ap.add_argument("--kernel", choices=["all", "gemm_bf16", "gemm_mxfp8", "transpose",
                                         "gemm_mxfp4", "gemm_nvfp4"],
                    default="all", help="run one part of the step only (profiling)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.size < 256 or args.size % 256:
        ap.error("--size must be a positive multiple of 256")
    global SIZE
    SIZE = args.size
    rank, world, _ = dist_env()
    if args.impl == "reference":
        # the oracle on host cores: rank 0 only, whatever the launch
        run_reference(args, rank, world)
        return
    if args.gpus > 1 or world > 1:
        # Single-GPU library: no multi-GPU run (its multicast TMA kernels are
        # 1-GPU code), so nothing is launched on any GPU.
        if rank == 0:
            print(json.dumps({"metric": METRIC, "n_gpus": max(args.gpus, world),
                              "unavailable": "the library is single-GPU code (one process "
                                             "drives one GPU); run bench.py with --gpus 1"}),
                  flush=True)
        return
    if args.configs:
        run_configs(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
