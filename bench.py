#!/usr/bin/env python3
"""Benchmark of the GB300 software-pipelined tiled GEMM.

Default workload: fp16 C = A.B^T at M = N = K = 8192, entries N(0,1)/sqrt(K)
from seed 2, fp32 accumulation, fp16 output, pipelined kernel.  One step is
one full GEMM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--stages S] [--variant pipelined|single_buffer]
                  [--layout nt|nn] [--epilogue auto|none|gelu|relu] [--out-f32]

--impl reference times the CPU oracle (fp64, OpenMP) on a bounded sample of
the same workload: a block of output rows per step.

Multi-GPU (torchrun, one rank per GPU): every rank runs its own independent
replica of the workload (the GEMM has no exchange step); the job's value is
all ranks' flops over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gemm_inputs  # noqa: E402

METRIC = "GEMM TFLOP/s (2MNK/time) at fp16 8192^3 on 1 GB300; % of dense tensor-core peak"
UNIT = "TFLOP/s"
FALLBACK_TFLOPS = 1900.0
FALLBACK_HBM = 6800.0
NOMINAL_TFLOPS = 2250.0            # dense fp16/bf16, no sparsity
NOMINAL_HBM_GBS = 7900.0
TENSOR_FLOP_PER_SM_CYCLE = 8192    # dense fp16/bf16 tcgen05 rate of one SM
L2_BYTES = 126 * 1024 * 1024


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="gemm_8192_f16", choices=sorted(gemm_inputs.WORKLOADS))
    ap.add_argument("--stages", type=int, default=0,
                    help="K slices in flight; 0 = the workload's depth (DEFAULT_STAGES, else 6)")
    ap.add_argument("--variant", default="pipelined", choices=["pipelined", "single_buffer"])
    ap.add_argument("--tile-n", type=int, default=0)
    ap.add_argument("--raster-group", type=int, default=0)
    ap.add_argument("--cta-group", type=int, default=0, choices=[0, 1, 2])
    ap.add_argument("--k-serpentine", type=int, default=0, choices=[-1, 0, 1],
                    help="K order of successive waves: 0 auto, 1 alternate, -1 always ascending")
    ap.add_argument("--tail-split", type=int, default=0,
                    help="K-splitting of the last partial wave: 0 auto, -1 off, k >= 2 forced")
    ap.add_argument("--layout", default="nt", choices=["nt", "nn"],
                    help="nt: B is (N, K), C = A.B^T; nn: B is (K, N), C = A.B")
    ap.add_argument("--epilogue", default="auto", choices=["auto", "none", "gelu", "relu"],
                    help="auto: the workload's own epilogue")
    ap.add_argument("--out-f32", action="store_true", help="write C in fp32")
    ap.add_argument("--bias", action="store_true",
                    help="add a seeded per-column bias before the epilogue (no e2e figure)")
    ap.add_argument("--flush-l2", default="auto", choices=["auto", "on", "off"],
                    help="auto: flush L2 between steps when the operands fit in it")
    ap.add_argument("--dist-reps", type=int, default=30,
                    help="extra individually timed steps for the p10/p50/p90 spread")
    ap.add_argument("--no-cublas", action="store_true",
                    help="skip the torch.matmul (cuBLAS) context timing")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-other-configs", dest="other_configs", action="store_false",
                    help="skip the compact measurements of the other configurations")
    ap.add_argument("--other-steps", type=int, default=20,
                    help="timed steps of each other configuration")
    ap.add_argument("--sustained-seconds", type=float, default=1.5,
                    help="length of the back-to-back sustained window (0: none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_TFLOPS, "bf16_tflops_sustained": 1700.0,
                "hbm_gbs": FALLBACK_HBM}, "fallback"


def source_digest():
    from software_pipelined_tiled_gemm_gb300 import _build
    return _build.kernel_digest()


def traffic_from_profiles(workload, digest):
    """DRAM bytes per launch of the GEMM kernel from a committed ncu summary,
    if that summary was taken on the current kernel sources."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, fn)) as f:
            for line in f:
                if not line.startswith("bench-traffic:"):
                    continue
                kv = dict(x.split("=", 1) for x in line.split()[1:] if "=" in x)
                if kv.get("workload") == workload and kv.get("source_digest") == digest:
                    try:
                        return int(kv["dram_bytes_per_launch"])
                    except (KeyError, ValueError):
                        return None
    return None


# nvmlClocksEventReason* bits that matter for a measurement
NVML_REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                    0x40: "hw_thermal_slowdown"}


def nvml_reason_names(bits):
    return [n for b, n in sorted(NVML_REASON_BITS.items()) if bits & b]


def summarize_clocks(samples, t0, t1, max_mhz):
    """Clock record of a timed region from (time, sm_mhz, power_w, [reasons])
    samples: the samples inside [t0, t1], or -- when the region is shorter
    than the sampling period -- the two nearest to its middle."""
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": max_mhz, "reasons": ["no samples"]}
    inside = [x for x in samples if t0 is not None and t0 <= x[0] <= t1]
    window = "timed region"
    if not inside:
        mid = (t0 + t1) / 2 if t0 is not None else samples[-1][0]
        inside = sorted(samples, key=lambda x: abs(x[0] - mid))[:2]
        window = "nearest to the timed region"
    return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": max_mhz,
            "reasons": sorted({n for x in inside for n in x[3]}), "samples": len(inside),
            "window": window, "power_w_max": max(x[2] for x in inside)}


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read from NVML (the driver's
    libnvidia-ml, through ctypes; read-only queries) by a thread every 2 ms,
    kept only when they fall inside the timed region.  A region of a few tens
    of milliseconds -- a short bench run -- is too short for nvidia-smi's
    polling, which then yields one or two samples from outside the load."""

    def __init__(self, pci_bus_id, index):
        import ctypes
        import threading
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        rc = 1
        if pci_bus_id:
            rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h))
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h))
        if rc != 0:
            raise OSError("no NVML handle for the device")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        self.samples = []
        self.stop_evt = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.t0 = self.t1 = None

    def _run(self):
        ct = self.ct
        clk, mw, rs = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        while not self.stop_evt.is_set():
            ok = self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk)) == 0
            self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw))
            self.reasons_fn(self.h, ct.byref(rs))
            if ok:
                self.samples.append((time.time(), float(clk.value), mw.value / 1000.0,
                                     nvml_reason_names(int(rs.value))))
            time.sleep(0.002)

    def start(self):
        self.thread.start()
        time.sleep(0.05)

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def stop(self):
        self.stop_evt.set()
        self.thread.join(timeout=5)
        try:
            self.lib.nvmlShutdown()
        except Exception:
            pass
        out = summarize_clocks(self.samples, self.t0, self.t1, self.max_mhz)
        out["source"] = "nvml"
        return out


def make_clock_sampler(dev, index):
    """NVML sampler when the driver library loads, else nvidia-smi."""
    try:
        import torch
        props = torch.cuda.get_device_properties(dev)
        bus = None
        if hasattr(props, "pci_bus_id"):
            bus = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                         getattr(props, "pci_device_id", 0))
        return NvmlClockSampler(bus, index)
    except Exception:
        return ClockSampler(index)


class ClockSampler:
    """nvidia-smi clock/throttle samples, kept only when they fall inside the
    timed region (host wall-clock window marked with mark_start/mark_stop)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.5)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    @classmethod
    def parse_rows(cls, text):
        """(time, sm_mhz, max_mhz, power_w, [reasons]) from nvidia-smi's CSV
        rows (the FIELDS columns, no header, no units); bad rows skipped."""
        samples = []
        for r in (line.split(",") for line in text.splitlines() if line.strip()):
            try:
                samples.append((cls._parse_ts(r[0]), float(r[2]), float(r[3]), float(r[4]),
                                [n for i, n in enumerate(cls.REASONS)
                                 if len(r) > 6 + i and r[6 + i].strip().lower() == "active"]))
            except (ValueError, IndexError):
                continue
        return samples

    @staticmethod
    def _parse_ts(text):
        # "YYYY/MM/DD HH:MM:SS.mmm", local time of this host
        text = text.strip()
        main, _, frac = text.partition(".")
        t = time.mktime(time.strptime(main, "%Y/%m/%d %H:%M:%S"))
        return t + (float("0." + frac) if frac else 0.0)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        samples = self.parse_rows(self.tmp.read())
        os.unlink(self.tmp.name)
        max_mhz = max((x[2] for x in samples), default=None)
        return summarize_clocks([(t, mhz, w, rs) for t, mhz, _, w, rs in samples],
                                self.t0, self.t1, max_mhz)


def reduce_max(value, world_size, device=None):
    """Largest `value` over all ranks (the slowest rank decides the job time)."""
    if world_size <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step, steps, world_size, elapsed_ms):
    """Whole-job TFLOP/s: every rank's steps over the slowest rank's time."""
    return flops_per_step * steps * world_size / (elapsed_ms * 1e-3) / 1e12


def cpu_baseline(A, B, w, seconds, threads=0, epi=None, bias=None):
    """Time the oracle (as it is) on a block of output rows of this workload
    (A is (M, K), B is (N, K)): the first and the last `rows` / 2 rows, so the
    sample reaches both the first tiles and the last wave's.  Returns the
    record, the row indices and the oracle's fp64 values of those rows."""
    import oracle
    import torch
    oracle.build()
    # calibrate on a few rows, then size the sample to about `seconds`
    probe = max(1, min(w.M, max(2, oracle.max_threads())))
    t0 = time.perf_counter()
    oracle.gemm_nt(A[:probe], B, w.dtype, epilogue=epi, threads=threads, bias=bias)
    dt = max(time.perf_counter() - t0, 1e-3)
    rows = int(max(1, min(w.M, probe * seconds / dt)))
    head = (rows + 1) // 2
    idx = sorted(set(range(head)) | set(range(w.M - (rows - head), w.M)))
    block = torch.cat([A[:head], A[w.M - (rows - head):]]) if rows > head else A[:head]
    t0 = time.perf_counter()
    ref = oracle.gemm_nt(block, B, w.dtype, epilogue=epi, threads=threads, bias=bias)
    el = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K
    cores = oracle.max_threads()
    out = {"value": flops / el / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": "%d of %d output rows (the first %d and the last %d; all %d columns, "
                     "full K=%d), %.1f s" % (rows, w.M, head, rows - head, w.N, w.K, el)}
    # The same oracle on one core, on a smaller block (about seconds / 5).
    t0 = time.perf_counter()
    oracle.gemm_nt(A[:1], B, w.dtype, epilogue=epi, threads=1, bias=bias)
    dt1 = max(time.perf_counter() - t0, 1e-3)
    rows1 = int(max(1, min(w.M, seconds / 5 / dt1)))
    t0 = time.perf_counter()
    oracle.gemm_nt(A[:rows1], B, w.dtype, epilogue=epi, threads=1, bias=bias)
    el1 = time.perf_counter() - t0
    oracle.gemm_nt(A[:1], B, w.dtype, epilogue=epi, threads=cores)  # restore the thread count
    out["single_thread"] = {"value": 2.0 * rows1 * w.N * w.K / el1 / 1e12, "unit": UNIT,
                            "sample": "%d output rows, %.1f s" % (rows1, el1)}
    return out, idx, ref


def parity_of_rows(C_rows, ref, dtype, f32):
    """Per-element and Frobenius error of the rows of a result against the
    oracle's values of the same rows (the tolerance the parity tests use)."""
    import numpy as np
    import oracle
    from tests import tolerance
    if f32:
        got = C_rows.numpy().astype(np.float64)
        kind = "f32"
    else:
        import torch
        got = oracle.decode(C_rows.contiguous().view(torch.int16).numpy().view(np.uint16), dtype)
        kind = dtype
    st = tolerance.compare(got, ref, kind)
    return {"ok": st["ok"], "elements": int(got.size), "max_ulp": st["max_ulp"],
            "max_abs": st["max_abs"], "frob": st["frob"], "bad": st["bad"],
            "tolerance": "|gpu - oracle| <= 2 ulp(|oracle|) + 1e-3 per element; relative "
                         "Frobenius <= 1e-3"}


def run_reference(args, w, ws, rank):
    """CPU oracle arm: each step computes a bounded block of output rows."""
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    A, B = gemm_inputs.make(w)
    epi_name = w.epilogue if args.epilogue == "auto" else args.epilogue
    epi = None if epi_name == "none" else epi_name
    total_steps = args.steps + args.warmup
    per_step = max(0.5, min(8.0, 150.0 / max(total_steps, 1)))
    probe = max(1, min(w.M, max(2, oracle.max_threads())))
    t0 = time.perf_counter()
    oracle.gemm_nt(A[:probe], B, w.dtype, epilogue=epi)
    dt = max(time.perf_counter() - t0, 1e-3)
    rows = int(max(1, min(w.M, probe * per_step / dt)))
    for i in range(args.warmup):
        oracle.gemm_nt(A[(i * rows) % w.M:][:rows], B, w.dtype, epilogue=epi)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.gemm_nt(A[(i * rows) % w.M:][:rows], B, w.dtype, epilogue=epi)
    el = time.perf_counter() - t0
    flops = 2.0 * rows * w.N * w.K * args.steps
    value = flops / el / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "input_dtype": w.dtype,
                   "epilogue": epi_name, "layout": args.layout,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle",
                         "sample": "%d of %d output rows per step (all columns, full K)" % (rows, w.M)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# Ring depth (K slices in flight) each workload is measured at unless
# --stages says otherwise: 6 (the pages' 4-6 concurrent steps, measured
# best for the tensor-bound shapes on GB300), and 8 for the HBM-bound
# skinny shape, whose 64-row A slices leave room for two more slices of B
# (26.9 -> 26.2 us per launch back to back).
DEFAULT_STAGES = {"skinny_64x8192x8192_f16": 8}


def default_stages(name):
    return DEFAULT_STAGES.get(name, 6)


# The other configurations reported beside the headline in one run: the
# workloads the GEMM is specified on, plus the single-buffer contrast.
OTHER_CONFIGS = [("gemm_256_f16", "pipelined"), ("gemm_4096_f16", "pipelined"),
                 ("gemm_8192_f16", "single_buffer"), ("gelu_3072x16384x4096_bf16", "pipelined"),
                 ("ragged_4095x4097x8191_f16", "pipelined"), ("skinny_64x8192x8192_f16", "pipelined")]


def measure_config(sg, torch, dev, stream, w, variant, stages, steps, warmup, peaks, peak_src,
                   scrub):
    """A compact measurement of one configuration with the headline's
    protocol: inputs resident, `warmup` untimed steps, then `steps` steps back
    to back between two events on the launch stream, or -- when the operands
    fit in L2 -- each step after an L2 flush, bracketed by its own events.
    Reports TFLOP/s, the roofline of its bound and torch.matmul on the same
    operands as context."""
    epi = None if w.epilogue == "none" else w.epilogue
    if variant == "single_buffer":
        stages = 1
    A, B = gemm_inputs.make(w)
    a, b = A.to(dev), B.to(dev)
    c = torch.empty(w.M, w.N, dtype=a.dtype, device=dev)
    plan = sg.Plan(w.M, w.N, w.K, w.dtype, epi, stages, variant, dev.index)
    sptr = stream.cuda_stream
    operand_bytes = (w.M * w.K + w.N * w.K) * 2
    flush = operand_bytes <= L2_BYTES

    def timed(fn, n):
        with torch.cuda.stream(stream):
            for _ in range(max(warmup, 3)):
                fn()
            if not flush:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(n):
                    fn()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                return e0.elapsed_time(e1) / n
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n)]
            for e0, e1 in evs:
                scrub.fill_(1)
                e0.record(stream)
                fn()
                e1.record(stream)
        torch.cuda.synchronize(dev)
        return sum(e0.elapsed_time(e1) for e0, e1 in evs) / n

    try:
        ms = timed(lambda: plan.run_ptr(a.data_ptr(), b.data_ptr(), c.data_ptr(), sptr), steps)
        ds, detail = plan.check()
        if ds != 0:
            raise SystemExit("device status %d (detail %#x) in %s" % (ds, detail, w.name))
        info = plan.info()
    finally:
        plan.close()
    flops = 2.0 * w.M * w.N * w.K
    min_bytes = 2.0 * (w.M * w.K + w.N * w.K + w.M * w.N)
    tflops = flops / (ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_TFLOPS))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM))
    out = {"variant": variant, "stages": info["stages"], "value": tflops, "unit": UNIT,
           "ms_per_step": ms, "steps": steps, "kernels_per_step": info["kernels_per_run"],
           "l2": "flushed before every step" if flush else "operands larger than L2; no flush",
           "plan": "%dx%d tiles, cta_group %d, %d slice(s) per slot, %s" % (
               info["tile_m"], info["tile_n"], info["cta_group"], info["k_sub"],
               "stream-K tail" if info["stream_k"] else
               ("narrow tail tiles" if info["tail_splits"] > 1 else "whole tiles"))}
    if flops / min_bytes < peak * 1e12 / (hbm * 1e9):
        out["roofline"] = {"bound": "hbm", "achieved": min_bytes / (ms * 1e-3) / 1e9, "peak": hbm,
                           "unit": "GB/s", "peak_source": "%s hbm_gbs" % peak_src}
    else:
        out["roofline"] = {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": UNIT,
                           "peak_source": "%s bf16_tflops" % peak_src}
    out["roofline"]["frac"] = out["roofline"]["achieved"] / out["roofline"]["peak"]
    if epi is None and variant == "pipelined":
        bt = b.t()
        cms = timed(lambda: torch.matmul(a, bt), steps)
        out["cublas_context"] = {"ms": cms, "tflops": flops / (cms * 1e-3) / 1e12}
    del a, b, c
    return out


def main():
    args = parse()
    ws, rank, local = dist_env()
    w = gemm_inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w, ws, rank)

    import torch
    import torch.distributed as dist
    import software_pipelined_tiled_gemm_gb300 as sg

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if ws > 1:
            dist.barrier()

    epi_name = w.epilogue if args.epilogue == "auto" else args.epilogue
    epi = None if epi_name == "none" else epi_name
    if args.stages == 0:
        args.stages = default_stages(w.name)
    if args.variant == "single_buffer":
        args.stages = 1
    nn = args.layout == "nn"
    tuning = dict(tile_n=args.tile_n, raster_group=args.raster_group, cta_group=args.cta_group,
                  tail_split=args.tail_split, k_serpentine=args.k_serpentine, b_kn=1 if nn else 0,
                  out_f32=1 if args.out_f32 else 0)
    A_cpu, B_cpu = gemm_inputs.make(w)
    if nn:  # the same draw, stored (K, N)
        B_cpu = B_cpu.t().contiguous()
    A, B = A_cpu.to(dev), B_cpu.to(dev)
    c_dtype = torch.float32 if args.out_f32 else A.dtype
    C = torch.empty(w.M, w.N, dtype=c_dtype, device=dev)
    plan = sg.Plan(w.M, w.N, w.K, w.dtype, epi, args.stages, args.variant, local, **tuning)
    stream = torch.cuda.Stream(dev)
    sptr = stream.cuda_stream
    a_p, b_p, c_p = A.data_ptr(), B.data_ptr(), C.data_ptr()
    bias_cpu = gemm_inputs.bias(w.N, w.dtype, seed=w.seed) if args.bias else None
    bias_t = bias_cpu.to(dev) if bias_cpu is not None else None
    bias_p = bias_t.data_ptr() if bias_t is not None else 0
    operand_bytes = (w.M * w.K + w.N * w.K) * 2
    flush = args.flush_l2 == "on" or (args.flush_l2 == "auto" and operand_bytes <= L2_BYTES)
    scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev) if flush else None

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            plan.run_ptr(a_p, b_p, c_p, sptr, bias_p)
    stream.synchronize()
    ds, detail = plan.check()
    if ds != 0:
        raise SystemExit("device status %d (detail %#x) after warm-up" % (ds, detail))
    info = plan.info()

    # Without flushing, two events bracket the timed region on the launch
    # stream and nothing else runs on it, so the average launch duration is
    # elapsed / steps (events between launches would also cut the
    # programmatic-dependent-launch overlap of consecutive GEMMs).  With
    # flushing (operands that fit in L2), each step is bracketed by its own
    # events and a 2 x L2 write runs between steps, outside them.
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    clocks = make_clock_sampler(dev, local)
    clocks.start()
    barrier()
    torch.cuda.synchronize(dev)
    clocks.mark_start()
    if not flush:
        ev0.record(stream)
        for _ in range(args.steps):
            plan.run_ptr(a_p, b_p, c_p, sptr, bias_p)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        elapsed_ms = ev0.elapsed_time(ev1)
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                scrub.fill_(1)
                e0.record(stream)
                plan.run_ptr(a_p, b_p, c_p, sptr, bias_p)
                e1.record(stream)
        torch.cuda.synchronize(dev)
        elapsed_ms = sum(e0.elapsed_time(e1) for e0, e1 in evs)
    clocks.mark_stop()
    barrier()
    clk = clocks.stop()
    ds, detail = plan.check()
    if ds != 0:
        raise SystemExit("device status %d (detail %#x) after timed steps" % (ds, detail))
    elapsed_ms = reduce_max(elapsed_ms, ws, dev)
    # The result of the last timed step, for the parity check below.
    C_timed = C.cpu()

    flops = 2.0 * w.M * w.N * w.K
    value = job_throughput(flops, args.steps, ws, elapsed_ms)
    # Per-step device time; with padded operands a step is the padding copy
    # plus the GEMM (kernels_per_step 2), otherwise the GEMM kernel alone.
    kavg = elapsed_ms / args.steps
    achieved = flops / (kavg * 1e-3) / 1e12

    # Spread of single-step device times (outside the timed region): each
    # step bracketed by its own events, L2 flushed first when flushing.
    dist_ms = None
    if args.dist_reps > 0:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.dist_reps)]
        with torch.cuda.stream(stream):
            for e0, e1 in evs:
                if flush:
                    scrub.fill_(1)
                e0.record(stream)
                plan.run_ptr(a_p, b_p, c_p, sptr, bias_p)
                e1.record(stream)
        torch.cuda.synchronize(dev)
        t = sorted(e0.elapsed_time(e1) for e0, e1 in evs)
        q = lambda f: t[min(len(t) - 1, int(round(f * (len(t) - 1))))]  # noqa: E731
        dist_ms = {"p10": q(0.1), "p50": q(0.5), "p90": q(0.9), "reps": len(t)}

    # torch.matmul (cuBLAS) on the same operands: context only, not timed
    # as part of this library.
    # Same protocol as the timed region: back to back between two events, or
    # (when flushing) each rep after an L2 flush, bracketed by its own events.
    cublas = None

    def ref_mm():
        return torch.matmul(A, bt) if bias_t is None else torch.addmm(bias_t, A, bt)

    if not args.no_cublas and epi is None and not args.out_f32:
        bt = B if nn else B.t()
        reps = 20
        with torch.cuda.stream(stream):
            for _ in range(3):
                ref_mm()
            if not flush:
                c0 = torch.cuda.Event(enable_timing=True)
                c1 = torch.cuda.Event(enable_timing=True)
                c0.record(stream)
                for _ in range(reps):
                    ref_mm()
                c1.record(stream)
            else:
                cevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                        for _ in range(reps)]
                for e0, e1 in cevs:
                    scrub.fill_(1)
                    e0.record(stream)
                    ref_mm()
                    e1.record(stream)
        torch.cuda.synchronize(dev)
        if not flush:
            cms = c0.elapsed_time(c1) / reps
        else:
            cms = sum(e0.elapsed_time(e1) for e0, e1 in cevs) / reps
        cublas = {"tflops": 2.0 * w.M * w.N * w.K / (cms * 1e-3) / 1e12, "ms": cms,
                  "what": "torch.matmul on the same device operands, %d reps, %s" % (
                      reps, "L2 flushed before each" if flush else "back to back")}

    # end-to-end through the C ABI with host buffers (pinned)
    e2e = None
    if args.e2e_steps > 0 and not args.bias:
        hA, hB = A_cpu.pin_memory(), B_cpu.pin_memory()
        hC = torch.empty(w.M, w.N, dtype=c_dtype).pin_memory()
        eplan = sg.Plan(w.M, w.N, w.K, w.dtype, epi, args.stages, args.variant, local, **tuning)
        eplan.run_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), sptr)
        barrier()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            eplan.run_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), sptr)
        el = reduce_max(time.perf_counter() - t0, ws, dev)
        eplan.close()
        e2e = {"value": job_throughput(flops, args.e2e_steps, ws, el * 1e3), "unit": UNIT,
               "h2d_bytes_per_step": (w.M * w.K + w.N * w.K) * 2,
               "d2h_bytes_per_step": w.M * w.N * C.element_size()}

    peaks, peak_src = load_peaks()

    # Sustained: the same plan back to back for about --sustained-seconds,
    # long enough for the power controller to settle at its cap, with a
    # clock record of its own; reported against the measured sustained
    # cuBLAS rate.  The burst region above is too short for the power
    # sensor, so its clock record shows the boost clock.
    sustained = None
    if args.sustained_seconds > 0:
        n_sus = max(10, int(args.sustained_seconds * 1e3 / max(kavg, 1e-3)))
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        sclk = make_clock_sampler(dev, local)
        sclk.start()
        barrier()
        torch.cuda.synchronize(dev)
        sclk.mark_start()
        s0.record(stream)
        for _ in range(n_sus):
            plan.run_ptr(a_p, b_p, c_p, sptr, bias_p)
        s1.record(stream)
        torch.cuda.synchronize(dev)
        sclk.mark_stop()
        barrier()
        sus_clk = sclk.stop()
        ds, detail = plan.check()
        if ds != 0:
            raise SystemExit("device status %d (detail %#x) after sustained steps" % (ds, detail))
        sus_ms = reduce_max(s0.elapsed_time(s1), ws, dev)
        sus_val = job_throughput(flops, n_sus, ws, sus_ms)
        sus_peak = float(peaks.get("bf16_tflops_sustained", 1700.0))
        sustained = {"value": sus_val, "unit": UNIT, "steps": n_sus, "seconds": sus_ms * 1e-3,
                     "peak": sus_peak, "frac": sus_val / ws / sus_peak,
                     "peak_source": "%s bf16_tflops_sustained" % peak_src,
                     "l2": "back to back, no flush", "clocks": sus_clk}
        mhz = sus_clk.get("sm_mhz")
        if mhz:
            # Rate per clock: TFLOP/s per GHz of the median SM clock, and the
            # fraction of the tensor pipes' rate at that clock (152 SMs x 8192
            # flop per SM-cycle for dense fp16/bf16).
            sustained["tflops_per_ghz"] = sus_val / ws / (mhz * 1e-3)
            sustained["frac_of_pipe_at_clock"] = (
                sus_val / ws / (info["sm_count"] * TENSOR_FLOP_PER_SM_CYCLE * mhz * 1e6 / 1e12))

    # The other configurations, measured in the same run (single GPU only).
    others = None
    if args.other_configs and ws == 1 and args.workload == "gemm_8192_f16" and not nn \
            and args.variant == "pipelined" and not args.out_f32 and not args.bias:
        others = {}
        if scrub is None:
            scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
        for name, variant in OTHER_CONFIGS:
            others[name + ("" if variant == "pipelined" else ":" + variant)] = measure_config(
                sg, torch, dev, stream, gemm_inputs.WORKLOADS[name], variant, default_stages(name),
                args.other_steps, 3, peaks, peak_src, scrub)

    long_region = elapsed_ms > 1000.0
    peak_key = "bf16_tflops_sustained" if long_region else "bf16_tflops"
    peak = float(peaks.get(peak_key, FALLBACK_TFLOPS))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM))
    digest = source_digest()
    # Profile key: the workload plus whatever changes the kernel or its traffic.
    variant_key = (w.name + ("" if not nn else ":nn")
                   + ("" if epi_name == w.epilogue else ":" + epi_name)
                   + (":single" if args.variant == "single_buffer" else "")
                   + (":f32" if args.out_f32 else "")
                   + (":bias" if args.bias else ""))
    traffic = traffic_from_profiles(variant_key, digest)
    min_bytes = 2.0 * (w.M * w.K + w.N * w.K) + float(w.M * w.N * C.element_size())
    # Below the ridge point (peak flops / HBM bandwidth) the GEMM is bound by
    # moving its operands once; report it against the copy bandwidth.
    if flops / min_bytes < peak * 1e12 / (hbm * 1e9):
        roof = {"bound": "hbm", "achieved": min_bytes / (kavg * 1e-3) / 1e9, "peak": hbm,
                "unit": "GB/s", "traffic": traffic,
                "peak_source": "%s hbm_gbs" % peak_src,
                "tensor_tflops": achieved, "kernel_ms_avg": kavg,
                "kernels_per_step": info["kernels_per_run"]}
    else:
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                "traffic": traffic,
                "peak_source": "%s %s (fp16 and bf16 share the dense tensor rate)" % (
                    peak_src, peak_key),
                "kernel_ms_avg": kavg, "kernels_per_step": info["kernels_per_run"]}
    roof["frac"] = roof["achieved"] / roof["peak"]
    # Beside the measured denominators: the published nominal rate, and the
    # tensor pipes' rate at the maximum SM clock.
    max_mhz = float(clk.get("sm_max_mhz") or peaks.get("sm_max_mhz") or 2070.0)
    if roof["bound"] == "tensor":
        roof["nominal_peak"] = NOMINAL_TFLOPS
        roof["frac_of_nominal"] = achieved / NOMINAL_TFLOPS
        roof["nominal_source"] = ("GB300 dense fp16/bf16 tensor rate without sparsity, "
                                  "%.0f TFLOP/s (NVIDIA's published figure)" % NOMINAL_TFLOPS)
        clock_peak = info["sm_count"] * TENSOR_FLOP_PER_SM_CYCLE * max_mhz * 1e6 / 1e12
        roof["clock_peak"] = clock_peak
        roof["frac_of_clock_peak"] = achieved / clock_peak
        roof["clock_peak_source"] = ("%d SMs x %d flop per SM-cycle x %.0f MHz (maximum SM clock)"
                                     % (info["sm_count"], TENSOR_FLOP_PER_SM_CYCLE, max_mhz))
    else:
        roof["nominal_peak"] = NOMINAL_HBM_GBS
        roof["frac_of_nominal"] = roof["achieved"] / NOMINAL_HBM_GBS
        roof["nominal_source"] = "GB300 HBM3e nominal bandwidth, %.0f GB/s" % NOMINAL_HBM_GBS

    # The oracle timed on the host cores.  The rows it computes are also the
    # parity check of the timed result (and of the end-to-end call's): every
    # element of those rows against the oracle, at the parity tests' bound.
    cpu = None
    parity = None
    if rank == 0 and not args.no_cpu_baseline and ws == 1:
        cpu, rows_idx, ref_rows = cpu_baseline(A_cpu, B_cpu.t().contiguous() if nn else B_cpu, w,
                                               args.cpu_seconds, epi=epi, bias=bias_cpu)
        parity = parity_of_rows(C_timed[rows_idx], ref_rows, w.dtype, bool(args.out_f32))
        parity["what"] = ("the C of the last timed step, %d whole rows (the cpu_baseline "
                          "sample) against the fp64 oracle" % len(rows_idx))
        if e2e is not None:
            e2e["parity"] = parity_of_rows(hC[rows_idx], ref_rows, w.dtype, bool(args.out_f32))

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": elapsed_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic",
            "config": {
                "workload": w.name, "M": w.M, "N": w.N, "K": w.K, "input_dtype": w.dtype,
                "accumulate": "f32", "epilogue": epi_name, "variant": args.variant,
                "layout": args.layout, "output_dtype": "f32" if args.out_f32 else w.dtype,
                "bias": bool(args.bias),
                "stages": info["stages"], "tile": "%dx%dx%d" % (info["tile_m"], info["tile_n"],
                                                               info["tile_k"]),
                "grid": info["grid"], "raster_group": info["raster_group"],
                "k_serpentine": info["k_serpentine"],
                "cta_group": info["cta_group"], "k_slices_per_slot": info["k_sub"],
                "tail_splits": info["tail_splits"],
                "tail_tiles": info["tail_tiles"],
                "l2": ("L2 flushed (2 x %d MiB write) before every step" % (L2_BYTES >> 20))
                if flush else
                ("inputs larger than L2 (%d MiB of operands vs %d MiB L2); no flush"
                 % (operand_bytes >> 20, L2_BYTES >> 20))
                if operand_bytes > L2_BYTES else "operands fit in L2, not flushed (warm)",
                "parallelism": "replicas" if ws > 1 else "single-gpu",
            },
            "roofline": roof,
            "clocks": clk,
            "e2e": e2e,
            "gpu_launches": args.steps * info["kernels_per_run"],
            "cpu_baseline": cpu,
            "parity": parity,
            "sustained": sustained,
            "step_ms_dist": dist_ms,
            "cublas_context": cublas,
            "other_configs": others,
        }
        print(json.dumps(line), flush=True)
    plan.close()
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
