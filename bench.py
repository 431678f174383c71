"""Benchmark of the guarded W8A8 linear on B300.

Metric: W8A8 linear TOPS (activation quantisation + INT32-exact GEMM + fused
epilogue) on the video-branch projection, M=6144, K=N=4096, bf16 inputs with
1 % outlier columns, on one GPU.  One step = one call of w8a8_linear through
the C ABI: the activation-quantisation kernel, then the GEMM+epilogue kernel
as its programmatic dependent.  Inputs are resident in HBM, and L2 is flushed
(256 MiB written) before every step.  Each step is timed with CUDA events on
the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-cpu-baseline] [--no-per-workload] [--profile]

The JSON line also carries:
  int8_peak     the measured rates of every exact INT8 route on this GPU
                (warp-level mma.sync s8, torch._int_mm, and the bf16 tcgen05
                pipe that carries the codes here) and ptxas's answer on the
                integer tcgen05 MMA; the largest rate is the denominator of
                the metric's "% of INT8 tensor peak" (frac_of_int8_peak)
  per_workload  every workload (tiny, video, MLP up and down, high-res x2,
                audio x4): median step time of 50 cold-L2 steps and of 250
                hot-L2 steps (graph replays), the quantiser and the GEMM
                alone, the native BF16 linear on the same shape, and their
                rooflines
  roofline, quant_roofline, e2e, cpu_baseline, clocks, and the timings of
                the MLP pair, the norm prologue and the Query/Key blocks

--impl reference times the CPU oracle (plain C) on the host cores on a
bounded row sample of the same workload.  Under torchrun (N > 1) every rank
runs an independent replica of the workload (rows are independent, no
collective on the data path; "weak" scaling), rank 0 prints the line.
"""
import argparse
import ctypes
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import w8a8_workloads as wl  # noqa: E402

METRIC = "W8A8 linear TOPS (quant+GEMM+epilogue) at M=6144,K=N=4096; % INT8 tensor peak"
UNIT = "TOPS"
WORKLOAD = "video"
FLUSH_BYTES = 256 << 20
PER_WORKLOAD_COLD = 50        # cold-L2 steps per per-workload measurement
PER_WORKLOAD_GRAPH = 50       # steps per captured graph (hot L2)
PER_WORKLOAD_REPLAYS = 5      # graph replays per hot-L2 measurement
SPIN_BEFORE_STEPS_CYCLES = 4_000_000   # about 2 ms at the B300's 2032 MHz

# Algorithmic bytes (the method's own accounting, with INT8 codes of 1 B):
#   quantiser per activation element: input (2 B bf16, 4 B fp32) + 1 B int8 code; + 4 B per row (scale)
#   GEMM per launch: Xq (M K) + Wq (N K) + sx (4 M) + sw (4 N) + bias (2 N or 4 N) + Y (2 M N)
# Bytes as built (the codes are carried as bf16 for the tensor cores):
#   quantiser: input + 2 B per code + 4 B per row; GEMM: 2 B per code of Xq and Wq


def quant_bytes(M, K, in_size, code_size=1):
    return M * K * in_size + M * K * code_size + 4 * M


def gemm_bytes(M, N, K, bias_size=2, code_size=1):
    return code_size * (M * K + N * K) + 4 * M + 4 * N + bias_size * N + 2 * M * N


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one GEMM launch
# on the default workload, from one ncu capture of it.
# Valid only for the kernel sources it was taken on: the key is a digest of
# their code (comments excluded), and the bench reports null traffic when the
# code has changed since.
GEMM_SOURCES = ["w8a8_int8_linear_act_b300/csrc/gemm_tcgen05.cuh",
                "w8a8_int8_linear_act_b300/csrc/ptx_sm103.cuh"]
GEMM_TRAFFIC = {"4c6119a28db36d2a": 164.14e6, "fd3b36ebdcdd6b15": 167.30e6, "7b406bc72ed21ced": 167.26e6,
                "25c25b09727d8201": 168.16e6, "523c87070454c4cf": 165.93e6, "6bc2643ac23e769c": 167.38e6}


def sources_digest(paths):
    """Digest of the code in `paths` with // comments, trailing blanks and
    empty lines removed, so that editing a comment does not invalidate a
    measurement of the same code."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            for line in f:
                code = re.sub(r"//.*$", "", line).rstrip()
                if code:
                    h.update(code.encode("utf-8") + b"\n")
    return h.hexdigest()[:16]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# SM clock and throttle reasons (read-only queries)
# ---------------------------------------------------------------------------

class _NvmlCtypes:
    """The few read-only NVML queries the sampler needs, through ctypes on
    the driver's libnvidia-ml (used when the Python NVML module is absent)."""

    # nvmlClocksEventReason* bits
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, index, pci):
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.h = ctypes.c_void_p()
        rc = -1
        if pci:
            rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci.encode(), ctypes.byref(self.h))
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h))
        if rc != 0:
            raise RuntimeError("no NVML handle")
        try:
            self._reasons = self.lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self._reasons = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_clock(self):
        v = ctypes.c_uint()
        return v.value if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(v)) == 0 else None

    def max_sm_clock(self):
        v = ctypes.c_uint()
        return v.value if self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(v)) == 0 else None

    def power_w(self):
        v = ctypes.c_uint()
        return v.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(v)) == 0 else None

    def reasons(self):
        v = ctypes.c_ulonglong()
        if self._reasons(self.h, ctypes.byref(v)) != 0:
            return set()
        return {k for k, b in self.BITS.items() if v.value & b}

    def close(self):
        self.lib.nvmlShutdown()


class _NvmlModule:
    REASONS = {
        "hw_slowdown": "nvmlClocksEventReasonHwSlowdown",
        "hw_thermal_slowdown": "nvmlClocksEventReasonHwThermalSlowdown",
        "sw_thermal_slowdown": "nvmlClocksEventReasonSwThermalSlowdown",
        "sw_power_cap": "nvmlClocksEventReasonSwPowerCap",
        "hw_power_brake_slowdown": "nvmlClocksEventReasonHwPowerBrakeSlowdown",
    }

    def __init__(self, index, pci):
        import pynvml
        pynvml.nvmlInit()
        self.nv = pynvml
        self.h = (pynvml.nvmlDeviceGetHandleByPciBusId(pci.encode()) if pci
                  else pynvml.nvmlDeviceGetHandleByIndex(index))
        self.masks = {k: getattr(pynvml, v) for k, v in self.REASONS.items() if hasattr(pynvml, v)}

    def sm_clock(self):
        return self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM)

    def max_sm_clock(self):
        return self.nv.nvmlDeviceGetMaxClockInfo(self.h, self.nv.NVML_CLOCK_SM)

    def power_w(self):
        return self.nv.nvmlDeviceGetPowerUsage(self.h) / 1000.0

    def reasons(self):
        active = self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
        return {k for k, m in self.masks.items() if active & m}

    def close(self):
        self.nv.nvmlShutdown()


class ClockSampler:
    """Samples the SM clock, power and the clock-event (throttle) reasons every
    5 ms from before the first GPU work to after the last (read-only NVML
    queries: the Python module, else ctypes on libnvidia-ml, else
    `nvidia-smi -lms 20`).  `mark(name)` / `end(name)` bracket a region (the
    headline's timed steps); `summary()` reports the whole run and each
    region."""

    SMI_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
                  "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
                  "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int, pci_bus_id=None, period_s: float = 0.005):
        self.index = index
        self.pci = pci_bus_id
        self.period = period_s
        self.samples = []          # (t, sm_mhz, power_w, reasons)
        self.max_mhz = None
        self.source = None
        self.errors = []
        self.regions = {}
        self._stop = threading.Event()
        self._thread = None
        self._q = None
        self._proc = None

    def __enter__(self):
        for cls, name in ((_NvmlModule, "nvml"), (_NvmlCtypes, "nvml-ctypes")):
            try:
                self._q = cls(self.index, self.pci)
                self.max_mhz = self._q.max_sm_clock()
                self.source = name
                self._thread = threading.Thread(target=self._run_nvml, daemon=True)
                self._thread.start()
                return self
            except Exception as e:  # try the next source
                self.errors.append("%s: %s: %s" % (name, type(e).__name__, e))
                self._q = None
        self._start_smi()
        return self

    def _start_smi(self):
        import subprocess
        target = self.pci if self.pci else str(self.index)
        cmd = ["nvidia-smi", "-i", target, "--query-gpu=" + ",".join(self.SMI_FIELDS),
               "--format=csv,noheader,nounits", "-lms", "20"]
        try:
            self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self._thread = threading.Thread(target=self._run_smi, daemon=True)
            self._thread.start()
        except Exception as e:
            self.errors.append("nvidia-smi: %s" % e)

    def _run_nvml(self):
        q = self._q
        while not self._stop.is_set():
            try:
                self.samples.append((time.perf_counter(), q.sm_clock(), q.power_w(), q.reasons()))
            except Exception as e:
                self.errors.append("sample: %s" % e)
                if len(self.errors) > 20:
                    return
            time.sleep(self.period)

    def _run_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != len(self.SMI_FIELDS):
                continue
            try:
                mhz, self.max_mhz = float(parts[0]), float(parts[1])
                pw = float(parts[2])
            except ValueError:
                continue
            reasons = {n for n, v in zip(names, parts[3:]) if v.lower() == "active"}
            self.samples.append((time.perf_counter(), mhz, pw, reasons))

    def _sample_now(self):
        # One sample taken at once (NVML sources), so that a region shorter
        # than the sampling period still holds its first and last instants.
        if self._q is None:
            return
        try:
            self.samples.append((time.perf_counter(), self._q.sm_clock(), self._q.power_w(), self._q.reasons()))
        except Exception as e:
            self.errors.append("sample: %s" % e)

    def mark(self, name):
        self.regions[name] = [time.perf_counter(), None]
        self._sample_now()

    def end(self, name):
        self._sample_now()
        self.regions[name][1] = time.perf_counter()

    def __exit__(self, *exc):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if self._thread is not None:
            self._thread.join(timeout=5)
        if self._q is not None:
            try:
                self._q.close()
            except Exception:
                pass
        return False

    @staticmethod
    def _stats(samples, max_mhz):
        if not samples:
            return {"sm_mhz": None, "samples": 0, "reasons": ["unsampled"]}
        # Samples under load: power above the run's idle level (the lowest
        # tenth of the power readings plus 100 W), or all when power is unknown.
        pw = sorted(p for _, _, p, _ in samples if p is not None)
        idle = pw[len(pw) // 10] if pw else None
        load = [s for s in samples if idle is None or s[2] is None or s[2] > idle + 100.0] or samples
        reasons = set()
        for s in load:
            reasons |= s[3]
        return {"sm_mhz": statistics.median(s[1] for s in load if s[1] is not None),
                "sm_mhz_min": min(s[1] for s in load if s[1] is not None),
                "sm_max_mhz": max_mhz, "reasons": sorted(reasons), "samples": len(samples),
                "samples_under_load": len(load),
                "power_w_max": max(pw) if pw else None}

    def summary(self):
        out = self._stats(self.samples, self.max_mhz)
        out["source"] = self.source
        out["scope"] = ("every 5 ms from before the warm-up to after the last GPU pass of this run, and at the "
                        "start and end of each region")
        for name, (t0, t1) in self.regions.items():
            inside = [s for s in self.samples if t0 <= s[0] <= (t1 if t1 is not None else float("inf"))]
            st = self._stats(inside, self.max_mhz)
            st["seconds"] = (t1 - t0) if t1 is not None else None
            out["region_" + name] = st
        if self.errors:
            out["errors"] = self.errors[:3]
        return out


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (reported baseline; also the --impl reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(case, rows: int, X_bits, Wq, sw, bias_f32):
    """Oracle on the first `rows` rows: act quant + INT32 GEMM + epilogue.
    Returns (seconds, ops)."""
    import numpy as np

    import oracle
    t0 = time.perf_counter()
    xq, sx = oracle.quantize_rows(X_bits[:rows])
    acc = oracle.gemm_s32(xq, Wq, np.arange(rows, dtype=np.int64))
    oracle.epilogue(acc, sx, sw, bias_f32)
    dt = time.perf_counter() - t0
    return dt, 2 * rows * case.N * case.K


def oracle_inputs(case, X, W, b):
    import numpy as np

    import oracle

    def host(t):
        # bf16 as its bit patterns (uint16), fp32 as is: the oracle's two input forms
        t = t.contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()

    Wq, sw = oracle.quantize_rows(host(W))
    bias = host(b)
    return host(X), Wq, sw, oracle.bf16_bits_to_f32(bias) if bias.dtype == np.uint16 else bias


def calibrate_rows(case, inputs, target_s: float) -> int:
    rows = 8
    dt, _ = oracle_sample(case, min(rows, case.M), *inputs)
    while dt < target_s / 8 and rows < case.M:
        rows = min(case.M, rows * 4)
        dt, _ = oracle_sample(case, rows, *inputs)
    return max(1, min(case.M, int(rows * target_s / max(dt, 1e-6))))


def cpu_baseline(case, X, W, b, target_s=12.0):
    import oracle
    inputs = oracle_inputs(case, X, W, b)
    rows = calibrate_rows(case, inputs, target_s)
    dt, ops = oracle_sample(case, rows, *inputs)
    return {"value": ops / dt / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "first %d of %d rows of the %s workload (act quant + INT32 GEMM + epilogue), %.1f s"
                      % (rows, case.M, case.name, dt)}


def run_reference(args):
    rank, world, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        if rank != 0:
            dist.destroy_process_group()
            return
    import oracle
    case = wl.CASES[args.workload]
    X, W, b = wl.make(case)
    inputs = oracle_inputs(case, X, W, b)
    per_step = max(2.0, 150.0 / max(1, args.steps + args.warmup))
    rows = calibrate_rows(case, inputs, per_step)
    for _ in range(args.warmup):
        oracle_sample(case, rows, *inputs)
    times = []
    ops = 0
    for _ in range(args.steps):
        dt, ops = oracle_sample(case, rows, *inputs)
        times.append(dt)
    ms = statistics.mean(times) * 1e3
    value = ops / (statistics.mean(times)) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int64 scalar (CPU oracle)", "data": "synthetic",
        "config": config_dict(case),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": "first %d of %d rows per step" % (rows, case.M)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


WORKLOAD_TEXT = {
    "video": "video-branch projection",
    "mlp_up": "video-branch MLP up-projection",
    "mlp_down": "video-branch MLP down-projection",
    "hires_n4k": "high-resolution video tokens, projection",
    "hires_n16k": "high-resolution video tokens, MLP up-projection",
    "tiny": "tiny fp32 layer",
}


def config_dict(case):
    what = WORKLOAD_TEXT.get(case.name, "audio-branch ragged shape (last row all zero)")
    dt = "bf16" if case.dtype == torch.bfloat16 else "fp32"
    extra = " (1% outlier columns x20)" if case.outliers else ""
    return {"workload": "%s: X %s [%d,%d]%s x W [%d,%d]^T + bias" % (what, dt, case.M, case.K, extra, case.N, case.K),
            "M": case.M, "K": case.K, "N": case.N, "l2": "flushed before every step (256 MiB write)",
            "weights": "quantised offline (static), not timed"}


# ---------------------------------------------------------------------------
# GPU timing helpers
# ---------------------------------------------------------------------------

class Timer:
    """CUDA-event timing on one stream.  cold(): the 256 MiB flush before
    every call, events around the call alone.  hot(): `per_graph` calls
    captured back to back in one CUDA graph and replayed (no host work
    between calls, L2 warm from the previous call); returns per-call times
    of each replay."""

    def __init__(self, stream, flush):
        self.stream = stream
        self.flush = flush
        self.flush2 = None    # the clean flush's second buffer, made on first use
        self.sink = torch.zeros((), dtype=torch.int64, device=flush.device)
        self.graphs = []      # captured graphs stay alive with the buffers they use, until release()

    def cold(self, fn, n, warm=3):
        for _ in range(warm):
            self.flush.zero_()
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b in ev:
            self.flush.zero_()
            a.record(self.stream)
            fn()
            b.record(self.stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    def cold_split(self, fns, n, warm=3):
        """Each of `fns` in turn after one flush, an event between them:
        per-function times of each call."""
        for _ in range(warm):
            self.flush.zero_()
            for f in fns:
                f()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)] for _ in range(n)]
        for e in evs:
            self.flush.zero_()
            e[0].record(self.stream)
            for i, f in enumerate(fns):
                f()
                e[i + 1].record(self.stream)
        torch.cuda.synchronize()
        return [[e[i].elapsed_time(e[i + 1]) for e in evs] for i in range(len(fns))]

    def clean_flush(self):
        """The write flush, then a read of a second buffer of the same size,
        so that L2 is left holding clean lines (the next kernel's misses then
        evict without writing back)."""
        self.flush.zero_()
        if self.flush2 is None:
            self.flush2 = torch.ones_like(self.flush)
        torch.sum(self.flush2.view(torch.int32), dim=0, dtype=torch.int64, out=self.sink)

    def cold_graph(self, fns, n=PER_WORKLOAD_COLD, replays=7, clean=False):
        """Device time per call of each of `fns` in turn after a flush,
        without host launch latency: graph k holds n x (flush, fns[0], ...,
        fns[k-1]); fns[k-1] costs (T_k - T_{k-1}) / n, each T the median of
        `replays` replays, the graphs replayed in turn (so that slow drifts
        of the clock fall on all of them alike).  Returns one time (ms) per
        function."""
        cur = torch.cuda.current_stream()
        gs = torch.cuda.Stream()
        gs.wait_stream(self.stream)
        graphs = []
        for k in range(len(fns) + 1):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(gs):
                for f in fns[:k]:
                    f()
                gs.synchronize()
                with torch.cuda.graph(g, stream=gs):
                    for _ in range(n):
                        if clean:
                            self.clean_flush()
                        else:
                            self.flush.zero_()
                        for f in fns[:k]:
                            f()
            torch.cuda.synchronize()
            self.graphs.append(g)
            graphs.append(g)
            g.replay()
        torch.cuda.synchronize()
        ts = [[] for _ in graphs]
        for _ in range(replays):
            for k, g in enumerate(graphs):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(cur)
                g.replay()
                b.record(cur)
                b.synchronize()
                ts[k].append(a.elapsed_time(b))
        totals = [med(t) for t in ts]
        return [(totals[k + 1] - totals[k]) / n for k in range(len(fns))]

    def hot(self, fn, per_graph=PER_WORKLOAD_GRAPH, replays=PER_WORKLOAD_REPLAYS):
        g = torch.cuda.CUDAGraph()
        gs = torch.cuda.Stream()
        gs.wait_stream(self.stream)
        with torch.cuda.stream(gs):
            fn()
            gs.synchronize()
            with torch.cuda.graph(g, stream=gs):
                for _ in range(per_graph):
                    fn()
        torch.cuda.synchronize()
        self.graphs.append(g)
        cur = torch.cuda.current_stream()
        g.replay()
        torch.cuda.synchronize()
        out = []
        for _ in range(replays):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(cur)
            g.replay()
            b.record(cur)
            b.synchronize()
            out.append(a.elapsed_time(b) / per_graph)
        return out

    def release(self):
        torch.cuda.synchronize()
        self.graphs = []


def med(xs):
    return statistics.median(xs)


def int8_peaks(dev, pk):
    """Rates of every exact INT8 x INT8 -> INT32 route this GPU offers, and
    the denominator of the metric's "% of INT8 tensor peak": the largest."""
    from w8a8_int8_linear_act_b300 import peaks as pp
    out = {"unit": "TOPS"}
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, threads = 4 * sms, 256
    sink = torch.zeros(blocks * threads, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def probe(kind):
        iters = 256
        pp.mma_sync_launch(kind, blocks, threads, iters, sink, stream)
        torch.cuda.synchronize()
        best = 0.0
        for _ in range(2):                      # calibrate to about 40 ms per launch
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            pp.mma_sync_launch(kind, blocks, threads, iters, sink, stream)
            b.record(stream)
            b.synchronize()
            ms = a.elapsed_time(b)
            best = max(best, pp.mma_sync_ops(kind, blocks, threads, iters) / (ms * 1e-3) / 1e12)
            iters = int(min(1 << 22, max(iters, iters * 40.0 / max(ms, 1e-3))))
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            pp.mma_sync_launch(kind, blocks, threads, iters, sink, stream)
            b.record(stream)
            b.synchronize()
            best = max(best, pp.mma_sync_ops(kind, blocks, threads, iters) / (a.elapsed_time(b) * 1e-3) / 1e12)
        return best

    try:
        out["mma_sync_s8"] = probe(pp.MMA_S8)
        out["mma_sync_bf16_tflops"] = probe(pp.MMA_BF16)
        out["mma_sync_note"] = ("warp-level mma.sync (m16n8k32 s8 / m16n8k16 bf16) from registers, %d CTAs x 8 "
                                "warps x 8 independent MMAs, best of 3 launches of about 40 ms" % blocks)
    except Exception as e:
        out["mma_sync_error"] = "%s: %s" % (type(e).__name__, e)
    try:
        n = 8192
        g = torch.Generator(device=dev).manual_seed(5)
        A = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=dev, generator=g)
        B = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=dev, generator=g)
        for _ in range(3):
            torch._int_mm(A, B.t())
        torch.cuda.synchronize()
        ts = []
        for _ in range(10):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            torch._int_mm(A, B.t())
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        out["torch_int_mm"] = 2 * n ** 3 / (min(ts) * 1e-3) / 1e12
        out["torch_int_mm_note"] = "torch._int_mm int8 [8192,8192] x [8192,8192]^T -> int32, best of 10"
        del A, B
    except Exception as e:
        out["torch_int_mm_error"] = "%s: %s" % (type(e).__name__, e)
    ok, msg, ver = pp.ptxas_accepts_tcgen05("sm_103a", "i8")
    out["tcgen05_kind_i8_sm_103a"] = {"accepted": ok, "ptxas": msg, "ptxas_version": ver}
    out["tcgen05_bf16_codes"] = pk["bf16_tflops"]
    out["tcgen05_bf16_codes_note"] = ("the bf16 tcgen05 pipe carrying the INT8 codes exactly (the route this "
                                      "library uses): MEASURED_PEAKS.json bf16 dense burst (%s)" % pk["source"])
    cands = {k: out[k] for k in ("mma_sync_s8", "torch_int_mm", "tcgen05_bf16_codes") if k in out}
    out["denominator"] = max(cands, key=cands.get)
    out["denominator_tops"] = cands[out["denominator"]]
    out["rule"] = "the largest measured rate of any exact INT8 x INT8 -> INT32 route on this GPU"
    return out


# ---------------------------------------------------------------------------
# Per-workload table (all five configurations)
# ---------------------------------------------------------------------------

def measure_workload(w8, name, dev, stream, flush, pk, sampler=None):
    c = wl.CASES[name]
    M, K, N = c.M, c.K, c.N
    X, W, b = wl.make(c)
    Xd, bd = X.to(dev), b.to(dev)
    Wq, sw = w8.quantize_weight(W.to(dev))
    Wp = w8.pack_weight(Wq)
    ws = torch.empty(w8.workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    T = Timer(stream, flush)

    def step():
        w8.linear(Xd, Wp, sw, bd, out=Y, workspace=ws, stream=torch.cuda.current_stream())

    cur = torch.cuda.current_stream
    if sampler is not None:
        sampler.mark(name + ":cold")
    cold = T.cold_graph([step])[0]
    cold_ev = med(T.cold(step, PER_WORKLOAD_COLD))
    if sampler is not None:
        sampler.end(name + ":cold")
        sampler.mark(name + ":hot")
    hot = T.hot(step)
    if sampler is not None:
        sampler.end(name + ":hot")
    qg = T.cold_graph([lambda: w8.linear_quant_stage(Xd, ws, stream=cur()),
                       lambda: w8.linear_gemm_stage(M, K, Wp, sw, bd, Y, ws, stream=cur())])
    st, bits_ = w8.read_status(ws)
    if st != 0:
        raise RuntimeError("%s: device status %d bits %#x" % (name, st, bits_))
    Xb = Xd.to(torch.bfloat16)
    Wb = W.to(torch.bfloat16).to(dev)
    bb = bd.to(torch.bfloat16)
    wsb = torch.empty(w8.bf16_linear_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
    if sampler is not None:
        sampler.mark(name + ":bf16_cold")
    bf = T.cold_graph([lambda: w8.bf16_linear(Xb, Wb, bb, out=Y, workspace=wsb, stream=cur())])[0]
    if sampler is not None:
        sampler.end(name + ":bf16_cold")
        sampler.mark(name + ":bf16_hot")
    bf_hot = T.hot(lambda: w8.bf16_linear(Xb, Wb, bb, out=Y, workspace=wsb,
                                          stream=torch.cuda.current_stream()))
    if sampler is not None:
        sampler.end(name + ":bf16_hot")
    T.release()
    ops = c.ops
    in_size = X.element_size()
    bias_size = b.element_size()
    s_cold, s_hot, q_ms, g_ms, b_ms, b_hot = cold, med(hot), qg[0], qg[1], bf, med(bf_hot)
    qb = quant_bytes(M, K, in_size)
    gb = gemm_bytes(M, N, K, bias_size)
    # Roofline floors: the quantiser's bytes at the copy bandwidth; the GEMM at
    # the larger of its operations at the tensor peak and its bytes at the
    # copy bandwidth; the step = the two in sequence.
    q_floor = qb / (pk["hbm_gbs"] * 1e9) * 1e3
    g_floor_t = ops / (pk["bf16_tflops"] * 1e12) * 1e3
    g_floor_m = gb / (pk["hbm_gbs"] * 1e9) * 1e3
    g_floor = max(g_floor_t, g_floor_m)
    plan = w8.gemm_plan(M, N, K)
    form = w8.gemm_form(M, N, K)
    row = {
        "M": M, "K": K, "N": N, "x_dtype": "bf16" if in_size == 2 else "fp32", "ops": ops,
        "step_us_cold": s_cold * 1e3, "step_us_hot": s_hot * 1e3, "step_us_cold_events": cold_ev * 1e3,
        "tops_cold": ops / (s_cold * 1e-3) / 1e12, "tops_hot": ops / (s_hot * 1e-3) / 1e12,
        "quant_us": q_ms * 1e3, "gemm_us": g_ms * 1e3,
        "gemm_tflops": ops / (g_ms * 1e-3) / 1e12,
        "gemm_frac_of_tensor_peak": ops / (g_ms * 1e-3) / 1e12 / pk["bf16_tflops"],
        "gemm_bound": "tensor" if g_floor_t >= g_floor_m else "hbm",
        "gemm_floor_us": g_floor * 1e3, "gemm_frac_of_roofline": g_floor / g_ms,
        "quant_gbs": qb / (q_ms * 1e-3) / 1e9, "quant_frac": qb / (q_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
        "step_floor_us": (q_floor + g_floor) * 1e3, "step_frac_of_roofline_cold": (q_floor + g_floor) / s_cold,
        "bf16_linear_us_cold": b_ms * 1e3, "bf16_linear_us_hot": b_hot * 1e3,
        "w8a8_over_bf16_cold": b_ms / s_cold, "w8a8_over_bf16_hot": b_hot / s_hot,
        "gemm_form": ({"form": "cluster-K", "tile": [128, form[1]], "cluster_k": form[2], "ctas": form[3]}
                      if form[0] == 1 else
                      {"form": "persistent", "dp_tiles": plan[0], "splits": plan[1], "tail_units": plan[2],
                       "ctas": plan[3], "ctas_per_tile": plan[4]}),
        "n_cold": PER_WORKLOAD_COLD, "n_hot": PER_WORKLOAD_GRAPH * PER_WORKLOAD_REPLAYS,
    }
    del Xd, bd, Wq, sw, Wp, ws, Y, Xb, Wb, bb, wsb
    return row, (X, W, b)


PER_WORKLOAD_NOTE = (
    "cold L2: a CUDA graph of %d x (256 MiB flush, call) minus one of %d flushes, per call (median of 3 "
    "replays; no host launch latency inside), also step_us_cold_events: the median of %d event-timed "
    "calls after a flush (host-bound for the small shapes); hot L2: %d back-to-back calls per CUDA graph, "
    "median of %d replays (sustained load, where the power cap can lower the SM clock, see clocks_hot); "
    "quant_us / gemm_us: the two stage calls, each the difference of graphs with and without it; bytes: "
    "int8 codes (1 B) as the method moves them; GEMM floor = max(ops / bf16 tensor peak, bytes / HBM copy "
    "bandwidth); bf16_linear: the guard's native BF16 fallback on the same shape (w8a8_over_bf16 > 1: W8A8 "
    "faster)"
    % (PER_WORKLOAD_COLD, PER_WORKLOAD_COLD, PER_WORKLOAD_COLD, PER_WORKLOAD_GRAPH, PER_WORKLOAD_REPLAYS))


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import w8a8_int8_linear_act_b300 as w8

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    pk = peaks()
    case = wl.CASES[args.workload]
    X, W, b = wl.make(case)
    M, K, N = case.M, case.K, case.N
    Xd, Wd, bd = X.to(dev), W.to(dev), b.to(dev)
    Wq, sw = w8.quantize_weight(Wd)
    Wp = w8.pack_weight(Wq)
    del Wd
    ws = torch.empty(w8.workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    T = Timer(stream, flush)
    try:
        pr = torch.cuda.get_device_properties(dev)
        pci = "%08X:%02X:%02X.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
    except Exception:
        pci = None
    sampler = ClockSampler(dev.index, pci)
    sampler.__enter__()

    def step():
        # One call of the hot path: w8a8_linear (quantiser, then the GEMM as
        # its programmatic dependent).
        w8.linear(Xd, Wp, sw, bd, out=Y, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st, bits_ = w8.read_status(ws)
    if st != 0:
        raise RuntimeError("device status %d bits %#x after warm-up" % (st, bits_))

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark("timed_steps")
    t_wall0 = time.perf_counter()
    # A spin of about 2 ms on the stream, outside every timed interval: the
    # host then enqueues the steps while the GPU is busy, so that no step's
    # interval includes the host's launch latency (the first step's did).
    spin = getattr(torch.cuda, "_sleep", None)
    if spin is not None:
        spin(SPIN_BEFORE_STEPS_CYCLES)
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    sampler.end("timed_steps")
    barrier(world)
    launches = 2 * args.steps
    s_ms = [e[0].elapsed_time(e[1]) for e in evs]
    step_ms = max_over_ranks(statistics.mean(s_ms), world)
    st, bits_ = w8.read_status(ws)
    if st != 0:
        raise RuntimeError("device status %d bits %#x after timed steps" % (st, bits_))
    if args.profile:
        # A short run for a profiler: the warm-up and the timed steps only.
        sampler.__exit__(None, None, None)
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": world * case.ops / (step_ms * 1e-3) / 1e12, "unit": UNIT,
                              "ms_per_step": step_ms, "steps": args.steps, "warmup": args.warmup,
                              "config": config_dict(case), "gemm_form": w8.gemm_form(M, N, K),
                              "note": "--profile: warm-up and timed steps only; not a benchmark line"}), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    # Per-kernel durations for the rooflines: the same two kernels through
    # the two stage calls, an event between them (no overlap between them).
    # Each kernel's duration: the difference of CUDA graphs of n x (flush,
    # quantiser) and n x (flush, quantiser, GEMM) replays (no host launch
    # latency; the GEMM keeps its programmatic overlap with the quantiser),
    # and, beside it, event intervals around the two stage calls.
    n_split = max(args.steps, PER_WORKLOAD_COLD)
    cur = torch.cuda.current_stream
    quant_ms, gemm_ms = T.cold_graph([lambda: w8.linear_quant_stage(Xd, ws, stream=cur()),
                                      lambda: w8.linear_gemm_stage(M, K, Wp, sw, bd, Y, ws, stream=cur())], n_split)
    T.release()
    quant_clean_ms = T.cold_graph([lambda: w8.linear_quant_stage(Xd, ws, stream=cur())], n_split, clean=True)[0]
    T.release()
    q_all, g_all = T.cold_split([lambda: w8.linear_quant_stage(Xd, ws, stream=stream),
                                 lambda: w8.linear_gemm_stage(M, K, Wp, sw, bd, Y, ws, stream=stream)], n_split)
    quant_ev_ms, gemm_ev_ms = med(q_all), med(g_all)
    # Hot L2 and CUDA-graph replay of the headline step; the cold step by
    # graph replay too (no host launch latency), beside the event-timed one.
    hot_ms = med(T.hot(lambda: w8.linear(Xd, Wp, sw, bd, out=Y, workspace=ws, stream=torch.cuda.current_stream())))
    T.release()
    step_graph_ms = T.cold_graph([lambda: w8.linear(Xd, Wp, sw, bd, out=Y, workspace=ws, stream=cur())],
                                 n_split)[0]
    T.release()
    st, bits_ = w8.read_status(ws)
    if st != 0:
        raise RuntimeError("device status %d bits %#x after the per-kernel passes" % (st, bits_))

    # The guard's fallback on the same shape: the native BF16 linear (the
    # same tcgen05 GEMM in its BF16 mode), each call timed alone after a flush.
    bf16 = None
    if w8.bf16_linear_supported(M, N, K)[0]:
        Xb = Xd.to(torch.bfloat16)
        Wb = W.to(torch.bfloat16).to(dev)
        bb = bd.to(torch.bfloat16)
        wsb = torch.empty(w8.bf16_linear_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
        be_ms = med(T.cold(lambda: w8.bf16_linear(Xb, Wb, bb, out=Y, workspace=wsb, stream=stream),
                           max(PER_WORKLOAD_COLD, min(args.steps, 200))))
        b_ms = T.cold_graph([lambda: w8.bf16_linear(Xb, Wb, bb, out=Y, workspace=wsb, stream=cur())],
                            PER_WORKLOAD_COLD)[0]
        T.release()
        st, bits_ = w8.read_status(wsb)
        if st != 0:
            raise RuntimeError("device status %d bits %#x after BF16 linear calls" % (st, bits_))
        b_tf = case.ops / (b_ms * 1e-3) / 1e12
        bf16 = {"kernel": "gemm_w8a8_tcgen05_kernel (BF16 mode) via w8a8_bf16_linear", "ms": b_ms,
                "ms_events": be_ms, "achieved": b_tf, "unit": "TFLOP/s", "frac": b_tf / pk["bf16_tflops"],
                "w8a8_step_ms_graph": step_graph_ms,
                "w8a8_step_speedup": b_ms / step_graph_ms,
                "w8a8_step_speedup_events": be_ms / med(s_ms),
                "note": "the guard's native BF16 fallback on this shape (header clear + GEMM), L2 flushed; ms: "
                        "graph replays of n x (flush, call) minus n x flush, per call; ms_events: median of "
                        "event-timed calls; w8a8_step_speedup = BF16 time / W8A8 step time, both graph-timed "
                        "(_events: both event-timed medians)"}
        del Xb, Wb, bb, wsb

    # SageSLA's per-block INT8 Query/Key quantisation at the video branch's
    # attention shape (32 heads of 128 over this workload's tokens), each call
    # timed alone after a flush.
    qk = None
    if M >= 1024:
        heads, dh = 32, 128
        Xqk = torch.randn((1, heads, M, dh), generator=torch.Generator().manual_seed(77)).to(torch.bfloat16).to(dev)
        qk = {"shape": [1, heads, M, dh], "layout": "HND", "unit": "GB/s", "peak": pk["hbm_gbs"]}
        for qname, bt in (("query", 128), ("key", 64)):
            qe_ms = med(T.cold(lambda: w8.quantize_qk_blocks(Xqk, bt, stream=stream), PER_WORKLOAD_COLD))
            call = [lambda: w8.quantize_qk_blocks(Xqk, bt, stream=torch.cuda.current_stream())]
            q_ms = T.cold_graph(call, PER_WORKLOAD_COLD)[0]
            qc_ms = T.cold_graph(call, PER_WORKLOAD_COLD, clean=True)[0]
            T.release()
            nbytes = Xqk.numel() * 3 + heads * (-(-M // bt)) * 4   # bf16 in, int8 out, one scale per block
            gbs = nbytes / (q_ms * 1e-3) / 1e9
            qk[qname] = {"block_tokens": bt, "ms": q_ms, "ms_events": qe_ms, "achieved": gbs,
                         "frac": gbs / qk["peak"], "algorithmic_bytes": nbytes,
                         "clean_l2": {"ms": qc_ms, "frac": nbytes / (qc_ms * 1e-3) / 1e9 / qk["peak"]}}
        qk["timing"] = ("ms: graph replays of n x (flush, call) minus n x flush, per call; ms_events: median "
                        "event interval around one call after a flush (adds the launch gap)")
        del Xqk

    # The norm + modulation prologue fused into the activation quantisation
    # (RMS norm, bf16 scale and shift) on this workload: the kernel alone
    # (int8 codes), the fused layer, and the unfused pair it replaces (a
    # PyTorch RMS norm + modulation writing the bf16 activation, then
    # w8a8_linear reading it).
    normp = None
    if X.dtype == torch.bfloat16:
        gn = torch.Generator().manual_seed(21)
        scn = (torch.randn(K, generator=gn) * 0.1).to(torch.bfloat16).to(dev)
        shn = (torch.randn(K, generator=gn) * 0.1).to(torch.bfloat16).to(dev)
        ymod = torch.empty_like(Xd)
        one_plus = (1.0 + scn.float())
        shf = shn.float()

        def unfused():
            ymod.copy_(torch.nn.functional.rms_norm(Xd.float(), (K,), eps=1e-6).mul_(one_plus).add_(shf))
            w8.linear(ymod, Wp, sw, bd, out=Y, workspace=ws, stream=stream)

        def unfused_min():
            # the least the unfused form could cost here: one bf16 write and
            # one read of the activation on top of the plain step
            ymod.copy_(Xd)
            w8.linear(ymod, Wp, sw, bd, out=Y, workspace=ws, stream=stream)

        ke_ms = med(T.cold(lambda: w8.norm_quantize_act(Xd, "rms", 1e-6, scn, shn, stream=stream),
                           PER_WORKLOAD_COLD))
        call = [lambda: w8.norm_quantize_act(Xd, "rms", 1e-6, scn, shn, stream=torch.cuda.current_stream())]
        k_ms = T.cold_graph(call, PER_WORKLOAD_COLD)[0]
        kc_ms = T.cold_graph(call, PER_WORKLOAD_COLD, clean=True)[0]
        T.release()
        nl_ms = med(T.cold(lambda: w8.norm_linear(Xd, Wp, sw, bd, "rms", 1e-6, scn, shn, out=Y, workspace=ws,
                                                  stream=stream), PER_WORKLOAD_COLD))
        un_ms = med(T.cold(unfused, PER_WORKLOAD_COLD))
        um_ms = med(T.cold(unfused_min, PER_WORKLOAD_COLD))
        nbytes = M * K * 2 + M * K + M * 4 + 2 * K * 2
        normp = {"kernel": "norm_quant_rows_kernel (RMS norm, bf16 modulation, int8 codes)", "ms": k_ms,
                 "ms_events": ke_ms,
                 "achieved": nbytes / (k_ms * 1e-3) / 1e9, "unit": "GB/s", "peak": pk["hbm_gbs"],
                 "frac": nbytes / (k_ms * 1e-3) / 1e9 / pk["hbm_gbs"], "algorithmic_bytes": nbytes,
                 "clean_l2": {"ms": kc_ms, "frac": nbytes / (kc_ms * 1e-3) / 1e9 / pk["hbm_gbs"]},
                 "norm_linear_ms": nl_ms, "norm_linear_tops": case.ops / (nl_ms * 1e-3) / 1e12,
                 "unfused_torch_norm_then_linear_ms": un_ms,
                 "unfused_copy_then_linear_ms": um_ms,
                 "linear_step_ms": med(s_ms),
                 "note": "L2 flushed; ms: graph replays of n x (flush, call) minus n x flush, per call; the "
                         "rest: medians of event intervals; unfused_torch: PyTorch rms_norm x (1 + scale) + shift "
                         "written as bf16, then w8a8_linear; unfused_copy: a bf16 copy of X then w8a8_linear (a "
                         "floor for any separate norm kernel)"}
        del ymod

    # The MLP pair at the MLP workload's sizes (6144 x 4096 -> 16384 -> 4096):
    # w8a8_mlp (the down layer's codes from the up GEMM's gathered row maxima)
    # against the same two layers as separate w8a8_linear calls.
    mlp = None
    if case.name == WORKLOAD:
        Mm, Km, Fm, Nm = 6144, 4096, 16384, 4096
        Xm, _, _ = wl.make("mlp_up")
        gm = torch.Generator().manual_seed(12)
        Wu = (torch.randn(Fm, Km, generator=gm) * 0.02).to(torch.bfloat16).to(dev)
        Wdn = (torch.randn(Nm, Fm, generator=gm) * 0.02).to(torch.bfloat16).to(dev)
        bu = (torch.randn(Fm, generator=gm) * 0.01).to(torch.bfloat16).to(dev)
        bdn = (torch.randn(Nm, generator=gm) * 0.01).to(torch.bfloat16).to(dev)
        Wqu, swu = w8.quantize_weight(Wu)
        Wqd, swd = w8.quantize_weight(Wdn)
        Wpu, Wpd = w8.pack_weight(Wqu), w8.pack_weight(Wqd)
        del Wu, Wdn, Wqu, Wqd
        Xm = Xm.to(dev)
        Hm = torch.empty((Mm, Fm), dtype=torch.bfloat16, device=dev)
        Ym = torch.empty((Mm, Nm), dtype=torch.bfloat16, device=dev)
        wsm = torch.empty(w8.mlp_workspace_bytes(Mm, Km, Fm, Nm), dtype=torch.uint8, device=dev)
        wsu = torch.empty(w8.workspace_bytes(Mm, Fm, Km), dtype=torch.uint8, device=dev)
        wsd = torch.empty(w8.workspace_bytes(Mm, Nm, Fm), dtype=torch.uint8, device=dev)

        def fused():
            w8.mlp(Xm, Wpu, swu, bu, Wpd, swd, bdn, H=Hm, out=Ym, workspace=wsm, stream=stream)

        def separate():
            w8.linear(Xm, Wpu, swu, bu, out=Hm, workspace=wsu, stream=stream)
            w8.linear(Hm, Wpd, swd, bdn, out=Ym, workspace=wsd, stream=stream)

        mlp = {"shape": {"M": Mm, "K": Km, "F": Fm, "N": Nm}, "unit": "TOPS"}
        ops_m = 2 * Mm * Fm * Km + 2 * Mm * Nm * Fm
        # Interleaved, so that both see the same clock and power state.
        f_all, s_all = [], []
        for _ in range(5):
            f_all += T.cold(fused, 10, warm=1)
            s_all += T.cold(separate, 10, warm=1)
        for mname, xs in (("fused", f_all), ("separate", s_all)):
            mlp[mname] = {"ms": med(xs), "value": ops_m / (med(xs) * 1e-3) / 1e12, "n": len(xs)}
        mlp["fused_speedup"] = mlp["separate"]["ms"] / mlp["fused"]["ms"]
        st, bits_ = w8.read_status(wsm)
        if st != 0:
            raise RuntimeError("device status %d bits %#x after MLP-pair calls" % (st, bits_))
        mlp["note"] = ("both layers INT8 (4 launches fused: quant, up GEMM gathering row maxima, codes pass, "
                       "down GEMM); L2 flushed before each call; medians of 50, the two forms interleaved")
        del Xm, Hm, Ym, wsm, wsu, wsd, Wpu, Wpd

    # End to end through the public C call with host buffers
    # (w8a8_linear_host): the copy of X in and of Y out are inside the timed
    # region, pipelined over row chunks against the compute.
    Xh = X.pin_memory()
    Yh = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    Xe = torch.empty_like(Xd)
    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        w8.linear_host(Xh, Wp, sw, bd, out=Yh, X_dev=Xe, Y_dev=Y, workspace=ws, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    for _ in range(e2e_steps):
        flush.zero_()
        e0.record(stream)
        w8.linear_host(Xh, Wp, sw, bd, out=Yh, X_dev=Xe, Y_dev=Y, workspace=ws, stream=stream)
        e1.record(stream)
        e1.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    e2e_step = max_over_ranks(statistics.mean(e2e_ms), world)
    # The copy floor of that call: the same two transfers (pinned host X to
    # the device, device Y to pinned host) run concurrently with no compute.
    c_h2d, c_d2h = torch.cuda.Stream(), torch.cuda.Stream()
    Yd_src = torch.empty_like(Y)

    def copies():
        c_h2d.wait_stream(stream)
        c_d2h.wait_stream(stream)
        with torch.cuda.stream(c_h2d):
            Xe.copy_(Xh, non_blocking=True)
        with torch.cuda.stream(c_d2h):
            Yh.copy_(Yd_src, non_blocking=True)
        stream.wait_stream(c_h2d)
        stream.wait_stream(c_d2h)

    copies()
    torch.cuda.synchronize()
    floor_ms = []
    for _ in range(e2e_steps):
        e0.record(stream)
        copies()
        e1.record(stream)
        e1.synchronize()
        floor_ms.append(e0.elapsed_time(e1))
    copy_floor = statistics.mean(floor_ms)
    del Yd_src, Xe

    # The measured rates of the exact INT8 routes (the metric's denominator).
    i8 = int8_peaks(dev, pk)

    # Every workload of the five configurations.
    per_wl = None
    cpu_inputs = {}
    if not args.no_per_workload and world == 1:
        del ws, Y
        torch.cuda.empty_cache()
        per_wl = {"note": PER_WORKLOAD_NOTE}
        for name in ["tiny", "video", "mlp_up", "mlp_down", "hires_n4k", "hires_n16k", "audio_m126_n2048",
                     "audio_m126_n8192", "audio_m1001_n2048", "audio_m1001_n8192"]:
            per_wl[name], host = measure_workload(w8, name, dev, stream, flush, pk, sampler)
            if name in ("tiny", "hires_n4k", "audio_m126_n2048", "audio_m126_n8192", "audio_m1001_n2048",
                        "audio_m1001_n8192"):
                cpu_inputs[name] = host
            torch.cuda.empty_cache()
    sampler.__exit__(None, None, None)

    ops = case.ops
    gemm_tflops = ops / (gemm_ms * 1e-3) / 1e12
    qb_alg = quant_bytes(M, K, X.element_size(), 1)
    qb_built = quant_bytes(M, K, X.element_size(), 2)
    gb_alg = gemm_bytes(M, N, K, b.element_size(), 1)
    gb_built = gemm_bytes(M, N, K, b.element_size(), 2)
    quant_gbs = qb_alg / (quant_ms * 1e-3) / 1e9
    clocks = sampler.summary()
    if per_wl is not None:
        for name, row in per_wl.items():
            if name == "note":
                continue
            for kind in ("cold", "hot", "bf16_cold", "bf16_hot"):
                r = clocks.pop("region_%s:%s" % (name, kind), None)
                if r is not None:
                    row["clocks_" + kind] = {"sm_mhz": r["sm_mhz"], "sm_mhz_min": r.get("sm_mhz_min"),
                                             "reasons": r["reasons"], "samples": r["samples"],
                                             "power_w_max": r.get("power_w_max")}
    value = world * ops / (step_ms * 1e-3) / 1e12
    if rank == 0:
        base = None
        base_wl = None
        if world == 1 and not args.no_cpu_baseline:
            base = cpu_baseline(case, X, W, b)
            base_wl = {}
            for name, (Xc, Wc, bc) in cpu_inputs.items():
                c = wl.CASES[name]
                base_wl[name] = cpu_baseline(c, Xc, Wc, bc, target_s=0.5 if name != "hires_n4k" else 4.0)
        line = {
            "metric": METRIC,
            "value": value,
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": step_ms,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "int8 codes x int8 codes -> int32 (exact, on bf16 tcgen05 tensor cores)",
            "data": "synthetic",
            "config": config_dict(case),
            "step_stats_ms": {"mean": statistics.mean(s_ms), "median": med(s_ms), "min": min(s_ms),
                              "max": max(s_ms), "n": len(s_ms), "steps": [round(x, 5) for x in s_ms],
                              "hot_l2_graph_median": hot_ms,
                              "cold_graph": step_graph_ms},
            "frac_of_int8_peak": value / world / i8["denominator_tops"],
            "int8_peak": i8,
            "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": gemm_tflops / pk["bf16_tflops"],
                         "traffic": GEMM_TRAFFIC.get(sources_digest(GEMM_SOURCES)) if case.name == WORKLOAD else None,
                         "kernel": "gemm_w8a8_tcgen05_kernel (GEMM + fused epilogue)",
                         "algorithmic_bytes": gb_alg, "bytes_as_built": gb_built, "ms": gemm_ms,
                         "n": n_split, "ms_events": gemm_ev_ms,
                         "timing": "graph replays: n x (flush, quantiser, GEMM) minus n x (flush, quantiser), "
                                   "per launch; ms_events: median event interval around the stage call",
                         "peak_source": "%s bf16 dense burst (the MMA runs bf16 kind::f16)" % pk["source"],
                         "note": ("the plain GEMM of the two-stage path (w8a8_linear_gemm_stage); the timed step "
                                  "runs the same kernel with two quantiser warps added, which also quantise the rows "
                                  "past the first wave's while it multiplies (no clean roofline of its own); the "
                                  "step-level fraction is frac_of_int8_peak") if case.name == WORKLOAD else
                                 "the GEMM of the two-stage path (w8a8_linear_gemm_stage)"},
            "quant_roofline": {"bound": "hbm", "achieved": quant_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                               "frac": quant_gbs / pk["hbm_gbs"], "ms": quant_ms, "n": n_split,
                               "ms_events": quant_ev_ms,
                               "clean_l2": {"ms": quant_clean_ms,
                                            "frac": qb_alg / (quant_clean_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                                            "frac_as_built": qb_built / (quant_clean_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                                            "note": "after a flush that writes 256 MiB and then reads another "
                                                    "256 MiB, so L2 holds clean lines: the kernel's misses evict "
                                                    "without the write-backs the write flush's dirty lines cost"},
                               "kernel": "quant_rows_kernel (bf16 codes)", "algorithmic_bytes": qb_alg,
                               "bytes_as_built": qb_built,
                               "frac_as_built": qb_built / (quant_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                               "note": "algorithmic bytes count int8 codes (input + 1 B per code + 4 B per row); "
                                       "the kernel writes the codes as bf16 (2 B), the tensor-core operand"},
            "e2e": {"value": world * ops / (e2e_step * 1e-3) / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": Xh.numel() * Xh.element_size(),
                    "d2h_bytes_per_step": Yh.numel() * Yh.element_size(), "ms_per_step": e2e_step,
                    "copy_floor_ms": copy_floor, "frac_of_copy_floor": copy_floor / e2e_step,
                    "note": "w8a8_linear_host, default chunks: copies in, compute and copies out of different "
                            "chunks overlap; copy_floor_ms = the same two transfers alone, concurrently"},
            "gpu_launches": launches,
            "kernel_split_ms": {"quant": quant_ms, "gemm": gemm_ms, "quant_events": quant_ev_ms,
                                "gemm_events": gemm_ev_ms,
                                "note": "per launch from graph replays (see roofline.timing); *_events: medians of "
                                        "event intervals around each stage call (they include the launch after "
                                        "the event that separates the two kernels)"},
            "bf16_fallback": bf16,
            "qk_block_quant": qk,
            "mlp_pair": mlp,
            "norm_prologue": normp,
            "per_workload": per_wl,
            "clocks": clocks,
            "wall_s_timed": t_wall,
        }
        if base is not None:
            line["cpu_baseline"] = base
            line["cpu_baseline_per_workload"] = base_wl
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(wl.CASES))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="warm-up and timed steps only (a short run to capture under a profiler)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)      # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
