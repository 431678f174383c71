"""Benchmark of the guarded W8A8 linear on B300.

Metric: W8A8 linear TOPS (activation quantisation + INT32-exact GEMM + fused
epilogue) on the video-branch projection, M=6144, K=N=4096, bf16 inputs with
1 % outlier columns, on one GPU.  One step = one call of the whole hot path:
the activation-quantisation kernel and the GEMM+epilogue kernel, through the
C ABI's two stages (exactly what w8a8_linear runs), inputs resident in HBM,
L2 flushed (256 MiB written) before every step, each kernel timed with CUDA
events on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (plain C) on the host cores on a
bounded row sample of the same workload.  Under torchrun (N > 1) every rank
runs an independent replica of the workload (rows are independent, no
collective on the data path; "weak" scaling), rank 0 prints the line.
"""
import argparse
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

# Algorithmic bytes per unit, for the rooflines:
#   quant kernel per activation element: 2 B read (bf16; 4 B for fp32) + 2 B written (bf16 code); + 4 B per row (scale)
#   GEMM per launch: codes A (2 M K) + codes B (2 N K) + sx (4 M) + sw (4 N) + bias (2 N) + Y (2 M N)


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one GEMM launch
# on the default workload, from one ncu capture of it.
# Valid only for the kernel sources it was taken on: the key is a digest of
# their code (comments excluded), and the bench reports null traffic when the
# code has changed since.
GEMM_SOURCES = ["w8a8_int8_linear_act_b300/csrc/gemm_tcgen05.cuh",
                "w8a8_int8_linear_act_b300/csrc/ptx_sm103.cuh"]
GEMM_TRAFFIC = {"4c6119a28db36d2a": 164.14e6}


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


class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons while the
    timed region runs (read-only queries).  NVML first, every 5 ms; if NVML
    cannot be opened, `nvidia-smi --query-gpu ... -lms 50` in a child process."""

    REASONS = {
        "hw_slowdown": "nvmlClocksEventReasonHwSlowdown",
        "hw_thermal_slowdown": "nvmlClocksEventReasonHwThermalSlowdown",
        "sw_thermal_slowdown": "nvmlClocksEventReasonSwThermalSlowdown",
        "sw_power_cap": "nvmlClocksEventReasonSwPowerCap",
        "hw_power_brake_slowdown": "nvmlClocksEventReasonHwPowerBrakeSlowdown",
    }
    SMI_FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
                  "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
                  "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int, pci_bus_id=None, period_s: float = 0.005):
        self.index = index
        self.pci = pci_bus_id
        self.period = period_s
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.source = None
        self.error = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._proc = None

    def __enter__(self):
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nvml = pynvml
            if self.pci:
                self._h = pynvml.nvmlDeviceGetHandleByPciBusId(self.pci.encode() if isinstance(self.pci, str)
                                                              else self.pci)
            else:
                self._h = pynvml.nvmlDeviceGetHandleByIndex(self.index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
            self.source = "nvml"
            self._thread = threading.Thread(target=self._run_nvml, daemon=True)
            self._thread.start()
        except Exception as e:  # fall back to nvidia-smi
            self.error = "nvml: %s: %s" % (type(e).__name__, e)
            self._nvml = None
            self._start_smi()
        return self

    def _start_smi(self):
        import subprocess
        target = self.pci if self.pci else str(self.index)
        cmd = ["nvidia-smi", "-i", target, "--query-gpu=" + ",".join(self.SMI_FIELDS),
               "--format=csv,noheader,nounits", "-lms", "50"]
        try:
            self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self._thread = threading.Thread(target=self._run_smi, daemon=True)
            self._thread.start()
        except Exception as e:
            self.error = (self.error or "") + "; nvidia-smi: %s" % e

    def _run_nvml(self):
        nv = self._nvml
        masks = {k: getattr(nv, v) for k, v in self.REASONS.items() if hasattr(nv, v)}
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self._h, nv.NVML_CLOCK_SM))
                active = nv.nvmlDeviceGetCurrentClocksEventReasons(self._h)
                for name, m in masks.items():
                    if active & m:
                        self.reasons.add(name)
            except Exception as e:
                self.error = "nvml sample: %s" % e
            time.sleep(self.period)

    def _run_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != len(self.SMI_FIELDS):
                continue
            try:
                self.samples.append(float(parts[0]))
                self.max_mhz = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[2:]):
                if val.lower() == "active":
                    self.reasons.add(name)

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
        if self._nvml is not None:
            try:
                self._nvml.nvmlShutdown()
            except Exception:
                pass
        return False

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"], "samples": 0,
                    "source": self.source, "error": self.error}
        out = {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
               "reasons": sorted(self.reasons), "samples": len(self.samples), "source": self.source}
        if self.error:
            out["error"] = self.error
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
    dt, _ = oracle_sample(case, rows, *inputs)
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

    def step():
        # One call of the hot path: w8a8_linear (quantiser, then the GEMM as
        # its programmatic dependent).
        w8.linear(Xd, Wp, sw, bd, out=Y, workspace=ws, stream=stream)

    def staged(evs):
        # The same two kernels through the two stage calls, with an event
        # between them: each kernel's own duration (no overlap between them).
        evs[0].record(stream)
        w8.linear_quant_stage(Xd, ws, stream=stream)
        evs[1].record(stream)
        w8.linear_gemm_stage(M, K, Wp, sw, bd, Y, ws, stream=stream)
        evs[2].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    st, bits_ = w8.read_status(ws)
    if st != 0:
        raise RuntimeError("device status %d bits %#x after warm-up" % (st, bits_))

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    kevs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    try:
        pr = torch.cuda.get_device_properties(dev)
        pci = "%08X:%02X:%02X.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
    except Exception:
        pci = None
    sampler = ClockSampler(dev.index, pci)
    barrier(world)
    torch.cuda.synchronize()
    with sampler:
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            evs[i][0].record(stream)
            step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
        barrier(world)
        # per-kernel durations, for the rooflines (a second timed pass)
        for i in range(args.steps):
            flush.zero_()
            staged(kevs[i])
        torch.cuda.synchronize()
    barrier(world)
    launches = 2 * args.steps
    s_ms = [e[0].elapsed_time(e[1]) for e in evs]
    q_ms = [e[0].elapsed_time(e[1]) for e in kevs]
    g_ms = [e[1].elapsed_time(e[2]) for e in kevs]
    step_ms = max_over_ranks(statistics.mean(s_ms), world)
    gemm_ms = statistics.mean(g_ms)
    quant_ms = statistics.mean(q_ms)
    st, bits_ = w8.read_status(ws)
    if st != 0:
        raise RuntimeError("device status %d bits %#x after timed steps" % (st, bits_))

    # The same step replayed from a CUDA graph (flush + w8a8_linear captured
    # once): GPU time alone, without the binding's per-call host work, which
    # dominates the event intervals of the small audio shapes.
    graph = {"value": None, "ms_per_step": None}
    try:
        g = torch.cuda.CUDAGraph()
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            step_on = lambda: w8.linear(Xd, Wp, sw, bd, out=Y, workspace=ws, stream=gs)  # noqa: E731
            flush.zero_()
            step_on()
            gs.synchronize()
            with torch.cuda.graph(g, stream=gs):
                flush.zero_()
                step_on()
        torch.cuda.synchronize()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(min(args.steps, 500))]
        cur = torch.cuda.current_stream()
        for a, b_ in gev:
            a.record(cur)
            g.replay()
            b_.record(cur)
        torch.cuda.synchronize()
        g_ms = statistics.mean(a.elapsed_time(b_) for a, b_ in gev)
        # the captured step includes the 256 MiB flush: time it alone the same way
        fg = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs):
            with torch.cuda.graph(fg, stream=gs):
                flush.zero_()
        torch.cuda.synchronize()
        fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(50)]
        for a, b_ in fev:
            a.record(cur)
            fg.replay()
            b_.record(cur)
        torch.cuda.synchronize()
        f_ms = statistics.mean(a.elapsed_time(b_) for a, b_ in fev)
        graph = {"value": case.ops / ((g_ms - f_ms) * 1e-3) / 1e12, "ms_per_step": g_ms - f_ms,
                 "note": "graph replay of flush + w8a8_linear, minus the flush replayed alone"}
        st, bits_ = w8.read_status(ws)
        if st != 0:
            raise RuntimeError("device status %d bits %#x after graph replays" % (st, bits_))
    except RuntimeError:
        raise
    except Exception as exc:  # capture unsupported: report why
        graph = {"value": None, "ms_per_step": None, "error": "%s: %s" % (type(exc).__name__, exc)}

    # The guard's fallback on the same shape: the native BF16 linear (the
    # same tcgen05 GEMM in its BF16 mode), each call timed alone after a flush.
    bf16 = None
    if w8.bf16_linear_supported(M, N, K)[0]:
        Xb = Xd.to(torch.bfloat16)
        Wb = W.to(torch.bfloat16).to(dev)
        bb = bd.to(torch.bfloat16)
        wsb = torch.empty(w8.bf16_linear_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
        for _ in range(3):
            flush.zero_()
            w8.bf16_linear(Xb, Wb, bb, out=Y, workspace=wsb, stream=stream)
        bev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(min(args.steps, 200))]
        for a, b_ in bev:
            flush.zero_()
            a.record(stream)
            w8.bf16_linear(Xb, Wb, bb, out=Y, workspace=wsb, stream=stream)
            b_.record(stream)
        torch.cuda.synchronize()
        st, bits_ = w8.read_status(wsb)
        if st != 0:
            raise RuntimeError("device status %d bits %#x after BF16 linear calls" % (st, bits_))
        b_ms = statistics.mean(a.elapsed_time(b_) for a, b_ in bev)
        b_tf = case.ops / (b_ms * 1e-3) / 1e12
        bf16 = {"kernel": "gemm_w8a8_tcgen05_kernel (BF16 mode) via w8a8_bf16_linear", "ms": b_ms,
                "achieved": b_tf, "unit": "TFLOP/s", "frac": b_tf / peaks()["bf16_tflops"],
                "w8a8_step_speedup": b_ms / step_ms,
                "note": "the guard's native BF16 fallback on this shape, header clear + GEMM, L2 flushed"}
        del Xb, Wb, bb, wsb

    pk_hbm = peaks()["hbm_gbs"]

    # SageSLA's per-block INT8 Query/Key quantisation at the video branch's
    # attention shape (32 heads of 128 over this workload's tokens), each call
    # timed alone after a flush.
    qk = None
    if M >= 1024:
        heads, dh = 32, 128
        Xqk = torch.randn((1, heads, M, dh), generator=torch.Generator().manual_seed(77)).to(torch.bfloat16).to(dev)
        qk = {"shape": [1, heads, M, dh], "layout": "HND", "unit": "GB/s", "peak": peaks()["hbm_gbs"]}
        for name, bt in (("query", 128), ("key", 64)):
            for _ in range(3):
                flush.zero_()
                w8.quantize_qk_blocks(Xqk, bt, stream=stream)
            qev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(min(args.steps, 200))]
            for a, b_ in qev:
                flush.zero_()
                a.record(stream)
                w8.quantize_qk_blocks(Xqk, bt, stream=stream)
                b_.record(stream)
            torch.cuda.synchronize()
            q_ms = statistics.mean(a.elapsed_time(b_) for a, b_ in qev)
            nbytes = Xqk.numel() * 3 + heads * (-(-M // bt)) * 4   # bf16 in, int8 out, one scale per block
            gbs = nbytes / (q_ms * 1e-3) / 1e9
            qk[name] = {"block_tokens": bt, "ms": q_ms, "achieved": gbs, "frac": gbs / qk["peak"],
                        "algorithmic_bytes": nbytes}
        del Xqk

    # The norm + modulation prologue fused into the activation quantisation
    # (RMS norm, bf16 scale and shift) on this workload: the kernel alone
    # (int8 codes) and the whole layer against the plain linear step.
    normp = None
    if X.dtype == torch.bfloat16:
        gn = torch.Generator().manual_seed(21)
        scn = (torch.randn(K, generator=gn) * 0.1).to(torch.bfloat16).to(dev)
        shn = (torch.randn(K, generator=gn) * 0.1).to(torch.bfloat16).to(dev)

        def timed(fn, n):
            for _ in range(3):
                flush.zero_()
                fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            for a, b_ in ev:
                flush.zero_()
                a.record(stream)
                fn()
                b_.record(stream)
            torch.cuda.synchronize()
            return statistics.mean(a.elapsed_time(b_) for a, b_ in ev)

        n_it = min(args.steps, 200)
        k_ms = timed(lambda: w8.norm_quantize_act(Xd, "rms", 1e-6, scn, shn, stream=stream), n_it)
        nl_ms = timed(lambda: w8.norm_linear(Xd, Wp, sw, bd, "rms", 1e-6, scn, shn, out=Y, workspace=ws,
                                             stream=stream), n_it)
        nbytes = M * K * 2 + M * K + M * 4 + 2 * K * 2
        normp = {"kernel": "norm_quant_rows_kernel (RMS norm, bf16 modulation, int8 codes)", "ms": k_ms,
                 "achieved": nbytes / (k_ms * 1e-3) / 1e9, "unit": "GB/s", "peak": pk_hbm,
                 "frac": nbytes / (k_ms * 1e-3) / 1e9 / pk_hbm, "algorithmic_bytes": nbytes,
                 "norm_linear_ms": nl_ms, "norm_linear_tops": case.ops / (nl_ms * 1e-3) / 1e12,
                 "linear_step_ms": step_ms,
                 "note": "w8a8_norm_linear = the prologue + GEMM in one call; the unfused form would add a "
                         "write and a read of the modulated activation (2 B each per element)"}

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
        for name, fn in (("fused", fused), ("separate", separate)):
            for _ in range(3):
                flush.zero_()
                fn()
            mev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(min(args.steps, 50))]
            for a, b_ in mev:
                flush.zero_()
                a.record(stream)
                fn()
                b_.record(stream)
            torch.cuda.synchronize()
            m_ms = statistics.mean(a.elapsed_time(b_) for a, b_ in mev)
            mlp[name] = {"ms": m_ms, "value": ops_m / (m_ms * 1e-3) / 1e12}
        st, bits_ = w8.read_status(wsm)
        if st != 0:
            raise RuntimeError("device status %d bits %#x after MLP-pair calls" % (st, bits_))
        mlp["note"] = ("both layers INT8 (4 launches fused: quant, up GEMM gathering row maxima, codes pass, "
                       "down GEMM); L2 flushed before each call")
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
    del Yd_src

    ops = case.ops
    pk = peaks()
    gemm_tflops = ops / (gemm_ms * 1e-3) / 1e12
    quant_bytes = M * K * X.element_size() + M * K * 2 + M * 4
    gemm_bytes = 2 * M * K + 2 * N * K + 4 * M + 4 * N + 2 * N + 2 * M * N
    quant_gbs = quant_bytes / (quant_ms * 1e-3) / 1e9
    clocks = sampler.summary()
    if rank == 0:
        base = cpu_baseline(case, X, W, b) if (world == 1 and not args.no_cpu_baseline) else None
        line = {
            "metric": METRIC,
            "value": world * ops / (step_ms * 1e-3) / 1e12,
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
            "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": gemm_tflops / pk["bf16_tflops"],
                         "traffic": GEMM_TRAFFIC.get(sources_digest(GEMM_SOURCES)) if case.name == WORKLOAD else None,
                         "kernel": "gemm_w8a8_tcgen05_kernel (GEMM + fused epilogue)",
                         "algorithmic_bytes": gemm_bytes, "ms": gemm_ms,
                         "peak_source": "%s bf16 dense burst (the MMA runs bf16 kind::f16)" % pk["source"]},
            "quant_roofline": {"bound": "hbm", "achieved": quant_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                               "frac": quant_gbs / pk["hbm_gbs"], "ms": quant_ms,
                               "kernel": "quant_rows_kernel (bf16 codes)", "algorithmic_bytes": quant_bytes},
            "e2e": {"value": world * ops / (e2e_step * 1e-3) / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": Xh.numel() * Xh.element_size(),
                    "d2h_bytes_per_step": Yh.numel() * Yh.element_size(), "ms_per_step": e2e_step,
                    "copy_floor_ms": copy_floor, "frac_of_copy_floor": copy_floor / e2e_step,
                    "note": "w8a8_linear_host, default chunks: copies in, compute and copies out of different "
                            "chunks overlap; copy_floor_ms = the same two transfers alone, concurrently"},
            "gpu_launches": launches,
            "graph": graph,
            "kernel_split_ms": {"quant": quant_ms, "gemm": gemm_ms,
                                "note": "each kernel alone (event between them); the step overlaps the "
                                        "GEMM's set-up with the quantiser's tail"},
            "bf16_fallback": bf16,
            "qk_block_quant": qk,
            "mlp_pair": mlp,
            "norm_prologue": normp,
            "clocks": clocks,
            "wall_s_timed": t_wall,
        }
        if base is not None:
            line["cpu_baseline"] = base
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(wl.CASES))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)      # at least three untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
