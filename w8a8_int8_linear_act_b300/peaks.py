"""ctypes binding of libw8a8_peaks.so (include/w8a8_peaks.h): throughput
probes of the warp-level tensor-core MMA (mma.sync) on INT8 and on bf16
operands, and the toolchain's answer on the integer tcgen05 MMA, used to
measure the roofline denominators.  Not part of the layer."""
import ctypes
import os
import shutil
import subprocess
import tempfile

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libw8a8_peaks.so")
_lib = None

MMA_S8 = 0
MMA_BF16 = 1


def lib_path() -> str:
    return _LIB_PATH


def load():
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError("libw8a8_peaks.so is not built (expected at %s)" % _LIB_PATH)
        lib = ctypes.CDLL(_LIB_PATH)
        i32, i64, p = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        lib.w8a8_peak_mma_sync_ops.argtypes = [i32, i32, i32, i64]
        lib.w8a8_peak_mma_sync_ops.restype = i64
        lib.w8a8_peak_mma_sync.argtypes = [i32, i32, i32, i64, p, p]
        lib.w8a8_peak_mma_sync.restype = i32
        _lib = lib
    return _lib


def mma_sync_ops(kind: int, blocks: int, threads: int, iters: int) -> int:
    return int(load().w8a8_peak_mma_sync_ops(kind, blocks, threads, iters))


def mma_sync_launch(kind: int, blocks: int, threads: int, iters: int, sink: torch.Tensor, stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    st = load().w8a8_peak_mma_sync(kind, blocks, threads, iters, ctypes.c_void_p(sink.data_ptr()),
                                   ctypes.c_void_p(s.cuda_stream))
    if st != 0:
        raise RuntimeError("w8a8_peak_mma_sync failed with status %d" % st)


# A kernel whose only instruction of interest is one tcgen05 integer MMA
# (all operands zero; it is assembled, never run).
_TCGEN05_I8_PTX = """.version 9.0
.target {target}
.address_size 64
.visible .entry probe_tcgen05_i8()
{{
  .reg .b32 r<2>;
  .reg .b64 rd<2>;
  .reg .pred p;
  mov.u32 r0, 0;
  mov.u64 rd0, 0;
  mov.u64 rd1, 0;
  mov.u32 r1, 0;
  setp.ne.b32 p, r1, 0;
  tcgen05.mma.cta_group::1.kind::{kind} [r0], rd0, rd1, r1, p;
  ret;
}}
"""


def ptxas_accepts_tcgen05(target: str, kind: str = "i8"):
    """Assemble a one-instruction tcgen05.mma of the given kind for `target`
    (e.g. "sm_103a") with this toolkit's ptxas.  Returns (accepted, first
    line of ptxas's message, ptxas version line); (None, why, None) when no
    ptxas is found."""
    ptxas = shutil.which("ptxas") or "/usr/local/cuda/bin/ptxas"
    if not os.path.exists(ptxas):
        return None, "no ptxas found", None
    ver = subprocess.run([ptxas, "--version"], capture_output=True, text=True).stdout.strip().splitlines()
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "probe.ptx")
        with open(src, "w") as f:
            f.write(_TCGEN05_I8_PTX.format(target=target, kind=kind))
        r = subprocess.run([ptxas, "-arch=" + target, src, "-o", os.path.join(d, "probe.cubin")],
                           capture_output=True, text=True)
    msg = (r.stderr or r.stdout).strip().splitlines()
    first = msg[0].split(": ", 1)[-1] if msg else ""
    if "error" in first:
        first = first[first.index("error"):]
    return r.returncode == 0, first, ver[-1] if ver else None
