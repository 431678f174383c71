"""Builds the package's two C-ABI libraries in-tree.

  libw8a8.so        the layer: the sm_103a kernels and the entry points of
                    include/w8a8.h
  libw8a8_peaks.so  throughput probes for the roofline denominators
                    (include/w8a8_peaks.h); not part of the layer

nvcc cross-compiles for sm_103a without a GPU.  IEEE division and square
root, no flush-to-zero, no fast math: the quantiser's codes depend on exact
fp32 division.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libw8a8.so")
PEAKS_LIB = os.path.join(HERE, "libw8a8_peaks.so")
SOURCES = [os.path.join(CSRC, "w8a8_api.cu"), os.path.join(CSRC, "noalloc.cu")]
PEAKS_SOURCES = [os.path.join(CSRC, "peaks.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + \
    [os.path.join(ROOT, "include", "w8a8.h")]
PEAKS_DEPS = PEAKS_SOURCES + [os.path.join(ROOT, "include", "w8a8_peaks.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
    "-Xcompiler", "-fPIC,-fvisibility=hidden",
    "-shared", "-cudart", "static",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _build_one(lib: str, sources, deps, force: bool, verbose: bool) -> str:
    if not force and os.path.exists(lib):
        lib_t = os.path.getmtime(lib)
        if all(os.path.getmtime(d) <= lib_t for d in deps):
            return lib
    tmp = lib + ".tmp.%d" % os.getpid()
    cmd = [nvcc(), *NVCC_FLAGS, *(["-Xptxas", "-v"] if verbose else []), *sources, "-o", tmp, "-lcuda"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libw8a8.so and libw8a8_peaks.so if any source is newer;
    return the path of libw8a8.so."""
    _build_one(PEAKS_LIB, PEAKS_SOURCES, PEAKS_DEPS, force, verbose)
    return _build_one(LIB, SOURCES, DEPS, force, verbose)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
