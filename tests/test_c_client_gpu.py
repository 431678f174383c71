"""The library used from plain C on the GPU (CUDA runtime and the public
header only, no Python in the process): its W8A8 linear agrees with the
oracle within one bf16 ulp."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import w8a8_int8_linear_act_b300 as w8
import w8a8_workloads as wl
from helpers import bias_f32, bits

pytestmark = pytest.mark.gpu


def test_c_client_linear_matches_oracle(cuda_device, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if cc is None or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime.h")):
        pytest.skip("no C compiler or CUDA headers")
    here = os.path.dirname(os.path.abspath(__file__))
    libdir = os.path.dirname(w8.lib_path())
    exe = tmp_path / "gpu_client"
    r = subprocess.run([cc, "-std=c99", "-O1", "-Wall", "-I", os.path.join(os.path.dirname(here), "include"),
                        "-I", os.path.join(cuda, "include"), os.path.join(here, "c_abi", "gpu_client.c"),
                        "-L", libdir, "-l:libw8a8.so", "-Wl,-rpath," + libdir,
                        "-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64"),
                        "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    M, K, N = 300, 1024, 520
    X, W, b = wl.make("video", M=M, N=N, K=K)
    inp, outp = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([M, K, N], dtype=np.int64).tobytes())
        for t in (X, W, b):
            f.write(bits(t).tobytes())
    run = subprocess.run([str(exe), str(inp), str(outp)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    Y = np.fromfile(outp, dtype=np.uint16).reshape(M, N)
    wq, sw = oracle.quantize_rows(bits(W))
    ref = oracle.linear(bits(X), wq, sw, bias_f32(b), exact_f64=True)
    err = np.abs(oracle.bf16_bits_to_f32(Y).astype(np.float64) - ref["y32"].astype(np.float64))
    assert (err <= oracle.ulp_bf16(ref["y32"])).all()
