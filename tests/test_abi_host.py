"""Host-only checks of the C ABI: the library loads, exports every symbol the
header declares, and the shape guard and argument checks behave as
documented.  No call here reaches a kernel or needs a GPU."""
import ctypes
import os
import re

import pytest
import torch

import w8a8_int8_linear_act_b300 as w8

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w8a8.h")


def declared_symbols():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"W8A8_API\s+[\w\s\*]+?\b(w8a8_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from w8a8_int8_linear_act_b300 import build
    build.build()
    return w8.load()


def test_header_declares_the_api():
    names = declared_symbols()
    for required in ("w8a8_quantize_weight", "w8a8_quantize_act", "w8a8_linear", "w8a8_shape_supported",
                     "w8a8_pack_weight", "w8a8_gemm_s32", "w8a8_linear_workspace_bytes"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(w8.lib_path())
    for name in declared_symbols():
        assert hasattr(raw, name), name


def test_version_and_status_strings(lib):
    assert lib.w8a8_version() == 1
    for s in range(9):
        assert lib.w8a8_status_str(s)
    assert b"unknown" in lib.w8a8_status_str(99)


@pytest.mark.parametrize("M,N,K", [(64, 128, 256), (6144, 4096, 4096), (6144, 16384, 4096), (6144, 4096, 16384),
                                   (28672, 4096, 4096), (28672, 16384, 4096), (126, 2048, 2048), (126, 8192, 2048),
                                   (1001, 2048, 2048), (1001, 8192, 2048), (1, 8, 16)])
def test_guard_accepts_workload_shapes(lib, M, N, K):
    ok, reasons = w8.shape_supported(M, N, K, torch.bfloat16, torch.bfloat16)
    assert ok and reasons == []


@pytest.mark.parametrize("M,N,K,expect", [
    (0, 128, 256, ["M"]),
    (64, 12, 256, ["N"]),
    (64, 0, 256, ["N"]),
    (64, 128, 250, ["K"]),
    (64, 128, 8, ["K"]),
    (64, 128, 133152, ["K_RANGE"]),
    (0, 3, 7, ["M", "N", "K"]),
])
def test_guard_rejects_with_reasons(lib, M, N, K, expect):
    ok, reasons = w8.shape_supported(M, N, K)
    assert not ok and reasons == expect


def test_guard_k_limit_boundary(lib):
    assert (2 ** 31 - 1) // (127 * 127) == 133144
    assert w8.shape_supported(8, 8, 133136)[0]          # largest multiple of 16 <= 133144
    assert not w8.shape_supported(8, 8, 133152)[0]


def test_guard_dtypes(lib):
    assert w8.shape_supported(8, 8, 16, torch.float32, torch.float32)[0]
    ok, r = w8.shape_supported(8, 8, 16, torch.float16, torch.bfloat16)
    assert not ok and r == ["X_DTYPE"]
    ok, r = w8.shape_supported(8, 8, 16, torch.bfloat16, torch.int8)
    assert not ok and r == ["BIAS_DTYPE"]


def test_workspace_bytes(lib):
    assert w8.workspace_bytes(6144, 4096) == 1024 + 1024 + 6144 * 4 + 6144 * 4096 * 2
    assert w8.workspace_bytes(126, 2048) == 1024 + 1024 + 1024 + 126 * 2048 * 2
    assert w8.workspace_bytes(0, 16) == 0


def test_argument_errors_return_before_any_launch(lib):
    """Null pointers, bad dtypes, rejected shapes and short workspaces are
    reported without touching the device (this runs without a GPU)."""
    p = ctypes.c_void_p(0x10000)     # never dereferenced: every call below fails validation first
    null = None
    assert lib.w8a8_linear(null, 1, 64, 256, p, p, 128, null, 1, p, p, 1 << 20, null) == 1
    assert lib.w8a8_linear(p, 7, 64, 256, p, p, 128, null, 1, p, p, 1 << 20, null) == 2
    assert lib.w8a8_linear(p, 1, 64, 250, p, p, 128, null, 1, p, p, 1 << 20, null) == 4
    assert lib.w8a8_linear(p, 1, 64, 256, p, p, 12, null, 1, p, p, 1 << 20, null) == 4
    assert lib.w8a8_linear(p, 1, 64, 256, p, p, 128, null, 1, p, p, 100, null) == 5
    assert lib.w8a8_linear(p, 1, 64, 256, p, p, 128, null, 1, p, null, 1 << 20, null) == 5
    assert lib.w8a8_linear(ctypes.c_void_p(0x10008), 1, 64, 256, p, p, 128, null, 1, p, p, 1 << 20, null) == 3
    assert lib.w8a8_quantize_act(null, 1, 4, 16, p, p, null) == 1
    assert lib.w8a8_quantize_act(p, 3, 4, 16, p, p, null) == 2
    assert lib.w8a8_quantize_act(p, 1, 4, 24, p, p, null) == 4
    assert lib.w8a8_quantize_weight(p, 1, 4, 133152, p, p, null) == 4
    assert lib.w8a8_pack_weight(p, 4, 20, p, null) == 4
    assert lib.w8a8_gemm_s32(p, p, 4, 8, 16, p, p, 10, null) == 5
    assert lib.w8a8_read_status(null, null, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    """No silent fallback: a missing library is an ImportError."""
    monkeypatch.setattr(w8, "_lib", None)
    monkeypatch.setattr(w8, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        w8.load()
