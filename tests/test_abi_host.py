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
                     "w8a8_pack_weight", "w8a8_gemm_s32", "w8a8_linear_workspace_bytes",
                     "w8a8_linear_workspace_min_bytes", "w8a8_gemm_plan", "w8a8_bf16_linear",
                     "w8a8_bf16_linear_supported", "w8a8_mlp", "w8a8_norm_linear", "w8a8_norm_quantize_act",
                     "w8a8_quantize_qk_blocks", "w8a8_linear_host", "w8a8_linear_noalloc",
                     "w8a8_noalloc_read_status"):
        assert required in names


def test_header_is_plain_c(tmp_path):
    """The boundary is a C ABI: the header compiles as C99 with no warnings."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use.c"
    src.write_text('#include "w8a8.h"\nint main(void) { return w8a8_version() > 0 ? 0 : 1; }\n')
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I", inc, str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(w8.lib_path())
    for name in declared_symbols():
        assert hasattr(raw, name), name


def test_peaks_library_exports_every_declared_symbol():
    """The throughput probes' library (roofline denominators) loads on a
    machine without a GPU and exports what its header declares."""
    from w8a8_int8_linear_act_b300 import build, peaks
    build.build()
    src = open(os.path.join(ROOT, "include", "w8a8_peaks.h")).read()
    names = sorted(set(re.findall(r"W8A8_PEAKS_API\s+[\w\s\*]+?\b(w8a8_\w+)\s*\(", src)))
    assert names == ["w8a8_peak_mma_sync", "w8a8_peak_mma_sync_ops"]
    raw = ctypes.CDLL(peaks.lib_path())
    for name in names:
        assert hasattr(raw, name), name
    # ops = blocks x warps x steps x 8 MMAs x (2 * 16 * 8 * 32) for INT8, (2 * 16 * 8 * 16) for bf16
    assert peaks.mma_sync_ops(peaks.MMA_S8, 148, 256, 1000) == 148 * 8 * 1000 * 8 * 8192
    assert peaks.mma_sync_ops(peaks.MMA_BF16, 2, 64, 3) == 2 * 2 * 3 * 8 * 4096
    assert peaks.mma_sync_ops(peaks.MMA_S8, 1, 48, 1) == 0      # not a whole number of warps


def test_gemm_form_choice(lib):
    """The GEMM form per shape (host-only planner, a 148-SM device when none
    is current): the cluster-K form for the few-tile audio and tiny shapes,
    the persistent form for the rest; the test switch pins a form."""
    w8.debug_force_gemm_form(-1)
    try:
        assert w8.gemm_form(126, 2048, 2048)[0] == 1
        assert w8.gemm_form(126, 8192, 2048)[0] == 1
        assert w8.gemm_form(1001, 2048, 2048)[0] == 1
        assert w8.gemm_form(64, 128, 256)[0] == 1
        for M, N, K in [(1001, 8192, 2048), (6144, 4096, 4096), (6144, 16384, 4096), (28672, 4096, 4096)]:
            assert w8.gemm_form(M, N, K) == (0, 0, 0, 0)
        for M, N, K in [(126, 2048, 2048), (1001, 2048, 2048), (300, 520, 1040), (1, 8, 16)]:
            f, bn, ks, ctas = w8.gemm_form(M, N, K)
            if f:
                assert bn in (64, 128, 256) and ks in (1, 2, 4, 8)
                assert ctas == -(-M // 128) * -(-N // bn) * ks <= 148
        w8.debug_force_gemm_form(1, 64, 8)
        assert w8.gemm_form(300, 520, 1040) == (1, 64, 8, 3 * 9 * 8)
        w8.debug_force_gemm_form(0)
        assert w8.gemm_form(126, 2048, 2048) == (0, 0, 0, 0)
    finally:
        w8.debug_force_gemm_form(-1)


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


SLOT = 128 * 256 * 4          # one INT32 partial tile


def test_workspace_min_bytes(lib):
    assert w8.workspace_min_bytes(6144, 4096) == 1024 + 1024 + 6144 * 4 + 6144 * 4096 * 2
    assert w8.workspace_min_bytes(126, 2048) == 1024 + 1024 + 1024 + 126 * 2048 * 2
    assert w8.workspace_min_bytes(0, 16) == 0


@pytest.mark.parametrize("M,N,K,plan", [
    # 256 x 256 tiles on CTA pairs (74 pairs on 148 SMs), whatever M.
    # 384 tiles: 5 full waves, the 14 tiles left are cut in 5 (<= sqrt(64) k-blocks)
    (6144, 4096, 4096, (370, 5, 70, 148, 2)),
    (6144, 4096, 16384, (370, 5, 70, 148, 2)),
    (28672, 4096, 4096, (1776, 4, 64, 148, 2)),        # 1792 tiles, 16 left: 74 // 16 = 4
    (6144, 16384, 4096, (1536, 1, 0, 148, 2)),         # 56 left > 37: the last wave is mostly full
    (28672, 16384, 4096, (7168, 1, 0, 148, 2)),
    (1001, 2048, 2048, (32, 1, 0, 64, 2)),             # 32 k-blocks: tiles this short are never cut
    (1001, 8192, 2048, (128, 1, 0, 148, 2)),           # 128 tiles: 54 left > 37
    (256 * 37, 512, 4096, (74, 1, 0, 148, 2)),         # exactly one wave
    # M <= 128 too: the odd CTA of each pair holds rows past M.
    (126, 2048, 2048, (8, 1, 0, 16, 2)),               # 8 tiles of 32 k-blocks: too short to cut
    (126, 8192, 2048, (32, 1, 0, 64, 2)),
    (64, 128, 256, (1, 1, 0, 2, 2)),
    (126, 2048, 4096, (0, 8, 64, 128, 2)),             # 64 k-blocks: cut in sqrt(64) = 8
    (128, 256, 133136, (0, 45, 45, 90, 2)),            # 2081 k-blocks: sqrt caps at 45
])
def test_gemm_plan_for_workload_shapes(lib, M, N, K, plan):
    assert w8.gemm_plan(M, N, K, num_sms=148) == plan
    dp, splits, units, grid, pair = plan
    assert w8.workspace_bytes(M, N, K) == w8.workspace_min_bytes(M, K) + units * pair * SLOT


def test_gemm_plan_single_cta_switch(lib):
    w8.debug_force_single_cta(True)
    try:
        assert w8.gemm_plan(6144, 4096, 4096, num_sms=148) == (740, 5, 140, 148, 1)
        assert w8.gemm_plan(128 * 37, 1024, 4096, num_sms=148) == (148, 1, 0, 148, 1)
    finally:
        w8.debug_force_single_cta(False)
    assert w8.gemm_plan(6144, 4096, 4096, num_sms=148)[4] == 2


def test_gemm_plan_respects_workspace_room(lib):
    # a pair unit needs two slots (one per CTA)
    assert w8.gemm_plan(6144, 4096, 4096, 148, max_slots=100) == (370, 3, 42, 148, 2)
    assert w8.gemm_plan(6144, 4096, 4096, 148, max_slots=55) == (384, 1, 0, 148, 2)
    assert w8.gemm_plan(6144, 4096, 4096, 148, max_slots=0) == (384, 1, 0, 148, 2)
    assert w8.gemm_plan(126, 2048, 4096, 148, max_slots=16) == (8, 1, 0, 16, 2)   # 16 slots: 8 pair units
    assert w8.gemm_plan(126, 2048, 4096, 148, max_slots=32) == (0, 2, 16, 32, 2)


def test_gemm_plan_invariants(lib):
    """Every tile is either whole or cut into `splits` segments of >= 2
    k-blocks; the segment units fit the workers; no more than half a wave is
    cut; CTA pairs whenever the device can hold them."""
    for sms in (148, 132, 8):
        for M in (1, 127, 128, 129, 1000, 6144, 28672):
            for N in (8, 256, 264, 2048, 4096, 16384):
                for K in (16, 64, 128, 1024, 4096, 16384):
                    dp, s, units, grid, pair = w8.gemm_plan(M, N, K, sms)
                    assert pair == 2
                    workers = sms // pair
                    tiles = -(-M // (128 * pair)) * -(-N // 256)
                    kb = -(-K // 64)
                    assert grid % pair == 0 and 1 <= grid // pair <= workers
                    if s == 1:
                        assert dp == tiles and units == 0 and grid == min(tiles, workers) * pair
                    else:
                        rem = tiles - dp
                        assert rem == tiles % workers and 0 < 2 * rem <= workers
                        assert units == rem * s <= workers and kb // s >= 2 and kb >= 48
                        assert s * s <= kb and rem * pair <= 240
                        assert grid == (workers if tiles >= workers else units) * pair


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


def test_host_pipeline_argument_errors(lib):
    """w8a8_linear_host validates before any copy or launch (no GPU here)."""
    p = ctypes.c_void_p(0x10000)
    null = None
    f = lib.w8a8_linear_host
    assert f(null, 1, 64, 256, p, p, 128, null, 1, p, p, p, p, 1 << 20, 0, null) == 1
    assert f(p, 1, 64, 256, p, p, 128, null, 1, null, p, p, p, 1 << 20, 0, null) == 1
    assert f(p, 1, 64, 256, p, p, 128, null, 1, p, p, p, p, 1 << 20, -1, null) == 1
    assert f(p, 5, 64, 256, p, p, 128, null, 1, p, p, p, p, 1 << 20, 0, null) == 2
    assert f(p, 1, 64, 250, p, p, 128, null, 1, p, p, p, p, 1 << 20, 0, null) == 4
    assert f(p, 1, 64, 256, p, p, 128, null, 1, p, p, p, p, 64, 0, null) == 5
    assert f(p, 1, 64, 256, p, p, 128, null, 1, p, ctypes.c_void_p(0x10008), p, p, 1 << 20, 0, null) == 3


@pytest.mark.parametrize("M,N,K,bias,ok,reasons", [
    (1, 8, 8, w8.BF16, True, []),
    (6144, 4096, 4096, w8.F32, True, []),
    (64, 128, 1032, w8.BF16, True, []),          # the INT8 guard rejects K = 8 (mod 16)
    (128, 256, 140000, w8.BF16, True, []),       # past the INT8 path's K limit
    (0, 8, 8, w8.BF16, False, ["M"]),
    (4, 12, 8, w8.BF16, False, ["N"]),
    (4, 8, 20, w8.BF16, False, ["K"]),
    (4, 8, 8, 7, False, ["BIAS_DTYPE"]),
])
def test_bf16_linear_guard(lib, M, N, K, bias, ok, reasons):
    r = ctypes.c_int(0)
    assert bool(lib.w8a8_bf16_linear_supported(M, N, K, bias, ctypes.byref(r))) == ok
    assert [v for k, v in w8.REASONS.items() if r.value & k] == reasons
    assert (w8.bf16_linear_workspace_bytes(M, N, K) > 0) == (ok or reasons == ["BIAS_DTYPE"])


def test_bf16_linear_workspace_sizes(lib):
    """Header only (2 KB with the alignment slack), plus 128 KB per CTA of
    each K-segment when the plan cuts the last wave."""
    assert w8.bf16_linear_workspace_bytes(1, 8, 8) == 2048
    assert w8.bf16_linear_workspace_bytes(6144, 4096, 4096) == 2048 + 70 * 2 * SLOT   # 14 tiles x 5 segments, two CTAs each
    assert w8.bf16_linear_workspace_bytes(64, 128, 1032) == 2048


def test_bf16_linear_argument_errors(lib):
    p = ctypes.c_void_p(0x10000)
    null = None
    f = lib.w8a8_bf16_linear
    assert f(null, 64, 256, p, 128, null, 1, p, p, 1 << 20, null) == 1
    assert f(p, 64, 256, p, 128, p, 9, p, p, 1 << 20, null) == 2
    assert f(p, 64, 250, p, 128, null, 1, p, p, 1 << 20, null) == 4
    assert f(p, 64, 256, p, 12, null, 1, p, p, 1 << 20, null) == 4
    assert f(p, 64, 256, p, 128, null, 1, p, p, 100, null) == 5
    assert f(p, 64, 256, p, 128, null, 1, p, null, 1 << 20, null) == 5
    assert f(p, 64, 256, ctypes.c_void_p(0x10008), 128, null, 1, p, p, 1 << 20, null) == 3


def test_qk_blocks_argument_errors(lib):
    p = ctypes.c_void_p(0x10000)
    null = None
    f = lib.w8a8_quantize_qk_blocks
    assert f(p, w8.BF16, 1, 2, 0, 64, 0, 64, null, null, null) == 0     # empty: no-op
    assert f(null, w8.BF16, 1, 2, 8, 64, 0, 64, p, p, null) == 1
    assert f(p, w8.BF16, 1, 2, 8, 64, 2, 64, p, p, null) == 1          # unknown layout
    assert f(p, 5, 1, 2, 8, 64, 0, 64, p, p, null) == 2
    assert f(p, w8.BF16, 1, 2, 8, 60, 0, 64, p, p, null) == 4          # D % 8
    assert f(p, w8.BF16, 1, 2, 8, 4096, 0, 64, p, p, null) == 4        # D > 2048
    assert f(p, w8.F32, 1, 2, 8, 2048, 0, 64, p, p, null) == 4         # fp32 D > 1024
    assert f(p, w8.BF16, 1, 2, 8, 64, 0, 0, p, p, null) == 4           # block_tokens 0
    assert f(p, w8.BF16, 1, 1, 1 << 31, 64, 0, 64, p, p, null) == 4    # L past int32
    assert f(ctypes.c_void_p(0x10008), w8.BF16, 1, 2, 8, 64, 0, 64, p, p, null) == 3


def test_mlp_workspace_and_argument_errors(lib):
    # both layers' activation codes and scales, the row maxima, and the slots
    # of whichever GEMM plan wants more
    M, K, F, N = 6144, 4096, 16384, 4096
    base = w8.workspace_min_bytes(M, K) + 2 * 24576 + M * F * 2
    up = w8.gemm_plan(M, F, K, num_sms=148)
    dn = w8.gemm_plan(M, N, F, num_sms=148)
    assert w8.mlp_workspace_bytes(M, K, F, N) == base + max(up[2] * up[4], dn[2] * dn[4]) * SLOT
    assert w8.mlp_workspace_bytes(M, K, 1000, N) == 0          # F % 16
    p = ctypes.c_void_p(0x10000)
    null = None
    f = lib.w8a8_mlp
    args = [p, w8.BF16, 64, 256, p, p, 512, null, 1, p, p, 128, null, 1, p, p, p, 1 << 26, null]
    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    assert call(a14=null) == 1                                  # no H
    assert call(a1=7) == 2
    assert call(a6=520) == 4                                    # F % 16 (down layer's K)
    assert call(a11=12) == 4
    assert call(a17=64) == 5
    assert call(a15=ctypes.c_void_p(0x10008)) == 3


def test_norm_argument_errors(lib):
    p = ctypes.c_void_p(0x10000)
    null = None
    f = lib.w8a8_norm_quantize_act
    assert f(null, 4, 64, 1, 1e-6, null, null, 1, null, p, p, null) == 1
    assert f(p, 4, 64, 3, 1e-6, null, null, 1, null, p, p, null) == 1         # unknown norm
    assert f(p, 4, 64, 1, -1.0, null, null, 1, null, p, p, null) == 1         # negative eps
    assert f(p, 4, 64, 1, 1e-6, p, null, 7, null, p, p, null) == 2            # modulation dtype
    assert f(p, 4, 72, 1, 1e-6, null, null, 1, null, p, p, null) == 4         # K % 16
    assert f(p, 4, 32784, 1, 1e-6, null, null, 1, null, p, p, null) == 4      # K > 32768
    assert f(p, 4, 64, 1, 1e-6, ctypes.c_void_p(0x10008), null, 1, null, p, p, null) == 3
    assert f(p, 4, 64, 1, 1e-6, null, null, 1, null, null, p, null) == 1
    g = lib.w8a8_norm_linear
    assert g(p, 4, 64, 1, 1e-6, null, null, 1, p, p, 12, null, 1, p, p, 1 << 20, null) == 4
    assert g(p, 4, 64, 1, 1e-6, null, null, 1, p, p, 128, null, 1, p, p, 64, null) == 5


def test_c_client_links_and_agrees_with_the_binding(tmp_path):
    """A C program built against include/w8a8.h and libw8a8.so alone sees the
    same guard, plan and workspace sizes as the Python binding."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    inc = os.path.join(os.path.dirname(here), "include")
    libdir = os.path.dirname(w8.lib_path())
    exe = tmp_path / "host_client"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", inc, os.path.join(here, "c_abi", "host_client.c"),
                        "-L", libdir, "-l:libw8a8.so", "-Wl,-rpath," + libdir, "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    lines = dict(line.split(" ", 1) for line in out.stdout.strip().splitlines())
    assert lines["version"] == "1"
    assert lines["guard"].split()[:2] == ["1", "0"]
    assert tuple(int(v) for v in lines["plan"].split()[1:]) == w8.gemm_plan(6144, 4096, 4096, num_sms=148)
    assert [int(v) for v in lines["workspace"].split()] == [w8.workspace_min_bytes(6144, 4096),
                                                            w8.workspace_bytes(6144, 4096, 4096)]
    assert int(lines["bf16"].split()[2]) == w8.bf16_linear_workspace_bytes(64, 128, 1032)
    assert int(lines["mlp"]) == w8.mlp_workspace_bytes(6144, 4096, 16384, 4096)
    assert lines["errors"] == "1 1"
