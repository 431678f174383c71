"""Guarded W8A8 linear layer for B300 (sm_103a): thin Python binding.

Every entry point here marshals torch tensors into the C ABI of
``libw8a8.so`` (declared in ``include/w8a8.h``) and raises on a non-OK
status.  All arithmetic runs in the library's CUDA kernels; PyTorch only
provides device memory and the current stream.  There is no CPU path: if the
library cannot be loaded, importing the functions fails loudly.

The layer (zhidx TurboT2VA article, section 01 item 3 "量化策略"): the weight
is quantised once to INT8 per output channel, the activation per row on every
call, the product accumulates in INT32, and the two scales and the bias are
applied once after the full accumulation.  Shapes the guard rejects raise
``UnsupportedShape`` from ``linear``; ``bf16_linear`` runs them natively on
the same tensor-core GEMM with fp32 accumulation, and ``GuardedLinear``
chooses between the two paths.
"""
import ctypes
import os

import torch

__all__ = [
    "W8A8Error", "UnsupportedShape", "lib_path", "load", "shape_supported", "quantize_weight",
    "quantize_act", "pack_weight", "workspace_bytes", "workspace_min_bytes", "gemm_plan", "linear", "linear_quant_stage",
    "linear_gemm_stage", "gemm_s32", "linear_noalloc", "noalloc_read_status", "linear_host", "bf16_linear", "bf16_linear_supported",
    "bf16_linear_workspace_bytes", "quantize_qk_blocks", "mlp", "mlp_workspace_bytes", "norm_quantize_act",
    "norm_linear", "read_status", "set_wait_limit_ns", "debug_skip_loads", "debug_force_single_cta",
    "gemm_form", "debug_force_gemm_form",
    "W8A8Linear", "GuardedLinear", "F32", "BF16", "MAX_K",
]

F32 = 0
BF16 = 1
MAX_K = 133144

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libw8a8.so")
_lib = None

_STATUS = {
    0: "OK", 1: "INVALID_ARG", 2: "DTYPE", 3: "ALIGNMENT", 4: "UNSUPPORTED_SHAPE",
    5: "WORKSPACE", 6: "CUDA", 7: "TIMEOUT", 8: "NO_DEVICE",
}

REASONS = {
    0x01: "M", 0x02: "N", 0x04: "K", 0x08: "K_RANGE", 0x10: "X_DTYPE", 0x20: "BIAS_DTYPE",
}


class W8A8Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s (%s)" % (what, _STATUS.get(status, status), _load().w8a8_status_str(status).decode()))


class UnsupportedShape(W8A8Error):
    pass


def lib_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            "libw8a8.so is not built (expected at %s); run "
            "`python w8a8_int8_linear_act_b300/build.py` or __graft_entry__.build()" % _LIB_PATH)
    lib = ctypes.CDLL(_LIB_PATH)
    p, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    sigs = {
        "w8a8_shape_supported": ([i64, i64, i64, i32, i32, ctypes.POINTER(ctypes.c_int)], i32),
        "w8a8_quantize_weight": ([p, i32, i64, i64, p, p, p], i32),
        "w8a8_quantize_act": ([p, i32, i64, i64, p, p, p], i32),
        "w8a8_pack_weight": ([p, i64, i64, p, p], i32),
        "w8a8_linear_workspace_min_bytes": ([i64, i64], sz),
        "w8a8_linear_workspace_bytes": ([i64, i64, i64], sz),
        "w8a8_gemm_plan": ([i64, i64, i64, i32, i64, ctypes.POINTER(ctypes.c_int64)], i32),
        "w8a8_linear": ([p, i32, i64, i64, p, p, i64, p, i32, p, p, sz, p], i32),
        "w8a8_linear_quant_stage": ([p, i32, i64, i64, p, sz, p], i32),
        "w8a8_linear_gemm_stage": ([i64, i64, p, p, i64, p, i32, p, p, sz, p], i32),
        "w8a8_gemm_s32": ([p, p, i64, i64, i64, p, p, sz, p], i32),
        "w8a8_linear_noalloc": ([p, i32, i64, i64, p, p, i64, p, i32, p, p], i32),
        "w8a8_noalloc_read_status": ([p, ctypes.POINTER(ctypes.c_uint32)], i32),
        "w8a8_linear_host": ([p, i32, i64, i64, p, p, i64, p, i32, p, p, p, p, sz, i64, p], i32),
        "w8a8_bf16_linear_supported": ([i64, i64, i64, i32, ctypes.POINTER(ctypes.c_int)], i32),
        "w8a8_bf16_linear_workspace_bytes": ([i64, i64, i64], sz),
        "w8a8_bf16_linear": ([p, i64, i64, p, i64, p, i32, p, p, sz, p], i32),
        "w8a8_quantize_qk_blocks": ([p, i32, i64, i64, i64, i64, i32, i64, p, p, p], i32),
        "w8a8_mlp_workspace_bytes": ([i64, i64, i64, i64], sz),
        "w8a8_norm_quantize_act": ([p, i64, i64, i32, ctypes.c_float, p, p, i32, p, p, p, p], i32),
        "w8a8_norm_linear": ([p, i64, i64, i32, ctypes.c_float, p, p, i32, p, p, i64, p, i32, p, p, sz, p], i32),
        "w8a8_mlp": ([p, i32, i64, i64, p, p, i64, p, i32, p, p, i64, p, i32, p, p, p, sz, p], i32),
        "w8a8_read_status": ([p, p, ctypes.POINTER(ctypes.c_uint32)], i32),
        "w8a8_set_wait_limit_ns": ([ctypes.c_uint64], None),
        "w8a8_debug_skip_loads": ([i32], None),
        "w8a8_debug_force_single_cta": ([i32], None),
        "w8a8_gemm_form": ([i64, i64, i64, ctypes.POINTER(ctypes.c_int64)], i32),
        "w8a8_debug_force_gemm_form": ([i32, i32, i32], None),
        "w8a8_status_str": ([i32], ctypes.c_char_p),
        "w8a8_version": ([], i32),
    }
    for name, (args, res) in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def load():
    """Load libw8a8.so (raises ImportError if it is missing)."""
    return _load()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError("dtype %s not supported (float32 or bfloat16)" % t.dtype)


def _check(st: int, what: str):
    if st != 0:
        if st == 4:
            raise UnsupportedShape(st, what)
        raise W8A8Error(st, what)


def _cuda2d(t, name):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError("%s must be a contiguous 2-D tensor" % name)


def shape_supported(M: int, N: int, K: int, x_dtype=torch.bfloat16, bias_dtype=torch.bfloat16):
    """(supported, [reason names]) from the library's shape guard (host only)."""
    r = ctypes.c_int(0)
    xd = {torch.float32: F32, torch.bfloat16: BF16}.get(x_dtype, 99)
    bd = {torch.float32: F32, torch.bfloat16: BF16}.get(bias_dtype, 99)
    ok = _load().w8a8_shape_supported(M, N, K, xd, bd, ctypes.byref(r))
    return bool(ok), [v for k, v in REASONS.items() if r.value & k]


def quantize_weight(W: torch.Tensor, stream=None):
    """Static per-output-channel quantisation: W [N, K] -> (Wq int8 [N, K], sw float32 [N])."""
    _cuda2d(W, "W")
    N, K = W.shape
    Wq = torch.empty((N, K), dtype=torch.int8, device=W.device)
    sw = torch.empty((N,), dtype=torch.float32, device=W.device)
    _check(_load().w8a8_quantize_weight(_ptr(W), _dt(W), N, K, _ptr(Wq), _ptr(sw), _stream(stream)),
           "w8a8_quantize_weight")
    return Wq, sw


def quantize_act(X: torch.Tensor, stream=None):
    """Dynamic per-row quantisation: X [M, K] -> (Xq int8 [M, K], sx float32 [M])."""
    _cuda2d(X, "X")
    M, K = X.shape
    Xq = torch.empty((M, K), dtype=torch.int8, device=X.device)
    sx = torch.empty((M,), dtype=torch.float32, device=X.device)
    _check(_load().w8a8_quantize_act(_ptr(X), _dt(X), M, K, _ptr(Xq), _ptr(sx), _stream(stream)),
           "w8a8_quantize_act")
    return Xq, sx


def pack_weight(Wq: torch.Tensor, stream=None) -> torch.Tensor:
    """INT8 codes -> the same integers as bf16 (the tensor-core operand)."""
    _cuda2d(Wq, "Wq")
    N, K = Wq.shape
    Wp = torch.empty((N, K), dtype=torch.bfloat16, device=Wq.device)
    _check(_load().w8a8_pack_weight(_ptr(Wq), N, K, _ptr(Wp), _stream(stream)), "w8a8_pack_weight")
    return Wp


def workspace_bytes(M: int, N: int, K: int) -> int:
    """Workspace for full speed: codes, scales and the GEMM's split partial tiles."""
    return int(_load().w8a8_linear_workspace_bytes(M, N, K))


def workspace_min_bytes(M: int, K: int) -> int:
    """Smallest workspace accepted (no K-split of the GEMM's last wave)."""
    return int(_load().w8a8_linear_workspace_min_bytes(M, K))


def gemm_plan(M: int, N: int, K: int, num_sms: int = 0, max_slots: int = -1):
    """(whole tiles, K-segments per remaining tile, segment units, CTAs,
    CTAs per tile) of the GEMM's tile schedule, from the library's planner.
    num_sms > 0 plans for that many SMs; 0 for the current device."""
    out = (ctypes.c_int64 * 5)()
    if not _load().w8a8_gemm_plan(M, N, K, num_sms, max_slots, out):
        raise ValueError("invalid sizes for a plan: %d x %d x %d" % (M, N, K))
    return tuple(int(v) for v in out)


def gemm_form(M: int, N: int, K: int):
    """(form, tile width, cluster size, CTAs) of the GEMM kernel a launch
    takes for (M, N, K): form 0 the persistent form (see ``gemm_plan``), 1
    the cluster-K form for problems with few output tiles."""
    out = (ctypes.c_int64 * 4)()
    if not _load().w8a8_gemm_form(M, N, K, out):
        raise ValueError("invalid sizes: %d x %d x %d" % (M, N, K))
    return tuple(int(v) for v in out)


def debug_force_gemm_form(form: int = -1, bn: int = 0, ks: int = 0):
    """Test switch: -1 chooses the GEMM form per shape (default), 0 forces
    the persistent form, 1 the cluster-K form (tile width bn, cluster size
    ks; 0 = chosen)."""
    _load().w8a8_debug_force_gemm_form(int(form), int(bn), int(ks))


def _workspace(M, N, K, device, ws):
    if ws is None:
        need = workspace_bytes(M, N, K)
        if need == 0:
            raise UnsupportedShape(4, "workspace size")
        ws = torch.empty((need,), dtype=torch.uint8, device=device)
    elif ws.numel() * ws.element_size() < workspace_min_bytes(M, K):
        raise W8A8Error(5, "workspace")
    return ws


def linear(X: torch.Tensor, Wp: torch.Tensor, sw: torch.Tensor, bias=None, out=None, workspace=None,
           stream=None) -> torch.Tensor:
    """Y [M, N] bf16 = W8A8 linear of X [M, K] with packed weight Wp [N, K] and scales sw [N]."""
    _cuda2d(X, "X")
    _cuda2d(Wp, "Wp")
    M, K = X.shape
    N = Wp.shape[0]
    if Wp.shape[1] != K:
        raise ValueError("K mismatch: X %s, Wp %s" % (tuple(X.shape), tuple(Wp.shape)))
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    ws = _workspace(M, N, K, X.device, workspace)
    bdt = _dt(bias) if bias is not None else BF16
    _check(_load().w8a8_linear(_ptr(X), _dt(X), M, K, _ptr(Wp), _ptr(sw), N, _ptr(bias), bdt, _ptr(out),
                               _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "w8a8_linear")
    return out


def linear_quant_stage(X: torch.Tensor, workspace: torch.Tensor, stream=None):
    """First half of ``linear``: activation codes and row scales into the workspace."""
    _cuda2d(X, "X")
    M, K = X.shape
    _check(_load().w8a8_linear_quant_stage(_ptr(X), _dt(X), M, K, _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream(stream)),
           "w8a8_linear_quant_stage")


def linear_gemm_stage(M: int, K: int, Wp: torch.Tensor, sw: torch.Tensor, bias, out: torch.Tensor,
                      workspace: torch.Tensor, stream=None):
    """Second half of ``linear``: GEMM and epilogue from the workspace's codes."""
    N = Wp.shape[0]
    bdt = _dt(bias) if bias is not None else BF16
    _check(_load().w8a8_linear_gemm_stage(M, K, _ptr(Wp), _ptr(sw), N, _ptr(bias), bdt, _ptr(out),
                                          _ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _stream(stream)), "w8a8_linear_gemm_stage")


def gemm_s32(Xq: torch.Tensor, Wp: torch.Tensor, out=None, workspace=None, stream=None) -> torch.Tensor:
    """acc [M, N] int32 = Xq [M, K] (int8) x Wq^T, from the packed weight Wp [N, K]."""
    _cuda2d(Xq, "Xq")
    _cuda2d(Wp, "Wp")
    M, K = Xq.shape
    N = Wp.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.int32, device=Xq.device)
    ws = _workspace(M, N, K, Xq.device, workspace)
    _check(_load().w8a8_gemm_s32(_ptr(Xq), _ptr(Wp), M, N, K, _ptr(out), _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream)), "w8a8_gemm_s32")
    return out


def linear_host(X_host: torch.Tensor, Wp: torch.Tensor, sw: torch.Tensor, bias=None, out=None,
                X_dev=None, Y_dev=None, workspace=None, chunk_rows: int = 0, stream=None) -> torch.Tensor:
    """``linear`` from a host (CPU) X to a host Y, pipelined over row chunks:
    each chunk's copy in, W8A8 linear and copy out overlap the other chunks'
    (one C call, ``w8a8_linear_host``).  X_host and ``out`` should be pinned
    (``pin_memory()``).  X_dev / Y_dev / workspace are the device staging
    buffers (allocated here when not given).  Ordered on ``stream``."""
    if X_host.is_cuda or X_host.dim() != 2 or not X_host.is_contiguous():
        raise ValueError("X_host must be a contiguous 2-D CPU tensor")
    _cuda2d(Wp, "Wp")
    M, K = X_host.shape
    N = Wp.shape[0]
    dev = Wp.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, pin_memory=True)
    if out.is_cuda or tuple(out.shape) != (M, N) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, N] bfloat16 CPU tensor")
    if X_dev is None:
        X_dev = torch.empty((M, K), dtype=X_host.dtype, device=dev)
    if Y_dev is None:
        Y_dev = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = torch.empty((workspace_bytes(M, N, K),), dtype=torch.uint8, device=dev)
    bdt = _dt(bias) if bias is not None else BF16
    _check(_load().w8a8_linear_host(_ptr(X_host), _dt(X_host), M, K, _ptr(Wp), _ptr(sw), N, _ptr(bias), bdt,
                                    _ptr(out), _ptr(X_dev), _ptr(Y_dev), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), int(chunk_rows),
                                    _stream(stream)), "w8a8_linear_host")
    return out


def bf16_linear_supported(M: int, N: int, K: int, bias_dtype=torch.bfloat16):
    """(supported, [reason names]) for the native BF16 linear (host only)."""
    r = ctypes.c_int(0)
    bd = {torch.float32: F32, torch.bfloat16: BF16}.get(bias_dtype, 99)
    ok = _load().w8a8_bf16_linear_supported(M, N, K, bd, ctypes.byref(r))
    return bool(ok), [v for k, v in REASONS.items() if r.value & k]


def bf16_linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(_load().w8a8_bf16_linear_workspace_bytes(M, N, K))


def bf16_linear(X: torch.Tensor, W: torch.Tensor, bias=None, out=None, workspace=None,
                stream=None) -> torch.Tensor:
    """The native BF16 linear on the same tcgen05 GEMM: Y = bf16(X W^T + bias)
    with fp32 accumulation, for the layers and shapes that do not take the
    W8A8 path (X [M, K] and W [N, K] bfloat16)."""
    _cuda2d(X, "X")
    _cuda2d(W, "W")
    if X.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("bf16_linear takes bfloat16 X and W")
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("K mismatch: X %s, W %s" % (tuple(X.shape), tuple(W.shape)))
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    if workspace is None:
        need = bf16_linear_workspace_bytes(M, N, K)
        if need == 0:
            raise UnsupportedShape(4, "bf16 linear workspace size")
        workspace = torch.empty((need,), dtype=torch.uint8, device=X.device)
    bdt = _dt(bias) if bias is not None else BF16
    _check(_load().w8a8_bf16_linear(_ptr(X), M, K, _ptr(W), N, _ptr(bias), bdt, _ptr(out), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)),
           "w8a8_bf16_linear")
    return out


def mlp_workspace_bytes(M: int, K: int, F: int, N: int) -> int:
    return int(_load().w8a8_mlp_workspace_bytes(M, K, F, N))


def mlp(X: torch.Tensor, Wp_up: torch.Tensor, sw_up: torch.Tensor, bias_up, Wp_down: torch.Tensor,
        sw_down: torch.Tensor, bias_down, H=None, out=None, workspace=None, stream=None):
    """MLP pair Y = down(up(X)) on the W8A8 path, the down layer's row
    quantisation fed by the up GEMM's row maxima.  Returns (Y, H)."""
    _cuda2d(X, "X")
    M, K = X.shape
    F = Wp_up.shape[0]
    N = Wp_down.shape[0]
    if Wp_up.shape[1] != K or Wp_down.shape[1] != F:
        raise ValueError("shape mismatch: X %s, Wp_up %s, Wp_down %s"
                         % (tuple(X.shape), tuple(Wp_up.shape), tuple(Wp_down.shape)))
    if H is None:
        H = torch.empty((M, F), dtype=torch.bfloat16, device=X.device)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    if workspace is None:
        need = mlp_workspace_bytes(M, K, F, N)
        if need == 0:
            raise UnsupportedShape(4, "mlp workspace size")
        workspace = torch.empty((need,), dtype=torch.uint8, device=X.device)
    bu = _dt(bias_up) if bias_up is not None else BF16
    bdn = _dt(bias_down) if bias_down is not None else BF16
    _check(_load().w8a8_mlp(_ptr(X), _dt(X), M, K, _ptr(Wp_up), _ptr(sw_up), F, _ptr(bias_up), bu, _ptr(Wp_down),
                            _ptr(sw_down), N, _ptr(bias_down), bdn, _ptr(H), _ptr(out), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _stream(stream)), "w8a8_mlp")
    return out, H


NORMS = {"rms": 1, "layer": 2}


def _mod_dtype(scale, shift):
    t = scale if scale is not None else shift
    if t is None:
        return BF16
    if scale is not None and shift is not None and scale.dtype != shift.dtype:
        raise TypeError("scale and shift must share a dtype")
    return _dt(t)


def norm_quantize_act(X: torch.Tensor, norm: str = "rms", eps: float = 1e-6, scale=None, shift=None,
                      want_y: bool = False, stream=None):
    """RMS norm or LayerNorm of each row of X (bf16 [M, K]), modulated by
    (1 + scale) and shift ([K] or None), rounded to bf16 and quantised per
    row.  Returns (Xq int8, sx float32) or (Xq, sx, y bf16) with want_y."""
    _cuda2d(X, "X")
    if X.dtype != torch.bfloat16:
        raise TypeError("norm_quantize_act takes bfloat16 X")
    M, K = X.shape
    Xq = torch.empty((M, K), dtype=torch.int8, device=X.device)
    sx = torch.empty((M,), dtype=torch.float32, device=X.device)
    y = torch.empty((M, K), dtype=torch.bfloat16, device=X.device) if want_y else None
    _check(_load().w8a8_norm_quantize_act(_ptr(X), M, K, NORMS[norm], eps, _ptr(scale), _ptr(shift),
                                          _mod_dtype(scale, shift), _ptr(y), _ptr(Xq), _ptr(sx), _stream(stream)),
           "w8a8_norm_quantize_act")
    return (Xq, sx, y) if want_y else (Xq, sx)


def norm_linear(X: torch.Tensor, Wp: torch.Tensor, sw: torch.Tensor, bias=None, norm: str = "rms",
                eps: float = 1e-6, scale=None, shift=None, out=None, workspace=None, stream=None) -> torch.Tensor:
    """The W8A8 linear with the norm + modulation prologue fused into its
    activation quantisation: Y = linear(bf16(norm(X) * (1 + scale) + shift))."""
    _cuda2d(X, "X")
    M, K = X.shape
    N = Wp.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    if workspace is None:
        workspace = torch.empty((workspace_bytes(M, N, K),), dtype=torch.uint8, device=X.device)
    bdt = _dt(bias) if bias is not None else BF16
    _check(_load().w8a8_norm_linear(_ptr(X), M, K, NORMS[norm], eps, _ptr(scale), _ptr(shift),
                                    _mod_dtype(scale, shift), _ptr(Wp), _ptr(sw), N, _ptr(bias), bdt, _ptr(out),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "w8a8_norm_linear")
    return out


LAYOUTS = {"HND": 0, "NHD": 1}


def quantize_qk_blocks(X: torch.Tensor, block_tokens: int, layout: str = "HND", stream=None):
    """Per-block INT8 quantisation of attention Query or Key (the SageSLA
    path's INT8 Q/K).  X is [B, H, L, D] ("HND") or [B, L, H, D] ("NHD"),
    contiguous.  Returns (codes int8, same shape; scales float32
    [B, H, ceil(L / block_tokens)])."""
    if not X.is_cuda or X.dim() != 4 or not X.is_contiguous():
        raise ValueError("X must be a contiguous 4-D CUDA tensor")
    if layout not in LAYOUTS:
        raise ValueError("layout must be 'HND' or 'NHD'")
    if layout == "HND":
        B, H, L, D = X.shape
    else:
        B, L, H, D = X.shape
    if block_tokens < 1:
        raise ValueError("block_tokens must be >= 1")
    nblk = -(-L // block_tokens) if L > 0 else 0
    Xq = torch.empty(X.shape, dtype=torch.int8, device=X.device)
    S = torch.empty((B, H, nblk), dtype=torch.float32, device=X.device)
    _check(_load().w8a8_quantize_qk_blocks(_ptr(X), _dt(X), B, H, L, D, LAYOUTS[layout], block_tokens, _ptr(Xq),
                                           _ptr(S), _stream(stream)), "w8a8_quantize_qk_blocks")
    return Xq, S


NOALLOC_SCRATCH_BYTES = 64 << 20


def linear_noalloc(X: torch.Tensor, Wp: torch.Tensor, sw: torch.Tensor, bias=None, out=None,
                   stream=None) -> torch.Tensor:
    """``linear`` without a workspace argument, for callers that cannot get
    device memory at the call site (a plugin whose host runtime owns all device
    memory, or a path that must not call cudaMalloc).  The library uses its own
    built-in 64 MiB scratch array; the caller still provides X, Wp, sw, bias
    and (optionally) Y.  Calls that may overlap on the GPU must be serialised:
    they share that one array.  Shapes whose workspace would exceed it raise
    ``W8A8Error`` (WORKSPACE)."""
    _cuda2d(X, "X")
    _cuda2d(Wp, "Wp")
    M, K = X.shape
    N = Wp.shape[0]
    if Wp.shape[1] != K:
        raise ValueError("K mismatch: X %s, Wp %s" % (tuple(X.shape), tuple(Wp.shape)))
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    bdt = _dt(bias) if bias is not None else BF16
    _check(_load().w8a8_linear_noalloc(_ptr(X), _dt(X), M, K, _ptr(Wp), _ptr(sw), N, _ptr(bias), bdt,
                                       _ptr(out), _stream(stream)), "w8a8_linear_noalloc")
    return out


def noalloc_read_status(stream=None):
    """(status, device bits) of ``linear_noalloc``'s built-in workspace, as
    ``read_status`` gives them for a caller-owned one: synchronises the
    stream, then status 0 (OK) with bits 0, or 7 (TIMEOUT) with the
    W8A8_DEV_* bits of the device-side waits that ran out."""
    v = ctypes.c_uint32(0)
    st = _load().w8a8_noalloc_read_status(_stream(stream), ctypes.byref(v))
    if st not in (0, 7):
        _check(st, "w8a8_noalloc_read_status")
    return st, v.value


def read_status(workspace: torch.Tensor, stream=None):
    """(status, device bits) of the last call that used this workspace (synchronises the stream)."""
    bits = ctypes.c_uint32(0)
    st = _load().w8a8_read_status(_ptr(workspace), _stream(stream), ctypes.byref(bits))
    return st, bits.value


def set_wait_limit_ns(ns: int):
    _load().w8a8_set_wait_limit_ns(int(ns))


def debug_skip_loads(on: bool):
    _load().w8a8_debug_skip_loads(1 if on else 0)


def debug_force_single_cta(on: bool):
    """Test hook: run every GEMM in the single-CTA form (128-row tiles)."""
    _load().w8a8_debug_force_single_cta(1 if on else 0)


class W8A8Linear:
    """A linear layer with static INT8 weights: quantises W once, then
    ``layer(X)`` runs the guarded W8A8 path (activation quantisation, tensor-core
    INT32-exact GEMM, fused dequantisation + bias + bf16 store)."""

    def __init__(self, weight: torch.Tensor, bias=None):
        self.Wq, self.sw = quantize_weight(weight)
        self.Wp = pack_weight(self.Wq)
        self.bias = bias
        self.out_features, self.in_features = weight.shape
        self._ws = None

    def supported(self, M: int, x_dtype=torch.bfloat16) -> bool:
        bdt = self.bias.dtype if self.bias is not None else torch.bfloat16
        return shape_supported(M, self.out_features, self.in_features, x_dtype, bdt)[0]

    def __call__(self, X: torch.Tensor, out=None) -> torch.Tensor:
        M, K = X.shape
        need = workspace_bytes(M, self.out_features, K)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty((need,), dtype=torch.uint8, device=X.device)
        return linear(X, self.Wp, self.sw, self.bias, out=out, workspace=self._ws)


class GuardedLinear:
    """A linear layer that takes the W8A8 path where the library's shape
    guard accepts it and the native BF16 linear (same tensor-core GEMM, fp32
    accumulation) where it does not: the guarded W8A8 layer of the TurboT2VA
    pages (zhidx article, section 01 item 3; arXiv paper, appendix C).
    The choice per layer follows from (N, K, bias dtype); per call, a row
    count the guard rejects also takes the BF16 path.

    ``policy``:
      "int8"     (default) the W8A8 path wherever the guard accepts: the method
                 as the pages give it.
      "fastest"  per row count, whichever of the two paths is faster on this
                 GPU, timed (CUDA events, median of 5 calls each after 3
                 warm-up calls) on the first call with that row count and
                 kept.  On B300 the bf16 tensor pipe carries both paths, so
                 W8A8 wins only where its lower power draw holds the clock
                 up under the power cap (the longest GEMMs) and loses where
                 the activation quantisation is a large share of the call.
                 Both outputs are correct; they differ by the quantisation
                 error.  Needs a bfloat16 weight (kept for the BF16 path)."""

    POLICIES = ("int8", "fastest")

    def __init__(self, weight: torch.Tensor, bias=None, policy: str = "int8"):
        _cuda2d(weight, "weight")
        if policy not in self.POLICIES:
            raise ValueError("policy must be one of %s" % (self.POLICIES,))
        self.policy = policy
        self.out_features, self.in_features = weight.shape
        bdt = bias.dtype if bias is not None else torch.bfloat16
        self.int8 = shape_supported(1, self.out_features, self.in_features, torch.bfloat16, bdt)[0]
        self.bias = bias
        self.weight = weight if weight.dtype == torch.bfloat16 else None
        self._w8a8 = W8A8Linear(weight, bias) if self.int8 else None
        self._ws = None
        self.choice = {}   # (rows, activation dtype) -> "int8" or "bf16", for policy "fastest"
        if (not self.int8 or policy == "fastest") and self.weight is None:
            raise TypeError("the BF16 path of this layer needs a bfloat16 weight")

    def _bf16(self, X: torch.Tensor, out=None) -> torch.Tensor:
        M = X.shape[0]
        need = bf16_linear_workspace_bytes(M, self.out_features, self.in_features)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty((max(need, 1),), dtype=torch.uint8, device=X.device)
        Xb = X if X.dtype == torch.bfloat16 else X.to(torch.bfloat16)
        return bf16_linear(Xb, self.weight, self.bias, out=out, workspace=self._ws)

    def _fastest(self, X: torch.Tensor) -> str:
        key = (X.shape[0], X.dtype)
        if key not in self.choice:
            stream = torch.cuda.current_stream()
            times = {}
            for name, fn in (("int8", lambda: self._w8a8(X)), ("bf16", lambda: self._bf16(X))):
                for _ in range(3):
                    fn()
                ts = []
                for _ in range(5):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    fn()
                    b.record(stream)
                    b.synchronize()
                    ts.append(a.elapsed_time(b))
                times[name] = sorted(ts)[2]
            self.choice[key] = "int8" if times["int8"] <= times["bf16"] else "bf16"
        return self.choice[key]

    def __call__(self, X: torch.Tensor, out=None) -> torch.Tensor:
        M = X.shape[0]
        if self._w8a8 is not None and self._w8a8.supported(M, X.dtype):
            if self.policy == "int8" or self._fastest(X) == "int8":
                return self._w8a8(X, out=out)
        if self.weight is None:
            raise UnsupportedShape(4, "GuardedLinear: no bfloat16 weight kept for the BF16 path")
        return self._bf16(X, out=out)
