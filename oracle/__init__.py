"""CPU oracle for the guarded W8A8 linear layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg (and its ``--impl reference`` arm) import this
package.  The product library never does, and the two share no code: the
arithmetic lives in ``w8a8_oracle.c`` (plain scalar C), called here through
ctypes on numpy arrays.

Definition followed (zhidx article "音视频生成提速54倍！浙大等团队开源联合蒸馏方案
TurboT2VA", section 01 item 3 "量化策略"): weights INT8 per output channel
(static), activations INT8 per row (dynamic), INT32 accumulation, scales and
bias applied once after the full accumulation.  The readings the pages leave
open are listed in ``w8a8_oracle.c``'s header.

Functions:
  quantize_rows(A)          -> (q int8 [R,K], s float32 [R])      scalar C
  gemm_s32(Xq, Wq, rows)    -> int32 [len(rows), N]               scalar C, int64-checked
  gemm_s32_f64(Xq, Wq)      -> int32 [M, N]                       numpy float64 matmul of the
                               codes; exact because every partial sum is an integer below 2^53
  epilogue(acc, sx, sw, b)  -> (y32 float32, y bf16 bits uint16)  scalar C
  bf16_rne(x float32)       -> uint16 bf16 bits                   scalar C
  linear(X, Wq, sw, bias)   -> the whole path for chosen rows
  bf16_linear_f64(X, W, b)  -> the native BF16 linear that guard-rejected branches run:
                               sum_k X W + b in float64 (bf16 products are exact in
                               float64), and sum_k |X W| for the fp32-accumulation bound
  bf16_linear_tolerance(..) -> that bound, per output
  norm_modulate_f64(X, kind, eps, scale, shift)
                            -> the normalised and modulated rows in float64 (RMS norm or
                               LayerNorm, then x * (1 + scale) + shift), with mean and 1/std
  norm_quantize(X, ...)     -> codes and scales of bf16_rne of those rows (quantize_rows)
  quantize_qk_blocks(X, bt, layout)
                            -> per-block INT8 codes and scales of attention Query/Key:
                               quantize_rows applied to each block of bt tokens of one
                               (batch, head), flattened

bf16 tensors are passed as their raw 16-bit patterns (numpy uint16).
"""
import ctypes
import os

import numpy as np

from . import build_oracle

_lib = None

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def _load():
    global _lib
    if _lib is None:
        path = build_oracle.build()
        lib = ctypes.CDLL(path)
        lib.oracle_quantize_rows_f32.argtypes = [_p, _i64, _i64, _p, _p]
        lib.oracle_quantize_rows_f32.restype = ctypes.c_int
        lib.oracle_quantize_rows_bf16.argtypes = [_p, _i64, _i64, _p, _p]
        lib.oracle_quantize_rows_bf16.restype = ctypes.c_int
        lib.oracle_gemm_s32.argtypes = [_p, _p, _i64, _i64, _i64, _p, _i64, _p]
        lib.oracle_gemm_s32.restype = ctypes.c_int64
        lib.oracle_epilogue.argtypes = [_p, _i64, _i64, _p, _p, _p, _p, _p]
        lib.oracle_epilogue.restype = None
        lib.oracle_bf16_rne.argtypes = [ctypes.c_float]
        lib.oracle_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_bf16_rne_array.argtypes = [_p, _i64, _p]
        lib.oracle_bf16_rne_array.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_num_threads.restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def quantize_rows(A: np.ndarray, dtype: str = None):
    """Per-row symmetric INT8 quantisation of A[R, K].

    ``A`` is float32, or uint16 holding bf16 bit patterns (``dtype='bf16'``,
    the default for uint16 arrays).  Returns (codes int8 [R, K], scales
    float32 [R]).  Rows whose fp32 absmax/127 is 0 get scale 1 and zero codes.
    """
    A = np.ascontiguousarray(A)
    if A.ndim != 2:
        raise ValueError("A must be 2-D")
    R, K = A.shape
    q = np.empty((R, K), dtype=np.int8)
    s = np.empty((R,), dtype=np.float32)
    lib = _load()
    if A.dtype == np.float32 and dtype in (None, "f32"):
        rc = lib.oracle_quantize_rows_f32(_ptr(A), R, K, _ptr(q), _ptr(s))
    elif A.dtype == np.uint16 and dtype in (None, "bf16"):
        rc = lib.oracle_quantize_rows_bf16(_ptr(A), R, K, _ptr(q), _ptr(s))
    else:
        raise TypeError("A must be float32 or uint16 (bf16 bits), got %s" % A.dtype)
    if rc != 0:
        raise ValueError("non-finite input: the quantiser is not defined there")
    return q, s


def gemm_s32(Xq: np.ndarray, Wq: np.ndarray, rows=None) -> np.ndarray:
    """acc[i, n] = sum_k Xq[rows[i], k] * Wq[n, k], in int64, checked to fit INT32."""
    Xq = np.ascontiguousarray(Xq, dtype=np.int8)
    Wq = np.ascontiguousarray(Wq, dtype=np.int8)
    M, K = Xq.shape
    N, K2 = Wq.shape
    if K != K2:
        raise ValueError("K mismatch")
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    acc = np.empty((rows.shape[0], N), dtype=np.int32)
    over = _load().oracle_gemm_s32(_ptr(Xq), _ptr(Wq), M, N, K, _ptr(rows), rows.shape[0], _ptr(acc))
    if over != 0:
        raise OverflowError("%d accumulators (or row indices) outside INT32 / range" % over)
    return acc


def gemm_s32_f64(Xq: np.ndarray, Wq: np.ndarray) -> np.ndarray:
    """The same accumulators through a float64 matrix product of the codes.

    Every product is at most 127*127 = 16129 and |sum| <= K*16129, far below
    2^53 for any K the layer accepts, so every partial sum of the BLAS routine
    is an exactly representable integer and the result is exact whatever order
    it sums in.  Used for the large configurations; checked against
    ``gemm_s32`` by the tests.
    """
    K = Xq.shape[1]
    if K * 16129 >= 2 ** 53:
        raise ValueError("K too large for an exact float64 product")
    acc = Xq.astype(np.float64) @ Wq.astype(np.float64).T
    if np.abs(acc).max(initial=0.0) > 2 ** 31 - 1:
        raise OverflowError("accumulator outside INT32")
    return acc.astype(np.int32)


def epilogue(acc: np.ndarray, sx: np.ndarray, sw: np.ndarray, bias=None):
    """y32 = ((float)acc * sx[row]) * sw[n] + bias[n] in fp32 steps; Y = bf16_rne(y32).

    ``bias`` is float32 (bf16 biases are widened exactly by the caller with
    ``bf16_bits_to_f32``) or None.  Returns (y32 float32, Y uint16 bf16 bits).
    """
    acc = np.ascontiguousarray(acc, dtype=np.int32)
    nrows, N = acc.shape
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    if sx.shape != (nrows,) or sw.shape != (N,):
        raise ValueError("scale shapes")
    b = None
    if bias is not None:
        b = np.ascontiguousarray(bias, dtype=np.float32)
        if b.shape != (N,):
            raise ValueError("bias shape")
    y32 = np.empty((nrows, N), dtype=np.float32)
    y = np.empty((nrows, N), dtype=np.uint16)
    _load().oracle_epilogue(_ptr(acc), nrows, N, _ptr(sx), _ptr(sw),
                            _ptr(b) if b is not None else None, _ptr(y32), _ptr(y))
    return y32, y


def bf16_rne(x) -> np.ndarray:
    """bf16 round-to-nearest-even of float32 values, as uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_bf16_rne_array(_ptr(x), x.size, _ptr(out))
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def linear(X: np.ndarray, Wq: np.ndarray, sw: np.ndarray, bias=None, rows=None, exact_f64=False):
    """The hot path for a set of rows: act quant -> INT32 GEMM -> epilogue.

    X is float32 or uint16 (bf16 bits) [M, K]; Wq int8 [N, K]; sw float32 [N];
    bias float32 [N] or None.  Returns dict with xq, sx (all rows), acc, y32,
    y (bf16 bits) for the chosen rows.  ``exact_f64`` takes the float64-matmul
    accumulator path (same result, faster for large shapes).
    """
    xq, sx = quantize_rows(X)
    if rows is None:
        rows = np.arange(X.shape[0], dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    if exact_f64:
        acc = gemm_s32_f64(xq[rows], Wq)
    else:
        acc = gemm_s32(xq, Wq, rows)
    y32, y = epilogue(acc, sx[rows], sw, bias)
    return {"xq": xq, "sx": sx, "rows": rows, "acc": acc, "y32": y32, "y": y}


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v|: 2^(floor(log2|v|) - 7) for normal v,
    and the subnormal spacing 2^-133 below 2^-126."""
    v = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(v > 0, v, 1.0)))
    e = np.maximum(e, -126.0)
    return np.exp2(e - 7.0)


def bf16_linear_f64(X_bits: np.ndarray, W_bits: np.ndarray, bias=None, rows=None):
    """The native BF16 linear (the branches the guarded W8A8 path does not
    take fall back to it: zhidx article, section 01 item 3), exactly enough
    to bound an fp32-accumulating GPU result.

    X_bits [M, K], W_bits [N, K] are bf16 bit patterns (uint16); bias is
    float32 [N] or None.  Every product of two bf16 values has at most 16
    significant bits and is exact in float64; the float64 sum is within
    K * 2^-53 * sum|x w| of the exact sum.  Returns (y64 [R, N], absum
    [R, N]) for the chosen rows, with absum = sum_k |x_k w_k| + |bias|.
    """
    if rows is None:
        rows = np.arange(X_bits.shape[0], dtype=np.int64)
    x = bf16_bits_to_f32(np.ascontiguousarray(X_bits[rows])).astype(np.float64)
    w = bf16_bits_to_f32(np.ascontiguousarray(W_bits)).astype(np.float64)
    y = x @ w.T
    absum = np.abs(x) @ np.abs(w).T
    if bias is not None:
        b = np.asarray(bias, dtype=np.float64)
        y = y + b[None, :]
        absum = absum + np.abs(b)[None, :]
    return y, absum


def bf16_linear_tolerance(y64: np.ndarray, absum: np.ndarray, K: int) -> np.ndarray:
    """Bound on |Y - y64| for Y = bf16(fp32-accumulated sum + bias): one bf16
    ulp of the result (final rounding, with margin) plus 2 * (K + 1) * 2^-24 *
    sum|x w| (K + 1 fp32 additions of terms bounded by sum|x w|, each off by
    at most one fp32 ulp of the running sum: the usual recursive-summation
    bound, doubled for truncating adders)."""
    return ulp_bf16(y64) + 2.0 * (K + 1) * np.exp2(-24.0) * absum


def quantize_qk_blocks(X: np.ndarray, block_tokens: int, layout: str = "HND"):
    """Per-block INT8 quantisation of attention Query or Key (zhidx TurboT2VA
    article, section 01 item 4: SageSLA quantises Query and Key to INT8).

    X is [B, H, L, D] ("HND") or [B, L, H, D] ("NHD"), float32 or bf16 bits.
    Each block of ``block_tokens`` consecutive tokens of one (batch, head),
    the last one possibly shorter, is flattened to one row and quantised by
    ``quantize_rows`` (one scale per block).  Returns (codes int8 in X's
    shape, scales float32 [B, H, nblk])."""
    Xh = X if layout == "HND" else X.transpose(0, 2, 1, 3)
    B, H, L, D = Xh.shape
    bt = min(block_tokens, L)
    nblk = -(-L // bt)
    q = np.empty((B, H, L, D), dtype=np.int8)
    s = np.empty((B, H, nblk), dtype=np.float32)
    for j in range(nblk):
        t0, t1 = j * bt, min(L, (j + 1) * bt)
        rows = np.ascontiguousarray(Xh[:, :, t0:t1, :]).reshape(B * H, (t1 - t0) * D)
        qj, sj = quantize_rows(rows)
        q[:, :, t0:t1, :] = qj.reshape(B, H, t1 - t0, D)
        s[:, :, j] = sj.reshape(B, H)
    return (q if layout == "HND" else np.ascontiguousarray(q.transpose(0, 2, 1, 3))), s


def norm_modulate_f64(X_bits: np.ndarray, kind: str, eps: float, scale=None, shift=None):
    """Normalisation and modulation before a linear layer, as the TurboT2VA
    pages fuse them (zhidx article, section 01: normalisation and modulation
    fused to cut intermediate reads and writes; arXiv paper, appendix C).

    Per row x of X (bf16 bits [M, K]), in float64:
      kind "rms":   mu = 0;             v = mean(x^2)
      kind "layer": mu = mean(x);       v = mean((x - mu)^2)
      r = 1 / sqrt(v + eps)
      y = (x - mu) * r * (1 + scale) + shift     (scale, shift: [K] or None)
    Returns (y [M, K], mu [M], r [M]), all float64."""
    x = bf16_bits_to_f32(np.ascontiguousarray(X_bits)).astype(np.float64)
    K = x.shape[1]
    if kind == "rms":
        mu = np.zeros(x.shape[0])
    elif kind == "layer":
        mu = x.sum(axis=1) / K
    else:
        raise ValueError("kind must be 'rms' or 'layer'")
    d = x - mu[:, None]
    r = 1.0 / np.sqrt((d * d).sum(axis=1) / K + eps)
    y = d * r[:, None]
    if scale is not None:
        y = y * (1.0 + np.asarray(scale, dtype=np.float64))[None, :]
    if shift is not None:
        y = y + np.asarray(shift, dtype=np.float64)[None, :]
    return y, mu, r


def norm_quantize(X_bits: np.ndarray, kind: str, eps: float, scale=None, shift=None):
    """The rows above rounded to bf16 (nearest even) and quantised by the row
    rule (zhidx article, section 01 item 3).  Returns (y_bf16 bits, codes,
    scales, y float64)."""
    y, _, _ = norm_modulate_f64(X_bits, kind, eps, scale, shift)
    yb = bf16_rne(y.astype(np.float32).ravel()).reshape(y.shape)
    q, s = quantize_rows(yb)
    return yb, q, s, y

