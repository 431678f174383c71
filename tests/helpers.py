"""Shared test helpers: tensor <-> numpy views and oracle-side references.

Nothing here computes the method: it only moves data between torch and
numpy and calls the oracle."""
import numpy as np
import torch

import oracle


def bits(t: torch.Tensor) -> np.ndarray:
    """numpy view of a CPU tensor; bf16 tensors become their uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bias_f32(bias: torch.Tensor):
    """The bias as the oracle takes it: exact fp32 widening of bf16 or fp32."""
    if bias is None:
        return None
    b = bits(bias)
    return oracle.bf16_bits_to_f32(b) if b.dtype == np.uint16 else b.astype(np.float32)


def assert_within_one_bf16_ulp(y_gpu_bits: np.ndarray, y32: np.ndarray, what: str = ""):
    """|Y_gpu - y32| <= 1 bf16 ulp of y32, element by element; returns the
    fraction of outputs that are bit-identical to the oracle's bf16."""
    yg = oracle.bf16_bits_to_f32(y_gpu_bits).astype(np.float64)
    ref = y32.astype(np.float64)
    err = np.abs(yg - ref)
    tol = oracle.ulp_bf16(ref)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d outputs beyond 1 bf16 ulp, e.g. %s"
                             % (what, int(bad.sum()), [(tuple(i), yg[tuple(i)], ref[tuple(i)]) for i in idx]))
    same = (y_gpu_bits == oracle.bf16_rne(y32.ravel()).reshape(y32.shape)) if y32.size < 2_000_000 else None
    return None if same is None else float(same.mean())


def check_linear_in_row_blocks(X_bits: np.ndarray, wq: np.ndarray, sw: np.ndarray, bias32, y_gpu_bits: np.ndarray,
                               acc_gpu: np.ndarray = None, block_rows: int = 2048, what: str = ""):
    """Every output of a full-size layer against the oracle, a block of rows
    at a time (host memory stays bounded): the oracle's activation codes
    once, then per block the exact INT32 accumulators (float64 product of the
    codes, exact: every partial sum is an integer below 2^53) and the fp32
    epilogue.  GPU accumulators, when given, must equal them bit for bit; GPU
    outputs must lie within one bf16 ulp of y32.  Returns the fraction of
    outputs bit-identical to the oracle's bf16."""
    xq, sx = oracle.quantize_rows(X_bits)
    M = xq.shape[0]
    same = 0
    for r0 in range(0, M, block_rows):
        r1 = min(M, r0 + block_rows)
        acc = oracle.gemm_s32_f64(xq[r0:r1], wq)
        if acc_gpu is not None:
            bad = np.argwhere(acc_gpu[r0:r1] != acc)
            assert bad.size == 0, "%s: INT32 accumulators differ at rows %d.., e.g. %s" % (what, r0, bad[:5].tolist())
        y32, yb = oracle.epilogue(acc, sx[r0:r1], sw, bias32)
        assert_within_one_bf16_ulp(y_gpu_bits[r0:r1], y32, "%s rows %d..%d" % (what, r0, r1))
        same += int((y_gpu_bits[r0:r1] == yb).sum())
    return same / float(y_gpu_bits.size), xq, sx
