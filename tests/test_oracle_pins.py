"""Pins for the CPU oracle: each test checks it against something other than
itself (closed forms, brute force, invariants, textbook or library routines).

Method being pinned: the zhidx article "音视频生成提速54倍！浙大等团队开源联合蒸馏方案
TurboT2VA", section 01 item 3 ("量化策略"): per-output-channel static INT8
weights, per-row dynamic INT8 activations, INT32 accumulation, scales and bias
applied once after the full accumulation.  Readings the pages leave open
(symmetric absmax/127 scale, IEEE division, round half to even, clamp to
[-127, 127], zero row -> scale 1) are the ones stated in the oracle's header.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def f32(x):
    return np.float32(x)


# --------------------------------------------------------------------------
# Quantiser
# --------------------------------------------------------------------------

@pytest.mark.parametrize("e", [-20, -7, 0, 3, 10, 60, 120])
def test_quant_lossless_power_of_two_scale(e):
    """x = k * 2^e with one |k| = 127 per row: the scale is exactly 2^e, the
    codes are exactly k, and q * s reproduces x bit for bit."""
    rng = np.random.default_rng(100 + e)
    R, K = 9, 300
    k = rng.integers(-127, 128, size=(R, K))
    k[np.arange(R), rng.integers(0, K, size=R)] = rng.choice([-127, 127], size=R)
    x = (k * 2.0 ** e).astype(np.float32)
    assert np.array_equal(x.astype(np.float64), k * 2.0 ** e)   # inputs exact
    q, s = oracle.quantize_rows(x)
    assert np.array_equal(s, np.full(R, 2.0 ** e, dtype=np.float32))
    assert np.array_equal(q.astype(np.int64), k)
    assert np.array_equal(q.astype(np.float32) * s[:, None], x)


def test_quant_all_255_codes_brute_force():
    """Every code value -127..127 appears exactly where the closed form says."""
    codes = np.arange(-127, 128)
    for e in (-9, 0, 5):
        x = (codes * 2.0 ** e).astype(np.float32)[None, :]
        q, s = oracle.quantize_rows(x)
        assert s[0] == f32(2.0 ** e)
        assert np.array_equal(q[0].astype(np.int64), codes)


def test_quant_ties_round_half_to_even():
    """With s = 2^-4 exactly, x = (j + 0.5) * 2^-4 divides to exactly j + 0.5;
    the code must be the even neighbour.  Python's round() is round half to
    even, the textbook rule, and supplies the expected values."""
    js = np.arange(-127, 127)                       # j + 0.5 in (-127, 127)
    vals = (js + 0.5) * 2.0 ** -4
    x = np.concatenate([[127 * 2.0 ** -4], vals]).astype(np.float32)[None, :]
    q, s = oracle.quantize_rows(x)
    assert s[0] == f32(2.0 ** -4)
    expect = np.array([127] + [round(j + 0.5) for j in js])
    assert np.array_equal(q[0].astype(np.int64), expect)
    # spot values written out: 0.5 -> 0, 1.5 -> 2, 2.5 -> 2, -0.5 -> 0, -1.5 -> -2, 126.5 -> 126
    pos = {v: i + 1 for i, v in enumerate(js)}
    assert q[0, pos[0]] == 0 and q[0, pos[1]] == 2 and q[0, pos[2]] == 2
    assert q[0, pos[-1]] == 0 and q[0, pos[-2]] == -2 and q[0, pos[126]] == 126


def test_quant_zero_row_scale_one():
    x = np.zeros((3, 64), dtype=np.float32)
    x[1, 5] = 3.0
    q, s = oracle.quantize_rows(x)
    assert s[0] == 1.0 and s[2] == 1.0
    assert not q[0].any() and not q[2].any()
    assert q[1, 5] == 127 and np.count_nonzero(q[1]) == 1


def test_quant_negative_zero_row_is_zero_row():
    x = np.full((1, 16), -0.0, dtype=np.float32)
    q, s = oracle.quantize_rows(x)
    assert s[0] == 1.0 and not q.any()


def test_quant_underflowing_scale_is_zero_row():
    """fp32 absmax below 127 * 2^-150 makes amax/127 round to 0: the row is
    treated as a zero row (scale 1, codes 0).  One denormal step above that
    it is a normal row with a denormal scale."""
    tiny = np.float32(np.ldexp(1.0, -149))                # smallest denormal
    x = np.array([[tiny * 63, 0.0, -tiny]], dtype=np.float32)
    q, s = oracle.quantize_rows(x)
    assert s[0] == 1.0 and not q.any()
    x2 = np.array([[tiny * 127, -tiny * 127, 0.0]], dtype=np.float32)
    q2, s2 = oracle.quantize_rows(x2)
    assert s2[0] == tiny and list(q2[0]) == [127, -127, 0]


def test_quant_single_element_rows():
    """A one-element row quantises to +-127 with q*s within one rounding of x."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((200, 1)) * 10.0 ** rng.integers(-30, 30, size=(200, 1))).astype(np.float32)
    q, s = oracle.quantize_rows(x)
    assert np.array_equal(q[:, 0], np.where(x[:, 0] > 0, 127, -127).astype(np.int8))
    rel = np.abs(q[:, 0].astype(np.float64) * s - x[:, 0]) / np.abs(x[:, 0])
    assert rel.max() <= 2.0 ** -23


def test_quant_invariants_random():
    """Every non-zero row reaches |q| = 127; |x - q s| <= s/2 (plus the two
    fp32 roundings of s and x/s); odd symmetry; exact power-of-two scaling."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((50, 777)).astype(np.float32)
    x[:, rng.choice(777, 8, replace=False)] *= 20
    q, s = oracle.quantize_rows(x)
    assert (np.abs(q).max(axis=1) == 127).all()
    assert np.abs(q).max() <= 127 and q.min() >= -127
    err = np.abs(x.astype(np.float64) - q.astype(np.float64) * s[:, None].astype(np.float64))
    assert (err <= s[:, None] * (0.5 + 2.0 ** -20)).all()
    qn, sn = oracle.quantize_rows(-x)
    assert np.array_equal(qn, -q) and np.array_equal(sn, s)
    q4, s4 = oracle.quantize_rows(x * np.float32(4.0))
    assert np.array_equal(q4, q) and np.array_equal(s4, s * np.float32(4.0))


def test_quant_row_independence_and_order():
    """Each row uses its own absmax only: quantising rows one by one, or in a
    shuffled order, gives the same codes and scales (catches a shared or
    mis-indexed scale)."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((20, 65)) * rng.uniform(0.01, 100, size=(20, 1))).astype(np.float32)
    q, s = oracle.quantize_rows(x)
    perm = rng.permutation(20)
    qp, sp = oracle.quantize_rows(x[perm])
    assert np.array_equal(qp, q[perm]) and np.array_equal(sp, s[perm])
    for r in (0, 7, 19):
        q1, s1 = oracle.quantize_rows(x[r:r + 1])
        assert np.array_equal(q1[0], q[r]) and s1[0] == s[r]


def test_quant_bf16_entry_matches_exact_widening():
    """bf16 inputs quantise exactly like their exact fp32 widening (every bf16
    value is an fp32 value); the widening is torch's own conversion."""
    g = torch.Generator().manual_seed(5)
    xb = (torch.randn(40, 512, generator=g) * 3).to(torch.bfloat16)
    xb[3].zero_()
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    q1, s1 = oracle.quantize_rows(bits)
    q2, s2 = oracle.quantize_rows(xb.float().numpy())
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)
    assert s1[3] == 1.0 and not q1[3].any()


def test_quant_rejects_non_finite():
    x = np.ones((2, 8), dtype=np.float32)
    x[1, 3] = np.inf
    with pytest.raises(ValueError):
        oracle.quantize_rows(x)


# --------------------------------------------------------------------------
# INT32 GEMM
# --------------------------------------------------------------------------

def test_gemm_k1_all_code_pairs_brute_force():
    """K = 1: acc[m, n] is the product of the two codes, for all 255^2 pairs."""
    codes = np.arange(-127, 128, dtype=np.int8)[:, None]
    acc = oracle.gemm_s32(codes, codes)
    assert np.array_equal(acc.astype(np.int64), np.outer(np.arange(-127, 128), np.arange(-127, 128)))


def test_gemm_hand_expanded():
    """Xq = [[1,2,3],[4,5,6]], Wq rows = [1,0,-1], [2,1,0], [0,0,1], [-1,-1,-1]:
    row 0: 1-3 = -2, 2+2 = 4, 3, -6;  row 1: 4-6 = -2, 8+5 = 13, 6, -15."""
    X = np.array([[1, 2, 3], [4, 5, 6]], dtype=np.int8)
    W = np.array([[1, 0, -1], [2, 1, 0], [0, 0, 1], [-1, -1, -1]], dtype=np.int8)
    assert oracle.gemm_s32(X, W).tolist() == [[-2, 4, 3, -6], [-2, 13, 6, -15]]
    assert oracle.gemm_s32_f64(X, W).tolist() == [[-2, 4, 3, -6], [-2, 13, 6, -15]]


def test_gemm_identity_and_permutation():
    """Wq = I gives acc = Xq; a permuted identity permutes the columns
    (pins which operand is transposed and which index runs over N)."""
    Xq = torch.randint(-127, 128, (7, 24), generator=torch.Generator().manual_seed(1)).to(torch.int8).numpy()
    eye = np.eye(24, dtype=np.int8)
    assert np.array_equal(oracle.gemm_s32(Xq, eye), Xq.astype(np.int32))
    perm = np.random.default_rng(2).permutation(24)
    assert np.array_equal(oracle.gemm_s32(Xq, eye[perm]), Xq[:, perm].astype(np.int32))


def test_gemm_all_127_row_closed_form():
    """A row of all 127 gives acc[n] = 127 * sum_k Wq[n, k]."""
    Wq = torch.randint(-127, 128, (33, 1000), generator=torch.Generator().manual_seed(4)).to(torch.int8).numpy()
    X = np.full((1, 1000), 127, dtype=np.int8)
    assert np.array_equal(oracle.gemm_s32(X, Wq)[0].astype(np.int64), 127 * Wq.astype(np.int64).sum(axis=1))


def test_gemm_matches_numpy_int64_matmul():
    """Against numpy's own int64 matrix product on a non-square shape."""
    g = torch.Generator().manual_seed(9)
    Xq = torch.randint(-127, 128, (37, 203), generator=g).to(torch.int8).numpy()
    Wq = torch.randint(-127, 128, (19, 203), generator=g).to(torch.int8).numpy()
    ref = Xq.astype(np.int64) @ Wq.astype(np.int64).T
    assert np.array_equal(oracle.gemm_s32(Xq, Wq).astype(np.int64), ref)
    assert np.array_equal(oracle.gemm_s32_f64(Xq, Wq).astype(np.int64), ref)
    rows = np.array([36, 0, 17, 17])
    assert np.array_equal(oracle.gemm_s32(Xq, Wq, rows).astype(np.int64), ref[rows])


def test_gemm_int32_limit():
    """|acc| <= K * 127^2 fits INT32 up to K = floor((2^31 - 1) / 16129) = 133144;
    one more element of 127 * 127 overflows and the oracle reports it."""
    kmax = (2 ** 31 - 1) // 16129
    assert kmax == 133144
    x = np.full((1, kmax), 127, dtype=np.int8)
    assert oracle.gemm_s32(x, x)[0, 0] == kmax * 16129
    xn = np.full((1, kmax), -127, dtype=np.int8)
    assert oracle.gemm_s32(x, xn)[0, 0] == -kmax * 16129
    x1 = np.full((1, kmax + 1), 127, dtype=np.int8)
    with pytest.raises(OverflowError):
        oracle.gemm_s32(x1, x1)


def test_gemm_f64_path_equals_scalar_path_large_sums():
    """Adversarial codes near +-127 with K = 4096: sums near 6.6e7, well past
    2^24, still identical on both routes (both must be exact)."""
    g = torch.Generator().manual_seed(12)
    Xq = torch.randint(100, 128, (16, 4096), generator=g).to(torch.int8).numpy()
    Wq = torch.randint(100, 128, (24, 4096), generator=g).to(torch.int8).numpy()
    Wq[::2] *= -1
    a = oracle.gemm_s32(Xq, Wq)
    b = oracle.gemm_s32_f64(Xq, Wq)
    assert np.array_equal(a, b)
    assert np.abs(a.astype(np.int64)).min() > 2 ** 24


# --------------------------------------------------------------------------
# Epilogue and bf16 rounding
# --------------------------------------------------------------------------

def test_bf16_rne_matches_torch_conversion():
    """Against torch's float32 -> bfloat16 conversion (round to nearest even):
    random values over the whole exponent range, exact ties, subnormals,
    values that round up into the next binade, and infinities."""
    rng = np.random.default_rng(21)
    bits = rng.integers(0, 2 ** 32, size=200000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    ties = (np.arange(-300, 300, dtype=np.int64).astype(np.uint32) << 16 | 0x8000).view(np.float32)
    special = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, 3.3895314e38, 1e-40, -1e-45,
                        1.00390625, 1.01171875, 255.5, 65504.0], dtype=np.float32)
    allx = np.concatenate([x, ties[np.isfinite(ties)], special]).astype(np.float32)
    ours = oracle.bf16_rne(allx)
    ref = torch.from_numpy(allx).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_epilogue_zero_acc_gives_bias():
    """A zero accumulator (zero row or zero weight channel) outputs the bias
    itself: 0 * sx * sw + b = b exactly."""
    b = np.array([0.5, -1.25, 3.0e-3, 7.0], dtype=np.float32)
    acc = np.zeros((3, 4), dtype=np.int32)
    y32, y = oracle.epilogue(acc, np.array([1.0, 0.25, 3.0], np.float32), np.array([0.1, 2.0, 1e-3, 9.0], np.float32), b)
    assert np.array_equal(y32, np.broadcast_to(b, (3, 4)))
    assert np.array_equal(y, np.broadcast_to(oracle.bf16_rne(b), (3, 4)))


def test_epilogue_exact_powers_of_two():
    """acc = 1000, sx = 2^-10, sw = 2^-3, bias = 0.25: every step is exact,
    y32 = 1000 / 8192 + 0.25 = 0.3720703125; bf16 keeps 8 significant bits,
    spacing 2^-7 on [1, 2): 0.3720703125 = 1.48828125 * 2^-2 and
    1.48828125 = 190.5 * 2^-7, an exact tie, so it rounds to the even 190:
    1.484375 * 2^-2 = 0.37109375."""
    y32, y = oracle.epilogue(np.array([[1000]], np.int32), np.array([2.0 ** -10], np.float32),
                             np.array([2.0 ** -3], np.float32), np.array([0.25], np.float32))
    assert y32[0, 0] == np.float32(0.3720703125)
    assert oracle.bf16_bits_to_f32(y)[0, 0] == np.float32(0.37109375)


def test_epilogue_no_bias():
    y32, _ = oracle.epilogue(np.array([[-3, 5]], np.int32), np.array([0.5], np.float32),
                             np.array([2.0, 0.25], np.float32), None)
    assert y32.tolist() == [[-3.0, 0.625]]


def test_epilogue_indices_against_float64():
    """Row scales follow rows and channel scales follow columns: compare with
    an fp64 evaluation on a non-square case with distinct scales (each fp32
    step adds at most half an ulp, so three steps stay within 2 ulp)."""
    rng = np.random.default_rng(31)
    acc = rng.integers(-2 ** 20, 2 ** 20, size=(13, 29)).astype(np.int32)
    sx = rng.uniform(1e-3, 1.0, 13).astype(np.float32)
    sw = rng.uniform(1e-4, 1e-2, 29).astype(np.float32)
    b = rng.uniform(-1, 1, 29).astype(np.float32)
    y32, y = oracle.epilogue(acc, sx, sw, b)
    ref = acc.astype(np.float64) * sx[:, None].astype(np.float64) * sw[None, :].astype(np.float64) + b.astype(np.float64)
    scale = np.abs(acc.astype(np.float64) * sx[:, None] * sw[None, :]) + np.abs(b)
    assert (np.abs(y32 - ref) <= scale * 2.0 ** -22).all()
    yf = oracle.bf16_bits_to_f32(y).astype(np.float64)
    assert (np.abs(yf - y32) <= oracle.ulp_bf16(y32) / 2).all()


def test_epilogue_rounding_order():
    """The dequantisation takes its fp32 roundings in the stated order:
    (float)acc * sx, then * sw, then + bias, each rounded once (zhidx
    TurboT2VA article, section 01 item 3: scale and bias once after the full
    INT32 sum; the order is this build's reading of it).  The expected values
    are computed here in exact binary64 arithmetic: every product of an
    integer below 2^21 or an fp32 value with an fp32 value, and every sum of
    two fp32 values of these sizes, is exact in binary64, so converting each
    step to float32 rounds it once, to nearest even.  About a third of these
    random triples give a different fp32 result when sx * sw is formed first,
    so the test tells the orders apart."""
    rng = np.random.default_rng(77)
    acc = rng.integers(-2 ** 20, 2 ** 20, size=(16, 24)).astype(np.int32)
    sx = rng.uniform(1e-3, 1.0, 16).astype(np.float32)
    sw = rng.uniform(1e-4, 1e-2, 24).astype(np.float32)
    b = rng.uniform(-1, 1, 24).astype(np.float32)
    y32, _ = oracle.epilogue(acc, sx, sw, b)
    a64 = acc.astype(np.float64)
    step1 = (a64 * sx[:, None].astype(np.float64)).astype(np.float32)
    step2 = (step1.astype(np.float64) * sw[None, :].astype(np.float64)).astype(np.float32)
    expect = (step2.astype(np.float64) + b[None, :].astype(np.float64)).astype(np.float32)
    assert np.array_equal(y32, expect)
    s2 = (sx[:, None].astype(np.float64) * sw[None, :].astype(np.float64)).astype(np.float32)
    other = ((a64 * s2.astype(np.float64)).astype(np.float32).astype(np.float64)
             + b[None, :].astype(np.float64)).astype(np.float32)
    assert (other != expect).mean() > 0.1


# --------------------------------------------------------------------------
# Whole path
# --------------------------------------------------------------------------

def test_linear_zero_row_outputs_bias():
    rng = np.random.default_rng(41)
    X = rng.standard_normal((5, 64)).astype(np.float32)
    X[2] = 0
    Wq, sw = oracle.quantize_rows((rng.standard_normal((8, 64)) * 0.02).astype(np.float32))
    b = (rng.standard_normal(8) * 0.01).astype(np.float32)
    out = oracle.linear(X, Wq, sw, b)
    assert not out["acc"][2].any()
    assert np.array_equal(out["y32"][2], b)


def test_linear_approximates_float_product():
    """The W8A8 result approximates X W^T + b: the dequantisation error of each
    code is at most half its scale, so |Y - X W^T - b| is bounded by
    sum_k (|x| sw/2 + |w| sx/2 + sx sw/4) plus the bf16 rounding.  A dropped
    term, a wrong sign or a transposed operand breaks this bound."""
    g = torch.Generator().manual_seed(51)
    X = torch.randn(48, 256, generator=g).numpy()
    W = (torch.randn(40, 256, generator=g) * 0.02).numpy()
    b = (torch.randn(40, generator=g) * 0.01).numpy()
    Wq, sw = oracle.quantize_rows(W)
    out = oracle.linear(X, Wq, sw, b)
    sx = out["sx"].astype(np.float64)
    ref = X.astype(np.float64) @ W.astype(np.float64).T + b
    bound = (np.abs(X) @ np.ones((256, 40))) * sw[None, :] / 2 \
        + (np.ones((48, 256)) @ np.abs(W).T) * sx[:, None] / 2 \
        + 256 * sx[:, None] * sw[None, :] / 4
    yf = oracle.bf16_bits_to_f32(out["y"]).astype(np.float64)
    assert (np.abs(yf - ref) <= bound + oracle.ulp_bf16(ref) + 1e-6).all()
    assert np.corrcoef(yf.ravel(), ref.ravel())[0, 1] > 0.999


def test_linear_bf16_workload_recipe_small():
    """The workload generator's bf16 recipe (outlier columns) runs through the
    oracle with the f64 and scalar accumulator routes agreeing."""
    import w8a8_workloads as wl
    X, W, b = wl.make("video", M=32, N=48, K=512)
    xb = X.view(torch.int16).numpy().view(np.uint16)
    wb = W.view(torch.int16).numpy().view(np.uint16)
    Wq, sw = oracle.quantize_rows(wb)
    bf = oracle.bf16_bits_to_f32(b.view(torch.int16).numpy().view(np.uint16))
    o1 = oracle.linear(xb, Wq, sw, bf)
    o2 = oracle.linear(xb, Wq, sw, bf, exact_f64=True)
    assert np.array_equal(o1["acc"], o2["acc"]) and np.array_equal(o1["y"], o2["y"])
    # outlier columns: most activation codes are small, the outliers reach 127
    assert np.abs(o1["xq"]).max(axis=1).min() == 127
    assert np.median(np.abs(o1["xq"])) <= 8


def test_ulp_bf16():
    assert oracle.ulp_bf16(np.array([1.0]))[0] == 2.0 ** -7
    assert oracle.ulp_bf16(np.array([1.99]))[0] == 2.0 ** -7
    assert oracle.ulp_bf16(np.array([-2.0]))[0] == 2.0 ** -6
    assert oracle.ulp_bf16(np.array([0.3]))[0] == 2.0 ** -9
    assert math.isclose(oracle.ulp_bf16(np.array([1e-39]))[0], 2.0 ** -133)


# ---------------------------------------------------------------- native BF16 linear reference

def _bf16(a):
    """float values -> bf16 bit patterns by truncation of exactly representable values."""
    return (np.asarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_bf16_linear_brute_force():
    """Pure-Python triple loop on a small case (values exact in bf16)."""
    rng = np.random.default_rng(3)
    Xv = rng.integers(-8, 9, size=(3, 5)).astype(np.float32) / 4
    Wv = rng.integers(-8, 9, size=(4, 5)).astype(np.float32) / 8
    b = np.array([0.5, -1.0, 0.25, 0.0], dtype=np.float32)
    y, absum = oracle.bf16_linear_f64(_bf16(Xv), _bf16(Wv), b)
    for m in range(3):
        for n in range(4):
            want = sum(float(Xv[m, k]) * float(Wv[n, k]) for k in range(5)) + float(b[n])
            wabs = sum(abs(float(Xv[m, k]) * float(Wv[n, k])) for k in range(5)) + abs(float(b[n]))
            assert y[m, n] == want and absum[m, n] == wabs


def test_bf16_linear_identity_and_roles():
    """W = identity gives X (+ bias); a permuted identity permutes columns:
    pins the operand roles (Y = X W^T, not W X^T)."""
    rng = np.random.default_rng(4)
    Xv = rng.standard_normal((6, 8)).astype(np.float32)
    xb = _bf16(Xv)
    x = oracle.bf16_bits_to_f32(xb).astype(np.float64)
    eye = _bf16(np.eye(8, dtype=np.float32))
    y, _ = oracle.bf16_linear_f64(xb, eye)
    assert np.array_equal(y, x)
    perm = rng.permutation(8)
    y, _ = oracle.bf16_linear_f64(xb, eye[perm])
    assert np.array_equal(y, x[:, perm])
    y, _ = oracle.bf16_linear_f64(xb, eye, np.full(8, 2.0, dtype=np.float32))
    assert np.array_equal(y, x + 2.0)


def test_bf16_linear_closed_form_and_tolerance():
    """All-ones rows against all-0.5 weights sum to K / 2 exactly; the bound
    is at least one bf16 ulp and grows with K * sum|x w|."""
    K = 4096
    y, absum = oracle.bf16_linear_f64(_bf16(np.ones((2, K))), _bf16(np.full((3, K), 0.5)))
    assert (y == K / 2).all() and (absum == K / 2).all()
    tol = oracle.bf16_linear_tolerance(y, absum, K)
    assert (tol >= oracle.ulp_bf16(y)).all()
    assert np.allclose(tol, oracle.ulp_bf16(y) + 2 * (K + 1) * 2.0 ** -24 * absum)



# ---------------------------------------------------------------- per-block Query/Key quantisation

def _py_block_quant(vals):
    """Pure-Python restatement on one block: fp32 absmax / 127, then each
    code round-half-even of the fp32 quotient, clamped."""
    f32 = np.float32
    amax = max(abs(float(v)) for v in vals)
    s = f32(f32(amax) / f32(127.0))
    if s == 0:
        return [0] * len(vals), f32(1.0)
    codes = [max(-127, min(127, round(float(f32(f32(v) / s))))) for v in vals]
    return codes, s


def test_qk_blocks_brute_force():
    rng = np.random.default_rng(21)
    X = rng.standard_normal((2, 3, 5, 4)).astype(np.float32)
    X[1, 2, 2:4] = 0.0                                  # one all-zero block
    q, s = oracle.quantize_qk_blocks(X, 2, "HND")
    assert q.shape == X.shape and s.shape == (2, 3, 3)
    for b in range(2):
        for h in range(3):
            for j, (t0, t1) in enumerate([(0, 2), (2, 4), (4, 5)]):
                codes, sc = _py_block_quant(X[b, h, t0:t1].ravel())
                assert s[b, h, j] == sc
                assert list(q[b, h, t0:t1].ravel()) == codes
    assert s[1, 2, 1] == 1.0 and not q[1, 2, 2:4].any()


def test_qk_blocks_layouts_agree():
    """NHD input is the HND tensor with heads and tokens swapped: the codes
    swap the same way and the scales are identical."""
    rng = np.random.default_rng(22)
    X = rng.standard_normal((2, 4, 37, 16)).astype(np.float32)
    qh, sh = oracle.quantize_qk_blocks(X, 8, "HND")
    qn, sn = oracle.quantize_qk_blocks(np.ascontiguousarray(X.transpose(0, 2, 1, 3)), 8, "NHD")
    assert np.array_equal(sh, sn)
    assert np.array_equal(qn, qh.transpose(0, 2, 1, 3))


def test_qk_blocks_special_block_sizes():
    """One token per block is per-token quantisation; one block per head is
    the head flattened to one row."""
    rng = np.random.default_rng(23)
    X = (rng.standard_normal((1, 3, 10, 8)) * 3).astype(np.float32)
    q1, s1 = oracle.quantize_qk_blocks(X, 1)
    qr, sr = oracle.quantize_rows(X.reshape(30, 8))
    assert np.array_equal(q1.reshape(30, 8), qr) and np.array_equal(s1.reshape(30), sr)
    qa, sa = oracle.quantize_qk_blocks(X, 1000)
    qr, sr = oracle.quantize_rows(X.reshape(3, 80))
    assert np.array_equal(qa.reshape(3, 80), qr) and np.array_equal(sa.reshape(3), sr)


def test_qk_blocks_are_independent_and_saturate():
    """Scaling one block by 2^3 scales only its scale (codes unchanged), and
    every nonzero block reaches |q| = 127."""
    rng = np.random.default_rng(24)
    X = rng.standard_normal((1, 2, 12, 8)).astype(np.float32)
    q, s = oracle.quantize_qk_blocks(X, 4)
    Y = X.copy()
    Y[0, 1, 4:8] *= 8.0
    q2, s2 = oracle.quantize_qk_blocks(Y, 4)
    assert np.array_equal(q2, q)
    assert s2[0, 1, 1] == 8 * s[0, 1, 1]
    s2[0, 1, 1] = s[0, 1, 1]
    assert np.array_equal(s2, s)
    for h in range(2):
        for j in range(3):
            assert np.abs(q[0, h, 4 * j:4 * j + 4].astype(np.int32)).max() == 127


# ---------------------------------------------------------------- normalisation + modulation

def _bits(a):
    return oracle.bf16_rne(np.asarray(a, dtype=np.float32))


def test_norm_brute_force():
    """Pure-Python restatement of both norms with modulation on small rows."""
    import math
    rng = np.random.default_rng(31)
    xb = _bits(rng.standard_normal((3, 16)) * 2)
    x = oracle.bf16_bits_to_f32(xb).astype(np.float64)
    sc = rng.standard_normal(16) * 0.1
    sh = rng.standard_normal(16) * 0.1
    for kind in ("rms", "layer"):
        y, mu, r = oracle.norm_modulate_f64(xb, kind, 1e-6, sc, sh)
        for m in range(3):
            row = [float(v) for v in x[m]]
            mean = math.fsum(row) / 16 if kind == "layer" else 0.0
            var = math.fsum((v - mean) ** 2 for v in row) / 16
            rr = 1.0 / math.sqrt(var + 1e-6)
            for k in range(16):
                want = (row[k] - mean) * rr * (1.0 + sc[k]) + sh[k]
                assert abs(y[m, k] - want) <= 1e-12 * max(1.0, abs(want))
            assert abs(mu[m] - mean) <= 1e-12 and abs(r[m] - rr) <= 1e-12 * rr


def test_norm_closed_forms():
    """A constant row c under RMS norm gives c / sqrt(c^2 + eps); a row of two
    values a, b (half each) under LayerNorm gives +-1 / sqrt(1 + eps / d^2)
    with d = (a - b) / 2."""
    c, eps = 1.5, 1e-3
    y, _, _ = oracle.norm_modulate_f64(_bits(np.full((1, 32), c)), "rms", eps)
    assert np.allclose(y, c / np.sqrt(c * c + eps), rtol=1e-14, atol=0)
    a, b = 3.0, -1.0
    row = np.array([a, b] * 16)
    y, mu, _ = oracle.norm_modulate_f64(_bits(row[None, :]), "layer", eps)
    d = (a - b) / 2
    assert mu[0] == (a + b) / 2
    assert np.allclose(y[0], np.where(row == a, 1.0, -1.0) / np.sqrt(1.0 + eps / (d * d)), rtol=1e-14, atol=0)


def test_norm_invariances_and_modulation():
    """LayerNorm ignores a constant offset; RMS norm ignores a power-of-two
    gain (eps = 0); scale = -1 leaves exactly the shift; RMS output has unit
    mean square (eps = 0)."""
    rng = np.random.default_rng(32)
    xb = _bits(rng.integers(-64, 64, size=(4, 64)) / 16.0)
    x = oracle.bf16_bits_to_f32(xb).astype(np.float64)
    y1, _, _ = oracle.norm_modulate_f64(xb, "layer", 0.0)
    y2, _, _ = oracle.norm_modulate_f64(_bits(x + 8.0), "layer", 0.0)
    assert np.allclose(y1, y2, rtol=0, atol=1e-12)
    y3, _, _ = oracle.norm_modulate_f64(xb, "rms", 0.0)
    y4, _, _ = oracle.norm_modulate_f64(_bits(x * 4.0), "rms", 0.0)
    assert np.array_equal(y3, y4)
    assert np.allclose((y3 * y3).mean(axis=1), 1.0, rtol=1e-13)
    sh = rng.standard_normal(64)
    y5, _, _ = oracle.norm_modulate_f64(xb, "rms", 1e-6, np.full(64, -1.0), sh)
    assert np.array_equal(y5, np.broadcast_to(sh, y5.shape))


def test_norm_quantize_composes_the_pinned_parts():
    """norm_quantize is bf16_rne of the float64 rows followed by the pinned
    row quantiser."""
    rng = np.random.default_rng(33)
    xb = _bits(rng.standard_normal((5, 48)))
    yb, q, s, y = oracle.norm_quantize(xb, "layer", 1e-5, rng.standard_normal(48) * 0.1, None)
    assert np.array_equal(yb, oracle.bf16_rne(y.astype(np.float32)))
    q2, s2 = oracle.quantize_rows(yb)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)


def test_bf16_rne_array_matches_scalar():
    rng = np.random.default_rng(34)
    v = np.concatenate([rng.standard_normal(5000).astype(np.float32),
                        np.array([0.0, -0.0, 1.00390625, 1.01171875, np.inf, -np.inf, 3.4e38], dtype=np.float32)])
    lib = oracle._load()
    assert np.array_equal(oracle.bf16_rne(v), np.array([lib.oracle_bf16_rne(float(t)) for t in v], dtype=np.uint16))


# ---------------------------------------------------------------- stored fixture

def test_oracle_reproduces_the_golden_fixture():
    """tests/golden/linear_small.json was written by the oracle
    (make_golden.py); the oracle must still produce it bit for bit."""
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "linear_small.json")
    g = json.load(open(path))
    xb = np.array(g["X_bf16_bits"], dtype=np.uint16)
    wb = np.array(g["W_bf16_bits"], dtype=np.uint16)
    bb = np.array(g["bias_bf16_bits"], dtype=np.uint16)
    wq, sw = oracle.quantize_rows(wb)
    xq, sx = oracle.quantize_rows(xb)
    assert np.array_equal(xq, np.array(g["Xq"])) and np.array_equal(wq, np.array(g["Wq"]))
    assert np.array_equal(sx.view(np.uint32), np.array(g["sx_f32_bits"], dtype=np.uint32))
    assert np.array_equal(sw.view(np.uint32), np.array(g["sw_f32_bits"], dtype=np.uint32))
    assert np.array_equal(oracle.gemm_s32(xq, wq, np.arange(xq.shape[0])), np.array(g["acc"]))
    ref = oracle.linear(xb, wq, sw, oracle.bf16_bits_to_f32(bb))
    assert np.array_equal(ref["y"], np.array(g["Y_bf16_bits"], dtype=np.uint16))
