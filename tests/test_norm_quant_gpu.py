"""GPU parity of the norm + modulation prologue fused into the activation
quantisation (zhidx TurboT2VA article, section 01: normalisation and
modulation fused; arXiv paper, appendix C).

The kernel sums in fp32 in its own order, so its y can differ from the
oracle's bf16_rne(y64) where y64 lies within the kernel's error bound of a
bf16 rounding boundary.  The bound B per element follows from the fp32
steps: every thread adds at most 128 values in sequence and the reductions
add at most 16 more levels, so the sum of squares is within 146 u
(u = 2^-24) relative of exact, the variance within 150 u after the division
and the epsilon, 1/sqrt within 76 u, the mean within 146 u sum|x| / K + u
|mu|; each later step adds one rounding.  B is twice the sum of those
terms.  Outside the band y, the codes and the row scales are bit-exact;
inside it y may be any bf16 value between the rounded ends of the band and a
code may move by one."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_linear_act_b300 as w8
import w8a8_workloads as wl
from helpers import bits

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def bands(xb, kind, eps, scale, shift):
    y, mu, r = oracle.norm_modulate_f64(xb, kind, eps, scale, shift)
    x = oracle.bf16_bits_to_f32(xb).astype(np.float64)
    K = x.shape[1]
    d = np.abs(x - mu[:, None])
    dr = 76 * U + 2 * U
    dmu = (146 * U * np.abs(x).sum(axis=1) / K + U * np.abs(mu)) if kind == "layer" else np.zeros_like(mu)
    a = np.abs(1.0 + np.asarray(scale, dtype=np.float64)) if scale is not None else np.ones(K)
    z = d * r[:, None]
    B = a[None, :] * (d * r[:, None] * (dr + 2 * U) + dmu[:, None] * r[:, None]) + 2 * U * z * a[None, :] \
        + U * np.abs(y)
    return y, 2.0 * B


def candidates(y, B):
    lo = oracle.bf16_rne((y - B).astype(np.float32))
    hi = oracle.bf16_rne((y + B).astype(np.float32))
    return lo, hi


def check(X, kind, eps, scale, shift, dev, rows=None, max_band=0.05):
    sc = None if scale is None else scale.to(dev)
    sh = None if shift is None else shift.to(dev)
    Xq, sx, Yg = w8.norm_quantize_act(X.to(dev), kind, eps, sc, sh, want_y=True)
    torch.cuda.synchronize()
    xb = bits(X)
    rows = np.arange(X.shape[0]) if rows is None else rows
    scn = None if scale is None else oracle.bf16_bits_to_f32(bits(scale)) if scale.dtype == torch.bfloat16 \
        else scale.numpy()
    shn = None if shift is None else oracle.bf16_bits_to_f32(bits(shift)) if shift.dtype == torch.bfloat16 \
        else shift.numpy()
    yb, q, s, y64 = oracle.norm_quantize(xb[rows], kind, eps, scn, shn)
    _, B = bands(xb[rows], kind, eps, scn, shn)
    lo, hi = candidates(y64, B)
    amb = lo != hi
    # About 0.5 % of elements fall in the band under RMS norm; LayerNorm's
    # worst-case bound on the mean widens it for small |y| (about 3 %).
    assert amb.mean() < max_band, "band too wide to be a useful check: %.4f" % amb.mean()
    yg = bits(Yg)[rows]
    assert np.array_equal(yg[~amb], yb[~amb]), "y differs outside the band"
    # Inside the band y may be any bf16 value between the rounded ends (near
    # zero the band spans several bf16 steps).
    v = oracle.bf16_bits_to_f32
    assert np.all((v(yg[amb]) >= v(lo[amb])) & (v(yg[amb]) <= v(hi[amb]))), "y outside its band"
    qg = Xq.cpu().numpy()[rows].astype(np.int32)
    sg = sx.cpu().numpy()[rows]
    lo_v, hi_v = v(lo).astype(np.float64), v(hi).astype(np.float64)
    mag_lo = np.where((lo_v <= 0) & (hi_v >= 0), 0.0, np.minimum(np.abs(lo_v), np.abs(hi_v)))
    mag_hi = np.maximum(np.abs(lo_v), np.abs(hi_v))
    amax_lo = mag_lo.max(axis=1)
    amax_hi = mag_hi.max(axis=1)
    exact_row = amax_lo == amax_hi
    assert np.array_equal(sg[exact_row].view(np.uint32), s[exact_row].view(np.uint32)), "row scales differ"
    # Elsewhere the scale comes from some max inside the band (a zero max
    # gives the zero-row scale 1).
    in_range = (sg >= np.float32(amax_lo / 127) * (1 - 1e-6)) & (sg <= np.float32(amax_hi / 127) * (1 + 1e-6))
    zero_ok = (amax_lo == 0) & (sg == 1.0)
    assert np.all((in_range | zero_ok)[~exact_row]), "row scale outside the band"
    qo = q.astype(np.int32)
    same = exact_row[:, None] & ~amb
    assert np.array_equal(qg[same], qo[same]), "codes differ outside the band"
    assert np.abs(qg - qo).max() <= 1
    return amb.mean()


def mod_vectors(K, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(K, generator=g) * 0.1).to(dtype), (torch.randn(K, generator=g) * 0.1).to(dtype)


@pytest.mark.parametrize("M,K,kind,mod", [
    (64, 256, "rms", None),
    (300, 4096, "rms", torch.bfloat16),
    (300, 4096, "layer", torch.bfloat16),
    (257, 16384, "layer", torch.float32),   # a CTA per row
    (100, 2048, "layer", None),
    (5, 32768, "rms", torch.float32),       # the largest K
    (33, 1040, "rms", torch.bfloat16),      # ragged vector count per lane
    (3, 16, "layer", torch.float32),        # the smallest K: two vectors per row
    (129, 1024, "rms", torch.bfloat16),     # whole rows of 4 vectors per lane
    (77, 2048, "rms", torch.float32),       # whole rows of 8 vectors per lane
    (3001, 1040, "layer", torch.bfloat16),  # more rows than warps on the GPU, ragged lanes
    (5, 4096, "rms", torch.bfloat16),       # fewer rows than SMs: one CTA per row, one warp busy
    (126, 4096, "layer", None),             # the audio row count: most CTAs take one row
    (2500, 4096, "rms", torch.float32),     # just past one round of the sixteen-warp CTAs
    (2500, 3968, "layer", torch.bfloat16),  # the same with ragged lanes (496 vectors a row)
])
def test_norm_quant_shapes(cuda_device, M, K, kind, mod):
    g = torch.Generator().manual_seed(M + K)
    X = (torch.randn(M, K, generator=g) * 3 + 0.5).to(torch.bfloat16)
    sc, sh = mod_vectors(K, K, mod) if mod is not None else (None, None)
    # a few elements in the band are a large fraction of a tiny tensor
    check(X, kind, 1e-6, sc, sh, cuda_device, max_band=0.05 if M * K >= 4096 else 0.25)


def test_norm_quant_video_rows(cuda_device):
    """The video projection's activation (6144 x 4096, 1 % outlier columns)
    under RMS norm with bf16 modulation, every row."""
    X, _, _ = wl.make("video")
    sc, sh = mod_vectors(4096, 5, torch.bfloat16)
    check(X, "rms", 1e-6, sc, sh, cuda_device)


def test_norm_quant_zero_and_constant_rows(cuda_device):
    """A zero row normalises to 0 (r = 1/sqrt(eps)): scale 1, codes 0 (plus
    the shift's codes); a constant row under LayerNorm is all zero too."""
    X = torch.randn(8, 256, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    X[2] = 0.0
    X[5] = 1.25
    check(X, "rms", 1e-6, None, None, cuda_device)
    # The constant row is ill-conditioned under LayerNorm (r = 1/sqrt(eps)
    # amplifies the bound on the mean), so its whole row is in the band;
    # the exact result for it is checked below.
    check(X, "layer", 1e-5, None, None, cuda_device, max_band=0.2)
    Xq, sx = w8.norm_quantize_act(X.to(cuda_device), "layer", 1e-5)
    assert float(sx[5]) == 1.0 and not Xq[5].any() and float(sx[2]) == 1.0


@pytest.mark.parametrize("e", [-100, -101, -110])
def test_norm_quant_tiny_shift_rows(cuda_device, e):
    """Zero rows under RMS norm become y = shift exactly; with a shift of
    absmax 127 * 2^e their scale lies around 2^-100, where the codes switch
    from the division-free correction step to the tie test with IEEE
    division.  Checked like every other row (bit-exact outside the band)."""
    X = torch.randn(6, 1024, generator=torch.Generator().manual_seed(11)).to(torch.bfloat16)
    X[1:5] = 0.0
    sh = torch.randn(1024, generator=torch.Generator().manual_seed(12), dtype=torch.float64)
    sh = (sh / sh.abs().max() * 127.0 * 2.0 ** e).to(torch.float32)
    check(X, "rms", 1e-6, None, sh, cuda_device)


def test_norm_linear_is_linear_of_the_modulated_rows(cuda_device):
    """w8a8_norm_linear equals w8a8_linear applied to the prologue's own y,
    bit for bit (the GEMM half is the parity-tested linear)."""
    M, K, N = 300, 4096, 520
    X = (torch.randn(M, K, generator=torch.Generator().manual_seed(4)) * 2).to(torch.bfloat16).to(cuda_device)
    W = (torch.randn(N, K, generator=torch.Generator().manual_seed(5)) * 0.02).to(torch.bfloat16).to(cuda_device)
    b = (torch.randn(N, generator=torch.Generator().manual_seed(6)) * 0.01).to(torch.bfloat16).to(cuda_device)
    sc, sh = mod_vectors(K, 7, torch.bfloat16)
    sc, sh = sc.to(cuda_device), sh.to(cuda_device)
    Wq, sw = w8.quantize_weight(W)
    Wp = w8.pack_weight(Wq)
    for kind in ("rms", "layer"):
        Y = w8.norm_linear(X, Wp, sw, b, kind, 1e-6, sc, sh)
        _, _, y = w8.norm_quantize_act(X, kind, 1e-6, sc, sh, want_y=True)
        Y2 = w8.linear(y, Wp, sw, b)
        torch.cuda.synchronize()
        assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))
