"""GPU parity of the MLP pair Y = down(up(X)) on the W8A8 path, the down
layer's row quantisation fed by the up GEMM's gathered row maxima (each layer:
zhidx TurboT2VA article, section 01 item 3).  Bar: H and Y bit-identical to
two separate w8a8_linear calls, and within one bf16 ulp of the oracle chain
(oracle linear, then oracle row quantisation of its bf16 output, then oracle
linear)."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_linear_act_b300 as w8
import w8a8_workloads as wl
from helpers import bias_f32, bits

pytestmark = pytest.mark.gpu


def weights(F, K, N, seed, dev, bias=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    Wu = (torch.randn(F, K, generator=g) * 0.02).to(torch.bfloat16)
    Wd = (torch.randn(N, F, generator=g) * 0.02).to(torch.bfloat16)
    bu = (torch.randn(F, generator=g) * 0.01).to(bias) if bias is not None else None
    bd = (torch.randn(N, generator=g) * 0.01).to(bias) if bias is not None else None
    Wqu, swu = w8.quantize_weight(Wu.to(dev))
    Wqd, swd = w8.quantize_weight(Wd.to(dev))
    return dict(Wu=Wu, Wd=Wd, bu=bu, bd=bd, Wqu=Wqu, swu=swu, Wqd=Wqd, swd=swd,
                Wpu=w8.pack_weight(Wqu), Wpd=w8.pack_weight(Wqd))


def dev_or_none(t, dev):
    return None if t is None else t.to(dev)


def run_pair(X, w, dev, workspace=None):
    Y, H = w8.mlp(X.to(dev), w["Wpu"], w["swu"], dev_or_none(w["bu"], dev), w["Wpd"], w["swd"],
                  dev_or_none(w["bd"], dev), workspace=workspace)
    Hs = w8.linear(X.to(dev), w["Wpu"], w["swu"], dev_or_none(w["bu"], dev))
    Ys = w8.linear(Hs, w["Wpd"], w["swd"], dev_or_none(w["bd"], dev))
    torch.cuda.synchronize()
    return Y.cpu(), H.cpu(), Ys.cpu(), Hs.cpu()


def oracle_chain(X, w, rows):
    wqu, swu = w["Wqu"].cpu().numpy(), w["swu"].cpu().numpy()
    wqd, swd = w["Wqd"].cpu().numpy(), w["swd"].cpu().numpy()
    h = oracle.linear(bits(X), wqu, swu, bias_f32(w["bu"]), rows=rows, exact_f64=True)
    y = oracle.linear(h["y"], wqd, swd, bias_f32(w["bd"]), exact_f64=True)
    return h, y


def check(X, w, dev, rows=None, workspace=None):
    Y, H, Ys, Hs = run_pair(X, w, dev, workspace)
    assert torch.equal(H.view(torch.int16), Hs.view(torch.int16)), "H differs from the separate up layer"
    assert torch.equal(Y.view(torch.int16), Ys.view(torch.int16)), "Y differs from the separate layers"
    if rows is None:
        rows = np.arange(X.shape[0])
    h, y = oracle_chain(X, w, rows)
    assert np.array_equal(bits(H)[rows], h["y"]), "H differs from the oracle"
    yg = oracle.bf16_bits_to_f32(bits(Y)[rows]).astype(np.float64)
    assert (np.abs(yg - y["y32"]) <= oracle.ulp_bf16(y["y32"])).all(), "Y beyond one bf16 ulp of the oracle"


@pytest.mark.parametrize("M,K,F,N", [
    (1, 256, 512, 128),      # one row
    (64, 256, 512, 128),
    (300, 256, 528, 264),    # ragged M, F and N tiles
    (129, 512, 1040, 136),   # one row past a 128-row tile: the single-CTA form for neither layer
    (1001, 2048, 8192, 2048),
])
def test_mlp_pair_shapes(cuda_device, M, K, F, N):
    X = torch.randn(M, K, generator=torch.Generator().manual_seed(M)).to(torch.bfloat16)
    check(X, weights(F, K, N, seed=F, dev=cuda_device), cuda_device)


def test_mlp_pair_mlp_workload_every_row(cuda_device):
    """The MLP workload's sizes (6144 x 4096 -> 16384 -> 4096, 1 % outlier
    columns), every row: H and Y bit-identical to the separate layers, H
    bit-identical to the oracle's up layer, Y within one bf16 ulp of the
    oracle chain (checked in blocks of rows; the chain is row-independent)."""
    X, _, _ = wl.make("mlp_up")
    w = weights(16384, 4096, 4096, seed=2, dev=cuda_device)
    Y, H, Ys, Hs = run_pair(X, w, cuda_device)
    assert torch.equal(H.view(torch.int16), Hs.view(torch.int16)), "H differs from the separate up layer"
    assert torch.equal(Y.view(torch.int16), Ys.view(torch.int16)), "Y differs from the separate layers"
    wqu, swu = w["Wqu"].cpu().numpy(), w["swu"].cpu().numpy()
    wqd, swd = w["Wqd"].cpu().numpy(), w["swd"].cpu().numpy()
    xq, sx = oracle.quantize_rows(bits(X))
    hb, yb = bits(H), bits(Y)
    for r0 in range(0, 6144, 1024):
        r1 = r0 + 1024
        acc = oracle.gemm_s32_f64(xq[r0:r1], wqu)
        _, h = oracle.epilogue(acc, sx[r0:r1], swu, bias_f32(w["bu"]))
        assert np.array_equal(hb[r0:r1], h), "H differs from the oracle in rows %d.." % r0
        y = oracle.linear(h, wqd, swd, bias_f32(w["bd"]), exact_f64=True)
        yg = oracle.bf16_bits_to_f32(yb[r0:r1]).astype(np.float64)
        assert (np.abs(yg - y["y32"]) <= oracle.ulp_bf16(y["y32"])).all(), "Y beyond one ulp in rows %d.." % r0


def test_mlp_pair_zero_rows_and_no_bias(cuda_device):
    """A zero row of X without biases makes a zero row of H (scale 1, codes
    0) and a zero row of Y; fp32 X and fp32 biases take the same path."""
    X = torch.randn(200, 256, generator=torch.Generator().manual_seed(9))
    X[7] = 0.0
    X[199] = 0.0
    w = weights(512, 256, 264, seed=10, dev=cuda_device, bias=None)
    check(X, w, cuda_device)
    Y, H, _, _ = run_pair(X, w, cuda_device)
    assert not H[7].float().any() and not Y[199].float().any()
    wf = weights(512, 256, 264, seed=11, dev=cuda_device, bias=torch.float32)
    check(X, wf, cuda_device)


def test_mlp_pair_minimum_workspace_and_repeats(cuda_device):
    """With no room for split-tile slots the result is the same; repeated
    calls on one workspace give identical results (the row maxima are
    cleared by every call)."""
    M, K, F, N = 300, 3072, 3072, 512
    X = torch.randn(M, K, generator=torch.Generator().manual_seed(12)).to(torch.bfloat16)
    w = weights(F, K, N, seed=13, dev=cuda_device)
    full = w8.mlp_workspace_bytes(M, K, F, N)
    ws = torch.empty(full, dtype=torch.uint8, device=cuda_device)
    Y1, H1 = w8.mlp(X.to(cuda_device), w["Wpu"], w["swu"], w["bu"].to(cuda_device), w["Wpd"], w["swd"],
                    w["bd"].to(cuda_device), workspace=ws)
    Y1 = Y1.clone()
    for _ in range(3):
        Y2, _ = w8.mlp(X.to(cuda_device), w["Wpu"], w["swu"], w["bu"].to(cuda_device), w["Wpd"], w["swd"],
                       w["bd"].to(cuda_device), workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    up, dn = w8.gemm_plan(M, F, K), w8.gemm_plan(M, N, F)
    slots = max(up[2] * up[4], dn[2] * dn[4])
    assert slots > 0, "this shape is expected to cut tiles along K"
    small = torch.empty(full - slots * 128 * 256 * 4, dtype=torch.uint8, device=cuda_device)
    check(X, w, cuda_device, workspace=small)
    st, bits_ = w8.read_status(ws)
    assert st == 0 and bits_ == 0
