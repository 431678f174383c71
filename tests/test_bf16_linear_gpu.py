"""GPU parity of the native BF16 linear (Y = bf16(X W^T + bias), fp32
accumulation on the same tcgen05 GEMM) that guard-rejected branches run
(zhidx TurboT2VA article, section 01 item 3: branches that do not meet the
INT8 operator's requirements fall back to native BF16).

Bar: every output within oracle.bf16_linear_tolerance of the float64 sum:
one bf16 ulp for the final rounding plus 2 (K + 1) 2^-24 sum|x w| for fp32
accumulation in any order.  The order of the fp32 additions is not fixed by
the method, so results are not compared bit for bit with the oracle; they
are with themselves (repeated calls, any split arrival order)."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_linear_act_b300 as w8
import w8a8_workloads as wl
from helpers import bias_f32, bits

pytestmark = pytest.mark.gpu


def make(M, N, K, seed, bias="bf16", scale=1.0):
    g = torch.Generator().manual_seed(seed)
    X = (torch.randn(M, K, generator=g) * scale).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    b = torch.randn(N, generator=g) * 0.01
    b = None if bias is None else b.to(torch.float32 if bias == "f32" else torch.bfloat16)
    return X, W, b


def run(X, W, b, dev, workspace=None):
    Y = w8.bf16_linear(X.to(dev), W.to(dev), None if b is None else b.to(dev), workspace=workspace)
    torch.cuda.synchronize()
    return Y.cpu()


def check(Y, X, W, b, rows=None, what=""):
    K = X.shape[1]
    y64, absum = oracle.bf16_linear_f64(bits(X), bits(W), bias_f32(b), rows=rows)
    yb = bits(Y) if rows is None else bits(Y)[rows]
    yg = oracle.bf16_bits_to_f32(yb).astype(np.float64)
    tol = oracle.bf16_linear_tolerance(y64, absum, K)
    err = np.abs(yg - y64)
    bad = ~(err <= tol)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d outputs beyond the bound, e.g. %s" % (
            what, int(bad.sum()), [(tuple(i), yg[tuple(i)], y64[tuple(i)], tol[tuple(i)]) for i in idx]))
    # Most outputs are the correctly rounded bf16 of the exact sum.
    near = (yb == oracle.bf16_rne(y64.astype(np.float32).ravel()).reshape(y64.shape)).mean()
    assert near > 0.9, "%s: only %.3f correctly rounded" % (what, near)


@pytest.mark.parametrize("M,N,K,bias", [
    (64, 128, 256, "bf16"),
    (1, 8, 16, None),          # smallest accepted shape
    (77, 40, 264, "f32"),      # K = 8 (mod 16): the INT8 guard rejects this K
    (300, 520, 1040, "bf16"),  # ragged M and N tiles, CTA pairs
    (129, 264, 2056, "f32"),   # one row / 8 columns past a tile, K = 8 (mod 64)
    (1000, 2048, 3200, None),
])
def test_bf16_linear_shapes(cuda_device, M, N, K, bias):
    X, W, b = make(M, N, K, seed=M + N, bias=bias)
    check(run(X, W, b, cuda_device), X, W, b, what="%dx%dx%d" % (M, N, K))


def test_bf16_linear_rejected_int8_shape_is_accepted_here(cuda_device):
    """A shape the INT8 guard rejects (K not a multiple of 16) runs here."""
    assert not w8.shape_supported(256, 512, 1032)[0]
    assert w8.bf16_linear_supported(256, 512, 1032)[0]
    X, W, b = make(256, 512, 1032, seed=2)
    check(run(X, W, b, cuda_device), X, W, b)


def test_bf16_linear_video_sampled_rows(cuda_device):
    """The video projection shape (6144 x 4096 x 4096, 1 % outlier columns)
    on CTA pairs with the last wave cut along K; 97 rows checked in full."""
    X, W, b = wl.make("video")
    rows = np.unique(np.concatenate([np.random.default_rng(0).choice(X.shape[0], 96, replace=False),
                                     [X.shape[0] - 1]]))
    check(run(X, W, b, cuda_device), X, W, b, rows=rows, what="video")


def test_bf16_linear_k_beyond_int8_limit(cuda_device):
    """K = 140000 (past the INT8 path's exact-accumulation limit), one
    128-row tile cut into many K-segments."""
    X, W, b = make(128, 256, 140000, seed=9)
    assert not w8.shape_supported(128, 256, 140000)[0]
    check(run(X, W, b, cuda_device), X, W, b, what="K=140000")


@pytest.mark.parametrize("M,N,K", [(256 * 75, 256, 4096), (100, 264, 4096), (300, 520, 3072)])
def test_bf16_linear_split_and_whole_tiles_agree(cuda_device, M, N, K):
    """The same shape with room for K-split partials and with the minimum
    workspace (whole tiles only): both within the bound; repeated split runs
    are bit-identical (partials are added in segment order)."""
    X, W, b = make(M, N, K, seed=K + M)
    rows = np.arange(0, M, max(1, M // 150))
    full = run(X, W, b, cuda_device)
    assert w8.gemm_plan(M, N, K)[1] > 1, "this shape is expected to cut tiles along K"
    again = run(X, W, b, cuda_device)
    assert torch.equal(full.view(torch.int16), again.view(torch.int16))
    ws = torch.empty(w8.bf16_linear_workspace_bytes(1, 8, 8), dtype=torch.uint8, device=cuda_device)
    whole = run(X, W, b, cuda_device, workspace=ws)
    check(full, X, W, b, rows=rows, what="split")
    check(whole, X, W, b, rows=rows, what="whole")


def test_bf16_linear_pair_and_single_cta(cuda_device):
    X, W, b = make(512, 768, 2048, seed=4)
    pair = run(X, W, b, cuda_device)
    w8.debug_force_single_cta(True)
    try:
        single = run(X, W, b, cuda_device)
    finally:
        w8.debug_force_single_cta(False)
    check(pair, X, W, b, what="pair")
    check(single, X, W, b, what="single")


def test_bf16_linear_identity_weight_is_exact(cuda_device):
    """W = permuted identity: every output is one input value (+ 0), exact."""
    K = 512
    g = torch.Generator().manual_seed(8)
    X = torch.randn(200, K, generator=g).to(torch.bfloat16)
    perm = torch.randperm(K, generator=g)
    W = torch.eye(K, dtype=torch.bfloat16)[perm]
    Y = run(X, W, None, cuda_device)
    assert torch.equal(Y.view(torch.int16), X[:, perm].view(torch.int16))


def test_bf16_linear_guarded_layer_dispatch(cuda_device):
    """GuardedLinear takes the INT8 path where the guard accepts the shape and
    the BF16 path where it rejects it; both outputs meet their own bars."""
    X, W, b = make(64, 128, 1032, seed=5)
    layer = w8.GuardedLinear(W.to(cuda_device), b.to(cuda_device))
    assert not layer.int8
    Y = layer(X.to(cuda_device))
    torch.cuda.synchronize()
    check(Y.cpu(), X, W, b)
    X, W, b = make(64, 128, 1024, seed=6)
    layer = w8.GuardedLinear(W.to(cuda_device), b.to(cuda_device))
    assert layer.int8
    Y = layer(X.to(cuda_device))
    torch.cuda.synchronize()
    wq, sw = oracle.quantize_rows(bits(W))
    ref = oracle.linear(bits(X), wq, sw, bias_f32(b))
    yg = oracle.bf16_bits_to_f32(bits(Y)).astype(np.float64)
    assert (np.abs(yg - ref["y32"]) <= oracle.ulp_bf16(ref["y32"])).all()


def test_guarded_layer_fastest_policy(cuda_device):
    """policy="fastest": per row count, the layer times both paths once and
    keeps the faster; each call's output is then exactly that path's output
    (the W8A8 path within one bf16 ulp of the oracle, the BF16 path within
    its accumulation bound)."""
    X, W, b = make(300, 512, 1024, seed=9)
    dev = cuda_device
    layer = w8.GuardedLinear(W.to(dev), b.to(dev), policy="fastest")
    assert layer.int8
    Y = layer(X.to(dev))
    torch.cuda.synchronize()
    choice = layer.choice[(300, torch.bfloat16)]
    assert choice in ("int8", "bf16")
    if choice == "int8":
        wq, sw = oracle.quantize_rows(bits(W))
        ref = oracle.linear(bits(X), wq, sw, bias_f32(b))
        yg = oracle.bf16_bits_to_f32(bits(Y)).astype(np.float64)
        assert (np.abs(yg - ref["y32"]) <= oracle.ulp_bf16(ref["y32"])).all()
    else:
        check(Y.cpu(), X, W, b)
    Y2 = layer(X.to(dev))          # the cached choice, same bytes
    torch.cuda.synchronize()
    assert torch.equal(Y2.view(torch.int16), Y.view(torch.int16))
    with pytest.raises(ValueError):
        w8.GuardedLinear(W.to(dev), b.to(dev), policy="sometimes")
