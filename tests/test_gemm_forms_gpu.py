"""GPU parity of the cluster-K GEMM form (problems with few output tiles:
the audio branch's 126- and 1001-row shapes; zhidx TurboT2VA article,
section 01 item 3: INT32 accumulation, scales and bias once after the full
sum; the audio and video branches have different shapes).

Each 128 x bn output tile is computed by a cluster of ks CTAs that split K
and add their INT32 partials through distributed shared memory.  Bar: the
INT32 accumulators equal the oracle's exactly, every bf16 output equals the
oracle's bf16 (within one ulp is the stated margin; the fp32 epilogue is the
same sequence of operations), for every tile width and cluster size, and
the bytes equal the persistent form's on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_linear_act_b300 as w8
import w8a8_workloads as wl
from helpers import assert_within_one_bf16_ulp, bias_f32, bits

pytestmark = pytest.mark.gpu

WIDTHS = [64, 128, 256]
SIZES = [1, 2, 4, 8]


@pytest.fixture
def form():
    """Restores the per-shape choice after a test that forces a form."""
    yield w8.debug_force_gemm_form
    w8.debug_force_gemm_form(-1)


def _layer(case, M, N, K, dev):
    X, W, b = wl.make(case, M=M, N=N, K=K)
    Wq, sw = w8.quantize_weight(W.to(dev))
    return (X, W, b), (X.to(dev), w8.pack_weight(Wq), sw, b.to(dev))


def _oracle(host):
    X, W, b = host
    wq, sw = oracle.quantize_rows(bits(W))
    return oracle.linear(bits(X), wq, sw, bias_f32(b), exact_f64=True)


@pytest.mark.parametrize("bn", WIDTHS)
@pytest.mark.parametrize("ks", SIZES)
def test_every_width_and_cluster_size_matches_oracle(cuda_device, form, bn, ks):
    """Ragged M (300: three 128-row tiles, the last partly past M), ragged N
    (520: a partial last tile for every width) and a K of 17 k-blocks, the
    last one partly past K, cut into ks ranges of 2 or 3 k-blocks."""
    M, N, K = 300, 520, 1040
    host, (Xd, Wp, sw, bd) = _layer("video", M, N, K, cuda_device)
    form(1, bn, ks)
    assert w8.gemm_form(M, N, K)[:3] == (1, bn, ks)
    Y = w8.linear(Xd, Wp, sw, bd)
    Xq, _ = w8.quantize_act(Xd)
    acc = w8.gemm_s32(Xq, Wp)
    torch.cuda.synchronize()
    ref = _oracle(host)
    assert np.array_equal(acc.cpu().numpy(), ref["acc"])
    assert_within_one_bf16_ulp(bits(Y), ref["y32"], "bn=%d ks=%d" % (bn, ks))
    assert np.array_equal(bits(Y), ref["y"])


@pytest.mark.parametrize("name", ["tiny", "audio_m126_n2048", "audio_m126_n8192", "audio_m1001_n2048",
                                  "audio_m1001_n8192"])
def test_planned_form_equals_persistent_form(cuda_device, form, name):
    """The audio and tiny workloads at full size: the form the planner picks
    (the cluster-K form for the few-tile shapes) gives the bytes of the
    persistent form, and both match the oracle."""
    c = wl.CASES[name]
    host, (Xd, Wp, sw, bd) = _layer(name, c.M, c.N, c.K, cuda_device)
    form(-1)
    planned = w8.gemm_form(c.M, c.N, c.K)
    if name != "audio_m1001_n8192":
        assert planned[0] == 1, planned
    y_auto = w8.linear(Xd, Wp, sw, bd)
    form(0)
    y_pers = w8.linear(Xd, Wp, sw, bd)
    torch.cuda.synchronize()
    assert torch.equal(y_auto.view(torch.int16), y_pers.view(torch.int16))
    ref = _oracle(host)
    assert_within_one_bf16_ulp(bits(y_auto), ref["y32"], name)
    assert np.array_equal(bits(y_auto), ref["y"])
    if c.zero_last_row:
        assert np.array_equal(bits(y_auto)[-1], oracle.bf16_rne(bias_f32(host[2])))


def test_forced_cluster_form_many_waves(cuda_device, form):
    """The video projection (6144 x 4096 x 4096) through the cluster-K form,
    384 clusters of 4 (several waves): identical to the persistent form."""
    M, N, K = 6144, 4096, 4096
    _, (Xd, Wp, sw, bd) = _layer("video", M, N, K, cuda_device)
    form(0)
    y_pers = w8.linear(Xd, Wp, sw, bd)
    form(1, 256, 4)
    assert w8.gemm_form(M, N, K) == (1, 256, 4, 48 * 16 * 4)
    y_kc = w8.linear(Xd, Wp, sw, bd)
    torch.cuda.synchronize()
    assert torch.equal(y_kc.view(torch.int16), y_pers.view(torch.int16))


@pytest.mark.parametrize("bn,ks", [(64, 8), (128, 4), (256, 2), (256, 1)])
def test_bf16_linear_cluster_form(cuda_device, form, bn, ks):
    """The native BF16 linear through the cluster-K form: fp32 partials
    added in rank order; within the fp32-accumulation bound of the float64
    sum, and repeated calls bit-identical."""
    M, N, K = 126, 264, 2048
    g = torch.Generator().manual_seed(bn + ks)
    X = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    b = (torch.randn(N, generator=g) * 0.01).to(torch.bfloat16)
    form(1, bn, ks)
    dev = cuda_device
    Y1 = w8.bf16_linear(X.to(dev), W.to(dev), b.to(dev))
    Y2 = w8.bf16_linear(X.to(dev), W.to(dev), b.to(dev))
    torch.cuda.synchronize()
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    y64, absum = oracle.bf16_linear_f64(bits(X), bits(W), bias_f32(b))
    err = np.abs(oracle.bf16_bits_to_f32(bits(Y1)).astype(np.float64) - y64)
    assert (err <= oracle.bf16_linear_tolerance(y64, absum, K)).all()


def test_cluster_form_output_guard_band(cuda_device, form):
    """Ragged tiles of the cluster-K form write nothing outside Y."""
    M, N, K = 131, 264, 320
    host, (Xd, Wp, sw, bd) = _layer("video", M, N, K, cuda_device)
    big = torch.full((M * N + 4096,), 0x5A5A, dtype=torch.int16, device=cuda_device)
    Y = big[2048:2048 + M * N].view(torch.bfloat16).view(M, N)
    form(1, 256, 2)
    w8.linear(Xd, Wp, sw, bd, out=Y)
    torch.cuda.synchronize()
    assert (big[:2048] == 0x5A5A).all() and (big[2048 + M * N:] == 0x5A5A).all()
    assert_within_one_bf16_ulp(bits(Y), _oracle(host)["y32"], "guard band")


def test_cluster_form_timeout_reported_and_context_survives(cuda_device, form):
    """The producer issues no copies (test hook): the bounded waits of the
    cluster-K form run out, the status word says so, every CTA still meets
    its cluster at both barriers and frees its tensor memory, and the next
    call is correct."""
    dev = cuda_device
    M, N, K = 126, 512, 2048
    _, (Xd, Wp, sw, bd) = _layer("audio_m126_n2048", M, N, K, dev)
    form(1, 128, 4)
    ws = torch.empty(w8.workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
    good = w8.linear(Xd, Wp, sw, bd, workspace=ws).clone()
    assert w8.read_status(ws) == (0, 0)
    w8.set_wait_limit_ns(20_000_000)
    w8.debug_skip_loads(True)
    try:
        w8.linear(Xd, Wp, sw, bd, workspace=ws)
        st, dev_bits = w8.read_status(ws)
    finally:
        w8.debug_skip_loads(False)
        w8.set_wait_limit_ns(2_000_000_000)
    assert st == 7 and dev_bits & 0x2 and dev_bits & 0x4
    again = w8.linear(Xd, Wp, sw, bd, workspace=ws)
    assert w8.read_status(ws) == (0, 0)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), good.view(torch.int16))
