"""GPU parity of the whole W8A8 linear (activation quantisation -> tcgen05 GEMM
-> fused dequantisation, bias, bf16 store) against the CPU oracle.

Bar: activation codes and scales bit-exact; every bf16 output within one bf16
ulp of the oracle's fp32 epilogue value y32 = ((float)acc * sx) * sw + bias
(zhidx TurboT2VA article, section 01 item 3: scales and bias applied once
after the full INT32 accumulation).  The kernel evaluates the same fp32
steps in the same order, so in practice the outputs are bit-identical; the
ulp is the stated margin."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_linear_act_b300 as w8
import w8a8_workloads as wl
from helpers import assert_within_one_bf16_ulp, bias_f32, bits, check_linear_in_row_blocks

pytestmark = pytest.mark.gpu


def gpu_linear(X, W, bias, dev, out=None, workspace=None):
    Wq, sw = w8.quantize_weight(W.to(dev))
    Wp = w8.pack_weight(Wq)
    Y = w8.linear(X.to(dev), Wp, sw, None if bias is None else bias.to(dev), out=out, workspace=workspace)
    torch.cuda.synchronize()
    return Y, Wq.cpu().numpy(), sw.cpu().numpy()


def oracle_linear(X, W, bias, rows=None, exact_f64=True):
    wq, sw = oracle.quantize_rows(bits(W))
    return oracle.linear(bits(X), wq, sw, bias_f32(bias), rows=rows, exact_f64=exact_f64), wq, sw


def compare(X, W, bias, dev, rows=None, what=""):
    Y, wq_g, sw_g = gpu_linear(X, W, bias, dev)
    ref, wq, sw = oracle_linear(X, W, bias, rows=rows)
    assert np.array_equal(wq_g, wq) and np.array_equal(sw_g.view(np.uint32), sw.view(np.uint32))
    yb = bits(Y)
    if rows is not None:
        yb = yb[rows]
    same = assert_within_one_bf16_ulp(yb, ref["y32"], what)
    return Y, ref, same


@pytest.mark.parametrize("name", list(wl.CASES))
def test_linear_reduced_sizes(cuda_device, name):
    """Every workload recipe with M and N cut to span several tiles plus a
    ragged tail (K kept), checked in full."""
    c = wl.CASES[name]
    M = min(c.M, 300)
    N = min(c.N, 520)
    X, W, b = wl.make(c, M=M, N=N)
    _, ref, same = compare(X, W, b, cuda_device, what=name)
    assert same is None or same == 1.0, "bit-identical fraction %.6f" % same


@pytest.mark.parametrize("name", ["tiny", "video", "audio_m126_n2048", "audio_m126_n8192",
                                  "audio_m1001_n2048", "audio_m1001_n8192"])
def test_linear_full_size(cuda_device, name):
    """Full-size workloads, every output checked."""
    c = wl.CASES[name]
    X, W, b = wl.make(c)
    Y, ref, _ = compare(X, W, b, cuda_device, what=name)
    if c.zero_last_row:
        assert np.array_equal(bits(Y)[-1], oracle.bf16_rne(bias_f32(b)))


@pytest.mark.parametrize("name", ["mlp_up", "mlp_down", "hires_n4k", "hires_n16k"])
def test_linear_full_size_every_output(cuda_device, name):
    """The MLP and high-resolution workloads at full size, in the launch
    configuration the benchmark times, every element checked: activation
    and weight codes and scales bit-exact, the INT32 accumulators of the
    same codes through w8a8_gemm_s32 bit-exact, every bf16 output within one
    bf16 ulp of the oracle's fp32 epilogue value (and bit-identical to its
    bf16 in practice)."""
    c = wl.CASES[name]
    dev = cuda_device
    X, W, b = wl.make(c)
    Xd = X.to(dev)
    Wq, sw = w8.quantize_weight(W.to(dev))
    Wp = w8.pack_weight(Wq)
    Xq, sx = w8.quantize_act(Xd)
    acc = w8.gemm_s32(Xq, Wp)
    Y = w8.linear(Xd, Wp, sw, b.to(dev))
    torch.cuda.synchronize()
    wq_ref, sw_ref = oracle.quantize_rows(bits(W))
    assert np.array_equal(Wq.cpu().numpy(), wq_ref)
    assert np.array_equal(sw.cpu().numpy().view(np.uint32), sw_ref.view(np.uint32))
    same, xq_ref, sx_ref = check_linear_in_row_blocks(bits(X), wq_ref, sw_ref, bias_f32(b), bits(Y),
                                                      acc_gpu=acc.cpu().numpy(), what=name)
    assert np.array_equal(Xq.cpu().numpy(), xq_ref)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), sx_ref.view(np.uint32))
    assert same == 1.0, "bit-identical fraction %.8f" % same


def test_linear_no_bias_and_f32_bias(cuda_device):
    c = wl.CASES["video"]
    X, W, b = wl.make(c, M=200, N=264, K=512)
    compare(X, W, None, cuda_device, what="no bias")
    compare(X, W, b.float(), cuda_device, what="f32 bias")


def test_linear_zero_rows_output_bias(cuda_device):
    X, W, b = wl.make("audio_m126_n2048", M=130, N=64, K=256)
    X[0].zero_()
    X[129].zero_()
    Y, ref, _ = compare(X, W, b, cuda_device)
    bb = oracle.bf16_rne(bias_f32(b))
    assert np.array_equal(bits(Y)[0], bb) and np.array_equal(bits(Y)[129], bb)


def test_linear_zero_weight_channel(cuda_device):
    X, W, b = wl.make("video", M=64, N=256, K=256)
    W[17].zero_()
    Y, ref, _ = compare(X, W, b, cuda_device)
    assert np.array_equal(bits(Y)[:, 17], np.full(64, oracle.bf16_rne(bias_f32(b)[17:18])[0]))


def test_linear_stages_equal_fused_call(cuda_device):
    """quant_stage + gemm_stage on one workspace gives the same bytes as linear()."""
    X, W, b = wl.make("video", M=256, N=512, K=1024)
    Xd, bd = X.to(cuda_device), b.to(cuda_device)
    Wq, sw = w8.quantize_weight(W.to(cuda_device))
    Wp = w8.pack_weight(Wq)
    Y1 = w8.linear(Xd, Wp, sw, bd)
    ws = torch.empty(w8.workspace_bytes(256, 512, 1024), dtype=torch.uint8, device=cuda_device)
    Y2 = torch.empty_like(Y1)
    w8.linear_quant_stage(Xd, ws)
    w8.linear_gemm_stage(256, 1024, Wp, sw, bd, Y2, ws)
    torch.cuda.synchronize()
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    assert w8.read_status(ws) == (0, 0)


@pytest.mark.parametrize("M,N", [(1600, 4096), (3000, 4096), (6150, 1024), (9000, 2048)])
def test_linear_in_gemm_quantisation_equals_two_stages(cuda_device, M, N):
    """With bf16 X and K = 4096, linear() quantises only the rows of the
    GEMM's first wave up front and the rest inside the GEMM while it runs
    (ragged last tiles, rows past the first wave in one or several tile
    groups).  Y, the codes and the row scales are the same bytes as the two
    stages give, and Y matches the oracle on sampled row blocks."""
    K = 4096
    X, W, b = wl.make("video", M=M, N=N, K=K)
    Xd, bd = X.to(cuda_device), b.to(cuda_device)
    Wq, sw = w8.quantize_weight(W.to(cuda_device))
    Wp = w8.pack_weight(Wq)
    ws1 = torch.empty(w8.workspace_bytes(M, N, K), dtype=torch.uint8, device=cuda_device)
    ws2 = torch.empty_like(ws1)
    ws1.fill_(0x5A)   # stale contents must not matter
    Y1 = w8.linear(Xd, Wp, sw, bd, workspace=ws1)
    Y2 = torch.empty_like(Y1)
    w8.linear_quant_stage(Xd, ws2)
    w8.linear_gemm_stage(M, K, Wp, sw, bd, Y2, ws2)
    torch.cuda.synchronize()
    assert w8.read_status(ws1) == (0, 0)
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    # the row scales and the codes in the workspace (layout: 1 KB header,
    # then sx, then the codes from the next 1 KB boundary)
    codes_off = 1024 + ((M * 4 + 1023) // 1024) * 1024
    assert torch.equal(ws1[1024:1024 + M * 4], ws2[1024:1024 + M * 4])
    assert torch.equal(ws1[codes_off:codes_off + M * K * 2], ws2[codes_off:codes_off + M * K * 2])
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(1500, 1600), np.arange(M - 64, M),
                                     np.random.default_rng(M).choice(M, 64, replace=False)]))
    compare(X, W, b, cuda_device, rows=rows[rows < M], what="in-GEMM quantisation")


def test_linear_in_gemm_quantisation_timeout_reported(cuda_device):
    """The in-GEMM quantisation path with the producer issuing no copies (test
    hook): the rows are still quantised and published, the MMA issuer's and
    the epilogue's bounded waits run out, the status says so, and the next
    call is clean and equal to the two-stage result."""
    M, N, K = 3000, 1024, 4096
    X, W, b = wl.make("video", M=M, N=N, K=K)
    Xd, bd = X.to(cuda_device), b.to(cuda_device)
    Wq, sw = w8.quantize_weight(W.to(cuda_device))
    Wp = w8.pack_weight(Wq)
    ws = torch.empty(w8.workspace_bytes(M, N, K), dtype=torch.uint8, device=cuda_device)
    w8.set_wait_limit_ns(20_000_000)
    w8.debug_skip_loads(True)
    try:
        w8.linear(Xd, Wp, sw, bd, workspace=ws)
        st, bits_ = w8.read_status(ws)
    finally:
        w8.debug_skip_loads(False)
        w8.set_wait_limit_ns(2_000_000_000)
    assert st == 7 and bits_ & 0x2 and bits_ & 0x4
    again = w8.linear(Xd, Wp, sw, bd, workspace=ws)
    assert w8.read_status(ws) == (0, 0)
    ws2 = torch.empty_like(ws)
    Y2 = torch.empty_like(again)
    w8.linear_quant_stage(Xd, ws2)
    w8.linear_gemm_stage(M, K, Wp, sw, bd, Y2, ws2)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), Y2.view(torch.int16))


def test_linear_output_guard_band(cuda_device):
    """Ragged M/N tiles write nothing outside Y: Y sits inside a larger buffer
    filled with a canary pattern that must survive."""
    M, N, K = 131, 264, 320
    X, W, b = wl.make("video", M=M, N=N, K=K)
    big = torch.full((M * N + 4096,), 0x5A5A, dtype=torch.int16, device=cuda_device)
    Y = big[2048:2048 + M * N].view(torch.bfloat16).view(M, N)
    Wq, sw = w8.quantize_weight(W.to(cuda_device))
    w8.linear(X.to(cuda_device), w8.pack_weight(Wq), sw, b.to(cuda_device), out=Y)
    torch.cuda.synchronize()
    assert (big[:2048] == 0x5A5A).all() and (big[2048 + M * N:] == 0x5A5A).all()
    ref, _, _ = oracle_linear(X, W, b)
    assert_within_one_bf16_ulp(bits(Y), ref["y32"], "guard band")


def test_linear_repeat_calls_reuse_workspace(cuda_device):
    """Back-to-back calls on one workspace and one stream give identical results."""
    X, W, b = wl.make("audio_m1001_n2048", M=300, N=256, K=512)
    dev = cuda_device
    Wq, sw = w8.quantize_weight(W.to(dev))
    Wp = w8.pack_weight(Wq)
    ws = torch.empty(w8.workspace_bytes(300, 256, 512), dtype=torch.uint8, device=dev)
    Xd, bd = X.to(dev), b.to(dev)
    outs = [w8.linear(Xd, Wp, sw, bd, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_layer_object(cuda_device):
    X, W, b = wl.make("video", M=100, N=256, K=256)
    layer = w8.W8A8Linear(W.to(cuda_device), b.to(cuda_device))
    assert layer.supported(100)
    Y = layer(X.to(cuda_device))
    torch.cuda.synchronize()
    ref, _, _ = oracle_linear(X, W, b)
    assert_within_one_bf16_ulp(bits(Y), ref["y32"], "layer")


def test_guard_rejects_without_launch(cuda_device):
    X = torch.randn(8, 24, device=cuda_device, dtype=torch.bfloat16)
    Wp = torch.zeros(16, 24, device=cuda_device, dtype=torch.bfloat16)
    sw = torch.ones(16, device=cuda_device)
    with pytest.raises(w8.UnsupportedShape):
        w8.linear(X, Wp, sw)


def test_linear_k_split_workspace_sizes_identical(cuda_device):
    """The full-size video projection with the workspace that w8a8_linear
    asks for (last wave cut along K), with a smaller one (fewer segments) and
    with the smallest accepted (whole tiles only): identical bytes."""
    dev = cuda_device
    M, N, K = 6144, 4096, 4096
    X, W, b = wl.make("video")
    Xd, bd = X.to(dev), b.to(dev)
    Wq, sw = w8.quantize_weight(W.to(dev))
    Wp = w8.pack_weight(Wq)
    slot = 128 * 256 * 4
    outs = []
    for size in (w8.workspace_bytes(M, N, K), w8.workspace_min_bytes(M, K) + 100 * slot,
                 w8.workspace_min_bytes(M, K)):
        ws = torch.empty(size, dtype=torch.uint8, device=dev)
        outs.append(w8.linear(Xd, Wp, sw, bd, workspace=ws))
        assert w8.read_status(ws) == (0, 0)
    torch.cuda.synchronize()
    assert w8.gemm_plan(M, N, K)[1] == 5
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_linear_pair_and_single_cta_forms_identical(cuda_device):
    """The video projection through the CTA-pair GEMM and through the
    single-CTA GEMM: identical bytes (both are the exact INT32 accumulator
    followed by the same fp32 epilogue)."""
    dev = cuda_device
    X, W, b = wl.make("video")
    Xd, bd = X.to(dev), b.to(dev)
    Wq, sw = w8.quantize_weight(W.to(dev))
    Wp = w8.pack_weight(Wq)
    pair = w8.linear(Xd, Wp, sw, bd)
    w8.debug_force_single_cta(True)
    try:
        single = w8.linear(Xd, Wp, sw, bd)
    finally:
        w8.debug_force_single_cta(False)
    torch.cuda.synchronize()
    assert torch.equal(pair.view(torch.int16), single.view(torch.int16))


@pytest.mark.parametrize("case,M,N,K", [
    ("video", 1000, 520, 1024),         # ragged tiles, CTA pairs
    ("video", 6144, 4096, 4096),        # the benchmark's layer
    ("tiny", 64, 128, 256),             # fp32 activations, one 256-row pair tile for 64 rows
    ("audio_m126_n2048", 126, 2048, 2048),
    ("audio_m1001_n8192", 1001, 8192, 2048),
])
def test_linear_repeated_calls_equal_stage_calls(cuda_device, case, M, N, K):
    """Twenty w8a8_linear calls in a row on one workspace must each give the
    bytes of the two stage calls (quantiser kernel, then GEMM) on the same
    inputs, with a clean status word: the workspace header (status word,
    split-tile counters) is cleared by every call's first kernel, and the
    GEMM, launched as that kernel's programmatic dependent, waits for it."""
    dev = cuda_device
    X, W, b = wl.make(case, M=M, N=N, K=K)
    Xd, bd = X.to(dev), b.to(dev)
    Wq, sw = w8.quantize_weight(W.to(dev))
    Wp = w8.pack_weight(Wq)
    ws = torch.empty(w8.workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
    ref = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    w8.linear_quant_stage(Xd, ws)
    w8.linear_gemm_stage(M, K, Wp, sw, bd, ref, ws)
    outs = [w8.linear(Xd, Wp, sw, bd, workspace=ws) for _ in range(20)]
    assert w8.read_status(ws) == (0, 0)
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16)), "call %d differs" % i


def test_linear_matches_the_golden_fixture(cuda_device):
    """The CUDA path on tests/golden/linear_small.json (written by the
    oracle): codes, scales and accumulators bit-exact, outputs within one
    bf16 ulp (identical in practice)."""
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "linear_small.json")
    g = json.load(open(path))
    as_bf16 = lambda a: torch.from_numpy(np.array(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)  # noqa: E731
    X, W, b = as_bf16(g["X_bf16_bits"]), as_bf16(g["W_bf16_bits"]), as_bf16(g["bias_bf16_bits"])
    dev = cuda_device
    Wq, sw = w8.quantize_weight(W.to(dev))
    Xq, sx = w8.quantize_act(X.to(dev))
    Wp = w8.pack_weight(Wq)
    acc = w8.gemm_s32(Xq, Wp)
    Y = w8.linear(X.to(dev), Wp, sw, b.to(dev))
    torch.cuda.synchronize()
    assert np.array_equal(Xq.cpu().numpy(), np.array(g["Xq"])) and np.array_equal(Wq.cpu().numpy(), np.array(g["Wq"]))
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), np.array(g["sx_f32_bits"], dtype=np.uint32))
    assert np.array_equal(sw.cpu().numpy().view(np.uint32), np.array(g["sw_f32_bits"], dtype=np.uint32))
    assert np.array_equal(acc.cpu().numpy(), np.array(g["acc"]))
    want = oracle.bf16_bits_to_f32(np.array(g["Y_bf16_bits"], dtype=np.uint16)).astype(np.float64)
    got = oracle.bf16_bits_to_f32(bits(Y)).astype(np.float64)
    assert (np.abs(got - want) <= oracle.ulp_bf16(want)).all()
