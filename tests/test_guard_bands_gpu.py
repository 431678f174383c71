"""Outputs of the §8(f) entry points at ragged shapes write nothing outside
their tensors: each output sits inside a larger buffer filled with a canary
pattern that must survive, and the values inside are checked against the
entry point's own parity test reference."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_linear_act_b300 as w8
import w8a8_workloads as wl
from helpers import bits

pytestmark = pytest.mark.gpu

PAD = 4096   # bytes of canary on each side (keeps 16-byte alignment)


def banded(numel, dtype, dev):
    """(buffer, view): a view of `numel` elements inside a canary-filled buffer."""
    esize = torch.empty((), dtype=dtype).element_size()
    pad = PAD // esize
    raw = torch.full((numel * esize + 2 * PAD,), 0xA5, dtype=torch.uint8, device=dev)
    return raw, raw[PAD:PAD + numel * esize].view(dtype)


def intact(raw, numel_bytes):
    return bool((raw[:PAD] == 0xA5).all()) and bool((raw[PAD + numel_bytes:] == 0xA5).all())


def test_bf16_linear_guard_band(cuda_device):
    M, N, K = 131, 264, 328
    g = torch.Generator().manual_seed(1)
    X = torch.randn(M, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    raw, Y = banded(M * N, torch.bfloat16, cuda_device)
    w8.bf16_linear(X.to(cuda_device), W.to(cuda_device), None, out=Y.view(M, N))
    torch.cuda.synchronize()
    assert intact(raw, M * N * 2)
    y64, absum = oracle.bf16_linear_f64(bits(X), bits(W))
    assert (np.abs(oracle.bf16_bits_to_f32(bits(Y.view(M, N))) - y64) <= oracle.bf16_linear_tolerance(y64, absum, K)).all()


def test_mlp_guard_bands(cuda_device):
    M, K, F, N = 131, 256, 528, 136
    X, _, _ = wl.make("video", M=M, N=8, K=K)
    g = torch.Generator().manual_seed(2)
    Wu = (torch.randn(F, K, generator=g) * 0.02).to(torch.bfloat16).to(cuda_device)
    Wd = (torch.randn(N, F, generator=g) * 0.02).to(torch.bfloat16).to(cuda_device)
    Wqu, swu = w8.quantize_weight(Wu)
    Wqd, swd = w8.quantize_weight(Wd)
    Wpu, Wpd = w8.pack_weight(Wqu), w8.pack_weight(Wqd)
    rawh, H = banded(M * F, torch.bfloat16, cuda_device)
    rawy, Y = banded(M * N, torch.bfloat16, cuda_device)
    w8.mlp(X.to(cuda_device), Wpu, swu, None, Wpd, swd, None, H=H.view(M, F), out=Y.view(M, N))
    torch.cuda.synchronize()
    assert intact(rawh, M * F * 2) and intact(rawy, M * N * 2)
    Hs = w8.linear(X.to(cuda_device), Wpu, swu, None)
    Ys = w8.linear(Hs, Wpd, swd, None)
    torch.cuda.synchronize()
    assert torch.equal(H.view(M, F).view(torch.int16), Hs.view(torch.int16))
    assert torch.equal(Y.view(M, N).view(torch.int16), Ys.view(torch.int16))


def test_qk_blocks_guard_bands(cuda_device):
    B, L, H, D, bt = 1, 77, 3, 80, 16
    X = torch.randn((B, L, H, D), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    nblk = -(-L // bt)
    rawq, Q = banded(X.numel(), torch.int8, cuda_device)
    raws, S = banded(B * H * nblk, torch.float32, cuda_device)
    Xd = X.to(cuda_device)
    lib = w8.load()
    st = lib.w8a8_quantize_qk_blocks(ctypes.c_void_p(Xd.data_ptr()), w8.BF16, B, H, L, D, 1, bt,
                                     ctypes.c_void_p(Q.data_ptr()), ctypes.c_void_p(S.data_ptr()), None)
    torch.cuda.synchronize()
    assert st == 0
    assert intact(rawq, X.numel()) and intact(raws, B * H * nblk * 4)
    qr, sr = oracle.quantize_qk_blocks(bits(X), bt, "NHD")
    assert np.array_equal(Q.cpu().numpy().reshape(X.shape), qr)
    assert np.array_equal(S.cpu().numpy().reshape(B, H, nblk), sr)


def test_norm_guard_bands(cuda_device):
    M, K = 33, 1040
    X = (torch.randn(M, K, generator=torch.Generator().manual_seed(4)) * 2).to(torch.bfloat16)
    rawq, Q = banded(M * K, torch.int8, cuda_device)
    raws, S = banded(M, torch.float32, cuda_device)
    rawy, Yb = banded(M * K, torch.bfloat16, cuda_device)
    Xd = X.to(cuda_device)
    lib = w8.load()
    st = lib.w8a8_norm_quantize_act(ctypes.c_void_p(Xd.data_ptr()), M, K, 1, ctypes.c_float(1e-6), None, None, 1,
                                    ctypes.c_void_p(Yb.data_ptr()), ctypes.c_void_p(Q.data_ptr()),
                                    ctypes.c_void_p(S.data_ptr()), None)
    torch.cuda.synchronize()
    assert st == 0
    assert intact(rawq, M * K) and intact(raws, M * 4) and intact(rawy, M * K * 2)
    # inside: y within one bf16 step of the float64 rows, codes within one step
    yb_ref, q_ref, _, y64 = oracle.norm_quantize(bits(X), "rms", 1e-6)
    assert (np.abs(oracle.bf16_bits_to_f32(bits(Yb.view(M, K))) - y64) <= oracle.ulp_bf16(y64)).all()
    assert np.abs(Q.cpu().numpy().reshape(M, K).astype(np.int32) - q_ref.astype(np.int32)).max() <= 1
