"""GPU parity of the per-block INT8 quantisation of attention Query and Key
(zhidx TurboT2VA article, section 01 item 4: SageSLA's INT8 Q/K) against the
CPU oracle: codes and scales bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_linear_act_b300 as w8
from helpers import bits

pytestmark = pytest.mark.gpu


def make(shape, seed, dtype=torch.bfloat16, outlier_tokens=0):
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(shape, generator=g)
    if outlier_tokens:
        idx = torch.randperm(X.numel() // shape[-1], generator=g)[:outlier_tokens]
        X.view(-1, shape[-1])[idx] *= 20.0
    return X.to(dtype)


def check(X, bt, layout, dev):
    q, s = w8.quantize_qk_blocks(X.to(dev), bt, layout)
    torch.cuda.synchronize()
    qr, sr = oracle.quantize_qk_blocks(bits(X), bt, layout)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), sr.view(np.uint32)), "scales differ"
    qg = q.cpu().numpy()
    assert np.array_equal(qg, qr), "codes differ at %d places" % int((qg != qr).sum())


@pytest.mark.parametrize("shape,bt,layout", [
    ((1, 32, 6144, 128), 128, "HND"),   # video Query, 128-token blocks
    ((1, 32, 6144, 128), 64, "HND"),    # video Key, 64-token blocks
    ((1, 6144, 32, 128), 128, "NHD"),   # same, token-major
    ((2, 1001, 4, 64), 64, "NHD"),      # audio: ragged last block
    ((1, 3, 126, 64), 128, "HND"),      # fewer tokens than one block
    ((1, 77, 2, 80), 16, "NHD"),        # D = 80: 10 vectors per token
    ((1, 2, 300, 128), 1, "HND"),       # one token per block
    ((1, 1, 4096, 128), 4096, "HND"),   # one block longer than the registers hold: read twice
    ((1, 2, 40, 2048), 8, "HND"),       # D = 2048: a token is 256 vectors
    ((2, 300, 3, 128), 128, "NHD"),     # 512-thread CTAs, ragged last block
    ((1, 2, 600, 128), 256, "HND"),     # 4096-vector blocks: 256 threads of 16 vectors
])
def test_qk_blocks_bf16(cuda_device, shape, bt, layout):
    check(make(shape, seed=sum(shape) + bt, outlier_tokens=3), bt, layout, cuda_device)


@pytest.mark.parametrize("shape,bt,layout", [
    ((1, 8, 1024, 128), 128, "HND"),   # 512-thread CTAs of 4 vectors
    ((1, 8, 1024, 128), 256, "HND"),   # 256 threads of 16 vectors
    ((1, 6, 300, 64), 64, "NHD"),      # ragged last blocks
])
def test_qk_blocks_tiny_scales(cuda_device, shape, bt, layout):
    """Blocks whose scale lies on either side of 2^-100 (the correction step
    against the out-of-line tie test with division), bit-exact."""
    X = make(shape, seed=sum(shape) + bt).to(torch.float32)
    tok_axis = 2 if layout == "HND" else 1
    L = shape[tok_axis]
    exps = [0, -100, -101, -110, -126, 15]
    for j, t0 in enumerate(range(0, L, bt)):
        sl = [slice(None)] * 4
        sl[tok_axis] = slice(t0, t0 + bt)
        X[tuple(sl)] *= 2.0 ** exps[j % len(exps)]
    check(X.to(torch.bfloat16), bt, layout, cuda_device)


def test_qk_blocks_fp32_and_zero_block(cuda_device):
    X = make((1, 4, 200, 64), seed=5, dtype=torch.float32)
    X[0, 2, 64:128] = 0.0
    check(X, 64, "HND", cuda_device)
    q, s = w8.quantize_qk_blocks(X.to(cuda_device), 64, "HND")
    assert float(s[0, 2, 1]) == 1.0 and not q[0, 2, 64:128].any()


def test_qk_blocks_empty_and_errors(cuda_device):
    q, s = w8.quantize_qk_blocks(torch.empty((1, 2, 0, 64), dtype=torch.bfloat16, device=cuda_device), 64)
    assert q.numel() == 0 and s.shape == (1, 2, 0)
    with pytest.raises(w8.UnsupportedShape):
        w8.quantize_qk_blocks(torch.zeros((1, 2, 8, 12), dtype=torch.bfloat16, device=cuda_device), 4)
