"""The host-buffer entry point w8a8_linear_host: X copied in and Y copied out
in row chunks, pipelined against the W8A8 linear of the other chunks, must give
the same bytes as w8a8_linear on device buffers (same kernels, same inputs)."""
import pytest
import torch

import w8a8_int8_linear_act_b300 as w8
import w8a8_workloads as wl
from helpers import bits
from test_linear_gpu import oracle_linear
from helpers import assert_within_one_bf16_ulp

pytestmark = pytest.mark.gpu


def _layer(case, M, N, K, dev):
    X, W, b = wl.make(case, M=M, N=N, K=K)
    Wq, sw = w8.quantize_weight(W.to(dev))
    return X, W, b, w8.pack_weight(Wq), sw


@pytest.mark.parametrize("case,M,N,K,chunk", [
    ("video", 1000, 520, 1024, 0),        # default chunks (256 rows), ragged last chunk
    ("video", 1000, 520, 1024, 300),      # chunks that are not tile multiples
    ("video", 6144, 4096, 4096, 0),       # the benchmark's layer, 768-row chunks
    ("tiny", 64, 128, 256, 16),           # fp32 X, four chunks
    ("audio_m126_n2048", 126, 2048, 2048, 0),   # one chunk, zero last row
])
def test_host_pipeline_equals_device_call(cuda_device, case, M, N, K, chunk):
    dev = cuda_device
    X, W, b, Wp, sw = _layer(case, M, N, K, dev)
    bd = b.to(dev)
    ref = w8.linear(X.to(dev), Wp, sw, bd)
    Xh = X.pin_memory()
    Yh = w8.linear_host(Xh, Wp, sw, bd, chunk_rows=chunk)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(Yh.view(torch.int16), ref.cpu().view(torch.int16))


def test_host_pipeline_no_bias_and_repeat(cuda_device):
    """No bias; two calls in a row on the same staging buffers; checked
    against the oracle."""
    dev = cuda_device
    M, N, K = 700, 264, 512
    X, W, b, Wp, sw = _layer("video", M, N, K, dev)
    Xh = X.pin_memory()
    Xd = torch.empty((M, K), dtype=X.dtype, device=dev)
    Yd = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(w8.workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
    outs = []
    for _ in range(2):
        outs.append(w8.linear_host(Xh, Wp, sw, None, X_dev=Xd, Y_dev=Yd, workspace=ws, chunk_rows=200))
    torch.cuda.current_stream().synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    ref, _, _ = oracle_linear(X, W, None)
    assert_within_one_bf16_ulp(bits(outs[0]), ref["y32"], "host pipeline, no bias")
