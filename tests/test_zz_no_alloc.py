"""The entry point for callers that cannot allocate device memory.

Some users of this library cannot hand it a workspace: a plugin whose host
runtime owns the device memory budget, or a path that must not call
cudaMalloc.  ``w8a8_linear_noalloc`` serves them from a scratch array built
into the library.  These checks call it through the C ABI twice in a row,
with different shapes, and compare each result with ``w8a8_linear`` (which
takes a caller-owned workspace) within one bf16 ulp; they also check that a
shape too large for the built-in array is refused with nothing launched, and
that the call takes no device memory of its own.  The file is named so that
pytest collects it last."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_linear_act_b300 as w8
import w8a8_workloads as wl
from helpers import bits

pytestmark = pytest.mark.gpu


def _layer(case, M, N, K, dev):
    X, W, b = wl.make(case, M=M, N=N, K=K)
    Wq, sw = w8.quantize_weight(W.to(dev))
    return X.to(dev), w8.pack_weight(Wq), sw, b.to(dev)


def _within_one_ulp(y_new: torch.Tensor, y_ref: torch.Tensor):
    a = oracle.bf16_bits_to_f32(bits(y_new)).astype(np.float64)
    r = oracle.bf16_bits_to_f32(bits(y_ref)).astype(np.float64)
    assert (np.abs(a - r) <= oracle.ulp_bf16(r)).all()


def test_noalloc_matches_workspace_entry_point_twice(cuda_device):
    dev = cuda_device
    first = _layer("video", 300, 520, 1040, dev)        # ragged tiles, two K-chunks
    second = _layer("audio_m1001_n2048", 1001, 264, 512, dev)

    refs = [w8.linear(X, Wp, sw, b) for X, Wp, sw, b in (first, second)]
    torch.cuda.synchronize()

    y1 = w8.linear_noalloc(*first)
    y2 = torch.empty_like(refs[1])
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    w8.linear_noalloc(*second, out=y2)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()

    _within_one_ulp(y1, refs[0])
    _within_one_ulp(y2, refs[1])
    assert free_after == free_before        # the call itself takes no device memory


def test_noalloc_full_video_projection(cuda_device):
    """The bench's workload (M=6144, K=N=4096) fits the built-in array."""
    X, Wp, sw, b = _layer("video", 6144, 4096, 4096, cuda_device)
    assert w8.workspace_min_bytes(6144, 4096) <= w8.NOALLOC_SCRATCH_BYTES
    y = w8.linear_noalloc(X, Wp, sw, b)
    ref = w8.linear(X, Wp, sw, b)
    torch.cuda.synchronize()
    _within_one_ulp(y, ref)


def test_noalloc_refuses_oversized_shape(cuda_device):
    M, K = 8192, 4096                     # workspace 64 MiB + headers: one byte too many is enough
    assert w8.workspace_min_bytes(M, K) > w8.NOALLOC_SCRATCH_BYTES
    X = torch.zeros((M, K), dtype=torch.bfloat16, device=cuda_device)
    Wp = torch.zeros((64, K), dtype=torch.bfloat16, device=cuda_device)
    sw = torch.ones(64, device=cuda_device)
    Y = torch.full((M, 64), 7.0, dtype=torch.bfloat16, device=cuda_device)
    with pytest.raises(w8.W8A8Error) as e:
        w8.linear_noalloc(X, Wp, sw, None, out=Y)
    assert e.value.status == 5
    torch.cuda.synchronize()
    assert (Y == 7.0).all()               # nothing was launched
