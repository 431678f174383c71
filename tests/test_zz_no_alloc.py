"""The entry points for callers that cannot allocate device memory.

Some users of this library cannot hand it a workspace: a plugin whose host
runtime owns the device memory budget and gives it no scratch space, or a
path that must not call cudaMalloc (it can synchronise the device, and there
may be no memory pool to draw from).  ``w8a8_linear_noalloc`` serves them
from a scratch array built into the library, and ``w8a8_noalloc_read_status``
reads that array's device status word.

These checks call both through the C ABI: two calls in a row with different
shapes, each output compared with the CPU oracle (within one bf16 ulp, and
bit-identical to the oracle's bf16 in practice) and with ``w8a8_linear`` on
a caller-owned workspace (bit-identical); a call whose plan cuts the last
wave along K, run right after a different shape, so that split partials and
arrival counters left in the shared array by earlier calls would show; a
shape too large for the array, refused with nothing launched; and a forced
device-side timeout reported through the status reader, after which the
next call is clean and correct.  The file is named so that pytest collects
it last."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_linear_act_b300 as w8
import w8a8_workloads as wl
from helpers import assert_within_one_bf16_ulp, bias_f32, bits

pytestmark = pytest.mark.gpu

SLOT_BYTES = 128 * 256 * 4   # one INT32 partial tile of the GEMM's K-split


def _layer(case, M, N, K, dev):
    X, W, b = wl.make(case, M=M, N=N, K=K)
    Wq, sw = w8.quantize_weight(W.to(dev))
    return (X, W, b), (X.to(dev), w8.pack_weight(Wq), sw, b.to(dev))


def _check_against_oracle(host, y):
    X, W, b = host
    wq, sw = oracle.quantize_rows(bits(W))
    ref = oracle.linear(bits(X), wq, sw, bias_f32(b), exact_f64=True)
    same = assert_within_one_bf16_ulp(bits(y), ref["y32"], "noalloc")
    assert same is None or same == 1.0, "bit-identical fraction %.6f" % same
    if same is None:   # large outputs: compare the bf16 bits directly
        assert np.array_equal(bits(y), ref["y"])


def test_noalloc_two_calls_match_oracle_and_workspace_entry_point(cuda_device):
    dev = cuda_device
    first_host, first = _layer("video", 300, 520, 1040, dev)                 # ragged tiles, two K-chunks
    second_host, second = _layer("audio_m1001_n2048", 1001, 264, 512, dev)   # zero last row

    refs = [w8.linear(X, Wp, sw, b) for X, Wp, sw, b in (first, second)]
    torch.cuda.synchronize()

    y1 = w8.linear_noalloc(*first)
    y2 = torch.empty_like(refs[1])
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    w8.linear_noalloc(*second, out=y2)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert w8.noalloc_read_status() == (0, 0)

    assert torch.equal(y1.view(torch.int16), refs[0].view(torch.int16))
    assert torch.equal(y2.view(torch.int16), refs[1].view(torch.int16))
    _check_against_oracle(first_host, y1)
    _check_against_oracle(second_host, y2)
    assert free_after == free_before        # the call itself takes no device memory


def test_noalloc_k_split_after_another_shape(cuda_device):
    """The video projection (M=6144, K=N=4096) fits the built-in array with
    room for some of the split partial tiles, so its last wave is cut along
    K.  It runs right after a smaller shape, and twice, and must equal the
    oracle each time: nothing left in the shared array may leak into it."""
    dev = cuda_device
    M, N, K = 6144, 4096, 4096
    min_ws = w8.workspace_min_bytes(M, K)
    assert min_ws <= w8.NOALLOC_SCRATCH_BYTES
    slots = (w8.NOALLOC_SCRATCH_BYTES - min_ws) // SLOT_BYTES
    plan = w8.gemm_plan(M, N, K, max_slots=slots)
    assert plan[1] > 1, "this shape is expected to cut its last wave along K"

    _, small = _layer("audio_m126_n2048", 126, 2048, 2048, dev)
    host, big = _layer("video", M, N, K, dev)
    w8.linear_noalloc(*small)
    y1 = w8.linear_noalloc(*big).clone()
    w8.linear_noalloc(*small)
    y2 = w8.linear_noalloc(*big)
    torch.cuda.synchronize()
    assert w8.noalloc_read_status() == (0, 0)
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    _check_against_oracle(host, y1)


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


def test_noalloc_timeout_is_reported_and_next_call_is_clean(cuda_device):
    """A test hook makes the GEMM's TMA producer issue no copies, so its
    bounded waits run out (20 ms limit): the built-in array's status word
    must say so, and the next call must be clean and correct."""
    host, layer = _layer("video", 256, 512, 512, cuda_device)
    good = w8.linear_noalloc(*layer).clone()
    assert w8.noalloc_read_status() == (0, 0)
    w8.set_wait_limit_ns(20_000_000)
    w8.debug_skip_loads(True)
    try:
        w8.linear_noalloc(*layer)
        st, dev_bits = w8.noalloc_read_status()
    finally:
        w8.debug_skip_loads(False)
        w8.set_wait_limit_ns(2_000_000_000)
    assert st == 7                                  # W8A8_ERR_TIMEOUT
    assert dev_bits & 0x2 and dev_bits & 0x4        # MMA issuer and epilogue both gave up
    again = w8.linear_noalloc(*layer)
    assert w8.noalloc_read_status() == (0, 0)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), good.view(torch.int16))
    _check_against_oracle(host, again)
