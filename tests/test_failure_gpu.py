"""Failure detection without a GPU fault: every device wait in the GEMM has a
wall-clock limit.  A test hook makes the TMA producer issue no copies, so the
MMA issuer's and the epilogue's waits run out; the kernel must record that in
the workspace's status word, free its tensor memory and return, leaving the
context usable for the next call."""
import numpy as np
import pytest
import torch

import w8a8_int8_linear_act_b300 as w8
import w8a8_workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[True, False], ids=["single-CTA form", "CTA-pair form"])
def single_cta(request):
    w8.debug_force_single_cta(request.param)
    yield request.param
    w8.debug_force_single_cta(False)


def test_bounded_wait_reports_timeout_and_context_survives(cuda_device, single_cta):
    dev = cuda_device
    M = 256
    X, W, b = wl.make("video", M=M, N=512, K=512)
    Xd, bd = X.to(dev), b.to(dev)
    Wq, sw = w8.quantize_weight(W.to(dev))
    Wp = w8.pack_weight(Wq)
    assert w8.gemm_plan(M, 512, 512)[4] == (1 if single_cta else 2)
    ws = torch.empty(w8.workspace_bytes(M, 512, 512), dtype=torch.uint8, device=dev)
    good = w8.linear(Xd, Wp, sw, bd, workspace=ws)
    assert w8.read_status(ws) == (0, 0)

    w8.set_wait_limit_ns(20_000_000)          # 20 ms
    w8.debug_skip_loads(True)
    try:
        w8.linear(Xd, Wp, sw, bd, workspace=ws)
        st, bits_ = w8.read_status(ws)
    finally:
        w8.debug_skip_loads(False)
        w8.set_wait_limit_ns(2_000_000_000)
    assert st == 7                             # W8A8_ERR_TIMEOUT
    assert bits_ & 0x2 and bits_ & 0x4         # MMA issuer and epilogue both gave up

    # The context still works and the next call is correct and clean.
    again = w8.linear(Xd, Wp, sw, bd, workspace=ws)
    assert w8.read_status(ws) == (0, 0)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), good.view(torch.int16))
