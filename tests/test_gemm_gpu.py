"""GPU parity of the INT32 accumulators: the tcgen05 GEMM (bf16-carried codes,
fp32 tensor-memory chunks of at most 1024 drained exactly into INT32) must
equal the oracle's exact integer dot products bit for bit (zhidx TurboT2VA
article, section 01 item 3: "INT32 accumulation")."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_linear_act_b300 as w8
import w8a8_workloads as wl

pytestmark = pytest.mark.gpu


def run_gemm(Xq: torch.Tensor, Wq: torch.Tensor, dev):
    Wp = w8.pack_weight(Wq.to(dev))
    acc = w8.gemm_s32(Xq.to(dev), Wp)
    torch.cuda.synchronize()
    return acc.cpu().numpy()


def ref_gemm(Xq, Wq, rows=None):
    xq = Xq.numpy()
    wq = Wq.numpy()
    if rows is None:
        return oracle.gemm_s32_f64(xq, wq)
    return oracle.gemm_s32(xq, wq, rows)


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 64),      # one tile, one k-block
    (128, 256, 1024),    # one full chunk
    (1, 8, 16),          # smallest accepted shape
    (77, 40, 272),       # ragged everything, K tail inside a k-block
    (300, 520, 1040),    # ragged M and N tiles, K just over one chunk
    (256, 512, 4096),    # four chunks
    (129, 264, 2064),    # one row / 8 columns past a tile, K past two chunks
    (1000, 2048, 3200),
])
def test_s32_random_codes(cuda_device, M, N, K):
    Xq = wl.random_codes((M, K), seed=M)
    Wq = wl.random_codes((N, K), seed=N + 1)
    acc = run_gemm(Xq, Wq, cuda_device)
    ref = ref_gemm(Xq, Wq)
    assert np.array_equal(acc, ref), "mismatches: %d" % int((acc != ref).sum())


def test_s32_chunk_sums_near_2_24(cuda_device):
    """Adversarial: codes in [100, 127] of one sign, so each 1024-long chunk
    sums to 1.0e7..1.65e7 (just under 2^24 = 1.68e7) with odd low bits, and the
    full K = 4096 sum reaches 6.6e7 (past fp32's exact-integer range)."""
    Xq = wl.random_codes((256, 4096), seed=11, low=100, high=127)
    Wq = wl.random_codes((512, 4096), seed=12, low=100, high=127)
    Wq[1::2] = -Wq[1::2]
    Xq[::3] = -Xq[::3]
    acc = run_gemm(Xq, Wq, cuda_device)
    ref = ref_gemm(Xq, Wq)
    assert np.abs(ref.astype(np.int64)).min() > 4 * 10 ** 7
    assert (ref % 2 != 0).any()
    assert np.array_equal(acc, ref), "mismatches: %d" % int((acc != ref).sum())


def test_s32_extreme_codes(cuda_device):
    """All +-127: every chunk reaches 1024 * 16129 = 16,516,096 exactly."""
    Xq = torch.full((128, 8192), 127, dtype=torch.int8)
    Wq = torch.full((256, 8192), 127, dtype=torch.int8)
    Wq[7] = -127
    acc = run_gemm(Xq, Wq, cuda_device)
    assert (acc[:, 0] == 8192 * 16129).all() and (acc[:, 7] == -8192 * 16129).all()


def test_s32_identity_and_permutation(cuda_device):
    """Wq = permuted identity: acc is Xq with permuted columns (pins operand
    roles and the output column order)."""
    K = 256
    Xq = wl.random_codes((130, K), seed=5)
    perm = torch.randperm(K, generator=torch.Generator().manual_seed(6))
    Wq = torch.eye(K, dtype=torch.int8)[perm]
    acc = run_gemm(Xq, Wq, cuda_device)
    assert np.array_equal(acc, Xq[:, perm].numpy().astype(np.int32))


def test_s32_max_k(cuda_device):
    """K = 133136, the largest accepted multiple of 16: 131 chunks, worst-case
    magnitudes 2.1e9, still exact."""
    K = 133136
    Xq = torch.full((2, K), 127, dtype=torch.int8)
    Xq[1, ::2] = -127
    Wq = torch.full((8, K), 127, dtype=torch.int8)
    Wq[3] = wl.random_codes((K,), seed=9)
    acc = run_gemm(Xq, Wq, cuda_device)
    ref = ref_gemm(Xq, Wq)
    assert acc[0, 0] == K * 16129
    assert np.array_equal(acc, ref)


@pytest.mark.parametrize("name", ["video", "audio_m1001_n8192", "audio_m126_n2048"])
def test_s32_workload_codes_full(cuda_device, name):
    """The accumulators of a real workload (quantised by the oracle), in full."""
    c = wl.CASES[name]
    X, W, _ = wl.make(c)
    from helpers import bits
    xq, _ = oracle.quantize_rows(bits(X))
    wq, _ = oracle.quantize_rows(bits(W))
    acc = run_gemm(torch.from_numpy(xq), torch.from_numpy(wq), cuda_device)
    ref = oracle.gemm_s32_f64(xq, wq)
    assert np.array_equal(acc, ref), "mismatches: %d" % int((acc != ref).sum())


@pytest.mark.parametrize("M,N,K", [
    (300, 520, 3072),        # 6 pair tiles on 74 pairs: every tile cut in 6 along K
    (256 * 75, 256, 4096),   # 74 whole pair tiles, then 1 tile cut in 8
    (100, 264, 4096),        # single-CTA tiles, 2 tiles cut in 8
    (128, 256, 133136),      # one tile cut into 45 segments of ~46 k-blocks
])
def test_s32_k_split_and_whole_tiles_agree(cuda_device, M, N, K):
    """The K-split of the last wave (INT32 partial tiles added by the last
    segment to finish) and whole-tile accumulation give the exact INT32
    accumulator: run once with room for the partial tiles and once with the
    smallest workspace (no split), both against the oracle."""
    dev = cuda_device
    assert w8.gemm_plan(M, N, K)[1] > 1
    assert w8.gemm_plan(M, N, K, max_slots=0)[1] == 1
    Xq = wl.random_codes((M, K), seed=M + 3)
    Wq = wl.random_codes((N, K), seed=N + 4)
    Wp = w8.pack_weight(Wq.to(dev))
    Xd = Xq.to(dev)
    split = w8.gemm_s32(Xd, Wp)
    ws_min = torch.empty(w8.workspace_min_bytes(M, K), dtype=torch.uint8, device=dev)
    whole = w8.gemm_s32(Xd, Wp, workspace=ws_min)
    again = w8.gemm_s32(Xd, Wp)                # a second split launch: same bytes
    torch.cuda.synchronize()
    ref = ref_gemm(Xq, Wq)
    for name, acc in (("split", split), ("whole", whole), ("split again", again)):
        acc = acc.cpu().numpy()
        assert np.array_equal(acc, ref), "%s: mismatches %d" % (name, int((acc != ref).sum()))


@pytest.mark.parametrize("M,N,K", [
    (1, 8, 16),           # one row: the pair's second CTA holds no row of X or Y
    (126, 2048, 2048),    # the audio rows, all inside the first CTA of each pair
    (64, 264, 1040),
    (129, 264, 2064),     # one row past a pair's first CTA: the second CTA's rows are all ragged
    (300, 520, 1040),
    (1000, 2048, 3200),
    (2048, 2048, 4096),
])
def test_s32_pair_and_single_cta_forms_agree(cuda_device, M, N, K):
    """The 2-CTA form (256 x 256 tiles, cta_group::2 MMA across two SMs) and
    the single-CTA form (128 x 256 tiles) on the same codes, both exact."""
    dev = cuda_device
    assert w8.gemm_plan(M, N, K)[4] == 2
    Xq = wl.random_codes((M, K), seed=M + 7)
    Wq = wl.random_codes((N, K), seed=N + 8)
    Wp = w8.pack_weight(Wq.to(dev))
    Xd = Xq.to(dev)
    pair = w8.gemm_s32(Xd, Wp)
    w8.debug_force_single_cta(True)
    try:
        assert w8.gemm_plan(M, N, K)[4] == 1
        single = w8.gemm_s32(Xd, Wp)
    finally:
        w8.debug_force_single_cta(False)
    torch.cuda.synchronize()
    ref = ref_gemm(Xq, Wq)
    for name, acc in (("pair", pair), ("single", single)):
        acc = acc.cpu().numpy()
        assert np.array_equal(acc, ref), "%s: mismatches %d" % (name, int((acc != ref).sum()))
