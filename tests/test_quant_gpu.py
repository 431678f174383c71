"""GPU parity of the per-row quantisation kernel against the CPU oracle:
codes and scales bit-exact (zhidx TurboT2VA article, section 01 item 3:
activations per row, weights per output channel, INT8)."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_int8_linear_act_b300 as w8
import w8a8_workloads as wl
from helpers import bits

pytestmark = pytest.mark.gpu


def check_rows(A: torch.Tensor, dev, weight=False):
    q_ref, s_ref = oracle.quantize_rows(bits(A))
    Ad = A.to(dev)
    q, s = (w8.quantize_weight if weight else w8.quantize_act)(Ad)
    torch.cuda.synchronize()
    q = q.cpu().numpy()
    s = s.cpu().numpy()
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32)), "scales differ"
    bad = np.argwhere(q != q_ref)
    assert bad.size == 0, "codes differ at %s" % bad[:5].tolist()
    return q, s


@pytest.mark.parametrize("name", list(wl.CASES))
def test_act_and_weight_codes_reduced(cuda_device, name):
    """Every workload's recipe at a reduced M/N (K kept): a few CTAs, ragged row counts."""
    c = wl.CASES[name]
    X, W, _ = wl.make(c, M=min(c.M, 77), N=min(c.N, 40))
    check_rows(X, cuda_device)
    check_rows(W, cuda_device, weight=True)


@pytest.mark.parametrize("name", ["tiny", "video", "mlp_up", "mlp_down", "hires_n4k", "hires_n16k",
                                  "audio_m1001_n8192", "audio_m126_n2048"])
def test_act_codes_full_size(cuda_device, name):
    """Activation and weight codes and scales of every workload at full
    size, bit-exact (the [16384, 4096] weights of mlp_up and hires_n16k, the
    [28672, 4096] high-resolution activations)."""
    c = wl.CASES[name]
    X, W, _ = wl.make(c)
    q, s = check_rows(X, cuda_device)
    if c.zero_last_row:
        assert s[-1] == 1.0 and not q[-1].any()
    check_rows(W, cuda_device, weight=True)


@pytest.mark.parametrize("K", [16, 32, 48, 256, 272, 2048, 4096, 8192, 16384, 65536, 70016, 133136])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_codes_many_row_lengths(cuda_device, K, dtype):
    """Row lengths covering every register-tile variant and the two-pass path."""
    g = torch.Generator().manual_seed(K)
    R = 3 if K > 60000 else 9
    X = torch.randn(R, K, generator=g) * torch.logspace(-3, 3, R).unsqueeze(1)
    X[0, K // 3] = 40.0
    check_rows(X.to(dtype), cuda_device)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_lossless_and_ties(cuda_device, dtype):
    """x = k 2^e (one |k| = 127): codes are k exactly; x = (j + 1/2) 2^e: codes
    round half to even — the same inputs the oracle's pins use."""
    codes = torch.arange(-127, 128, dtype=torch.float64)
    rows = [codes * 2.0 ** e for e in (-10, 0, 7)]
    half = torch.cat([torch.tensor([127.0]), torch.arange(-127, 127, dtype=torch.float64) + 0.5]) * 2.0 ** -4
    rows.append(torch.cat([half, torch.zeros(1)]))
    X = torch.stack([r[:255] for r in rows]).to(torch.float32)
    X = torch.nn.functional.pad(X, (0, 1)).to(dtype)   # K = 256
    q, s = check_rows(X, cuda_device)
    assert (q[0, :255].astype(int) == np.arange(-127, 128)).all()
    assert s[0] == np.float32(2.0 ** -10)


def test_zero_and_denormal_rows(cuda_device):
    """Zero rows, negative-zero rows and fp32 rows whose scale underflows to 0
    become zero rows (scale 1); one step larger gives a denormal scale."""
    tiny = float(np.ldexp(np.float32(1.0), -149))
    X = torch.zeros(5, 32, dtype=torch.float32)
    X[1] = -0.0
    X[2, 3] = tiny * 63
    X[3, 0] = tiny * 127
    X[3, 1] = -tiny * 127
    X[4, 7] = 1e-30
    q, s = check_rows(X, cuda_device)
    assert s[0] == 1.0 and s[1] == 1.0 and s[2] == 1.0
    assert s[3] == np.float32(tiny) and q[3, 0] == 127 and q[3, 1] == -127
    Xb = X.to(torch.bfloat16)
    check_rows(Xb, cuda_device)


def scaled_rows(M, K, exps, seed):
    """bf16 rows of Gaussian values scaled to absmax 127 * 2^e for the given
    exponents (cycled), with exact ties and a lossless code sprinkled in."""
    g = torch.Generator().manual_seed(seed)
    X = torch.randn(M, K, generator=g, dtype=torch.float64)
    X = X / X.abs().amax(dim=1, keepdim=True) * 127.0
    X[:, 1] = 127.0
    X[:, 2:34] = torch.arange(32, dtype=torch.float64) - 15.5   # exact half-integers of s
    for i in range(M):
        X[i] *= 2.0 ** exps[i % len(exps)]
    return X.to(torch.float32).to(torch.bfloat16)


@pytest.mark.parametrize("M,K", [(8, 4096), (8, 1024), (7300, 512)])
def test_tiny_scales_both_code_paths(cuda_device, M, K):
    """bf16 rows whose scale lies on either side of 2^-100, where the kernels
    switch from the division-free correction step to the out-of-line tie
    test with IEEE division, in the CTA-per-row form (8 rows) and the warp
    form (7300 rows, more than 48 per SM): codes and scales bit-exact."""
    X = scaled_rows(M, K, [0, -100, -101, -110, -126, 20], seed=K + M)
    check_rows(X, cuda_device)


def test_empty_rows_call(cuda_device):
    """M = 0 is a no-op (nothing launched) for the quantiser."""
    X = torch.empty((0, 64), dtype=torch.bfloat16, device=cuda_device)
    q, s = w8.quantize_act(X)
    assert q.shape == (0, 64) and s.shape == (0,)


def test_pack_weight_exact(cuda_device):
    Wq = wl.random_codes((300, 512), seed=3)
    Wp = w8.pack_weight(Wq.to(cuda_device))
    torch.cuda.synchronize()
    assert torch.equal(Wp.cpu().float(), Wq.float())


def test_near_ties_take_exact_division_f32(cuda_device):
    """Elements whose quotient x/s lies within 2^-14 of a half-integer (and
    exactly on it) with a scale that is not a power of two: the kernel must
    decide them exactly like IEEE division followed by round-half-even."""
    rng = np.random.default_rng(77)
    R, K = 64, 1024
    rows = []
    for r in range(R):
        amax = np.float32(rng.uniform(0.3, 30.0))
        s = np.float32(amax) / np.float32(127.0)
        k = rng.integers(-127, 127, size=K - 1)
        delta = rng.choice([0.0, 1e-7, -1e-7, 3e-6, -3e-6, 2.0 ** -15, -2.0 ** -15, 1e-4, -1e-4], size=K - 1)
        x = ((k + 0.5 + delta) * np.float64(s)).astype(np.float32)
        rows.append(np.concatenate([[amax], x]).astype(np.float32))
    X = np.stack(rows)
    q_ref, s_ref = oracle.quantize_rows(X)
    v = X.astype(np.float64) / s_ref[:, None].astype(np.float64)
    near = np.abs(np.abs(v - np.floor(v)) - 0.5) < 2.0 ** -14
    assert near.sum() > 1000            # the fallback is really exercised
    check_rows(torch.from_numpy(X), cuda_device)


def test_near_ties_bf16(cuda_device):
    """bf16 rows: exact ties (x = (k + 1/2) 2^e, s = 2^e; every such value has
    at most 8 significant bits, so it is a bf16 value) and a large random block
    whose quotients fall near half-integers by chance."""
    e = -5
    ks = np.arange(-127, 127) + 0.5
    tie_row = np.concatenate([[127.0], ks, np.zeros(256 - 1 - ks.size)]) * 2.0 ** e
    ties = torch.from_numpy(np.tile(tie_row, (8, 1)).astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(ties.float(), torch.from_numpy(np.tile(tie_row, (8, 1)).astype(np.float32)))
    q, s = check_rows(ties, cuda_device)
    assert s[0] == np.float32(2.0 ** e)
    assert list(q[0, 1:5]) == [round(k) for k in ks[:4]]
    g = torch.Generator().manual_seed(78)
    Xr = (torch.randn(1024, 2048, generator=g) * torch.rand(1024, 1, generator=g) * 10).to(torch.bfloat16)
    xb = oracle.bf16_bits_to_f32(bits(Xr)).astype(np.float64)
    _, s_ref = oracle.quantize_rows(bits(Xr))
    v = xb / s_ref[:, None]
    assert (np.abs(np.abs(v - np.floor(v)) - 0.5) < 2.0 ** -14).sum() > 50
    check_rows(Xr, cuda_device)
