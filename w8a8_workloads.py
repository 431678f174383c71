"""Seeded synthetic inputs for the W8A8 linear layer.

This module holds no arithmetic of the method: it only draws random tensors
with the shapes and value distributions of the workloads below, on the CPU,
with ``torch.Generator`` so that every consumer (tests, bench, smoke check)
sees identical inputs.  Both the CUDA path and the CPU oracle are fed from
here; neither is imported by it.

Workloads (transformer-branch projections of a joint video/audio generator;
activations X [M, K], weights W [N, K] as in a linear layer, bias [N]):

  tiny      X f32 [64, 256] ~ N(0,1); W f32 [128, 256] ~ N(0, 0.02); bias f32 ~ N(0, 0.01)
  video     X bf16 [6144, 4096] ~ N(0,1) with 1 % of the K columns scaled x20
            (outlier channels); W bf16 [4096, 4096] ~ N(0, 0.02); bias bf16 ~ N(0, 0.01)
  mlp_up    X bf16 [6144, 4096] (outliers as video) -> W [16384, 4096]
  mlp_down  X bf16 [6144, 16384] (outliers as video) -> W [4096, 16384]
  hires_n4k X bf16 [28672, 4096] (outliers) -> W [4096, 4096]
  hires_n16k X bf16 [28672, 4096] (outliers) -> W [16384, 4096]
  audio_*   X bf16 [126 | 1001, 2048] ~ N(0,1), no outliers, last row all zero;
            W bf16 [2048 | 8192, 2048]

Recipe for one case, seed s: g = torch.Generator().manual_seed(s); draw X, then
W, then bias, then (if outliers) randperm(K)[:round(0.01 K)] as the outlier
columns; all draws in float32, the outlier columns multiplied by 20 in float32,
then the whole tensor cast to the case dtype.  Seeds: tiny 0, video 1,
mlp_up 2, mlp_down 3, hires_n4k 4, hires_n16k 5, audio_* 6..9.
"""
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Case:
    name: str
    M: int
    K: int
    N: int
    dtype: torch.dtype          # of X, W and bias
    outliers: bool
    zero_last_row: bool
    seed: int

    @property
    def ops(self) -> int:
        """Integer multiply-adds counted as two operations: 2*M*N*K."""
        return 2 * self.M * self.N * self.K


CASES = {
    "tiny": Case("tiny", 64, 256, 128, torch.float32, False, False, 0),
    "video": Case("video", 6144, 4096, 4096, torch.bfloat16, True, False, 1),
    "mlp_up": Case("mlp_up", 6144, 4096, 16384, torch.bfloat16, True, False, 2),
    "mlp_down": Case("mlp_down", 6144, 16384, 4096, torch.bfloat16, True, False, 3),
    "hires_n4k": Case("hires_n4k", 28672, 4096, 4096, torch.bfloat16, True, False, 4),
    "hires_n16k": Case("hires_n16k", 28672, 4096, 16384, torch.bfloat16, True, False, 5),
    "audio_m126_n2048": Case("audio_m126_n2048", 126, 2048, 2048, torch.bfloat16, False, True, 6),
    "audio_m126_n8192": Case("audio_m126_n8192", 126, 2048, 8192, torch.bfloat16, False, True, 7),
    "audio_m1001_n2048": Case("audio_m1001_n2048", 1001, 2048, 2048, torch.bfloat16, False, True, 8),
    "audio_m1001_n8192": Case("audio_m1001_n8192", 1001, 2048, 8192, torch.bfloat16, False, True, 9),
}

# The five workload groups in the order they are listed above.
GROUPS = {
    "tiny": ["tiny"],
    "video": ["video"],
    "mlp_pair": ["mlp_up", "mlp_down"],
    "hires": ["hires_n4k", "hires_n16k"],
    "audio": ["audio_m126_n2048", "audio_m126_n8192", "audio_m1001_n2048", "audio_m1001_n8192"],
}


def make(case, M: int = None, N: int = None, K: int = None, seed: int = None):
    """Draw (X, W, bias) for a case on the CPU.  M/N/K/seed override the
    case's own (used for reduced-size parity runs of the same recipe)."""
    if isinstance(case, str):
        case = CASES[case]
    M = case.M if M is None else M
    N = case.N if N is None else N
    K = case.K if K is None else K
    g = torch.Generator().manual_seed(case.seed if seed is None else seed)
    X = torch.randn(M, K, generator=g, dtype=torch.float32)
    W = torch.randn(N, K, generator=g, dtype=torch.float32) * 0.02
    bias = torch.randn(N, generator=g, dtype=torch.float32) * 0.01
    if case.outliers:
        n_out = int(round(0.01 * K))
        cols = torch.randperm(K, generator=g)[:n_out]
        X[:, cols] *= 20.0
    if case.zero_last_row:
        X[M - 1].zero_()
    return X.to(case.dtype), W.to(case.dtype), bias.to(case.dtype)


def random_codes(shape, seed: int, low: int = -127, high: int = 127) -> torch.Tensor:
    """Uniform INT8 codes in [low, high] (inclusive), drawn on the CPU."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(low, high + 1, shape, generator=g, dtype=torch.int16).to(torch.int8)
