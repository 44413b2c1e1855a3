"""Seeded synthetic inputs for fused linear cross-entropy.

This module only draws random numbers and lays them out; it holds none of the
loss or gradient arithmetic, so both the CPU oracle and the CUDA path can take
their inputs from here without sharing any of the method.

The workloads stand in for the Qwen-family SFT and pre-training runs the pages
talk about (ms-swift PR #9784 "feat(sft): Add optional fused linear ce for
qwen2/qwen3 on npu", sections Background and Scope; the Qwen3.5-35B-A3B LoRA SFT
blog post, listings `load_model` and `train`).  No dataset is read: token ids are
drawn from a seeded generator with the stated distribution and mask pattern.

Every tensor is drawn in float32 on the CPU from a seeded ``torch.Generator`` and
rounded to bfloat16 with round-to-nearest-even (``Tensor.to(torch.bfloat16)``).
Both sides read the same bf16 tensors.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

IGNORE_INDEX = -100


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int             # sequences per call
    S: int             # tokens per sequence (the shift boundary)
    H: int             # hidden size
    V: int             # vocabulary size
    x_std: float       # std of the hidden states
    w_std: float       # std of the LM-head weight
    x_rms_norm: bool   # rescale each hidden row to unit RMS (RMSNorm-like)
    labels: str        # "uniform" | "zipf"
    mask: str          # "random" | "prefix" | "turn_prefix"
    mask_frac: float   # fraction of raw label positions set to IGNORE_INDEX
    shift: bool
    reduction: str     # "mean" | "sum"
    seed: int
    zipf_s: float = 1.1
    turns: int = 4     # for mask == "turn_prefix": turns per sequence

    @property
    def N(self) -> int:
        return self.B * self.S

    @property
    def flops(self) -> int:
        """Algorithmic FLOPs of one forward + backward: 2NHV forward, 6NHV backward."""
        return 8 * self.N * self.H * self.V


# The five workloads: a small one the oracle finishes in seconds, three shaped
# like the pages' Qwen2 / Qwen3 / 32K-context runs, and a wide-logit stress case.
WORKLOADS = [
    Workload("tiny", 1, 256, 256, 4096, 1.0, 0.02, False, "uniform", "random",
             0.10, False, "mean", 1000),
    Workload("qwen2_7b", 1, 8192, 3584, 152064, 1.0, 0.02, False, "uniform", "random",
             0.05, True, "mean", 1001),
    Workload("qwen3_8b", 2, 8192, 4096, 151936, 1.0, 0.02, True, "zipf", "turn_prefix",
             0.20, True, "mean", 1002),
    Workload("long_ctx", 1, 32768, 2048, 151936, 1.0, 0.02, False, "uniform", "prefix",
             0.40, True, "mean", 1003),
    Workload("stress", 1, 4096, 8192, 128256, 4.0, 0.05, False, "uniform", "random",
             0.50, False, "sum", 1004),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def get(name: str) -> Workload:
    return BY_NAME[name]


def _draw_labels(wl: Workload, g: torch.Generator, N: int, V: int) -> torch.Tensor:
    if wl.labels == "uniform":
        return torch.randint(0, V, (N,), generator=g, dtype=torch.int64)
    if wl.labels == "zipf":
        # P(rank r) proportional to r^-s over ranks 1..V; id = rank - 1, so low
        # ids are the frequent ones, as in BPE vocabularies.
        ranks = torch.arange(1, V + 1, dtype=torch.float64)
        cdf = torch.cumsum(ranks.pow(-wl.zipf_s), 0)
        u = torch.rand(N, generator=g, dtype=torch.float64) * cdf[-1]
        return torch.searchsorted(cdf, u).clamp_(max=V - 1).to(torch.int64)
    raise ValueError(wl.labels)


def _mask_positions(wl: Workload, g: torch.Generator, labels: torch.Tensor, B: int,
                    S: int) -> None:
    N = labels.numel()
    if wl.mask == "random":
        k = int(wl.mask_frac * N)
        idx = torch.randperm(N, generator=g)[:k]
        labels[idx] = IGNORE_INDEX
    elif wl.mask == "prefix":
        # the first mask_frac of every sequence (a long prompt before the answer)
        k = int(wl.mask_frac * S)
        labels.view(B, S)[:, :k] = IGNORE_INDEX
    elif wl.mask == "turn_prefix":
        # each sequence is `turns` chat turns; the prompt at the start of each
        # turn is masked, as SFT collators do.
        T = S // wl.turns
        k = round(wl.mask_frac * T)
        labels.view(B, wl.turns, T)[:, :, :k] = IGNORE_INDEX
    else:
        raise ValueError(wl.mask)


def make_inputs(wl: Workload, *, N: Optional[int] = None, H: Optional[int] = None,
                V: Optional[int] = None, seed: Optional[int] = None):
    """Return (X bf16 [N,H], W bf16 [V,H], labels int64 [N]) on the CPU.

    N, H, V and seed may be overridden to get smaller cases with the same
    distributions; N must then stay a multiple of the sequence count B.
    """
    N = wl.N if N is None else N
    H = wl.H if H is None else H
    V = wl.V if V is None else V
    B = wl.B if N % wl.B == 0 else 1
    S = N // B
    g = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    X = torch.randn(N, H, generator=g, dtype=torch.float32) * wl.x_std
    if wl.x_rms_norm:
        X = X / X.pow(2).mean(dim=1, keepdim=True).sqrt()
    W = torch.randn(V, H, generator=g, dtype=torch.float32) * wl.w_std
    labels = _draw_labels(wl, g, N, V)
    _mask_positions(wl, g, labels, B, S)
    return X.to(torch.bfloat16), W.to(torch.bfloat16), labels


def random_case(N: int, H: int, V: int, *, seed: int, x_std: float = 1.0,
                w_std: float = 0.05, ignore_frac: float = 0.1,
                ignore_index: int = IGNORE_INDEX):
    """A small uniform case of arbitrary shape for edge-case tests."""
    g = torch.Generator().manual_seed(seed)
    X = (torch.randn(N, H, generator=g) * x_std).to(torch.bfloat16)
    W = (torch.randn(V, H, generator=g) * w_std).to(torch.bfloat16)
    labels = torch.randint(0, V, (N,), generator=g, dtype=torch.int64)
    k = int(ignore_frac * N)
    if k:
        labels[torch.randperm(N, generator=g)[:k]] = ignore_index
    return X, W, labels
