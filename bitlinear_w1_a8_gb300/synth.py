"""Seeded synthetic inputs for the BitLinear workloads.

This module holds no arithmetic of the method: it only draws random numbers
(torch CPU generators, fixed seeds) in the shapes, scales and outlier
structure of the BitNet-3B / 1.3B workloads, so that the CUDA library and the
CPU oracle can be fed the same bytes.  Shapes follow the model tables of the
"Hesper.Models.BitNet" page (section "Model Configurations": dim 2560, FFN
10240, vocabulary 50000 for 3B; dim 2048, FFN 8192 for 1.3B).
"""
from __future__ import annotations

import torch

# BitNet-3B and 1.3B dimensions ("Model Configurations").
DIM_3B, FFN_3B, VOCAB, LAYERS_3B = 2560, 10240, 50000, 32
DIM_1B3, FFN_1B3 = 2048, 8192

WEIGHT_STD = 0.02
OUTLIER_FRACTION = 0.01
OUTLIER_FACTOR = 20.0


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, seed: int) -> torch.Tensor:
    """fp32 N(0, std^2) on the CPU, drawn from torch.Generator(seed)."""
    return torch.randn(*shape, generator=_gen(seed), dtype=torch.float32) * std


def normal_cuda(shape, std: float, seed: int, device) -> torch.Tensor:
    """fp32 N(0, std^2) drawn on a CUDA device from a seeded CUDA generator (for
    workloads too large to draw on the CPU; deterministic for a given device type
    and torch version)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randn(*shape, generator=g, dtype=torch.float32, device=device) * std


def uniform(shape, lo: float, hi: float, seed: int) -> torch.Tensor:
    """fp32 U(lo, hi) on the CPU."""
    return torch.rand(*shape, generator=_gen(seed), dtype=torch.float32) * (hi - lo) + lo


def weight(N: int, K: int, seed: int) -> torch.Tensor:
    """A [N, K] fp32 weight matrix ~ N(0, 0.02^2) (out features x in features)."""
    return normal((N, K), WEIGHT_STD, seed)


def outlier_channels(K: int, seed: int, fraction: float = OUTLIER_FRACTION) -> torch.Tensor:
    """The first round(fraction*K) entries of a seeded permutation of range(K)."""
    n = int(round(fraction * K))
    return torch.randperm(K, generator=_gen(seed))[:n]


def activations(M: int, K: int, seed: int, outlier_seed: int | None = None,
                factor: float = OUTLIER_FACTOR) -> torch.Tensor:
    """[M, K] fp32 ~ N(0, 1); if outlier_seed is given, 1% of the channels
    (the same channels in every row) are multiplied by `factor`."""
    x = torch.randn(M, K, generator=_gen(seed), dtype=torch.float32)
    if outlier_seed is not None:
        idx = outlier_channels(K, outlier_seed)
        x[:, idx] *= factor
    return x


# Seeds of the workloads (one per tensor, fixed).
SEEDS = {
    "small": {"W": 0, "x": 1},
    "decode": {"W_up_shape": 10, "W_down_shape": 11, "x": 12, "outliers": 13},
    "weight_set": {"base": 1000, "lm_head": 2000, "x": 3},
    "prefill": {"W_up_shape": 20, "W_down_shape": 21, "x": 22},
    "ffn_1b3": {"norm": 30, "subnorm": 31, "gate": 32, "up": 33, "down": 34, "x": 35},
}


def weight_set_seed(layer: int, proj: int) -> int:
    """Seed of projection `proj` (0..6 = q,k,v,o,gate,up,down) of `layer`."""
    return SEEDS["weight_set"]["base"] + 8 * layer + proj
