"""Seeded synthetic inputs for the FP8 W8A8 linear.

This module only draws random numbers and stores them as bf16; it holds none of
the quantization or GEMM arithmetic, so both the CUDA path and the CPU oracle
can consume its tensors without sharing any of the method's code.

Shapes are the public layer dimensions of the models the source pages run
("Prototype FP8Linear W8A8 runtime quantization": OpenHermes-2.5-Mistral-7B;
"[Kernel] Implement fallback for FP8 channelwise using torch._scaled_mm":
Llama-3-8B-Instruct; "Fp8 Quantization Support": TinyLlama-1.1B). No model
weights or datasets are used: values are drawn from the distributions below.

Generation: numpy PCG64 seeded from a SeedSequence of (workload id, layer,
role), drawn in float32, then rounded to bf16 with torch's round-to-nearest-
even conversion. Both sides of every parity test see the same bf16 bits.
"""

from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

# roles inside one (workload, layer) seed sequence
_ROLE_A, _ROLE_W, _ROLE_BIAS, _ROLE_COLS = 0, 1, 2, 3


def rng(*key: int) -> np.random.Generator:
    """PCG64 generator for an integer key tuple."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """float32 numpy array -> contiguous bf16 CPU tensor (round-to-nearest-even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def activations_normal(M: int, K: int, key: Sequence[int], outlier_cols: int = 0,
                       outlier_scale: float = 50.0) -> torch.Tensor:
    """A ~ N(0, 1) bf16 [M, K]; `outlier_cols` seeded input channels scaled by `outlier_scale`."""
    g = rng(*key, _ROLE_A)
    a = g.standard_normal((M, K), dtype=np.float32)
    if outlier_cols and K:
        cols = rng(*key, _ROLE_COLS).choice(K, size=min(outlier_cols, K), replace=False)
        a[:, cols] *= np.float32(outlier_scale)
    return to_bf16(a)


def activations_heavy_tail(M: int, K: int, key: Sequence[int], frac: float = 0.01,
                           nu: float = 3.0) -> torch.Tensor:
    """A ~ N(0, 1) bf16 [M, K] with round(frac*K) seeded channels ~ Student-t(nu)."""
    g = rng(*key, _ROLE_A)
    a = g.standard_normal((M, K), dtype=np.float32)
    n_heavy = int(round(frac * K))
    if n_heavy:
        cols = np.sort(rng(*key, _ROLE_COLS).choice(K, size=n_heavy, replace=False))
        a[:, cols] = g.standard_t(nu, size=(M, n_heavy)).astype(np.float32)
    return to_bf16(a)


def weights_normal(N: int, K: int, key: Sequence[int], std: float = 0.02) -> torch.Tensor:
    """W ~ N(0, std^2) bf16 [N, K] (nn.Linear layout: out_features x in_features)."""
    g = rng(*key, _ROLE_W)
    w = g.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(std)
    return to_bf16(w)


def weights_row_std(N: int, K: int, key: Sequence[int], lo: float = 0.005,
                    hi: float = 0.05) -> torch.Tensor:
    """W row j ~ N(0, sigma_j^2), sigma_j ~ U(lo, hi): rows with very different ranges."""
    g = rng(*key, _ROLE_W)
    sigma = g.uniform(lo, hi, size=(N, 1)).astype(np.float32)
    w = g.standard_normal((N, K), dtype=np.float32)
    w *= sigma
    return to_bf16(w)


def bias_normal(N: int, key: Sequence[int], std: float = 0.5) -> torch.Tensor:
    """Optional bias ~ N(0, std^2) bf16 [N]."""
    return to_bf16(rng(*key, _ROLE_BIAS).standard_normal(N, dtype=np.float32) * np.float32(std))


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Layer:
    name: str
    K: int  # in_features
    N: int  # out_features


# Mistral-7B / Llama-3-8B decoder linears: hidden 4096, intermediate 14336,
# 32 query heads and 8 KV heads of 128 -> fused qkv N = 4096 + 2*1024.
LLAMA8B_LAYERS: Tuple[Layer, ...] = (
    Layer("qkv", 4096, 6144),
    Layer("o_proj", 4096, 4096),
    Layer("gate_up", 4096, 28672),
    Layer("down", 14336, 4096),
)

# TinyLlama-1.1B: hidden 2048, intermediate 5632, 32 query / 4 KV heads of 64, 22 layers.
TINYLLAMA_LAYERS: Tuple[Layer, ...] = (
    Layer("qkv", 2048, 2560),
    Layer("o_proj", 2048, 2048),
    Layer("gate_up", 2048, 11264),
    Layer("down", 5632, 2048),
)
TINYLLAMA_DEPTH = 22
TINYLLAMA_MS = (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 4096, 16384)

DECODE_MS = (1, 2, 4, 8, 15)
PREFILL_M = 16 * 1024

UNALIGNED_SHAPES = ((1, 4100, 4097), (7, 2050, 3001), (13, 1000, 1027), (15, 4096, 4095))

# workload ids (seed roots)
TINY, UNALIGNED, DECODE, PREFILL, TINYLLAMA = 1000, 1001, 1002, 1003, 1004


@dataclasses.dataclass
class Case:
    """One linear problem: bf16 A [M, K], bf16 W [N, K], optional bias, weight scale mode."""
    name: str
    a: torch.Tensor
    w: torch.Tensor
    per_channel: bool
    bias: Optional[torch.Tensor] = None

    @property
    def M(self) -> int:
        return self.a.shape[0]

    @property
    def K(self) -> int:
        return self.a.shape[1]

    @property
    def N(self) -> int:
        return self.w.shape[0]


def tiny_case() -> Case:
    """16 x 256 x 256, per-tensor scales, A ~ N(0,1), W ~ N(0, 0.02)."""
    return Case("tiny_16x256x256", activations_normal(16, 256, (TINY, 0)),
                weights_normal(256, 256, (TINY, 0)), per_channel=False)


def unaligned_cases() -> List[Case]:
    """Dimensions that are not multiples of 16; 4 input channels of A scaled x50."""
    out = []
    for i, (M, K, N) in enumerate(UNALIGNED_SHAPES):
        out.append(Case(f"unaligned_{M}x{K}x{N}",
                        activations_normal(M, K, (UNALIGNED, i), outlier_cols=4),
                        weights_normal(N, K, (UNALIGNED, i)), per_channel=False))
    return out


def decode_weight(layer_idx: int, copy: int = 0) -> torch.Tensor:
    L = LLAMA8B_LAYERS[layer_idx]
    return weights_normal(L.N, L.K, (DECODE, layer_idx, copy))


def decode_activations(M: int, layer_idx: int, step: int = 0) -> torch.Tensor:
    L = LLAMA8B_LAYERS[layer_idx]
    return activations_normal(M, L.K, (DECODE, layer_idx, 100 + M, step))


def prefill_weight(layer_idx: int, copy: int = 0) -> torch.Tensor:
    L = LLAMA8B_LAYERS[layer_idx]
    return weights_row_std(L.N, L.K, (PREFILL, layer_idx, copy))


def prefill_activations(layer_idx: int, M: int = PREFILL_M, step: int = 0) -> torch.Tensor:
    L = LLAMA8B_LAYERS[layer_idx]
    return activations_heavy_tail(M, L.K, (PREFILL, layer_idx, step))


def tinyllama_weight(depth: int, layer_idx: int) -> torch.Tensor:
    L = TINYLLAMA_LAYERS[layer_idx]
    return weights_normal(L.N, L.K, (TINYLLAMA, depth, layer_idx))


def tinyllama_activations(M: int, depth: int, layer_idx: int) -> torch.Tensor:
    L = TINYLLAMA_LAYERS[layer_idx]
    return activations_normal(M, L.K, (TINYLLAMA, depth, layer_idx, M))


# ---------------------------------------------------------------------------
# Device-drawn tensors for timing-only workloads (never compared with the oracle)
# ---------------------------------------------------------------------------

def _device_seed(key: Sequence[int]) -> int:
    return int(np.random.SeedSequence(list(key)).generate_state(1, dtype=np.uint64)[0] >> 1)


def normal_device(rows: int, cols: int, key: Sequence[int], std: float, device) -> torch.Tensor:
    """bf16 [rows, cols] ~ N(0, std^2) drawn on `device` by torch's generator seeded from `key`.
    Used where only timing matters and host generation of gigabytes would dominate the run
    (the TinyLlama sweep's 22 weight sets); parity tests use the host draws above."""
    g = torch.Generator(device=device)
    g.manual_seed(_device_seed(key))
    x = torch.empty((rows, cols), dtype=torch.float32, device=device)
    x.normal_(0.0, std, generator=g)
    return x.to(torch.bfloat16)


def tinyllama_weight_device(depth: int, layer_idx: int, device) -> torch.Tensor:
    L = TINYLLAMA_LAYERS[layer_idx]
    return normal_device(L.N, L.K, (TINYLLAMA, depth, layer_idx, 7), 0.02, device)


def tinyllama_activations_device(M: int, copy: int, layer_idx: int, device) -> torch.Tensor:
    L = TINYLLAMA_LAYERS[layer_idx]
    return normal_device(M, L.K, (TINYLLAMA, copy, layer_idx, 8), 1.0, device)
