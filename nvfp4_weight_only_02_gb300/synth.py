"""Seeded synthetic inputs for the NVFP4 weight path.

This module draws random numbers and rounds them to bf16; it holds none of the
method's arithmetic.  Both the CUDA path and the CPU oracle consume the same
bytes produced here.

Shapes stand in for the Qwen2.5 models the RL-with-NVFP4 post evaluates on
(tggo.me/sberlogasci/42740, section "Эксперименты"); no checkpoint or dataset
is used.  Noise magnitudes follow the schedule end points of the same post
(section "Метод": 1e-2 down to 5e-4).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

# Qwen2.5-shaped projection matrices (out_features, in_features)
QWEN7B_UP = (18944, 3584)
QWEN7B_DOWN = (3584, 18944)
QWEN32B_UP = (27648, 5120)
QWEN32B_DOWN = (5120, 27648)
QWEN7B_LAYER = {
    "q": (3584, 3584), "k": (512, 3584), "v": (512, 3584), "o": (3584, 3584),
    "gate": (18944, 3584), "up": (18944, 3584), "down": (3584, 18944),
}


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_weight(shape, std: float, seed: int, outlier_frac: float = 0.0,
                  outlier_mult: float = 20.0) -> np.ndarray:
    """bf16 bits of N(0, std^2), with a fraction of entries (uniform random
    positions) multiplied by outlier_mult."""
    g = rng(seed)
    w = g.standard_normal(shape, dtype=np.float32) * np.float32(std)
    if outlier_frac > 0:
        n = w.size
        idx = g.integers(0, n, size=max(1, int(n * outlier_frac)))
        w.reshape(-1)[idx] *= np.float32(outlier_mult)
    return to_bf16_bits(w)


def student_t_weight(shape, scale: float, nu: float, seed: int) -> np.ndarray:
    g = rng(seed)
    w = (g.standard_t(nu, size=shape) * scale).astype(np.float32)
    return to_bf16_bits(w)


def activations(M: int, K: int, seed: int, std: float = 1.0) -> np.ndarray:
    g = rng(seed)
    return to_bf16_bits(g.standard_normal((M, K), dtype=np.float32) * np.float32(std))


def noise_vector(K: int, sigma: float, seed: int) -> np.ndarray:
    """Multiplicative noise z = 1 + sigma * N(0,1), fp32, one per input channel."""
    g = rng(seed)
    return (1.0 + sigma * g.standard_normal(K)).astype(np.float32)


@dataclass
class LinearCase:
    name: str
    w: np.ndarray            # (N, K) bf16 bits
    x: np.ndarray            # (M, K) bf16 bits
    a: np.ndarray | None     # (r, K) bf16 bits
    b: np.ndarray | None     # (N, r) bf16 bits
    lora_scale: float
    z: np.ndarray | None     # (K,) fp32


def lora_pair(N: int, K: int, r: int, std: float, seed: int):
    g = rng(seed)
    a = to_bf16_bits(g.standard_normal((r, K), dtype=np.float32) * np.float32(std))
    b = to_bf16_bits(g.standard_normal((N, r), dtype=np.float32) * np.float32(std))
    return a, b


def single_layer_case(seed: int = 0) -> LinearCase:
    """512 x 2048 layer: W ~ N(0, 0.02^2) (seed 0), X 4 x 2048 ~ N(0,1), LoRA
    r=16 with A, B ~ N(0, 0.01^2), s = 2, noise 1 + 1e-2 N(0,1)."""
    N, K, M, r = 512, 2048, 4, 16
    w = normal_weight((N, K), 0.02, seed)
    x = activations(M, K, seed + 1)
    a, b = lora_pair(N, K, r, 0.01, seed + 2)
    z = noise_vector(K, 1e-2, seed + 3)
    return LinearCase("single_512x2048", w, x, a, b, 2.0, z)


def qwen7b_case(which: str, M: int, seed: int = 0, r: int = 32) -> LinearCase:
    """7B-shaped decode: W ~ N(0, 0.02^2) with 0.1% outliers x20, LoRA r=32
    (A, B ~ N(0, 0.01^2), s = 2), noise sigma 5e-4."""
    N, K = QWEN7B_UP if which == "up" else QWEN7B_DOWN
    w = normal_weight((N, K), 0.02, seed, outlier_frac=1e-3, outlier_mult=20.0)
    x = activations(M, K, seed + 1)
    a, b = lora_pair(N, K, r, 0.01, seed + 2)
    z = noise_vector(K, 5e-4, seed + 3)
    return LinearCase(f"qwen7b_{which}_M{M}", w, x, a, b, 2.0, z)


def qwen32b_case(which: str, M: int, seed: int = 0, r: int = 64) -> LinearCase:
    """32B-shaped decode: W = 0.02 * Student-t(nu=4), LoRA r=64, noise 5e-4."""
    N, K = QWEN32B_UP if which == "up" else QWEN32B_DOWN
    w = student_t_weight((N, K), 0.02, 4.0, seed)
    x = activations(M, K, seed + 1)
    a, b = lora_pair(N, K, r, 0.01, seed + 2)
    z = noise_vector(K, 5e-4, seed + 3)
    return LinearCase(f"qwen32b_{which}_M{M}", w, x, a, b, 2.0, z)


def small_case(M: int, N: int, K: int, r: int, seed: int, w_std=0.02, sigma=1e-2,
               with_lora=True, with_noise=True) -> LinearCase:
    w = normal_weight((N, K), w_std, seed, outlier_frac=1e-3)
    x = activations(M, K, seed + 1)
    a, b = lora_pair(N, K, r, 0.01, seed + 2) if with_lora and r > 0 else (None, None)
    z = noise_vector(K, sigma, seed + 3) if with_noise else None
    return LinearCase(f"small_{M}x{N}x{K}_r{r}", w, x, a, b, 2.0, z)
