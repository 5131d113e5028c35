"""Seeded synthetic bf16 inputs with the shapes and value distributions of the
workloads the FP8 pages measure on (Llama 3 8B / 70B / 3.1 405B layer shapes,
"mastering FP8 LLM training 1.5x speedup", test setup and Figs. 1-4).

This module holds no quantization arithmetic: it only draws numbers.  Both
the CUDA library's tests and the oracle's tests take their inputs from here.

Every tensor is drawn as fp32 from numpy's PCG64 generator seeded with the
stated seed, optionally modified (outlier columns / elements, magnitude
walk) in fp32, then cast to bf16 with round-to-nearest-even by torch.
"""
from __future__ import annotations

import math

import numpy as np
import torch


def normal_f32(shape, seed: int, std: float = 1.0) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(seed))
    x = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def to_bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def normal_bf16(shape, seed: int, std: float = 1.0) -> torch.Tensor:
    return to_bf16(normal_f32(shape, seed, std))


def outlier_columns(cols: int, frac: float, seed: int) -> np.ndarray:
    """Indices of round(frac * cols) columns picked by a seeded permutation."""
    n = int(round(frac * cols))
    g = np.random.Generator(np.random.PCG64(seed))
    return np.sort(g.permutation(cols)[:n])


def with_outlier_columns(x: np.ndarray, frac: float, factor: float, seed: int) -> np.ndarray:
    cols = outlier_columns(x.shape[1], frac, seed)
    x[:, cols] *= np.float32(factor)
    return x


def with_outlier_elements(x: np.ndarray, frac: float, factor: float, seed: int) -> np.ndarray:
    flat = x.reshape(-1)
    n = max(1, int(round(frac * flat.size)))
    g = np.random.Generator(np.random.PCG64(seed))
    idx = g.choice(flat.size, size=n, replace=False)
    flat[idx] *= np.float32(factor)
    return x


# ------------------------------------------------------------- workloads

def pertensor_256(seed_a: int = 0, seed_b: int = 1):
    """A, B [256, 256] ~ N(0, 1): the per-tensor current-scaling case."""
    return normal_bf16((256, 256), seed_a), normal_bf16((256, 256), seed_b)


def llama8b_up_proj(tokens: int = 4096, hidden: int = 4096, ffn: int = 14336):
    """Blockwise case: X [tokens, hidden] ~ N(0,1) with 1% of its columns x100
    (outlier channels, column pick seed 2); W [ffn, hidden] ~ N(0, 0.02^2)."""
    x = with_outlier_columns(normal_f32((tokens, hidden), 0), 0.01, 100.0, 2)
    return to_bf16(x), normal_bf16((ffn, hidden), 1, 0.02)


def llama8b_mlp(tokens: int = 8192, hidden: int = 4096, ffn: int = 14336):
    """MXFP8 case: X [tokens, hidden] ~ N(0,1), W [ffn, hidden] ~ N(0, 0.02^2),
    dY [tokens, ffn] ~ N(0, 1e-4^2)."""
    return (normal_bf16((tokens, hidden), 0), normal_bf16((ffn, hidden), 1, 0.02),
            normal_bf16((tokens, ffn), 2, 1e-4))


DELAYED_SIGMA = (1.0, 0.02, 1e-4)     # X, W, dY


def delayed_magnitudes(steps: int = 32, walk_sigma: float = 0.3, spike_step: int = 20,
                       spike: float = 50.0) -> np.ndarray:
    """[steps, 3] multipliers of the X / W / dY base sigmas: a lognormal random
    walk m_t = m_{t-1} * exp(walk_sigma * z_t), z_t ~ N(0,1) drawn with seed
    1000 * (i + 1) + t, m_0 = 1, with step spike_step multiplied by spike."""
    m = np.ones((steps, 3), dtype=np.float64)
    for i in range(3):
        cur = 1.0
        for t in range(steps):
            if t > 0:
                z = float(np.random.Generator(np.random.PCG64(1000 * (i + 1) + t)).standard_normal())
                cur = cur * math.exp(walk_sigma * z)
            m[t, i] = cur
    m[spike_step, :] *= spike
    return m


def llama70b_ffn_bases(tokens: int = 4096, hidden: int = 8192, ffn: int = 28672):
    """Delayed-scaling case: the fp32 N(0,1) base tensors X [tokens, hidden],
    W [ffn, hidden], dY [tokens, ffn], seeds 0, 1, 2."""
    shapes = ((tokens, hidden), (ffn, hidden), (tokens, ffn))
    return tuple(torch.from_numpy(normal_f32(shapes[i], i)) for i in range(3))


def llama70b_ffn_step(t: int, bases, mags: np.ndarray | None = None):
    """Step t of the delayed-scaling case: each base tensor times its sigma
    (1, 0.02, 1e-4) times the step's walk multiplier, cast to bf16."""
    if mags is None:
        mags = delayed_magnitudes()
    return tuple((bases[i] * float(DELAYED_SIGMA[i] * mags[t, i])).to(torch.bfloat16) for i in range(3))


def sweep_tensor(mib: int, cols: int = 4096, seed: int = 5) -> torch.Tensor:
    """Quantize sweep: a bf16 tensor of `mib` MiB shaped [n / cols, cols],
    N(0,1) with 0.1% of the elements x1000 at seeded positions."""
    n = mib * (1 << 20) // 2
    x = normal_f32((n // cols, cols), seed)
    return to_bf16(with_outlier_elements(x, 0.001, 1000.0, seed + 1))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The uint16 bit patterns of a bf16 tensor (CPU copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
