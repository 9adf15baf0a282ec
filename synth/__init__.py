"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

This module only draws random numbers and arranges them into arrays. It holds none of
the quantisation, encoding or attention arithmetic: those live in ``oracle/`` (the CPU
checker) and in the CUDA library (the product), which never import each other.

Workload shapes follow the pages' workloads:

* LoopVQ (LoopVQ: Sub 1-bit KV Cache Quantization for Looped Transformers, research
  motivation and method step 1): KV of a looped LM whose consecutive loop steps are
  strongly correlated (adjacent-step correlation rising from 0.69 to 0.94; same channel
  across steps |r| = 0.85). We draw x_1 ~ N(0, 1) and
  x_{t+1} = rho_t x_t + sqrt(1 - rho_t^2) eps per (token, channel). Keys get a few fixed
  outlier channels scaled up (the fixed-outlier-channel structure of keys described on
  the KIVI page, "distribution evidence" section).
* KIVI (KIVI 完全拆解, "distribution evidence" section): keys N(0, 1) with fixed outlier
  channels, values N(0, 1).

Every function takes a ``numpy.random.Generator`` (PCG64) so a test is reproducible from
its seed alone.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rng",
    "rho_schedule",
    "loop_correlated",
    "outlier_channels",
    "scale_channels",
    "sample_codebooks",
    "kivi_kv",
    "gaussian",
    "random_indices",
    "bf16_round",
    "bf16_bits",
    "bf16_from_bits",
    "fp16_round",
]


def rng(seed: int) -> np.random.Generator:
    """PCG64 generator for ``seed``."""
    return np.random.Generator(np.random.PCG64(seed))


def rho_schedule(T: int, first: float = 0.69, last: float = 0.94) -> np.ndarray:
    """Correlation between loop step t and t+1 for t = 1..T-1, linear from ``first`` to ``last``.

    For T = 4 this gives 0.69, 0.815, 0.94. Pass ``first == last`` for a constant schedule
    (the long-context workload uses a constant 0.85).
    """
    if T <= 1:
        return np.zeros(0)
    if T == 2:
        return np.array([first])
    return np.linspace(first, last, T - 1)


def loop_correlated(g: np.random.Generator, T: int, n: int, D: int, rhos) -> np.ndarray:
    """Float64 array [T][n][D]: an AR(1) chain along the loop axis, unit variance per step."""
    rhos = np.asarray(rhos, dtype=np.float64)
    assert rhos.shape == (max(T - 1, 0),)
    x = np.empty((T, n, D), dtype=np.float64)
    x[0] = g.standard_normal((n, D))
    for t in range(1, T):
        r = rhos[t - 1]
        x[t] = r * x[t - 1] + np.sqrt(1.0 - r * r) * g.standard_normal((n, D))
    return x


def outlier_channels(g: np.random.Generator, D: int, k: int) -> np.ndarray:
    """``k`` distinct channel indices in [0, D), sorted."""
    return np.sort(g.choice(D, size=k, replace=False))


def scale_channels(x: np.ndarray, channels, factor: float) -> np.ndarray:
    """Copy of ``x`` with the last-axis ``channels`` multiplied by ``factor``."""
    y = np.array(x, dtype=np.float64, copy=True)
    y[..., channels] *= factor
    return y


def sample_codebooks(g: np.random.Generator, x: np.ndarray, Tc: int, G: int,
                     K: int = 256, noise_var: float = 0.01) -> np.ndarray:
    """Codebooks drawn from the data: K sampled tokens plus N(0, noise_var) noise.

    ``x`` is [T][n][D] (one layer and head). Returns float32 [NB][NG][K][G] with
    NB = T / Tc blocks and NG = D / c groups, c = G / Tc. Entry r of block b, group g is
    token tok_r's values arranged channel-major, loop-step-minor: coordinate i*Tc + m is
    channel g*c + i at 0-based loop step b*Tc + m. Any arrangement is a valid codebook;
    this one makes entries look like the vectors they will be matched against.
    """
    T, n, D = x.shape
    assert T % Tc == 0 and G % Tc == 0
    c = G // Tc
    assert D % c == 0
    NB, NG = T // Tc, D // c
    toks = g.choice(n, size=K, replace=(n < K))
    s = x[:, toks, :]                                   # [T][K][D]
    s = s.reshape(NB, Tc, K, NG, c)                     # [b][m][r][g][i]
    s = s.transpose(0, 3, 2, 4, 1).reshape(NB, NG, K, G)  # [b][g][r][i*Tc+m]
    noise = np.sqrt(noise_var) * g.standard_normal(s.shape)
    return (s + noise).astype(np.float32)


def kivi_kv(g: np.random.Generator, n: int, D: int, outliers, outlier_scale: float = 20.0):
    """(K, V) float64 [n][D]: N(0,1) with key outlier channels scaled by ``outlier_scale``."""
    k = g.standard_normal((n, D))
    k[:, outliers] *= outlier_scale
    v = g.standard_normal((n, D))
    return k, v


def gaussian(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return std * g.standard_normal(shape)


def random_indices(g: np.random.Generator, shape, K: int = 256) -> np.ndarray:
    """Uniform uint8 codeword indices."""
    return g.integers(0, K, size=shape, dtype=np.uint8)


# ---- storage-type rounding of generated inputs (round to nearest even) ----------------

def bf16_bits(x) -> np.ndarray:
    """uint16 bf16 bit patterns of ``x`` (rounded to nearest, ties to even)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    bias = ((u >> 16) & 1) + 0x7FFF
    r = ((u + bias) >> 16).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def bf16_from_bits(b) -> np.ndarray:
    """float64 values of uint16 bf16 bit patterns."""
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def bf16_round(x) -> np.ndarray:
    """``x`` rounded to bf16, returned as float64."""
    return bf16_from_bits(bf16_bits(x))


def fp16_round(x) -> np.ndarray:
    """``x`` rounded to fp16, returned as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


# ---- device-side generation for full-size workloads (same recipe, torch generator) ------

def torch_loop_correlated(gen, T: int, shape, rhos, device="cuda"):
    """Float32 tensor [T, *shape]: the loop-axis AR(1) chain of ``loop_correlated``, drawn
    with a seeded ``torch.Generator`` on ``device``."""
    import torch

    rhos = [float(r) for r in rhos]
    x = torch.empty((T, *shape), dtype=torch.float32, device=device)
    x[0].normal_(generator=gen)
    for t in range(1, T):
        r = rhos[t - 1]
        x[t] = r * x[t - 1] + (1.0 - r * r) ** 0.5 * torch.randn(shape, generator=gen, device=device)
    return x


def torch_sample_codebooks(gen, x, Tc: int, G: int, K: int = 256, noise_var: float = 0.01):
    """Device version of ``sample_codebooks``: x float [T][n][D] (one head) ->
    float32 [NB][NG][K][G], K tokens drawn with ``gen`` plus N(0, noise_var) noise."""
    import torch

    T, n, D = x.shape
    c = G // Tc
    NB, NG = T // Tc, D // c
    toks = torch.randint(0, n, (K,), generator=gen, device=x.device)
    s = x[:, toks, :].float().reshape(NB, Tc, K, NG, c).permute(0, 3, 2, 4, 1).reshape(NB, NG, K, G)
    return (s + noise_var ** 0.5 * torch.randn(s.shape, generator=gen, device=x.device)).contiguous()
