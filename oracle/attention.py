"""Full-softmax decode attention, RoPE and the split/logsumexp merge, in fp64 (oracle).

Test infrastructure only.
"""
from __future__ import annotations

import numpy as np


def rope_frequencies(D: int, base: float = 1.0e4) -> np.ndarray:
    """theta_i = base^(-2i/D) for i in [0, D/2), fp64.

    The pages do not give the RoPE convention. Reading used here: the rotate-half pairing
    (channel i with channel i + D/2) with the usual base of 1e4 (LoopVQ page, background
    "RoPE": keys are rotated by an angle that depends on their position).
    """
    i = np.arange(D // 2, dtype=np.float64)
    return base ** (-2.0 * i / D)


def rope(x: np.ndarray, pos, base: float = 1.0e4) -> np.ndarray:
    """Rotate the last axis of ``x`` by position ``pos`` (scalar or array broadcast over rows).

    Pair (i, i + D/2) is turned by pos * theta_i:
        y_i       = x_i cos - x_{i+D/2} sin
        y_{i+D/2} = x_{i+D/2} cos + x_i sin
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_frequencies(D, base)
    c, s = np.cos(ang), np.sin(ang)
    lo, hi = x[..., :h], x[..., h:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def softmax_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """o = softmax(scale * K q) V over every row of K and V, in fp64.

    One softmax over the whole key set: the KIVI page (core design, the note on eq. (3))
    stresses that the quantized and full-precision segments are normalised together.
    """
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    if K.shape[0] == 0:
        return np.zeros(V.shape[1])
    s = scale * (K @ q)
    p = np.exp(s - s.max())
    return (p @ V) / p.sum()


def partial_softmax(q, K, V, scale):
    """(m, l, o_unnormalised) of one split: m = max score, l = sum exp(s - m), o = sum exp(s - m) v."""
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    if K.shape[0] == 0:
        return -np.inf, 0.0, np.zeros(V.shape[1])
    s = scale * (K @ q)
    m = s.max()
    p = np.exp(s - m)
    return m, p.sum(), p @ V


def lse_merge(parts) -> np.ndarray:
    """Exact merge of split partials (Flash-Decoding, as the LoopVQ page describes it in the
    background on SGLang / Flash-Decoding and in method step 5):
        M = max_s m_s,  L = sum_s l_s e^{m_s - M},  o = (sum_s e^{m_s - M} o_s) / L.
    """
    ms = np.array([p[0] for p in parts], dtype=np.float64)
    M = ms.max()
    w = np.where(np.isfinite(ms), np.exp(ms - M), 0.0)
    L = sum(wi * p[1] for wi, p in zip(w, parts))
    o = sum(wi * p[2] for wi, p in zip(w, parts))
    return o / L


def split_attention(q, K, V, scale, cuts) -> np.ndarray:
    """Attention computed as partials over the row ranges between ``cuts`` and merged."""
    edges = [0] + list(cuts) + [K.shape[0]]
    parts = [partial_softmax(q, K[a:b], V[a:b], scale) for a, b in zip(edges[:-1], edges[1:])]
    return lse_merge(parts)
