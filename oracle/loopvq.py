"""LoopVQ: loop-axis coupled vectors, nearest-codeword encode, dequantize and decode
attention over the sink / index-page / recent cache (oracle; test infrastructure only).

Source: "LoopVQ: Sub 1-bit KV Cache Quantization for Looped Transformers" (paper digest),
background on vector quantization, method steps 1, 4 and 5, Figure 3, Algorithm 1 and
Figure 5. Notation follows the page: T loop steps (1-based t), blocks of Tc consecutive
steps (beta = block index), G coupled dimensions, c = G / Tc channels per codeword,
NG = D / c index groups per token, head and block, K = 256 codebook entries.

Readings where the page is silent or garbled, taken here:
* The coupled-vector map is printed as "channel g_{c+i}"; it is read as channel g*c + i.
* Keys and values have separate codebooks and separate indices of the same structure.
* Ties in the argmin go to the lowest index.
* Tokens [0, sink) stay bf16 (sink), then whole 8-token index pages, then the recent
  tokens in bf16; after a prefill of length L the recent window holds
  W + ((L - sink - W) mod 8) tokens.
"""
from __future__ import annotations

import numpy as np

from .attention import rope, softmax_attention


def step_to_block(t: int, Tc: int):
    """1-based loop step t -> (beta, m): block beta = (t-1) // Tc, offset m = (t-1) % Tc."""
    assert t >= 1
    return (t - 1) // Tc, (t - 1) % Tc


def coupled_vectors(x: np.ndarray, beta: int, Tc: int, G: int) -> np.ndarray:
    """Coupled vectors of block ``beta`` for every token and group.

    ``x`` is [T][n][D] (axis 0 is the 0-based loop step, i.e. step t is x[t-1]).
    Returns z [n][NG][G] with, for i < c and m < Tc (method step 1, Figure 3):
        z[j][g][i*Tc + m] = value of channel g*c + i at loop step beta*Tc + m + 1.
    """
    T, n, D = x.shape
    assert G % Tc == 0
    c = G // Tc
    assert D % c == 0 and (beta + 1) * Tc <= T
    NG = D // c
    z = np.empty((n, NG, G), dtype=np.float64)
    for g in range(NG):
        for i in range(c):
            for m in range(Tc):
                step = beta * Tc + m + 1            # 1-based loop step
                z[:, g, i * Tc + m] = x[step - 1, :, g * c + i]
    return z


def squared_distances(z: np.ndarray, cb: np.ndarray) -> np.ndarray:
    """d[j][r] = sum_k (z[j][k] - e_r[k])^2 in fp64 by brute force. z [n][G], cb [K][G]."""
    z = np.asarray(z, np.float64)
    e = np.asarray(cb, np.float64)
    return ((z[:, None, :] - e[None, :, :]) ** 2).sum(axis=-1)


def nearest_codeword(z: np.ndarray, cb: np.ndarray):
    """a(z) = argmin_r ||z - e_r||^2 (background, "vector quantization and codebooks").

    Returns (idx [n] int64, d [n][K] fp64). Exact ties go to the lowest r (numpy's argmin
    returns the first minimum).
    """
    d = squared_distances(z, cb)
    return np.argmin(d, axis=1), d


def tie_mask(d: np.ndarray, rel: float = 1e-6) -> np.ndarray:
    """Candidates r whose distance is within ``rel`` (relative) of the row minimum.

    An encoder that picks any of them is counted as a tie-match, not a mismatch.
    """
    dmin = d.min(axis=1, keepdims=True)
    return d <= dmin * (1.0 + rel)


def encode_block(x: np.ndarray, cb_block: np.ndarray, beta: int, Tc: int, rel: float = 1e-6):
    """Encode every token of block ``beta`` (method step 4).

    ``cb_block`` is [NG][K][G] (the codebooks B_{beta,l,h,g} of one layer and head).
    Returns (idx [n][NG] uint8, ties [n][NG][K] bool).
    """
    NG, K, G = cb_block.shape
    z = coupled_vectors(x, beta, Tc, G)
    n = z.shape[0]
    idx = np.empty((n, NG), dtype=np.uint8)
    ties = np.empty((n, NG, K), dtype=bool)
    for g in range(NG):
        a, d = nearest_codeword(z[:, g, :], cb_block[g])
        idx[:, g] = a
        ties[:, g, :] = tie_mask(d, rel)
    return idx, ties


def dequantize(idx: np.ndarray, cb_block: np.ndarray, m: int, Tc: int) -> np.ndarray:
    """Reconstruct the vectors of in-block loop step m from shared indices (method step 5,
    Figure 3: step t reads the indices through its own slice B_t of the codebook).

    idx [n][NG], cb_block [NG][K][G]. Returns [n][D] with, by explicit lookup,
        out[j][g*c + i] = cb_block[g][idx[j][g]][i*Tc + m].
    """
    NG, K, G = cb_block.shape
    c = G // Tc
    idx = np.asarray(idx).astype(np.int64)
    n = idx.shape[0]
    out = np.empty((n, NG * c), dtype=np.float64)
    for g in range(NG):
        rows = np.asarray(cb_block[g], np.float64)[idx[:, g]]     # e_{idx[j][g]} for every j
        for i in range(c):
            out[:, g * c + i] = rows[:, i * Tc + m]
    return out


def prefill_split(L: int, sink: int = 8, recent: int = 64, page: int = 8):
    """(n_sink, n_pages, n_recent) after a prefill of L tokens (method step 4, Figure 5).

    The first ``sink`` tokens stay bf16; the last ``recent`` tokens plus the remainder that
    does not fill a whole page stay bf16; the rest fill 8-token index pages.
    """
    n_sink = min(sink, L)
    n_pages = max(0, (L - sink - recent) // page)
    return n_sink, n_pages, L - n_sink - page * n_pages


def cache_positions(seq_len: int, n_pages: int, sink: int = 8, page: int = 8):
    """(bf16 positions, quantized positions) of a request's cache, in position order."""
    n_sink = min(sink, seq_len)
    q0, q1 = sink, sink + page * n_pages
    bf = np.concatenate([np.arange(0, n_sink), np.arange(q1, seq_len)]).astype(np.int64)
    return bf, np.arange(q0, q1, dtype=np.int64)


def decode_attention(q, t: int, Tc: int, seq_len: int, n_pages: int,
                     idx_k, idx_v, cb_k_block, cb_v_block, win_k, win_v,
                     rope_base: float = 1.0e4, sink: int = 8, page: int = 8) -> np.ndarray:
    """Decode attention of one (request, head) at loop step t, in fp64.

    q: [D] pre-RoPE query of the newest token, which sits at position seq_len - 1.
    idx_k, idx_v: [n_pages * page][NG] indices of the quantized tokens (positions
        sink .. sink + page*n_pages - 1) for block beta(t).
    cb_k_block, cb_v_block: [NG][K][G] codebooks of block beta(t).
    win_k, win_v: [seq_len][D] pre-RoPE bf16 values at step t; only the sink and recent
        positions are read.

    Keys are rebuilt by lookup (quantized) or read (bf16), every key and the query are
    RoPE-rotated at their positions (keys are cached pre-RoPE: background "RoPE" and
    method step 1), and one softmax with scale 1/sqrt(D) runs over all keys (method step 5
    merges the partials of the quantized pages and of the bf16 window exactly, so the result
    is the full softmax).
    """
    beta, m = step_to_block(t, Tc)
    q = np.asarray(q, np.float64)
    D = q.shape[0]
    bf_pos, q_pos = cache_positions(seq_len, n_pages, sink, page)
    assert len(q_pos) == np.asarray(idx_k).shape[0] == np.asarray(idx_v).shape[0]
    Kq = dequantize(np.asarray(idx_k), cb_k_block, m, Tc)
    Vq = dequantize(np.asarray(idx_v), cb_v_block, m, Tc)
    win_k = np.asarray(win_k, np.float64)
    win_v = np.asarray(win_v, np.float64)
    pos = np.concatenate([bf_pos, q_pos])
    K = np.concatenate([win_k[bf_pos], Kq], axis=0)
    V = np.concatenate([win_v[bf_pos], Vq], axis=0)
    qr = rope(q, seq_len - 1, rope_base)
    Kr = rope(K, pos, rope_base)
    return softmax_attention(qr, Kr, V, 1.0 / np.sqrt(D))
