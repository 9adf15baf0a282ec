"""KIVI: asymmetric 2- or 4-bit group quantization (keys per channel, values per token), its
dequantization, decode attention over the quantized + fp16 residual cache, grouped-query
head mapping and the streaming cache of Algorithm 1 (oracle; test infrastructure only).

Source: "KIVI 完全拆解：非对称 2-bit KV Cache 量化" (walkthrough of the KIVI paper):
the quantize / dequantize formula (section on per-token and per-channel quantization),
the grouped + residual cache, eq. (3) and Algorithm 1 (core design section), the memory
accounting, the configurable bit widths and GQA (implementation section).

Readings where the page is silent, taken here:
* The scale splits [min, max] evenly: s = (max - min) / (2^b - 1); the zero-point is
  z = -min / s, kept as fp16 like the scale, so that X_hat = s * (q - z) is the printed
  dequantization. A group whose fp16 scale rounds to 0 (all values equal) uses s = 1.
* The arithmetic is a fixed fp32 sequence (IEEE division, separate add, round half to
  even) so that an encoder that follows it reproduces the codes bit for bit.
* Keys are grouped over 32 consecutive tokens of one channel, values over 32 consecutive
  channels of one token. Codes are logical integers here; the byte packing belongs to
  the storage format, not to the arithmetic.
* Keys are taken as already rotated (KIVI quantizes post-RoPE keys), so no RoPE here.
"""
from __future__ import annotations

import numpy as np

from .attention import softmax_attention


def quantize_group(x, bits: int = 2):
    """Quantize one group of fp16 values.

    Returns (codes int64 [n], s16 np.float16, z16 np.float16). In fp32:
        s   = (max - min) / (2^b - 1)
        s16 = fp16(s), replaced by 1 when it is 0
        z16 = fp16(-min / s16)
        q   = clamp(rint(x / s16 + z16), 0, 2^b - 1)
    """
    x32 = np.asarray(x, dtype=np.float16).astype(np.float32)
    levels = np.float32(2 ** bits - 1)
    mn = x32.min()
    mx = x32.max()
    s = np.float32(np.float32(mx - mn) / levels)
    s16 = np.float16(s)
    if s16 == np.float16(0.0):
        s16 = np.float16(1.0)
    z16 = np.float16(np.float32(-mn) / np.float32(s16))
    t = np.float32(x32 / np.float32(s16))          # fp32 IEEE division, rounded
    t = np.float32(t + np.float32(z16))             # fp32 add, rounded (no fused multiply-add)
    q = np.clip(np.rint(t), 0, 2 ** bits - 1).astype(np.int64)   # rint: round half to even
    return q, s16, z16


def dequantize_group(q, s16, z16) -> np.ndarray:
    """X_hat = s * (q - z) in fp64 from the stored fp16 scale and zero-point."""
    return float(s16) * (np.asarray(q, np.float64) - float(z16))


def quantize_keys(K, group: int = 32, bits: int = 2):
    """Per-channel key quantization over groups of ``group`` consecutive tokens.

    K: [n][D] fp16 values, n a multiple of ``group``.
    Returns codes [n][D], scale [n/group][D] fp16, zero [n/group][D] fp16.
    """
    K = np.asarray(K, dtype=np.float16)
    n, D = K.shape
    assert n % group == 0
    codes = np.empty((n, D), dtype=np.int64)
    scale = np.empty((n // group, D), dtype=np.float16)
    zero = np.empty((n // group, D), dtype=np.float16)
    for gi in range(n // group):
        for ch in range(D):
            rows = slice(gi * group, (gi + 1) * group)
            q, s16, z16 = quantize_group(K[rows, ch], bits)
            codes[rows, ch] = q
            scale[gi, ch] = s16
            zero[gi, ch] = z16
    return codes, scale, zero


def quantize_values(V, group: int = 32, bits: int = 2):
    """Per-token value quantization over groups of ``group`` consecutive channels.

    V: [n][D] fp16 values, D a multiple of ``group``.
    Returns codes [n][D], scale [n][D/group] fp16, zero [n][D/group] fp16.
    """
    V = np.asarray(V, dtype=np.float16)
    n, D = V.shape
    assert D % group == 0
    codes = np.empty((n, D), dtype=np.int64)
    scale = np.empty((n, D // group), dtype=np.float16)
    zero = np.empty((n, D // group), dtype=np.float16)
    for j in range(n):
        for gi in range(D // group):
            cols = slice(gi * group, (gi + 1) * group)
            q, s16, z16 = quantize_group(V[j, cols], bits)
            codes[j, cols] = q
            scale[j, gi] = s16
            zero[j, gi] = z16
    return codes, scale, zero


def dequantize_keys(codes, scale, zero, group: int = 32) -> np.ndarray:
    """Token j, channel ch: scale[j // group][ch] * (codes[j][ch] - zero[j // group][ch])."""
    codes = np.asarray(codes, np.float64)
    n, D = codes.shape
    out = np.empty((n, D), dtype=np.float64)
    for j in range(n):
        gi = j // group
        out[j] = scale[gi].astype(np.float64) * (codes[j] - zero[gi].astype(np.float64))
    return out


def dequantize_values(codes, scale, zero, group: int = 32) -> np.ndarray:
    """Token j, channel ch: scale[j][ch // group] * (codes[j][ch] - zero[j][ch // group])."""
    codes = np.asarray(codes, np.float64)
    n, D = codes.shape
    ch_group = np.arange(D) // group
    out = np.empty((n, D), dtype=np.float64)
    for j in range(n):
        s = scale[j].astype(np.float64)[ch_group]
        z = zero[j].astype(np.float64)[ch_group]
        out[j] = s * (codes[j] - z)
    return out


def decode_attention(q, k_codes, k_scale, k_zero, v_codes, v_scale, v_zero,
                     k_resid, v_resid, group: int = 32) -> np.ndarray:
    """Decode attention of one (request, head) over the grouped + residual cache (eq. (3)).

    A_g = q Q(X_Kg)^T and A_r = q X_Kr^T are concatenated, one softmax (scale 1/sqrt(D))
    runs over the concatenation, and the output is A_g Q(X_Vg) + A_r X_Vr.
    """
    q = np.asarray(q, np.float64)
    D = q.shape[0]
    Kg = dequantize_keys(k_codes, k_scale, k_zero, group) if len(k_codes) else np.zeros((0, D))
    Vg = dequantize_values(v_codes, v_scale, v_zero, group) if len(v_codes) else np.zeros((0, D))
    K = np.concatenate([Kg, np.asarray(k_resid, np.float64).reshape(-1, D)], axis=0)
    V = np.concatenate([Vg, np.asarray(v_resid, np.float64).reshape(-1, D)], axis=0)
    return softmax_attention(q, K, V, 1.0 / np.sqrt(D))


# ------------------------------------------------------------------ grouped-query attention

def kv_head(h_q: int, n_q_heads: int, n_kv_heads: int) -> int:
    """KV head read by query head ``h_q`` under grouped-query attention.

    KIVI page, implementation section: the code base gained GQA support (the Llama-3
    family). Reading: the usual GQA layout, where each run of n_q_heads / n_kv_heads
    consecutive query heads shares one KV head, so query head h reads KV head
    h // (n_q_heads / n_kv_heads). With n_q_heads == n_kv_heads this is multi-head attention.
    """
    assert n_q_heads % n_kv_heads == 0 and 0 <= h_q < n_q_heads
    return h_q // (n_q_heads // n_kv_heads)


# ------------------------------------------------------------------ streaming (Algorithm 1)

class KiviStream:
    """The cache of one (request, KV head) as the page's Algorithm 1 builds it.

    KIVI page, core design section and Algorithm 1: the prefill quantizes all but the
    last R tokens (keys per channel in groups of G tokens, values per token) and keeps the
    last R in fp16; each decode token enters the fp16 residuals; a full key residual is
    quantized whole and appended to the grouped keys; the value window keeps the newest R
    tokens and quantizes the token that falls out of it.

    Readings where the pseudo-code leaves a step open:
    * Key flush timing. The prefill leaves R keys in the residual, and the pseudo-code's
      test "len == R" after appending would then never fire. Taken here: a key residual
      that already holds R tokens when a new token arrives is quantized and appended to the
      grouped keys, and the new token starts a fresh residual. The key residual therefore
      holds 1 to R tokens during decoding, always flushed in whole groups of G.
    * Prefill length. X_Kg = X_K[: l - R] needs l - R to be a multiple of G for the key
      groups. For other lengths the quantized prefix is l - R rounded up to a multiple of G
      (so the residuals never exceed R); for l <= R nothing is quantized. The values use
      the same prefix at prefill, then evict one token per decode step once the window
      exceeds R (pseudo-code: X_Vr[:-R] is quantized).
    Codes, scales and zero-points are those of quantize_keys / quantize_values; the bit
    widths of keys and values are set separately (implementation section: K and V bits
    are independently configurable, 2 or 4).
    """

    def __init__(self, D: int = 128, group: int = 32, residual: int = 128, k_bits: int = 2, v_bits: int = 2):
        assert residual % group == 0 and D % group == 0
        self.D, self.G, self.R = D, group, residual
        self.k_bits, self.v_bits = k_bits, v_bits
        z_i = np.zeros((0, D), np.int64)
        self.k_codes, self.k_scale, self.k_zero = z_i, np.zeros((0, D), np.float16), np.zeros((0, D), np.float16)
        self.v_codes = z_i
        self.v_scale = np.zeros((0, D // group), np.float16)
        self.v_zero = np.zeros((0, D // group), np.float16)
        self.k_resid = np.zeros((0, D), np.float16)
        self.v_resid = np.zeros((0, D), np.float16)

    @property
    def n_quant_k(self) -> int:
        return len(self.k_codes)

    @property
    def n_quant_v(self) -> int:
        return len(self.v_codes)

    @property
    def n_tok(self) -> int:
        return self.n_quant_k + len(self.k_resid)

    def _push_keys(self, K):
        c, s, z = quantize_keys(K, self.G, self.k_bits)
        self.k_codes = np.concatenate([self.k_codes, c])
        self.k_scale = np.concatenate([self.k_scale, s])
        self.k_zero = np.concatenate([self.k_zero, z])

    def _push_values(self, V):
        c, s, z = quantize_values(V, self.G, self.v_bits)
        self.v_codes = np.concatenate([self.v_codes, c])
        self.v_scale = np.concatenate([self.v_scale, s])
        self.v_zero = np.concatenate([self.v_zero, z])

    def prefill(self, K, V) -> None:
        """Cache the l prompt tokens K, V ([l][D] fp16) of an empty stream."""
        assert self.n_tok == 0
        K = np.asarray(K, np.float16)
        V = np.asarray(V, np.float16)
        l = K.shape[0]
        nq = 0 if l <= self.R else -(-(l - self.R) // self.G) * self.G
        if nq:
            self._push_keys(K[:nq])
            self._push_values(V[:nq])
        self.k_resid = K[nq:].copy()
        self.v_resid = V[nq:].copy()

    def append(self, k, v) -> None:
        """One decode token: k, v [D] fp16."""
        k = np.asarray(k, np.float16).reshape(1, self.D)
        v = np.asarray(v, np.float16).reshape(1, self.D)
        if len(self.k_resid) == self.R:            # full key residual: quantize it whole
            self._push_keys(self.k_resid)
            self.k_resid = self.k_resid[:0]
        self.k_resid = np.concatenate([self.k_resid, k])
        self.v_resid = np.concatenate([self.v_resid, v])
        if len(self.v_resid) > self.R:              # value window overflow: oldest token out
            self._push_values(self.v_resid[:-self.R])
            self.v_resid = self.v_resid[-self.R:]

    def attention(self, q) -> np.ndarray:
        """Decode attention of query q [D] over this stream (eq. (3), one softmax)."""
        return decode_attention(q, self.k_codes, self.k_scale, self.k_zero, self.v_codes, self.v_scale,
                                self.v_zero, self.k_resid, self.v_resid, self.G)
