"""Byte and bit accounting of the cache formats (oracle; test infrastructure only)."""
from __future__ import annotations


def kv_cache_bytes(n_layer: int, h_kv: int, d_head: int, seq_len: int, bytes_per_elem: float) -> float:
    """M_KV = 2 * N_layer * H_kv * d_head * S * b_dtype.

    KIVI page, background section (KV memory formula): one K and one V vector per layer,
    KV head and token.
    """
    return 2 * n_layer * h_kv * d_head * seq_len * bytes_per_elem


def vq_bits_per_element(code_bits: int, G: int) -> float:
    """b / G: one ``code_bits``-bit index per G-element sub-vector.

    LoopVQ page, background "vector quantization and codebooks": each index costs b/G
    bit per element. Loop-axis coupling keeps this unchanged (method, "core innovations").
    """
    return code_bits / G


def loopvq_index_bytes_per_token_head(T: int, Tc: int, G: int, D: int, code_bits: int = 8) -> float:
    """Bytes of K (or V) indices one token and head keeps for all T loop steps.

    LoopVQ method step 1: T / Tc loop blocks, each with D / c indices (c = G / Tc) of
    ``code_bits`` bits (method step 5: "D/c indices").
    """
    assert T % Tc == 0 and G % Tc == 0
    c = G // Tc
    assert D % c == 0
    return (T // Tc) * (D // c) * code_bits / 8


def kivi_bits_per_element(bits: int, group: int, scale_bits: int = 16, zero_bits: int = 16) -> float:
    """Quantized bits plus the per-group scale and zero-point spread over the group.

    KIVI page, memory accounting at the end of the core-design section: 2 bits plus one
    fp16 scale and one fp16 zero-point per 32 elements is 3 bits per element.
    """
    return bits + (scale_bits + zero_bits) / group
