"""Pins of the oracle's RoPE, softmax attention and split/LSE merge.

Checked against closed forms, invariants and an independent library formulation
(torch's scaled_dot_product_attention in fp64 and RoPE as complex multiplication).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import attention as att


def torch_rope_complex(x, pos, base=1e4):
    """RoPE as a complex product: (x_i + j x_{i+D/2}) * exp(j pos theta_i)."""
    x = torch.as_tensor(np.asarray(x), dtype=torch.float64)
    D = x.shape[-1]
    h = D // 2
    theta = base ** (-torch.arange(h, dtype=torch.float64) * 2 / D)
    ang = torch.as_tensor(np.asarray(pos, np.float64))[..., None] * theta
    zc = torch.complex(x[..., :h], x[..., h:]) * torch.polar(torch.ones_like(ang), ang)
    return torch.cat([zc.real, zc.imag], dim=-1).numpy()


def sdpa(q, K, V, scale):
    qt = torch.as_tensor(q, dtype=torch.float64)[None, None, None, :]
    Kt = torch.as_tensor(K, dtype=torch.float64)[None, None]
    Vt = torch.as_tensor(V, dtype=torch.float64)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)[0, 0, 0].numpy()


def test_rope_matches_complex_form():
    g = synth.rng(1)
    x = g.standard_normal((37, 128))
    pos = g.integers(0, 40000, size=37)
    # angles reach 4e4 rad, so the two evaluations differ by a few 1e-12 (fp64 angle ulp)
    assert np.allclose(att.rope(x, pos), torch_rope_complex(x, pos), atol=5e-11, rtol=0)


def test_rope_position_zero_is_identity_and_norm_preserved():
    g = synth.rng(2)
    x = g.standard_normal((5, 128))
    assert np.array_equal(att.rope(x, 0), x)
    y = att.rope(x, 1234)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)


def test_rope_relative_property():
    # <R(a) q, R(b) k> depends only on a - b
    g = synth.rng(3)
    q, k = g.standard_normal(128), g.standard_normal(128)
    d1 = att.rope(q, 700) @ att.rope(k, 300)
    d2 = att.rope(q, 5400) @ att.rope(k, 5000)
    d3 = att.rope(q, 400) @ k
    assert abs(d1 - d2) < 1e-10 and abs(d1 - d3) < 1e-10


def test_rope_pairs_rotate_half():
    # a vector with only channel i set rotates into channel i + D/2 (and not i + 1)
    x = np.zeros(128)
    x[5] = 1.0
    y = att.rope(x, 1)
    th = 1e4 ** (-2 * 5 / 128)
    assert abs(y[5] - np.cos(th)) < 1e-15 and abs(y[69] - np.sin(th)) < 1e-15
    assert np.count_nonzero(np.abs(y) > 1e-15) == 2


def test_attention_matches_library():
    g = synth.rng(4)
    q = g.standard_normal(128)
    K = 3 * g.standard_normal((300, 128))
    V = g.standard_normal((300, 128))
    s = 1 / np.sqrt(128)
    assert np.allclose(att.softmax_attention(q, K, V, s), sdpa(q, K, V, s), atol=1e-12)


def test_all_keys_equal_gives_mean_of_values():
    g = synth.rng(5)
    q = g.standard_normal(128)
    K = np.tile(g.standard_normal(128), (50, 1))
    V = g.standard_normal((50, 128))
    assert np.allclose(att.softmax_attention(q, K, V, 0.1), V.mean(axis=0), atol=1e-13)


def test_dominant_logit_selects_row():
    g = synth.rng(6)
    K = np.zeros((40, 128))
    q = np.zeros(128)
    q[0] = 1.0
    K[17, 0] = 1000.0
    V = g.standard_normal((40, 128))
    assert np.allclose(att.softmax_attention(q, K, V, 1.0), V[17], atol=1e-12)


@pytest.mark.parametrize("cuts", [[], [1], [100, 101], list(range(8, 600, 8)), [3, 200, 590]])
def test_split_lse_merge_invariance(cuts):
    g = synth.rng(7)
    q = g.standard_normal(128)
    K = 4 * g.standard_normal((600, 128))
    V = g.standard_normal((600, 128))
    s = 1 / np.sqrt(128)
    full = att.softmax_attention(q, K, V, s)
    assert np.max(np.abs(att.split_attention(q, K, V, s, cuts) - full)) < 1e-12


def test_lse_merge_handles_empty_split():
    g = synth.rng(8)
    q = g.standard_normal(16)
    K, V = g.standard_normal((9, 16)), g.standard_normal((9, 16))
    parts = [att.partial_softmax(q, K[:0], V[:0], 1.0), att.partial_softmax(q, K, V, 1.0)]
    assert np.allclose(att.lse_merge(parts), att.softmax_attention(q, K, V, 1.0), atol=1e-14)
