"""Pins of the KIVI oracle: the hand-worked group, code range, closed-form error bound,
constant groups, grouping axes, and attention over grouped + residual segments."""
import json
import os

import numpy as np
import pytest
import torch

import synth
from oracle import kivi

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_group():
    gd = json.load(open(os.path.join(GOLD, "kivi_group.json")))
    q, s16, z16 = kivi.quantize_group(np.array(gd["x"]), gd["bits"])
    assert float(s16) == gd["scale"] and float(z16) == gd["zero"]
    assert q.tolist() == gd["codes"]
    assert kivi.dequantize_group(q, s16, z16).tolist() == gd["x_hat"]


def _groups(seed, n=400, size=32):
    g = synth.rng(seed)
    out = []
    for k in range(n):
        scale = 10.0 ** g.uniform(-3, 1.5)
        shift = g.uniform(-3, 3) * scale * (k % 3)
        out.append(synth.fp16_round(shift + scale * g.standard_normal(size)))
    return out


def test_code_range_min_max_and_error_bound():
    for x in _groups(30):
        q, s16, z16 = kivi.quantize_group(x)
        assert q.min() >= 0 and q.max() <= 3
        xh = kivi.dequantize_group(q, s16, z16)
        if abs(float(z16)) < 512:   # zero-point rounding below a quarter level
            assert q[np.argmin(x)] == 0 and q[np.argmax(x)] == 3
            # |x - x_hat| <= s/2 (plus fp32 rounding of x/s + z)
            assert np.max(np.abs(x - xh)) <= float(s16) * (0.5 + 1e-6)


def test_constant_group_decodes_exactly():
    for v in [0.0, 1.0, -3.25, 1000.0, 6.1e-5]:
        x = synth.fp16_round(np.full(32, v))
        q, s16, z16 = kivi.quantize_group(x)
        assert float(s16) == 1.0
        assert np.array_equal(kivi.dequantize_group(q, s16, z16), x)


def test_four_levels_are_evenly_spaced():
    # X_hat takes at most 4 values per group, one level s apart
    x = synth.fp16_round(synth.rng(31).standard_normal(32))
    q, s16, z16 = kivi.quantize_group(x)
    levels = np.unique(kivi.dequantize_group(np.arange(4), s16, z16))
    assert np.allclose(np.diff(levels), float(s16), rtol=1e-12)


def test_grouping_axes_keys_per_channel_values_per_token():
    # per-channel grouping of K over tokens == per-token grouping of K^T over channels
    g = synth.rng(32)
    K = synth.fp16_round(g.standard_normal((64, 64)) * 3)
    ck, sk, zk = kivi.quantize_keys(K)
    cv, sv, zv = kivi.quantize_values(K.T)
    assert np.array_equal(ck, cv.T) and np.array_equal(sk, sv.T) and np.array_equal(zk, zv.T)
    # and one outlier channel only changes its own key group scales
    K2 = K.copy()
    K2[:, 7] *= 20
    ck2, sk2, _ = kivi.quantize_keys(synth.fp16_round(K2))
    changed = np.flatnonzero((sk2 != sk).any(axis=0))
    assert changed.tolist() == [7]


def _sdpa(q, K, V):
    t = lambda a: torch.as_tensor(np.asarray(a, np.float64))
    return torch.nn.functional.scaled_dot_product_attention(
        t(q)[None, None, None], t(K)[None, None], t(V)[None, None],
        scale=1 / np.sqrt(len(q)))[0, 0, 0].numpy()


@pytest.mark.parametrize("n_q,n_r", [(0, 20), (64, 0), (96, 31), (3968 // 31, 128)])
def test_attention_over_segments_equals_single_softmax(n_q, n_r):
    n_q = (n_q // 32) * 32
    g = synth.rng(33 + n_q + n_r)
    D = 128
    K, V = synth.kivi_kv(g, n_q + n_r, D, synth.outlier_channels(g, D, 6))
    K, V = synth.fp16_round(K), synth.fp16_round(V)
    q = synth.bf16_round(g.standard_normal(D))
    ck, sk, zk = kivi.quantize_keys(K[:n_q])
    cv, sv, zv = kivi.quantize_values(V[:n_q])
    out = kivi.decode_attention(q, ck, sk, zk, cv, sv, zv, K[n_q:], V[n_q:])
    Kh = np.concatenate([kivi.dequantize_keys(ck, sk, zk) if n_q else np.zeros((0, D)), K[n_q:]])
    Vh = np.concatenate([kivi.dequantize_values(cv, sv, zv) if n_q else np.zeros((0, D)), V[n_q:]])
    assert np.max(np.abs(out - _sdpa(q, Kh, Vh))) < 1e-12


def test_dequantize_keys_uses_token_groups():
    # group gi of keys covers tokens [32 gi, 32 gi + 32) with one scale per channel
    codes = np.tile(np.arange(4), (64, 32))[:, :128]
    scale = np.array([[1.0] * 128, [2.0] * 128], dtype=np.float16)
    zero = np.zeros((2, 128), dtype=np.float16)
    out = kivi.dequantize_keys(codes, scale, zero)
    assert np.array_equal(out[:32], codes[:32]) and np.array_equal(out[32:], 2 * codes[32:])
