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


@pytest.mark.parametrize("name", ["kivi_group.json", "kivi_group_4bit.json"])
def test_hand_worked_group(name):
    gd = json.load(open(os.path.join(GOLD, name)))
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


@pytest.mark.parametrize("bits", [2, 4])
def test_code_range_min_max_and_error_bound(bits):
    top = 2 ** bits - 1
    for x in _groups(30):
        q, s16, z16 = kivi.quantize_group(x, bits)
        assert q.min() >= 0 and q.max() <= top
        xh = kivi.dequantize_group(q, s16, z16)
        if abs(float(z16)) < 512:   # zero-point rounding below a quarter level
            assert q[np.argmin(x)] == 0 and q[np.argmax(x)] == top
            # |x - x_hat| <= s/2 (plus fp32 rounding of x/s + z)
            assert np.max(np.abs(x - xh)) <= float(s16) * (0.5 + 1e-6)


@pytest.mark.parametrize("bits", [2, 4])
def test_constant_group_decodes_exactly(bits):
    for v in [0.0, 1.0, -3.25, 1000.0, 6.1e-5]:
        x = synth.fp16_round(np.full(32, v))
        q, s16, z16 = kivi.quantize_group(x, bits)
        assert float(s16) == 1.0
        assert np.array_equal(kivi.dequantize_group(q, s16, z16), x)


@pytest.mark.parametrize("bits", [2, 4])
def test_levels_are_evenly_spaced(bits):
    # X_hat takes at most 2^b values per group, one level s apart
    x = synth.fp16_round(synth.rng(31).standard_normal(32))
    q, s16, z16 = kivi.quantize_group(x, bits)
    assert len(np.unique(q)) <= 2 ** bits
    levels = np.unique(kivi.dequantize_group(np.arange(2 ** bits), s16, z16))
    assert len(levels) == 2 ** bits
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


def test_gqa_runs_of_query_heads_share_a_kv_head():
    # the usual GQA layout (Llama-3: 32 query heads over 8 KV heads): query heads
    # 4k .. 4k+3 read KV head k; multi-head attention when the counts are equal
    assert [kivi.kv_head(h, 32, 8) for h in range(32)] == [h // 4 for h in range(32)]
    assert [kivi.kv_head(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [kivi.kv_head(h, 4, 4) for h in range(4)] == [0, 1, 2, 3]
    assert [kivi.kv_head(h, 6, 1) for h in range(6)] == [0] * 6


def _stream_lengths(l, m, R, G):
    """Closed form of the stream's lengths after a prefill of l tokens and m decode tokens,
    from the flush and eviction rules: the key residual cycles through 1..R once decoding
    starts, the value window holds min(R, tokens not quantized at prefill + m)."""
    nq0 = 0 if l <= R else -(-(l - R) // G) * G
    r0 = l - nq0
    rk = r0 if m == 0 else (r0 + m - 1) % R + 1
    rv = min(R, r0 + m)
    n = l + m
    return n, n - rk, n - rv


@pytest.mark.parametrize("l", [0, 5, 100, 128, 129, 160, 200])
def test_stream_lengths_follow_flush_and_eviction(l):
    R, G, D = 64, 32, 64
    g = synth.rng(40 + l)
    n_steps = 150
    K = synth.fp16_round(g.standard_normal((l + n_steps, D)))
    V = synth.fp16_round(g.standard_normal((l + n_steps, D)))
    st = kivi.KiviStream(D=D, group=G, residual=R)
    st.prefill(K[:l], V[:l])
    for m in range(n_steps + 1):
        if m:
            st.append(K[l + m - 1], V[l + m - 1])
        n, nqk, nqv = _stream_lengths(l, m, R, G)
        assert (st.n_tok, st.n_quant_k, st.n_quant_v) == (n, nqk, nqv), m
        assert nqk % G == 0 and 0 <= nqv <= nqk and n - nqv <= R and (n - nqk <= R)


@pytest.mark.parametrize("k_bits,v_bits", [(2, 2), (4, 2), (2, 4), (4, 4)])
def test_stream_contents_equal_one_shot_quantization(k_bits, v_bits):
    # keys are flushed in whole groups aligned to token 0 and values one token at a time,
    # so the streamed cache equals quantizing the same prefixes in one go, and every
    # token still in a residual is the token as it arrived
    R, G, D, l, n_steps = 64, 32, 64, 90, 170
    g = synth.rng(41)
    K = synth.fp16_round(g.standard_normal((l + n_steps, D)) * 2)
    V = synth.fp16_round(g.standard_normal((l + n_steps, D)))
    st = kivi.KiviStream(D=D, group=G, residual=R, k_bits=k_bits, v_bits=v_bits)
    st.prefill(K[:l], V[:l])
    for m in range(n_steps):
        st.append(K[l + m], V[l + m])
        if m % 37 and m != n_steps - 1:
            continue
        n, nqk, nqv = st.n_tok, st.n_quant_k, st.n_quant_v
        ck, sk, zk = kivi.quantize_keys(K[:nqk], G, k_bits)
        cv, sv, zv = kivi.quantize_values(V[:nqv], G, v_bits)
        assert np.array_equal(st.k_codes, ck) and np.array_equal(st.v_codes, cv)
        assert np.array_equal(st.k_scale.view(np.uint16), sk.view(np.uint16))
        assert np.array_equal(st.k_zero.view(np.uint16), zk.view(np.uint16))
        assert np.array_equal(st.v_scale.view(np.uint16), sv.view(np.uint16))
        assert np.array_equal(st.v_zero.view(np.uint16), zv.view(np.uint16))
        assert np.array_equal(st.k_resid, K[nqk:n]) and np.array_equal(st.v_resid, V[nqv:n])


def test_stream_attention_without_quantization_is_plain_attention():
    # while the prompt and the decoded tokens fit in the residuals nothing is quantized,
    # so attention is textbook softmax attention over the fp16 tokens
    R, D = 128, 128
    g = synth.rng(42)
    K = synth.fp16_round(g.standard_normal((100, D)))
    V = synth.fp16_round(g.standard_normal((100, D)))
    q = synth.bf16_round(g.standard_normal(D))
    st = kivi.KiviStream(D=D, residual=R)
    st.prefill(K[:60], V[:60])
    for j in range(60, 100):
        st.append(K[j], V[j])
    assert st.n_quant_k == st.n_quant_v == 0
    assert np.max(np.abs(st.attention(q) - _sdpa(q, K.astype(np.float64), V.astype(np.float64)))) < 1e-12
