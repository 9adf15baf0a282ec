"""Pins of the LoopVQ oracle: coupled-vector map, argmin, dequantize + RoPE + attention,
prefill split. Every check compares against the page's statement, a hand-derived table,
a library routine or a closed form, never against the oracle itself."""
import json
import os

import numpy as np
import pytest
import torch
from scipy.spatial.distance import cdist

import synth
from oracle import loopvq as lv
from oracle.attention import rope

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def marked_input(T, D):
    """x[t-1][0][ch] = 1000*t + ch: every value names its loop step (1-based) and channel."""
    t = np.arange(1, T + 1)[:, None, None]
    ch = np.arange(D)[None, None, :]
    return (1000.0 * t + ch).astype(np.float64)


def test_index_map_hand_table():
    gd = json.load(open(os.path.join(GOLD, "loopvq_index_map.json")))
    x = marked_input(gd["T"], gd["D"])
    for beta in range(gd["T"] // gd["Tc"]):
        z = lv.coupled_vectors(x, beta, gd["Tc"], gd["G"])[0]
        for g in range(gd["NG"]):
            assert z[g].tolist() == gd["z"][f"beta{beta}_g{g}"]


@pytest.mark.parametrize("T,Tc,G,D", [(4, 2, 16, 128), (4, 4, 32, 128), (4, 1, 16, 128), (4, 4, 16, 128), (32, 4, 16, 64)])
def test_index_map_codeword_spans_c_channels_by_Tc_steps(T, Tc, G, D):
    # one codeword spans c = G/Tc consecutive channels of group g across the Tc steps of
    # block beta, each (step, channel) pair exactly once, and no group overlaps another
    c = G // Tc
    x = marked_input(T, D)
    seen = set()
    for beta in range(T // Tc):
        z = lv.coupled_vectors(x, beta, Tc, G)[0]
        for g in range(D // c):
            pairs = {(int(v) // 1000, int(v) % 1000) for v in z[g]}
            want = {(beta * Tc + m + 1, g * c + i) for m in range(Tc) for i in range(c)}
            assert pairs == want
            seen |= pairs
    assert len(seen) == T * D


@pytest.mark.parametrize("T,Tc,G", [(4, 2, 16), (4, 4, 32), (4, 1, 16), (4, 4, 16)])
def test_one_index_serves_every_step_of_its_block(T, Tc, G):
    # codebook = the tokens' own coupled vectors -> indices are the token ids, and
    # dequantizing at each in-block step m returns that step's values exactly
    g = synth.rng(11)
    D, n = 64, 40
    x = g.standard_normal((T, n, D))
    c = G // Tc
    for beta in range(T // Tc):
        z = lv.coupled_vectors(x, beta, Tc, G)        # [n][NG][G]
        cb = np.transpose(z, (1, 0, 2))               # [NG][n][G], entry r = token r
        idx, _ = lv.encode_block(x, cb, beta, Tc)
        assert np.array_equal(idx, np.tile(np.arange(n)[:, None], (1, D // c)))
        for m in range(Tc):
            assert np.array_equal(lv.dequantize(idx, cb, m, Tc), x[beta * Tc + m])


def test_argmin_brute_force_exhaustive_grid_vs_library():
    g = synth.rng(12)
    for K, G in [(2, 2), (4, 2), (4, 4), (256, 16), (16, 3)]:
        cb = g.integers(-3, 4, size=(K, G)).astype(np.float64)
        if G <= 4:
            grid = np.stack(np.meshgrid(*[np.arange(-4, 5)] * G, indexing="ij"), -1).reshape(-1, G)
        else:
            grid = g.integers(-4, 5, size=(3000, G))
        z = grid.astype(np.float64)
        idx, d = lv.nearest_codeword(z, cb)
        ref = cdist(z, cb, "sqeuclidean")
        assert np.array_equal(d, ref)                  # integer grid: exact in fp64
        assert np.array_equal(idx, np.argmin(ref, axis=1))
        # lowest index among exact ties
        for j in np.flatnonzero((ref == ref.min(1, keepdims=True)).sum(1) > 1)[:50]:
            assert idx[j] == np.flatnonzero(ref[j] == ref[j].min())[0]


def test_codeword_encodes_to_itself_and_permutation_equivariance():
    g = synth.rng(13)
    cb = g.standard_normal((256, 16))
    idx, _ = lv.nearest_codeword(cb, cb)
    assert np.array_equal(idx, np.arange(256))
    z = g.standard_normal((500, 16))
    perm = g.permutation(256)
    a, _ = lv.nearest_codeword(z, cb)
    b, _ = lv.nearest_codeword(z, cb[perm])
    assert np.array_equal(perm[b], a)


def test_exact_tie_goes_to_lowest_index():
    cb = np.array([[1.0, 0.0], [-1.0, 0.0], [0.0, 5.0]])
    idx, _ = lv.nearest_codeword(np.zeros((1, 2)), cb)
    assert idx[0] == 0
    idx, _ = lv.nearest_codeword(np.zeros((1, 2)), cb[[1, 0, 2]])
    assert idx[0] == 0


def test_tie_mask_relative_window():
    d = np.array([[1.0, 1.0 + 5e-7, 1.0 + 2e-6, 3.0]])
    assert lv.tie_mask(d, 1e-6).tolist() == [[True, True, False, False]]


def torch_rope(x, pos, base=1e4):
    x = torch.as_tensor(x, dtype=torch.float64)
    h = x.shape[-1] // 2
    th = base ** (-torch.arange(h, dtype=torch.float64) * 2 / x.shape[-1])
    ang = torch.as_tensor(np.asarray(pos, np.float64))[..., None] * th
    zc = torch.complex(x[..., :h], x[..., h:]) * torch.polar(torch.ones_like(ang), ang)
    return torch.cat([zc.real, zc.imag], -1)


@pytest.mark.parametrize("T,Tc,G,t", [(4, 2, 16, 1), (4, 2, 16, 4), (4, 4, 32, 3), (4, 1, 16, 2), (4, 4, 16, 3)])
def test_attention_equals_plain_attention_when_tokens_are_codewords(T, Tc, G, t):
    # when every quantized token equals a codeword exactly, LoopVQ attention must equal
    # textbook RoPE attention on the unquantized cache (library SDPA, complex-form RoPE)
    g = synth.rng(14 + t)
    D, sink, W = 128, 8, 64
    seq_len = 8 + 8 * 30 + 64 + 3
    n_sink, n_pages, n_rec = lv.prefill_split(seq_len, sink, W)
    x = g.standard_normal((T, seq_len, D))          # keys, all loop steps
    y = g.standard_normal((T, seq_len, D))          # values
    beta, m = lv.step_to_block(t, Tc)
    qpos = np.arange(sink, sink + 8 * n_pages)
    # codebooks: the coupled vectors of the quantized tokens themselves (K = n_q entries)
    cbk = np.transpose(lv.coupled_vectors(x[:, qpos], beta, Tc, G), (1, 0, 2))
    cbv = np.transpose(lv.coupled_vectors(y[:, qpos], beta, Tc, G), (1, 0, 2))
    ik, _ = lv.encode_block(x[:, qpos], cbk, beta, Tc)
    iv, _ = lv.encode_block(y[:, qpos], cbv, beta, Tc)
    q = g.standard_normal(D)
    out = lv.decode_attention(q, t, Tc, seq_len, n_pages, ik, iv, cbk, cbv, x[t - 1], y[t - 1])
    pos = np.arange(seq_len)
    Kr = torch_rope(x[t - 1], pos)
    qr = torch_rope(q, seq_len - 1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        qr[None, None, None], Kr[None, None], torch.as_tensor(y[t - 1])[None, None],
        scale=1 / np.sqrt(D))[0, 0, 0].numpy()
    assert np.max(np.abs(out - ref)) < 1e-12


def test_attention_uses_step_slice_and_position_shift_invariance():
    # a different loop step of the same block reads a different slice (the output changes),
    # and shifting every position (query and keys) by the same amount changes nothing
    g = synth.rng(20)
    T, Tc, G, D = 4, 2, 16, 128
    x = g.standard_normal((T, 200, D))
    y = g.standard_normal((T, 200, D))
    cbk = synth.sample_codebooks(g, x, Tc, G)
    cbv = synth.sample_codebooks(g, y, Tc, G)
    seq_len = 200
    _, n_pages, _ = lv.prefill_split(seq_len)
    qpos = np.arange(8, 8 + 8 * n_pages)
    ik, _ = lv.encode_block(x[:, qpos], cbk[0], 0, Tc)
    iv, _ = lv.encode_block(y[:, qpos], cbv[0], 0, Tc)
    q = g.standard_normal(D)
    o1 = lv.decode_attention(q, 1, Tc, seq_len, n_pages, ik, iv, cbk[0], cbv[0], x[0], y[0])
    o2 = lv.decode_attention(q, 2, Tc, seq_len, n_pages, ik, iv, cbk[0], cbv[0], x[1], y[1])
    assert np.max(np.abs(o1 - o2)) > 1e-3
    # shift invariance, checked on an explicit rebuild: rotate by +500 everywhere
    Kq = lv.dequantize(ik, cbk[0], 0, Tc)
    bf, qp = lv.cache_positions(seq_len, n_pages)
    K = np.concatenate([x[0][bf], Kq])
    pos = np.concatenate([bf, qp])
    s1 = rope(K, pos) @ rope(q, seq_len - 1)
    s2 = rope(K, pos + 500) @ rope(q, seq_len - 1 + 500)
    assert np.max(np.abs(s1 - s2)) < 1e-9


@pytest.mark.parametrize("L,W,expect", [(512, 64, (8, 55, 64)), (6144, 64, (8, 759, 64)),
                                        (32768, 256, (8, 4063, 256)), (80, 64, (8, 1, 64)),
                                        (87, 64, (8, 1, 71)), (72, 64, (8, 0, 64)), (5, 64, (5, 0, 0))])
def test_prefill_split(L, W, expect):
    assert lv.prefill_split(L, 8, W) == expect


def test_step_to_block():
    assert [lv.step_to_block(t, 2) for t in (1, 2, 3, 4)] == [(0, 0), (0, 1), (1, 0), (1, 1)]
    assert [lv.step_to_block(t, 4) for t in (1, 4)] == [(0, 0), (0, 3)]
