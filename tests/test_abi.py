"""CPU checks of the C ABI: the library builds, loads and exports every function the header
declares, and host-side validation rejects bad arguments before anything is launched.
No call here reaches a kernel (there is no GPU in this suite)."""
import ctypes

import numpy as np
import pytest

import synth
from sub_bit_quantized_gb300 import _build, kvq
from tests import _layout


@pytest.fixture(scope="module")
def L():
    _build.build()
    return kvq.lib()


def test_exports_every_declared_function(L):
    names = kvq.header_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), n
    assert set(kvq._SIGS) == set(names)


def test_version_and_status_strings(L):
    assert L.kvq_version() >= 100
    for code, text in [(0, b"ok"), (1, b"invalid argument"), (2, b"capacity exceeded"),
                       (3, b"unsupported shape"), (4, b"CUDA error"), (5, b"workspace too small"),
                       (6, b"device wait timed out")]:
        assert L.kvq_status_string(code) == text


def cfg2(**kw):
    base = dict(D=128, T=4, Tc=2, G=16, K=256, n_layers=24, n_heads=16, sink=8, recent=64,
                max_pages=759, max_batch=64, max_ctx=6144)
    base.update(kw)
    return kvq.VqConfig(**base)


def test_cache_sizes_formula(L):
    c = cfg2()
    s = kvq.vq_cache_sizes(c)
    assert s.idx == 24 * 2 * 64 * 16 * 759 * 128
    assert s.win == 24 * 4 * 64 * 16 * 80 * 128 * 2
    assert s.bt == 24 * 4 * 16 * 256 * 128 * 4
    assert s.bt_v == 24 * 4 * 16 * 256 * 128 * 2
    assert s.cb == 24 * 2 * 16 * 16 * 256 * 16 * 4
    assert s.rope == 6144 * 64 * 4 and s.per_request == 64 * 4
    # three bf16 parts of each codebook, 256 rows x 4 chunks of 16 bytes (16 coordinates, the
    # -|e|^2/2 chunk, one padding chunk)
    assert s.cbp == 24 * 2 * 16 * 16 * 3 * 256 * 4 * 16
    # one call reads one (layer, block) of each index array: 199.0 MB at B=64, 6K
    assert s.idx / 24 / 2 * 2 == pytest.approx(199.0e6, rel=1e-3)


@pytest.mark.parametrize("Tc,NG", [(1, 8), (2, 16), (4, 32)])
def test_half_bit_loop_grouping_sizes(L, Tc, NG):
    # 0.5 bit (G = 16) at Tc = 1, 2, 4: c = 16, 8, 4 channels per codeword, NG = 8, 16, 32 index
    # bytes per (token, head, block), T / Tc blocks: the index arrays hold the same bytes
    s = kvq.vq_cache_sizes(cfg2(Tc=Tc, G=16))
    assert s.idx == 24 * (4 // Tc) * 64 * 16 * 759 * 8 * NG
    assert s.idx == kvq.vq_cache_sizes(cfg2()).idx
    assert s.cb == 24 * (4 // Tc) * 16 * NG * 256 * 16 * 4


@pytest.mark.parametrize("kw,code", [(dict(Tc=3), 1), (dict(G=12), 1), (dict(G=32), 3),
                                     (dict(D=64), 3), (dict(K=16), 3), (dict(max_ctx=1), 1),
                                     (dict(T=8, Tc=8, G=64), 3), (dict(max_batch=0), 1),
                                     (dict(Tc=2, G=8), 3), (dict(Tc=4, G=64), 3)])
def test_bad_configs_rejected(L, kw, code):
    with pytest.raises(kvq.KvqError) as e:
        kvq.vq_cache_sizes(cfg2(**kw))
    assert e.value.status == code


FAKE = 0x10000  # aligned, never dereferenced: every call below fails validation first


def fake_cache():
    return kvq.VqCacheC(*([FAKE] * 12))


def test_decode_attn_argument_checks(L):
    c = cfg2().to_c()
    kc = fake_cache()
    f = L.kvq_decode_attn
    B = ctypes.byref
    assert f(0, B(c), B(kc), 0, 1, None, 64, FAKE, 0, 0, None, 0, None) == 1   # null q
    assert f(0, B(c), B(kc), 0, 1, FAKE + 2, 64, FAKE, 0, 0, None, 0, None) == 1  # misaligned
    assert f(0, B(c), B(kc), 0, 1, FAKE, 64, FAKE, 7, 0, None, 0, None) == 1   # out dtype
    assert f(0, B(c), B(kc), 24, 1, FAKE, 64, FAKE, 0, 0, None, 0, None) == 1  # layer
    assert f(0, B(c), B(kc), 0, 5, FAKE, 64, FAKE, 0, 0, None, 0, None) == 1   # loop step 5 > T
    assert f(0, B(c), B(kc), 0, 0, FAKE, 64, FAKE, 0, 0, None, 0, None) == 1   # steps are 1-based
    assert f(0, B(c), B(kc), 0, 1, FAKE, 65, FAKE, 0, 0, None, 0, None) == 2   # B > max_batch
    assert f(0, B(c), B(kc), 0, 1, FAKE, 64, FAKE, 0, 3, None, 0, None) == 5   # split needs ws
    assert f(9, B(c), B(kc), 0, 1, FAKE, 64, FAKE, 0, 0, None, 0, None) == 1   # format
    assert b"workspace" in L.kvq_last_error() or b"format" in L.kvq_last_error()
    kc.seq_len = None
    assert f(0, B(c), B(kc), 0, 1, FAKE, 64, FAKE, 0, 0, None, 0, None) == 1   # cache pointer


def test_workspace_size_and_split_plan(L):
    c = cfg2()

    def a256(x):
        return (x + 255) // 256 * 256

    # LoopVQ: one merge counter per (request, head) segment, and two partial slots per block
    # (the segments a block shares with its neighbours), each (M, l, 2 pad, o[128]) floats
    for blocks in (1, 4, 152):
        want = a256(64 * 16 * 4) + a256(blocks * 2 * 132 * 4)
        assert kvq.kvq_decode_workspace_size(c, 64, blocks) == want
    auto = kvq.kvq_decode_auto_splits(c, 64)
    assert auto >= 1
    assert kvq.kvq_decode_workspace_size(c, 64, 0) == kvq.kvq_decode_workspace_size(c, 64, auto)
    # the decode kernel runs one block per SM by default, whatever the batch
    big = cfg2(max_pages=40000, max_ctx=400000)
    assert kvq.kvq_decode_auto_splits(big, 1) == auto


def test_encode_and_prefill_argument_checks(L):
    c = cfg2().to_c()
    B = ctypes.byref
    f = L.kvq_encode_vq
    # n_tok not a whole number of pages
    assert f(B(c), FAKE, 0, 0, 0, 0, 1, 12, FAKE, FAKE, 0, 0, 16, None, None) == 1
    # pages beyond max_pages
    assert f(B(c), FAKE, 0, 0, 0, 0, 1, 8 * 760, FAKE, FAKE, 0, 0, 16, None, None) == 2
    # groups outside [0, 16)
    assert f(B(c), FAKE, 0, 0, 0, 0, 1, 8, FAKE, FAKE, 0, 10, 8, None, None) == 1
    # stride not a multiple of 8 elements
    assert f(B(c), FAKE, 3, 0, 0, 0, 1, 8, FAKE, FAKE, 0, 0, 16, None, None) == 1
    kc = fake_cache()
    g = L.kvq_prefill_vq
    assert g(B(c), B(kc), 0, FAKE, FAKE, 0, 0, 0, 0, 1, 6145, None, None) == 2   # L > max_ctx
    big = cfg2(max_ctx=1 << 20).to_c()
    assert g(B(big), B(kc), 0, FAKE, FAKE, 0, 0, 0, 0, 1, 8 * 800, None, None) == 2  # pages
    assert g(B(c), B(kc), 0, FAKE, FAKE, 0, 0, 0, 60, 5, 100, None, None) == 2  # requests
    a = L.kvq_append_page
    assert a(B(c), B(kc), 0, 0, FAKE, FAKE, 1, None) == 1                        # step 0
    assert a(B(c), B(kc), 0, 1, FAKE, FAKE, 65, None) == 2                       # n_seq


def test_kivi_argument_checks(L):
    k = kvq.KiviConfig(n_heads=32, max_batch=16, max_tokens=3968).to_c()
    B = ctypes.byref
    f = L.kvq_quantize_kivi
    assert f(B(k), 0, FAKE, 0, 0, 16, 31, FAKE, FAKE, FAKE, 0, None) == 1   # keys need 32-token groups
    assert f(B(k), 0, FAKE, 0, 0, 16, 64, FAKE, FAKE, FAKE, 3936, None) == 2  # past capacity
    assert f(B(k), 2, FAKE, 0, 0, 16, 64, FAKE, FAKE, FAKE, 0, None) == 1   # axis
    k3 = kvq.KiviConfig(k_bits=3, max_tokens=64).to_c()
    assert f(B(k3), 1, FAKE, 0, 0, 1, 1, FAKE, FAKE, FAKE, 0, None) == 3    # 3-bit not built
    kq = kvq.KiviConfig(n_heads=8, n_q_heads=12, max_tokens=64).to_c()
    assert f(B(kq), 1, FAKE, 0, 0, 1, 1, FAKE, FAKE, FAKE, 0, None) == 1    # GQA ratio not whole
    kr = kvq.KiviConfig(residual=100, max_tokens=64).to_c()
    assert f(B(kr), 1, FAKE, 0, 0, 1, 1, FAKE, FAKE, FAKE, 0, None) == 1    # R not a multiple of 32
    kc = kvq.KiviCacheC(*([FAKE] * len(kvq.KIVI_CACHE_FIELDS)))
    p = L.kvq_kivi_prefill
    assert p(B(k), B(kc), FAKE, FAKE, 0, 0, 15, 2, 64, None) == 2            # b0 + B > max_batch
    assert p(B(k), B(kc), FAKE, FAKE, 0, 0, 0, 1, 3968 + 129, None) == 2     # quantized part too long
    assert p(B(k), B(kc), FAKE, FAKE, 0, 0, 0, 1, -1, None) == 1
    bad = kvq.KiviCacheC(*([FAKE] * (len(kvq.KIVI_CACHE_FIELDS) - 1) + [None]))
    assert p(B(k), B(bad), FAKE, FAKE, 0, 0, 0, 1, 64, None) == 1            # null length array
    k0 = kvq.KiviConfig(residual=0, max_tokens=64).to_c()
    a = L.kvq_kivi_append
    assert a(B(k0), B(kc), FAKE, FAKE, 1, None) == 1                         # streaming needs R > 0
    assert a(B(k), B(kc), FAKE, FAKE, 17, None) == 2                         # n_seq > max_batch
    assert a(B(k), B(kc), FAKE, FAKE, 0, None) == 0                          # nothing to do


def test_library_missing_fails_loudly(monkeypatch):
    monkeypatch.setattr(kvq, "_lib", None)
    monkeypatch.setattr(kvq, "LIB_PATH", "/nonexistent/libkvq.so")
    with pytest.raises(RuntimeError, match="libkvq.so not found"):
        kvq.lib()


def test_page_layout_round_trip():
    g = synth.rng(5)
    idx = synth.random_indices(g, (3, 40, 16))
    pages = _layout.pack_pages(idx)
    assert pages.shape == (3, 5, 128)
    assert np.array_equal(_layout.unpack_pages(pages), idx)
    # byte (s*8 + j)*2 + 1 holds group s + 8 of token j
    assert pages[0, 0, (3 * 8 + 5) * 2 + 1] == idx[0, 5, 11]


def test_code_packing_round_trip():
    g = synth.rng(6)
    codes = g.integers(0, 4, size=(7, 128))
    b = _layout.pack_codes(codes)
    assert b.shape == (7, 32) and np.array_equal(_layout.unpack_codes(b), codes)
    assert b[0, 0] == codes[0, 0] | (codes[0, 1] << 2) | (codes[0, 2] << 4) | (codes[0, 3] << 6)
    c4 = g.integers(0, 16, size=(7, 128))
    b4 = _layout.pack_codes(c4, 4)
    assert b4.shape == (7, 64) and np.array_equal(_layout.unpack_codes(b4, 4), c4)
    assert b4[2, 5] == c4[2, 10] | (c4[2, 11] << 4)
