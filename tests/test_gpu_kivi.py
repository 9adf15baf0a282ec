"""GPU parity of KIVI: group quantization with 2- and 4-bit codes (codes, fp16 scales and
zero-points bit-exact with the oracle's fixed fp32 sequence), the streaming cache of
Algorithm 1 (prefill and decode append: cache contents bit-exact with the oracle's stream),
and decode attention over quantized + fp16 segments with grouped-query heads (max-abs 2e-3,
relative L2 1e-3 against fp64)."""
import numpy as np
import pytest
import torch

import synth
from oracle import kivi as okivi
from sub_bit_quantized_gb300 import kvq
from tests import _cases as C
from tests import _layout

pytestmark = pytest.mark.gpu
D = 128


def kv_data(seed, B, H, n):
    g = synth.rng(seed)
    K = np.empty((B, H, n, D), np.float16)
    V = np.empty((B, H, n, D), np.float16)
    for h in range(H):
        outl = synth.outlier_channels(g, D, 6)
        for b in range(B):
            k, v = synth.kivi_kv(g, n, D, outl)
            K[b, h], V[b, h] = k.astype(np.float16), v.astype(np.float16)
    # degenerate groups: a constant key group, a constant value group, a wide-range group
    K[0, 0, 32:64, 5] = np.float16(0.75)
    V[0, 0, 3, 64:96] = np.float16(-2.5)
    K[-1, -1, :32, 9] = (np.arange(32) * 300.0 - 4000.0).astype(np.float16)
    return g, K, V


@pytest.mark.parametrize("bits", [2, 4])
def test_quantize_bit_exact(bits):
    B, H, n = 2, 3, 96
    g, K, V = kv_data(300, B, H, n)
    # groups whose scaled values x / s + z fall exactly on k + 1/2 (s a power of two, z = 0):
    # the rounding ties that the exact division decides (half to even)
    s0, top = 0.25, (1 << bits) - 1
    ties = (np.arange(32) % top + 0.5) * s0
    ties[0], ties[1] = 0.0, top * s0  # the group's minimum and maximum
    K[1, 2, 64:96, 17] = ties.astype(np.float16)  # a key group: channel 17, tokens 64..95
    V[1, 1, 7, 32:64] = ties.astype(np.float16)   # a value group: token 7, channels 32..63
    cfg = kvq.KiviConfig(n_heads=H, k_bits=bits, v_bits=bits, max_batch=B, max_tokens=160)
    cache = kvq.KiviCache(cfg)
    kvq.kvq_quantize_kivi(cfg, kvq.PER_CHANNEL, torch.from_numpy(K).cuda(), cache.k_codes, cache.k_scale,
                          cache.k_zero, tok_begin=32)
    kvq.kvq_quantize_kivi(cfg, kvq.PER_TOKEN, torch.from_numpy(V).cuda(), cache.v_codes, cache.v_scale,
                          cache.v_zero, tok_begin=32)
    torch.cuda.synchronize()
    kc = _layout.unpack_codes(cache.k_codes.cpu().numpy(), bits)
    vc = _layout.unpack_codes(cache.v_codes.cpu().numpy(), bits)
    ks, kz = cache.k_scale.cpu().numpy(), cache.k_zero.cpu().numpy()
    vs, vz = cache.v_scale.cpu().numpy(), cache.v_zero.cpu().numpy()
    for b in range(B):
        for h in range(H):
            c, s, z = okivi.quantize_keys(K[b, h], bits=bits)
            assert np.array_equal(kc[b, h, 32:32 + n], c)
            assert np.array_equal(ks[b, h, 1:1 + n // 32].view(np.uint16), s.view(np.uint16))
            assert np.array_equal(kz[b, h, 1:1 + n // 32].view(np.uint16), z.view(np.uint16))
            c, s, z = okivi.quantize_values(V[b, h], bits=bits)
            assert np.array_equal(vc[b, h, 32:32 + n], c)
            assert np.array_equal(vs[b, h, 32:32 + n].view(np.uint16), s.view(np.uint16))
            assert np.array_equal(vz[b, h, 32:32 + n].view(np.uint16), z.view(np.uint16))
    # untouched regions stay zero
    assert not kc[:, :, :32].any() and not vc[:, :, 128:].any()


@pytest.mark.parametrize("n", [5, 37, 70])
def test_quantize_values_ragged_tiles(n):
    # per-token quantization of a token count that leaves the last 32-row tile (and its last
    # 8-row block) partly empty: codes, scales and zero-points bit-exact, nothing written past
    # the last token
    B, H, bits = 2, 3, 2
    V = np.ascontiguousarray(kv_data(301, B, H, max(n, 32))[2][:, :, :n])
    cfg = kvq.KiviConfig(n_heads=H, k_bits=bits, v_bits=bits, max_batch=B, max_tokens=128)
    cache = kvq.KiviCache(cfg)
    kvq.kvq_quantize_kivi(cfg, kvq.PER_TOKEN, torch.from_numpy(V).cuda(), cache.v_codes, cache.v_scale,
                          cache.v_zero, tok_begin=8)
    torch.cuda.synchronize()
    vc = _layout.unpack_codes(cache.v_codes.cpu().numpy(), bits)
    vs, vz = cache.v_scale.cpu().numpy(), cache.v_zero.cpu().numpy()
    for b in range(B):
        for h in range(H):
            c, sc, z = okivi.quantize_values(V[b, h], bits=bits)
            assert np.array_equal(vc[b, h, 8:8 + n], c)
            assert np.array_equal(vs[b, h, 8:8 + n].view(np.uint16), sc.view(np.uint16))
            assert np.array_equal(vz[b, h, 8:8 + n].view(np.uint16), z.view(np.uint16))
    assert not vc[:, :, :8].any() and not vc[:, :, 8 + n:].any()
    assert not vs[:, :, 8 + n:].view(np.uint16).any() and not vz[:, :, 8 + n:].view(np.uint16).any()


def test_quantize_full_size_sampled():
    # prefill workload: K and V of 16 heads x 32768 tokens
    H, n = 16, 32768
    gen = torch.Generator(device="cuda").manual_seed(31)
    K = torch.randn((1, H, n, D), generator=gen, device="cuda")
    outl = torch.randperm(D, generator=gen, device="cuda")[:6]
    K[..., outl] *= 20.0
    K = K.half().contiguous()
    V = torch.randn((1, H, n, D), generator=gen, device="cuda").half().contiguous()
    cfg = kvq.KiviConfig(n_heads=H, max_batch=1, max_tokens=n)
    cache = kvq.KiviCache(cfg)
    kvq.kvq_quantize_kivi(cfg, kvq.PER_CHANNEL, K, cache.k_codes, cache.k_scale, cache.k_zero)
    kvq.kvq_quantize_kivi(cfg, kvq.PER_TOKEN, V, cache.v_codes, cache.v_scale, cache.v_zero)
    torch.cuda.synchronize()
    rs = np.random.default_rng(4)
    for h, gi in zip(rs.integers(0, H, 12), rs.integers(0, n // 32, 12)):
        blk = K[0, h, gi * 32:(gi + 1) * 32].cpu().numpy()
        c, s, z = okivi.quantize_keys(blk)
        got = _layout.unpack_codes(cache.k_codes[0, h, gi * 32:(gi + 1) * 32].cpu().numpy())
        assert np.array_equal(got, c)
        assert np.array_equal(cache.k_scale[0, h, gi].cpu().numpy().view(np.uint16), s[0].view(np.uint16))
        assert np.array_equal(cache.k_zero[0, h, gi].cpu().numpy().view(np.uint16), z[0].view(np.uint16))
    for h, j in zip(rs.integers(0, H, 12), rs.integers(0, n, 12)):
        row = V[0, h, j:j + 1].cpu().numpy()
        c, s, z = okivi.quantize_values(row)
        assert np.array_equal(_layout.unpack_codes(cache.v_codes[0, h, j:j + 1].cpu().numpy()), c)
        assert np.array_equal(cache.v_scale[0, h, j].cpu().numpy().view(np.uint16), s[0].view(np.uint16))


def run(case, cache, n_splits=0, dtype=torch.float32):
    B, Hq = len(case.n_tok), case.cfg.q_heads
    out = torch.empty((B, Hq, D), dtype=dtype, device="cuda")
    ws = kvq.make_workspace(case.cfg, B, n_splits)
    kvq.kvq_decode_attn(case.cfg, cache, 0, 1, C.bf16_tensor(case.q), out, n_splits, ws)
    torch.cuda.synchronize()
    assert kvq.device_error() == 0
    return out


def check_all(case, got):
    B, Hq = got.shape[:2]
    ref = np.stack([[C.oracle_kivi(case, b, h) for h in range(Hq)] for b in range(B)])
    C.check_close(got, ref)


@pytest.mark.parametrize("n_splits", [0, 1, 3, 7])
def test_attention_segments_and_splits(n_splits):
    case = C.make_kivi_case(310, B=4, H=2, n_quant=[0, 96, 32 * 40, 32], n_resid=[17, 0, 128, 1])
    check_all(case, run(case, C.fill_kivi_cache(case), n_splits).cpu().numpy())


@pytest.mark.parametrize("k_bits,v_bits,rep", [(2, 2, 1), (4, 4, 1), (2, 4, 2), (4, 2, 2), (4, 2, 4), (4, 4, 4),
                                               (2, 2, 8), (4, 4, 3)])
def test_attention_bits_and_gqa(k_bits, v_bits, rep):
    # query head h reads KV head h // rep; one block serves up to four query heads
    case = C.make_kivi_case(313 + rep, B=3, H=2, Hq=2 * rep, k_bits=k_bits, v_bits=v_bits,
                            n_quant=[32 * 9, 0, 32 * 21], n_resid=[40, 77, 128])
    for n_splits in (0, 2):
        check_all(case, run(case, C.fill_kivi_cache(case), n_splits).cpu().numpy())


@pytest.mark.parametrize("k_bits,v_bits,rep", [(2, 2, 1), (4, 4, 4)])
def test_attention_mixed_value_segment(k_bits, v_bits, rep):
    # the streaming cache's tail: keys quantized up to n_quant_k, values only up to n_quant_v,
    # tokens between them take their value from the fp16 window (ring rows t % R)
    nqk = [32 * 12, 32 * 5, 128, 64]
    nr = [1, 60, 128, 30]
    nqv = [32 * 12 - 127, 32 * 5 - 3, 128, 0]   # n - n_quant_v <= R
    case = C.make_kivi_case(320 + rep, B=4, H=2, Hq=2 * rep, k_bits=k_bits, v_bits=v_bits, n_quant=nqk,
                            n_resid=nr, n_quant_v=nqv)
    assert all(n - v <= 128 and 0 <= v <= k for n, v, k in zip(case.n_tok, nqv, nqk))
    for n_splits in (0, 1, 5):
        check_all(case, run(case, C.fill_kivi_cache(case), n_splits).cpu().numpy())


def test_attention_repeated_calls_identical():
    # splits merge in split order and warps in warp order: repeated calls agree bit for bit,
    # with the same workspace (its arrival counters reset by the last block) or a fresh one
    case = C.make_kivi_case(316, B=3, H=2, Hq=8, k_bits=4, v_bits=2, n_quant=[992, 640, 1504], n_resid=[77, 128, 5])
    cache = C.fill_kivi_cache(case)
    B, Hq = len(case.n_tok), case.cfg.q_heads
    ws = kvq.make_workspace(case.cfg, B, 5)
    outs = []
    for _ in range(3):
        out = torch.empty((B, Hq, D), dtype=torch.float32, device="cuda")
        kvq.kvq_decode_attn(case.cfg, cache, 0, 1, C.bf16_tensor(case.q), out, 5, ws)
        torch.cuda.synchronize()
        assert kvq.device_error() == 0
        outs.append(out)
    outs.append(run(case, cache, 5))
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    check_all(case, outs[0].cpu().numpy())


def test_attention_empty_cache_gives_zero():
    case = C.make_kivi_case(311, B=1, H=1, n_quant=[0], n_resid=[0])
    cache = C.fill_kivi_cache(case)
    assert torch.count_nonzero(run(case, cache)) == 0


def test_attention_full_size_sampled():
    # Llama-2-7B-shaped layer: 32 heads, batch 16, context 4096 = 3968 quantized + 128 fp16
    case = C.make_kivi_case(312, B=16, H=32, n_quant=[3968] * 16, n_resid=[128] * 16)
    cache = C.fill_kivi_cache(case)
    got = run(case, cache).cpu().numpy()
    got16 = run(case, cache, dtype=torch.bfloat16)
    assert torch.equal(torch.from_numpy(got).cuda().to(torch.bfloat16), got16)
    rs = np.random.default_rng(5)
    pairs = list(zip(rs.integers(0, 16, 6), rs.integers(0, 32, 6))) + [(0, 0), (15, 31)]
    C.check_close(np.stack([got[b, h] for b, h in pairs]), np.stack([C.oracle_kivi(case, b, h) for b, h in pairs]))


def test_attention_kivi4_gqa_full_size_sampled():
    # Llama-3-8B-shaped layer: 32 query heads over 8 KV heads, 4-bit keys and values,
    # batch 16, context 4096 = 3968 quantized + 128 fp16
    case = C.make_kivi_case(314, B=16, H=8, Hq=32, k_bits=4, v_bits=4, n_quant=[3968] * 16, n_resid=[128] * 16)
    got = run(case, C.fill_kivi_cache(case)).cpu().numpy()
    rs = np.random.default_rng(6)
    pairs = list(zip(rs.integers(0, 16, 6), rs.integers(0, 32, 6))) + [(0, 0), (15, 31)]
    C.check_close(np.stack([got[b, h] for b, h in pairs]), np.stack([C.oracle_kivi(case, b, h) for b, h in pairs]))


def _stream_state(cache, b, h, cfg):
    """The logical stream of (request b, KV head h) read back from the device cache."""
    n, nqk, nqv = (int(t[b]) for t in (cache.n_tok, cache.n_quant_k, cache.n_quant_v))
    R = cfg.residual
    kr = cache.k_resid[b, h, :n - nqk].cpu().numpy()
    rows = [(t % R) for t in range(nqv, n)]
    vr = cache.v_resid[b, h].cpu().numpy()[rows]
    kc = _layout.unpack_codes(cache.k_codes[b, h, :nqk].cpu().numpy(), cfg.k_bits)
    vc = _layout.unpack_codes(cache.v_codes[b, h, :nqv].cpu().numpy(), cfg.v_bits)
    return (n, nqk, nqv, kc, cache.k_scale[b, h, :nqk // 32].cpu().numpy(), cache.k_zero[b, h, :nqk // 32].cpu().numpy(),
            vc, cache.v_scale[b, h, :nqv].cpu().numpy(), cache.v_zero[b, h, :nqv].cpu().numpy(), kr, vr)


def _same_stream(got, st):
    n, nqk, nqv, kc, ks, kz, vc, vs, vz, kr, vr = got
    assert (n, nqk, nqv) == (st.n_tok, st.n_quant_k, st.n_quant_v)
    assert np.array_equal(kc, st.k_codes) and np.array_equal(vc, st.v_codes)
    for a, b in ((ks, st.k_scale), (kz, st.k_zero), (vs, st.v_scale), (vz, st.v_zero), (kr, st.k_resid),
                 (vr, st.v_resid)):
        assert np.array_equal(a.view(np.uint16), np.asarray(b, np.float16).view(np.uint16))


@pytest.mark.parametrize("k_bits,v_bits,rep", [(2, 2, 1), (4, 2, 2), (4, 4, 4)])
def test_streaming_prefill_and_append(k_bits, v_bits, rep):
    # requests of mixed prompt lengths (ragged, shorter than R, a multiple of R) stream decode
    # tokens through key flushes and value evictions; the device cache must equal the
    # oracle's Algorithm 1 stream bit for bit, and attention over it must match
    H, R, n_steps = 2, 128, 200
    prompts = [300, 37, 256, 129]
    B = len(prompts)
    cfg = kvq.KiviConfig(n_heads=H, n_q_heads=H * rep, k_bits=k_bits, v_bits=v_bits, residual=R, max_batch=B,
                         max_tokens=640)
    cache = kvq.KiviCache(cfg)
    g = synth.rng(330 + rep)
    total = max(prompts) + n_steps
    K = np.empty((B, H, total, D), np.float16)
    V = np.empty((B, H, total, D), np.float16)
    for h in range(H):
        outl = synth.outlier_channels(g, D, 6)
        for b in range(B):
            k, v = synth.kivi_kv(g, total, D, outl)
            K[b, h], V[b, h] = k, v
    streams = [[okivi.KiviStream(D, 32, R, k_bits, v_bits) for _ in range(H)] for _ in range(B)]
    for b, l in enumerate(prompts):
        kvq.kvq_kivi_prefill(cfg, cache, torch.from_numpy(K[b:b + 1, :, :l].copy()).cuda(),
                             torch.from_numpy(V[b:b + 1, :, :l].copy()).cuda(), b0=b)
        for h in range(H):
            streams[b][h].prefill(K[b, h, :l], V[b, h, :l])
    Kt, Vt = torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda()
    pos = torch.tensor(prompts, device="cuda")
    for m in range(n_steps):
        k_new = Kt[torch.arange(B), :, pos + m].contiguous()
        v_new = Vt[torch.arange(B), :, pos + m].contiguous()
        kvq.kvq_kivi_append(cfg, cache, k_new, v_new)
        for b, l in enumerate(prompts):
            for h in range(H):
                streams[b][h].append(K[b, h, l + m], V[b, h, l + m])
        if m in (0, 1, 90, 91, 128, 129, n_steps - 1):
            torch.cuda.synchronize()
            assert kvq.device_error() == 0
            for b in range(B):
                for h in range(H):
                    _same_stream(_stream_state(cache, b, h, cfg), streams[b][h])
            q = synth.bf16_round(synth.gaussian(g, (B, H * rep, D)))
            out = torch.empty((B, H * rep, D), dtype=torch.float32, device="cuda")
            kvq.kvq_decode_attn(cfg, cache, 0, 1, C.bf16_tensor(q), out)
            got = out.cpu().numpy()
            ref = np.stack([[streams[b][okivi.kv_head(hq, H * rep, H)].attention(q[b, hq]) for hq in range(H * rep)]
                            for b in range(B)])
            C.check_close(got, ref)


def test_append_beyond_capacity_reports_and_keeps_state():
    # a key flush that would pass max_tokens leaves the request as it is and raises
    # KVQ_ERR_CAPACITY through the device error word; other requests still advance
    H, R = 1, 128
    cfg = kvq.KiviConfig(n_heads=H, residual=R, max_batch=2, max_tokens=64)
    cache = kvq.KiviCache(cfg)
    g = synth.rng(340)
    x = torch.from_numpy(synth.fp16_round(g.standard_normal((2, H, 192, D))).astype(np.float16)).cuda()
    kvq.kvq_kivi_prefill(cfg, cache, x[:1].contiguous(), x[:1].contiguous(), b0=0)   # 64 quantized + 128
    kvq.kvq_kivi_prefill(cfg, cache, x[1:, :, :10].contiguous(), x[1:, :, :10].contiguous(), b0=1)
    torch.cuda.synchronize()
    assert kvq.device_error() == 0
    before = [t.clone() for t in (cache.n_tok, cache.n_quant_k, cache.n_quant_v, cache.k_resid, cache.v_resid)]
    kvq.kvq_kivi_append(cfg, cache, x[:, :, 0].contiguous(), x[:, :, 1].contiguous())
    assert kvq.device_error() == kvq.ERR_CAPACITY
    assert cache.n_tok.tolist() == [192, 11] and cache.n_quant_k.tolist() == [64, 0]
    assert torch.equal(before[3][0], cache.k_resid[0]) and torch.equal(before[4][0], cache.v_resid[0])


def test_prefill_then_attention_integration():
    # each side quantizes the same fp16 K/V itself (prefill: 256 quantized + 40 fp16), then attends
    B, H, l = 2, 2, 296
    g, K, V = kv_data(320, B, H, l)
    cfg = kvq.KiviConfig(n_heads=H, residual=40 + 24, max_batch=B, max_tokens=256)
    cache = kvq.KiviCache(cfg)
    kvq.kvq_kivi_prefill(cfg, cache, torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    torch.cuda.synchronize()
    assert cache.n_quant_k.tolist() == [256, 256] and cache.n_tok.tolist() == [l, l]
    q = synth.bf16_round(synth.gaussian(g, (B, H, D)))
    out = torch.empty((B, H, D), dtype=torch.float32, device="cuda")
    kvq.kvq_decode_attn(cfg, cache, 0, 1, C.bf16_tensor(q), out)
    got = out.cpu().numpy()
    for b in range(B):
        for h in range(H):
            st = okivi.KiviStream(D, 32, cfg.residual)
            st.prefill(K[b, h], V[b, h])
            assert st.n_quant_k == 256
            C.check_close(got[b, h], st.attention(q[b, h]))
