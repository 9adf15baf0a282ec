"""GPU parity of KIVI: group quantization (codes, fp16 scales and zero-points bit-exact with
the oracle's fixed fp32 sequence) and decode attention over quantized + fp16 residual
segments (max-abs 2e-3, relative L2 1e-3 against fp64)."""
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


def test_quantize_bit_exact():
    B, H, n = 2, 3, 96
    g, K, V = kv_data(300, B, H, n)
    cfg = kvq.KiviConfig(n_heads=H, max_batch=B, max_tokens=160)
    cache = kvq.KiviCache(cfg)
    kvq.kvq_quantize_kivi(cfg, kvq.PER_CHANNEL, torch.from_numpy(K).cuda(), cache.k_codes, cache.k_scale,
                          cache.k_zero, tok_begin=32)
    kvq.kvq_quantize_kivi(cfg, kvq.PER_TOKEN, torch.from_numpy(V).cuda(), cache.v_codes, cache.v_scale,
                          cache.v_zero, tok_begin=32)
    torch.cuda.synchronize()
    kc = _layout.unpack_codes(cache.k_codes.cpu().numpy())
    vc = _layout.unpack_codes(cache.v_codes.cpu().numpy())
    ks, kz = cache.k_scale.cpu().numpy(), cache.k_zero.cpu().numpy()
    vs, vz = cache.v_scale.cpu().numpy(), cache.v_zero.cpu().numpy()
    for b in range(B):
        for h in range(H):
            c, s, z = okivi.quantize_keys(K[b, h])
            assert np.array_equal(kc[b, h, 32:32 + n], c)
            assert np.array_equal(ks[b, h, 1:1 + n // 32].view(np.uint16), s.view(np.uint16))
            assert np.array_equal(kz[b, h, 1:1 + n // 32].view(np.uint16), z.view(np.uint16))
            c, s, z = okivi.quantize_values(V[b, h])
            assert np.array_equal(vc[b, h, 32:32 + n], c)
            assert np.array_equal(vs[b, h, 32:32 + n].view(np.uint16), s.view(np.uint16))
            assert np.array_equal(vz[b, h, 32:32 + n].view(np.uint16), z.view(np.uint16))
    # untouched regions stay zero
    assert not kc[:, :, :32].any() and not vc[:, :, 128:].any()


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
    B, H = len(case.n_quant), case.cfg.n_heads
    out = torch.empty((B, H, D), dtype=dtype, device="cuda")
    ws = kvq.make_workspace(case.cfg, B, n_splits)
    kvq.kvq_decode_attn(case.cfg, cache, 0, 1, C.bf16_tensor(case.q), out, n_splits, ws)
    torch.cuda.synchronize()
    assert kvq.device_error() == 0
    return out


@pytest.mark.parametrize("n_splits", [0, 1, 3, 7])
def test_attention_segments_and_splits(n_splits):
    case = C.make_kivi_case(310, B=4, H=2, n_quant=[0, 96, 32 * 40, 32], n_resid=[17, 0, 128, 1])
    cache = C.fill_kivi_cache(case)
    got = run(case, cache, n_splits).cpu().numpy()
    ref = np.stack([[C.oracle_kivi(case, b, h) for h in range(2)] for b in range(4)])
    C.check_close(got, ref)


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


def test_quantize_then_attention_integration():
    # each side quantizes the same fp16 K/V itself, then attends
    B, H, nq, nr = 2, 2, 256, 40
    g, K, V = kv_data(320, B, H, nq + nr)
    cfg = kvq.KiviConfig(n_heads=H, max_batch=B, max_tokens=nq)
    cache = kvq.KiviCache(cfg)
    Kt, Vt = torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda()
    kvq.kvq_quantize_kivi(cfg, kvq.PER_CHANNEL, Kt[:, :, :nq].contiguous(), cache.k_codes, cache.k_scale, cache.k_zero)
    kvq.kvq_quantize_kivi(cfg, kvq.PER_TOKEN, Vt[:, :, :nq].contiguous(), cache.v_codes, cache.v_scale, cache.v_zero)
    cache.k_resid[:, :, :nr].copy_(Kt[:, :, nq:])
    cache.v_resid[:, :, :nr].copy_(Vt[:, :, nq:])
    cache.n_quant.fill_(nq)
    cache.n_resid.fill_(nr)
    q = synth.bf16_round(synth.gaussian(g, (B, H, D)))
    out = torch.empty((B, H, D), dtype=torch.float32, device="cuda")
    kvq.kvq_decode_attn(cfg, cache, 0, 1, C.bf16_tensor(q), out)
    got = out.cpu().numpy()
    for b in range(B):
        for h in range(H):
            ck, sk, zk = okivi.quantize_keys(K[b, h, :nq])
            cv, sv, zv = okivi.quantize_values(V[b, h, :nq])
            ref = okivi.decode_attention(q[b, h], ck, sk, zk, cv, sv, zv, K[b, h, nq:], V[b, h, nq:])
            C.check_close(got[b, h], ref)
