"""GPU parity of LoopVQ encode (kvq_encode_vq), prefill (kvq_prefill_vq) and the decode-time
append / page roll (kvq_append_page) against the oracle. Indices must equal the oracle's
exact-arithmetic argmin; a different index is accepted only inside the oracle's 1e-6
relative tie set, and such ties are counted."""
import numpy as np
import pytest
import torch

import synth
from oracle import loopvq as olv
from sub_bit_quantized_gb300 import kvq
from tests import _cases as C
from tests import _layout

pytestmark = pytest.mark.gpu
D = 128


def gen_kv(seed, B, H, L, T, rho=(0.69, 0.94)):
    g = synth.rng(seed)
    rhos = synth.rho_schedule(T, *rho)
    xk = np.empty((T, B, H, L, D))
    xv = np.empty((T, B, H, L, D))
    outl = [synth.outlier_channels(g, D, 4) for _ in range(H)]
    for b in range(B):
        for h in range(H):
            xk[:, b, h] = synth.bf16_round(synth.scale_channels(synth.loop_correlated(g, T, L, D, rhos), outl[h], 15.0))
            xv[:, b, h] = synth.bf16_round(synth.loop_correlated(g, T, L, D, rhos))
    return g, xk, xv


def codebooks(g, x, Tc, G):
    """[NB][H][NG][256][G] from all requests of x [T][B][H][L][D]."""
    T, B, H, L, _ = x.shape
    out = []
    for h in range(H):
        pool = x[:, :, h].reshape(T, B * L, D)
        out.append(synth.sample_codebooks(g, pool, Tc, G))
    return np.stack(out, axis=1)


def check_indices(got, want, ties):
    """got/want [n][NG]; ties [n][NG][256]. Returns the number of tie decisions."""
    diff = got != want
    if diff.any():
        jj, gg = np.nonzero(diff)
        assert ties[jj, gg, got[jj, gg]].all(), "index outside the tie set"
    return int(diff.sum())


@pytest.mark.parametrize("Tc,G", [(2, 16), (4, 32), (1, 8), (1, 16), (4, 16)])
def test_encode_matches_oracle(Tc, G):
    T, B, H, L = 4, 2, 2, 96
    g, xk, _ = gen_kv(200 + Tc, B, H, L, T)
    cb = codebooks(g, xk, Tc, G)
    cfg = kvq.VqConfig(T=T, Tc=Tc, G=G, n_heads=H, max_pages=L // 8 + 2, max_batch=B, max_ctx=L + 80)
    x = C.bf16_tensor(xk)
    idx = torch.full((cfg.NB, B, H, cfg.max_pages, 8 * cfg.NG), 0xEE, dtype=torch.uint8, device="cuda")
    ties = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_encode_vq(cfg, x, (B * H * L * D, H * L * D, L * D), 0, B, L, torch.from_numpy(cb).cuda(), idx,
                      page_begin=1, n_ties=ties)
    torch.cuda.synchronize()
    pages = idx.cpu().numpy()
    assert (pages[:, :, :, 0] == 0xEE).all() and (pages[:, :, :, L // 8 + 1:] == 0xEE).all()
    got = _layout.unpack_pages(pages[:, :, :, 1:L // 8 + 1], cfg.NG)
    n_tie = 0
    for beta in range(cfg.NB):
        for b in range(B):
            for h in range(H):
                want, tie = olv.encode_block(xk[:, b, h], cb[beta, h], beta, Tc)
                n_tie += check_indices(got[beta, b, h], want, tie)
    assert n_tie <= int(ties.item())


def test_encode_group_subset_and_exact_ties():
    T, Tc, G, B, H, L = 4, 2, 16, 1, 1, 16
    g, xk, _ = gen_kv(210, B, H, L, T)
    cb = codebooks(g, xk, Tc, G)
    # duplicate entries: entry 200 copies entry 7, so an exact tie must resolve to 7
    cb[:, :, :, 200] = cb[:, :, :, 7]
    # make token 3's coupled vectors equal to entry 7 exactly (bf16-representable)
    cb[:, :, :, 7] = synth.bf16_round(cb[:, :, :, 7]).astype(np.float32)
    cb[:, :, :, 200] = cb[:, :, :, 7]
    for beta in range(T // Tc):
        for gg in range(D // 8):
            e = cb[beta, 0, gg, 7]
            for i in range(8):
                for m in range(Tc):
                    xk[beta * Tc + m, 0, 0, 3, gg * 8 + i] = e[i * Tc + m]
    cfg = kvq.VqConfig(T=T, Tc=Tc, G=G, n_heads=H, max_pages=4, max_batch=B, max_ctx=128)
    idx = torch.full((cfg.NB, B, H, 4, 128), 0xEE, dtype=torch.uint8, device="cuda")
    kvq.kvq_encode_vq(cfg, C.bf16_tensor(xk), (B * H * L * D, H * L * D, L * D), 0, B, L,
                      torch.from_numpy(cb).cuda(), idx, g_begin=3, g_count=9)
    torch.cuda.synchronize()
    got = _layout.unpack_pages(idx.cpu().numpy()[:, :, :, :2], 16)
    for beta in range(2):
        want, tie = olv.encode_block(xk[:, 0, 0], cb[beta, 0], beta, Tc)
        assert (got[beta, 0, 0, :, :3] == 0xEE).all() and (got[beta, 0, 0, :, 12:] == 0xEE).all()
        assert (got[beta, 0, 0, 3, 3:12] == 7).all()
        check_indices(got[beta, 0, 0, :, 3:12], want[:, 3:12], tie[:, 3:12])


@pytest.mark.parametrize("copies", [2, 3])
def test_encode_duplicated_codebook_ties(copies):
    """Every codeword repeated `copies` times (entry r + k * 256 // copies copies entry r), so
    every vector has `copies` exact-tie candidates: the lowest copy must win each one. Two
    copies fill a warp's near-tie list exactly (32 rows x 2 pairs); three overflow it and take
    the row-by-row path."""
    T, Tc, G, B, H, L = 4, 2, 16, 1, 1, 160
    g, xk, _ = gen_kv(220 + copies, B, H, L, T)
    cb = codebooks(g, xk, Tc, G)
    span = 256 // copies
    for k in range(1, copies):
        cb[:, :, :, k * span:(k + 1) * span] = cb[:, :, :, :span]
    cb[:, :, :, copies * span:] = cb[:, :, :, :256 - copies * span]  # the remainder copies too
    cfg = kvq.VqConfig(T=T, Tc=Tc, G=G, n_heads=H, max_pages=L // 8, max_batch=B, max_ctx=L + 80)
    idx = torch.zeros((cfg.NB, B, H, L // 8, 128), dtype=torch.uint8, device="cuda")
    ties = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_encode_vq(cfg, C.bf16_tensor(xk), (B * H * L * D, H * L * D, L * D), 0, B, L,
                      torch.from_numpy(cb).cuda(), idx, n_ties=ties)
    torch.cuda.synchronize()
    got = _layout.unpack_pages(idx.cpu().numpy(), 16)
    for beta in range(T // Tc):
        want, tie = olv.encode_block(xk[:, 0, 0], cb[beta, 0], beta, Tc)
        check_indices(got[beta, 0, 0], want, tie)
        assert (want < span).all()
        assert (got[beta, 0, 0] < span).all(), "an exact tie went to a higher copy"
    assert int(ties.item()) >= (T // Tc) * L * 16  # every vector has a tie


def test_encode_full_size_sampled():
    # prefill encode workload: 16 heads x 8 channel groups x 2 loop blocks x 32768 tokens
    T, Tc, G, H, L = 4, 2, 16, 16, 32768
    gen = torch.Generator(device="cuda").manual_seed(2024)
    x32 = synth.torch_loop_correlated(gen, T, (1, H, L, D), synth.rho_schedule(T))
    outl = torch.randperm(D, generator=gen, device="cuda")[:4]
    x32[..., outl] *= 15.0
    x = x32.to(torch.bfloat16).contiguous()
    del x32
    g = synth.rng(2025)
    cfg = kvq.VqConfig(T=T, Tc=Tc, G=G, n_heads=H, max_pages=L // 8, max_batch=1, max_ctx=L + 80)
    sample_tok = torch.randint(0, L, (4096,), generator=gen, device="cuda")
    xs = x[:, 0, :, sample_tok].float().cpu().numpy()           # [T][H][4096][D]
    cb = np.stack([synth.sample_codebooks(g, xs[:, h], Tc, G) for h in range(H)], axis=1)
    cb += synth.gaussian(g, cb.shape, 0.05).astype(np.float32)   # keep codewords off the data
    idx = torch.zeros((cfg.NB, 1, H, cfg.max_pages, 128), dtype=torch.uint8, device="cuda")
    ties = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_encode_vq(cfg, x, (H * L * D, H * L * D, L * D), 0, 1, L, torch.from_numpy(cb).cuda(), idx,
                      g_begin=0, g_count=8, n_ties=ties)
    torch.cuda.synchronize()
    rs = np.random.default_rng(3)
    toks = rs.integers(0, L, 400)
    heads = rs.integers(0, H, 400)
    pages = idx.cpu().numpy()
    n_tie = 0
    for tok, h in zip(toks, heads):
        xt = x[:, 0, int(h), int(tok)].float().cpu().numpy()[:, None, :]    # [T][1][D]
        for beta in range(2):
            want, tie = olv.encode_block(xt, cb[beta, h], beta, Tc)
            got = _layout.unpack_pages(pages[beta, 0, h, tok // 8][None], 16)[tok % 8][None]
            n_tie += check_indices(got[:, :8], want[:, :8], tie[:, :8])
    assert n_tie <= int(ties.item())


@pytest.mark.parametrize("Tc", [2, 1, 4])
def test_prefill_then_attention_integration(Tc):
    # each side runs its own pipeline from the same synthetic K/V: GPU prefill (encode +
    # windows) then GPU attention, against oracle encode then oracle attention; at 0.5 bit
    # with Tc = 2 (c = 8), Tc = 1 (c = 16) and Tc = 4 (c = 4)
    T, G, B, H = 4, 16, 3, 2
    lens = [200, 77, 8 + 64 + 8 * 20 + 3]
    Lmax = max(lens)
    g, xk, xv = gen_kv(220, B, H, Lmax, T)
    cbk = codebooks(g, xk, Tc, G)
    cbv = codebooks(g, xv, Tc, G)
    cfg = kvq.VqConfig(T=T, Tc=Tc, G=G, n_heads=H, max_pages=40, max_batch=B, max_ctx=Lmax + 8)
    cache = kvq.VqCache(cfg)
    C.load_codebooks(cache, cbk, cbv)
    xk_t, xv_t = C.bf16_tensor(xk), C.bf16_tensor(xv)
    for b, L in enumerate(lens):
        kvq.kvq_prefill_vq(cfg, cache, 0, xk_t[:, b:b + 1].contiguous(), xv_t[:, b:b + 1].contiguous(), b, L)
    torch.cuda.synchronize()
    n_pages = [olv.prefill_split(L)[1] for L in lens]
    assert cache.seq_len.tolist() == lens and cache.n_pages.tolist() == n_pages
    q = synth.bf16_round(synth.gaussian(g, (B, H, D)))
    out = torch.empty((B, H, D), dtype=torch.float32, device="cuda")
    pk = _layout.unpack_pages(cache.idx_k[0].cpu().numpy(), cfg.NG)
    pv = _layout.unpack_pages(cache.idx_v[0].cpu().numpy(), cfg.NG)
    for t in (1, 2, 3, 4):
        kvq.kvq_decode_attn(cfg, cache, 0, t, C.bf16_tensor(q), out)
        got = out.cpu().numpy()
        beta, _ = olv.step_to_block(t, Tc)
        for b, L in enumerate(lens):
            npg = n_pages[b]
            qpos = np.arange(8, 8 + 8 * npg)
            for h in range(H):
                ik, tk = olv.encode_block(xk[:, b, h, qpos], cbk[beta, h], beta, Tc)
                iv, tv = olv.encode_block(xv[:, b, h, qpos], cbv[beta, h], beta, Tc)
                assert check_indices(pk[beta, b, h, :8 * npg], ik, tk) == 0
                assert check_indices(pv[beta, b, h, :8 * npg], iv, tv) == 0
                ref = olv.decode_attention(q[b, h], t, Tc, L, npg, ik, iv, cbk[beta, h], cbv[beta, h],
                                           xk[t - 1, b, h, :L], xv[t - 1, b, h, :L])
                C.check_close(got[b, h], ref)


def test_split_codebook_parts_sum_back():
    # kvq_split_codebooks: in the tensor-core operand layout (row groups of 8 rows x 16-byte
    # chunks), hi + mid + lo of every coordinate is the fp32 entry exactly, and the augmented
    # chunk's first element carries -|e|^2/2 (its parts summed); the rest is zero
    for Tc, G in ((2, 16), (4, 32), (1, 8)):
        C_ = G // Tc
        cfg = kvq.VqConfig(T=4, Tc=Tc, G=G, n_layers=1, n_heads=1, max_pages=4, max_batch=1, max_ctx=64)
        rng = np.random.default_rng(11 + G)
        cb = (rng.standard_normal((1, cfg.NB, 1, cfg.NG, 256, G)) * rng.choice([1.0, 15.0], size=G)).astype(np.float32)
        cbp = torch.zeros(kvq.vq_cache_sizes(cfg).cbp, dtype=torch.uint8, device="cuda")
        kvq.kvq_split_codebooks(cfg, torch.from_numpy(cb).cuda(), cbp)
        raw = cbp.cpu().numpy()
        DC = G // 8
        KC = 2 * ((DC + 2) // 2)
        part = 256 * KC * 16
        n_cb = cfg.NB * cfg.NG
        words = raw.reshape(n_cb, 3, 256 // 8, KC, 8, 16).view(np.uint16)  # [cb][part][rg][chunk][row][8 bf16]
        vals = (words.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        total = vals.sum(axis=1)  # hi + mid + lo, exact in float64
        flat = cb.reshape(n_cb, 256, G).astype(np.float64)
        rows = np.arange(256)
        for c in range(DC):
            for i in range(8):
                kk = 8 * c + i
                coord = (kk % C_) * Tc + kk // C_
                got = total[:, rows // 8, c, rows % 8, i]
                assert np.array_equal(got, flat[:, :, coord]), (G, c, i)
        nh = total[:, rows // 8, DC, rows % 8, 0]
        want = -0.5 * (flat ** 2).sum(axis=2)
        assert np.allclose(nh, want, rtol=1e-6, atol=0)
        rest = total[:, :, DC:, :, :].copy()
        rest[:, :, 0, :, 0] = 0.0
        assert not rest.any()


@pytest.mark.parametrize("path", ["tensor", "cuda"])
@pytest.mark.parametrize("Tc", [2, 1, 4])
def test_append_and_roll_equal_prefill_encoding(Tc, path):
    # stream 40 tokens through kvq_append_page (2 layers x 4 loop steps each): the rolled
    # pages must equal the oracle's encoding of the same tokens, lengths must follow the
    # sink / page / recent rule, and attention must match the oracle at the end
    T, G, B, H, NL = 4, 16, 2, 2, 2
    L0 = [101, 90]
    n_new = 40
    Lmax = max(L0) + n_new
    g, xk, xv = gen_kv(230, B, H, Lmax, T)
    xk2 = np.stack([xk, np.flip(xk, axis=3)])          # layer 1 uses other data
    xv2 = np.stack([xv, np.flip(xv, axis=3)])
    cbk = np.stack([codebooks(g, xk2[l], Tc, G) for l in range(NL)])
    cbv = np.stack([codebooks(g, xv2[l], Tc, G) for l in range(NL)])
    cfg = kvq.VqConfig(T=T, Tc=Tc, G=G, n_layers=NL, n_heads=H, max_pages=16, max_batch=B, max_ctx=Lmax)
    cache = kvq.VqCache(cfg)
    cache.load_codebooks(torch.from_numpy(cbk).cuda(), torch.from_numpy(cbv).cuda())
    if path == "cuda":  # no split codebook parts: the roll runs on CUDA cores
        cache.cbp_k = cache.cbp_v = None
    xk_t = [C.bf16_tensor(np.ascontiguousarray(xk2[l])) for l in range(NL)]
    xv_t = [C.bf16_tensor(np.ascontiguousarray(xv2[l])) for l in range(NL)]
    for l in range(NL):
        for b in range(B):
            kvq.kvq_prefill_vq(cfg, cache, l, xk_t[l][:, b:b + 1].contiguous(), xv_t[l][:, b:b + 1].contiguous(),
                               b, L0[b])
    lens = list(L0)
    for step in range(n_new):
        for l in range(NL):
            for t in range(1, T + 1):
                kn = torch.stack([xk_t[l][t - 1, b, :, lens[b]] for b in range(B)]).contiguous()
                vn = torch.stack([xv_t[l][t - 1, b, :, lens[b]] for b in range(B)]).contiguous()
                kvq.kvq_append_page(cfg, cache, l, t, kn, vn)
        lens = [x + 1 for x in lens]
        torch.cuda.synchronize()
        assert cache.seq_len.tolist() == lens
        assert cache.n_pages.tolist() == [olv.prefill_split(x)[1] for x in lens]
    assert kvq.device_error() == 0
    for l in range(NL):
        for name, x2, cb in (("idx_k", xk2, cbk), ("idx_v", xv2, cbv)):
            pages = _layout.unpack_pages(getattr(cache, name)[l].cpu().numpy(), cfg.NG)
            for b in range(B):
                npg = olv.prefill_split(lens[b])[1]
                qpos = np.arange(8, 8 + 8 * npg)
                for h in range(H):
                    for beta in range(T // Tc):
                        want, tie = olv.encode_block(x2[l][:, b, h, qpos], cb[l, beta, h], beta, Tc)
                        assert check_indices(pages[beta, b, h, :8 * npg], want, tie) == 0
    q = synth.bf16_round(synth.gaussian(g, (B, H, D)))
    out = torch.empty((B, H, D), dtype=torch.float32, device="cuda")
    for l, t in ((0, 1), (1, 4)):
        kvq.kvq_decode_attn(cfg, cache, l, t, C.bf16_tensor(q), out)
        got = out.cpu().numpy()
        beta, _ = olv.step_to_block(t, Tc)
        for b in range(B):
            L = lens[b]
            npg = olv.prefill_split(L)[1]
            qpos = np.arange(8, 8 + 8 * npg)
            for h in range(H):
                ik, _ = olv.encode_block(xk2[l][:, b, h, qpos], cbk[l, beta, h], beta, Tc)
                iv, _ = olv.encode_block(xv2[l][:, b, h, qpos], cbv[l, beta, h], beta, Tc)
                ref = olv.decode_attention(q[b, h], t, Tc, L, npg, ik, iv, cbk[l, beta, h], cbv[l, beta, h],
                                           xk2[l][t - 1, b, h, :L], xv2[l][t - 1, b, h, :L])
                C.check_close(got[b, h], ref)
