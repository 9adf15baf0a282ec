"""Seeded LoopVQ / KIVI test cases: host data from ``synth``, GPU caches filled through the
library, and the oracle evaluated on the same host data (test infrastructure)."""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import synth
from oracle import kivi as okivi
from oracle import loopvq as olv
from sub_bit_quantized_gb300 import kvq
from tests import _layout

D = 128


def bf16_tensor(x: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(synth.bf16_bits(x).view(np.int16)).view(torch.bfloat16).to(device)


def fp16_tensor(x: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.asarray(x, dtype=np.float16)).to(device)


@dataclass
class VqCase:
    cfg: kvq.VqConfig
    lens: list
    n_pages: list
    bf_pos: list              # per request: positions kept in bf16 (sink + recent)
    wk: np.ndarray            # [B][H][T][max_nbf][D] bf16 values of those positions
    wv: np.ndarray
    cb_k: np.ndarray          # [NB][H][NG][256][G] float32
    cb_v: np.ndarray
    idx_k: np.ndarray         # [NB][B][H][max_pages*8][NG] logical indices
    idx_v: np.ndarray
    q: np.ndarray             # [B][H][D] bf16 values


def make_vq_case(seed, B, H, lens, T=4, Tc=2, G=16, recent=64, rho=(0.69, 0.94), pool=2048) -> VqCase:
    """Attention-only case: bf16 window tokens and codebooks from the loop-correlated
    generator (keys with 4 outlier channels x15), uniformly random index pages."""
    g = synth.rng(seed)
    n_pages = [olv.prefill_split(L, 8, recent)[1] for L in lens]
    cfg = kvq.VqConfig(T=T, Tc=Tc, G=G, n_heads=H, recent=recent, max_pages=max(max(n_pages), 1),
                       max_batch=B, max_ctx=max(max(lens), 2))
    rhos = synth.rho_schedule(T, *rho)
    bf_pos = [olv.cache_positions(L, n)[0] for L, n in zip(lens, n_pages)]
    nbf = max(len(p) for p in bf_pos)
    wk = np.zeros((B, H, T, nbf, D))
    wv = np.zeros_like(wk)
    cb_k = np.empty((cfg.NB, H, cfg.NG, 256, G), np.float32)
    cb_v = np.empty_like(cb_k)
    for h in range(H):
        outl = synth.outlier_channels(g, D, 4)
        pk = synth.scale_channels(synth.loop_correlated(g, T, pool, D, rhos), outl, 15.0)
        pv = synth.loop_correlated(g, T, pool, D, rhos)
        cb_k[:, h] = synth.sample_codebooks(g, pk, Tc, G)
        cb_v[:, h] = synth.sample_codebooks(g, pv, Tc, G)
        for b in range(B):
            n = len(bf_pos[b])
            k = synth.scale_channels(synth.loop_correlated(g, T, n, D, rhos), outl, 15.0)
            wk[b, h, :, :n] = synth.bf16_round(k)
            wv[b, h, :, :n] = synth.bf16_round(synth.loop_correlated(g, T, n, D, rhos))
    shape = (cfg.NB, B, H, cfg.max_pages * 8, cfg.NG)
    idx_k = synth.random_indices(g, shape)
    idx_v = synth.random_indices(g, shape)
    q = synth.bf16_round(synth.gaussian(g, (B, H, D)))
    return VqCase(cfg, list(lens), n_pages, bf_pos, wk, wv, cb_k, cb_v, idx_k, idx_v, q)


def load_codebooks(cache: kvq.VqCache, cb_k: np.ndarray, cb_v: np.ndarray):
    L = cache.cfg.n_layers
    cbk = np.array(np.broadcast_to(cb_k, (L,) + cb_k.shape))
    cbv = np.array(np.broadcast_to(cb_v, (L,) + cb_v.shape))
    cache.load_codebooks(torch.from_numpy(cbk).cuda(), torch.from_numpy(cbv).cuda())


def fill_vq_cache(case: VqCase, layer: int = 0) -> kvq.VqCache:
    """GPU cache holding the case's codebooks, bf16 windows and index pages."""
    c = case.cfg
    cache = kvq.VqCache(c)
    load_codebooks(cache, case.cb_k, case.cb_v)
    B, H = len(case.lens), c.n_heads
    win_k = np.zeros((c.T, B, H, c.win_slots, D))
    win_v = np.zeros_like(win_k)
    for b in range(B):
        for w, p in enumerate(case.bf_pos[b]):
            s = _layout.window_slot(int(p), c.sink, c.recent)
            win_k[:, b, :, s] = case.wk[b, :, :, w].transpose(1, 0, 2)
            win_v[:, b, :, s] = case.wv[b, :, :, w].transpose(1, 0, 2)
    cache.win_k[layer].copy_(bf16_tensor(win_k))
    cache.win_v[layer].copy_(bf16_tensor(win_v))
    cache.idx_k[layer].copy_(torch.from_numpy(_layout.pack_pages(case.idx_k)).cuda())
    cache.idx_v[layer].copy_(torch.from_numpy(_layout.pack_pages(case.idx_v)).cuda())
    cache.seq_len.copy_(torch.tensor(case.lens, dtype=torch.int32))
    cache.n_pages.copy_(torch.tensor(case.n_pages, dtype=torch.int32))
    return cache


def oracle_vq(case: VqCase, b: int, h: int, t: int) -> np.ndarray:
    c = case.cfg
    beta, _ = olv.step_to_block(t, c.Tc)
    L, npg = case.lens[b], case.n_pages[b]
    wk = np.zeros((L, D))
    wv = np.zeros((L, D))
    n = len(case.bf_pos[b])
    wk[case.bf_pos[b]] = case.wk[b, h, t - 1, :n]
    wv[case.bf_pos[b]] = case.wv[b, h, t - 1, :n]
    return olv.decode_attention(case.q[b, h], t, c.Tc, L, npg, case.idx_k[beta, b, h, :8 * npg],
                                case.idx_v[beta, b, h, :8 * npg], case.cb_k[beta, h], case.cb_v[beta, h],
                                wk, wv)


def check_close(got: np.ndarray, ref: np.ndarray, max_abs=2e-3, rel_l2=1e-3):
    err = np.abs(got - ref)
    rl2 = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err.max() <= max_abs, f"max-abs {err.max():.3e} > {max_abs}"
    assert rl2 <= rel_l2, f"rel-L2 {rl2:.3e} > {rel_l2}"
    return float(err.max()), float(rl2)


# ------------------------------------------------------------------------------------ KIVI

@dataclass
class KiviCase:
    cfg: kvq.KiviConfig
    n_tok: list
    n_quant_k: list
    n_quant_v: list
    k_codes: np.ndarray   # [B][H][N][D] int
    k_scale: np.ndarray   # [B][H][N/32][D] fp16
    k_zero: np.ndarray
    v_codes: np.ndarray
    v_scale: np.ndarray   # [B][H][N][D/32]
    v_zero: np.ndarray
    k_res: np.ndarray     # [B][H][R][D] fp16: row i is token n_quant_k + i
    v_res: np.ndarray     # [B][H][R][D] fp16: row i is token n_quant_v + i
    q: np.ndarray         # [B][Hq][D] bf16 values


def make_kivi_case(seed, B, H, n_quant, n_resid, max_tokens=None, residual=128, Hq=None, k_bits=2, v_bits=2,
                   n_quant_v=None) -> KiviCase:
    """Random codes and fp16 scales / zero-points of the shapes KIVI stores (attention-only).

    Request b holds n_quant[b] quantized keys and n_resid[b] fp16 keys; its values are
    quantized for tokens below n_quant_v[b] (default n_quant[b]) and fp16 above."""
    g = synth.rng(seed)
    N = max_tokens or max(max(n_quant), 32)
    Hq = Hq or H
    cfg = kvq.KiviConfig(n_heads=H, n_q_heads=Hq, k_bits=k_bits, v_bits=v_bits, residual=residual,
                         max_batch=B, max_tokens=N)
    kc = g.integers(0, 2 ** k_bits, size=(B, H, N, D), dtype=np.uint8)
    vc = g.integers(0, 2 ** v_bits, size=(B, H, N, D), dtype=np.uint8)
    # scales shrink with more levels so dequantized values keep the same range
    ks = (np.abs(synth.gaussian(g, (B, H, N // 32, D), 0.7)) * 3 / (2 ** k_bits - 1)).astype(np.float16)
    ks += np.float16(0.05)
    outl = synth.outlier_channels(g, D, 6)
    ks[..., outl] *= np.float16(20)
    kz = np.asarray(synth.gaussian(g, (B, H, N // 32, D), 1.5) * (2 ** k_bits - 1) / 3, np.float16)
    vs = ((np.abs(synth.gaussian(g, (B, H, N, D // 32), 0.7)) + 0.05) * 3 / (2 ** v_bits - 1)).astype(np.float16)
    vz = np.asarray(synth.gaussian(g, (B, H, N, D // 32), 1.5) * (2 ** v_bits - 1) / 3, np.float16)
    R = max(residual, 1)
    kr, vr = synth.kivi_kv(g, B * H * R, D, outl)
    kr = kr.reshape(B, H, R, D).astype(np.float16)
    vr = vr.reshape(B, H, R, D).astype(np.float16)
    q = synth.bf16_round(synth.gaussian(g, (B, Hq, D)))
    nqv = list(n_quant) if n_quant_v is None else list(n_quant_v)
    n_tok = [a + r for a, r in zip(n_quant, n_resid)]
    return KiviCase(cfg, n_tok, list(n_quant), nqv, kc, ks, kz, vc, vs, vz, kr, vr, q)


def fill_kivi_cache(case: KiviCase) -> kvq.KiviCache:
    cfg = case.cfg
    cache = kvq.KiviCache(cfg)
    cache.k_codes.copy_(torch.from_numpy(_layout.pack_codes(case.k_codes, cfg.k_bits)))
    cache.v_codes.copy_(torch.from_numpy(_layout.pack_codes(case.v_codes, cfg.v_bits)))
    for name in ("k_scale", "k_zero", "v_scale", "v_zero"):
        getattr(cache, name).copy_(fp16_tensor(getattr(case, name)))
    cache.k_resid.copy_(fp16_tensor(case.k_res))
    if cfg.residual > 0:   # value of token t at ring row t % R
        vr = np.zeros_like(case.v_res)
        for b, (n, nqv) in enumerate(zip(case.n_tok, case.n_quant_v)):
            for i in range(n - nqv):
                vr[b, :, (nqv + i) % cfg.residual] = case.v_res[b, :, i]
        cache.v_resid.copy_(fp16_tensor(vr))
    cache.n_tok.copy_(torch.tensor(case.n_tok, dtype=torch.int32))
    cache.n_quant_k.copy_(torch.tensor(case.n_quant_k, dtype=torch.int32))
    cache.n_quant_v.copy_(torch.tensor(case.n_quant_v, dtype=torch.int32))
    return cache


def oracle_kivi(case: KiviCase, b: int, hq: int) -> np.ndarray:
    hk = okivi.kv_head(hq, case.cfg.q_heads, case.cfg.n_heads)
    n, nqk, nqv = case.n_tok[b], case.n_quant_k[b], case.n_quant_v[b]
    return okivi.decode_attention(case.q[b, hq], case.k_codes[b, hk, :nqk], case.k_scale[b, hk, :nqk // 32],
                                  case.k_zero[b, hk, :nqk // 32], case.v_codes[b, hk, :nqv],
                                  case.v_scale[b, hk, :nqv], case.v_zero[b, hk, :nqv],
                                  case.k_res[b, hk, :n - nqk], case.v_res[b, hk, :n - nqv])
