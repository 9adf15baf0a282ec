"""GPU parity of LoopVQ decode attention (kvq_decode_attn, format LoopVQ) against the fp64
oracle, on the same seeded inputs. Tolerance: max-abs 2e-3 and relative L2 1e-3 on the
fp32-output mode; the bf16 output must be the bf16 rounding of the fp32 result."""
import os

import numpy as np
import pytest
import torch

from sub_bit_quantized_gb300 import kvq
from tests import _cases as C

pytestmark = pytest.mark.gpu
D = 128


def run_attn(case, cache, t, n_splits=0, out_dtype=torch.float32, ws=None):
    c = case.cfg
    B = len(case.lens)
    q = C.bf16_tensor(case.q)
    out = torch.empty((B, c.n_heads, 128), dtype=out_dtype, device="cuda")
    if ws is None:
        ws = kvq.make_workspace(c, B, n_splits)
    kvq.kvq_decode_attn(c, cache, 0, t, q, out, n_splits, ws)
    torch.cuda.synchronize()
    assert kvq.device_error() == 0
    return out


def check_all(case, cache, steps=(1, 2, 3, 4), n_splits=0, pairs=None):
    errs = []
    for t in steps:
        out = run_attn(case, cache, t, n_splits).cpu().numpy().astype(np.float64)
        sel = pairs or [(b, h) for b in range(len(case.lens)) for h in range(case.cfg.n_heads)]
        got = np.stack([out[b, h] for b, h in sel])
        ref = np.stack([C.oracle_vq(case, b, h, t) for b, h in sel])
        errs.append(C.check_close(got, ref))
    return errs


def test_tiny_config_every_loop_step():
    # 1 layer, 1 head, T=4, Tc=2, G=16, batch 1, context 512: 55 pages + 8 sink + 64 recent
    case = C.make_vq_case(100, B=1, H=1, lens=[512])
    assert case.n_pages == [55]
    cache = C.fill_vq_cache(case)
    check_all(case, cache)


@pytest.mark.parametrize("n_splits", [0, 1, 2, 3, 7, 64, 152])
def test_split_counts_and_odd_batch(n_splits):
    # ragged batch of 3; lengths give 0, 1 and 55 pages (112 pages over 2 heads: with 64 blocks
    # segments are merged across many blocks, with 152 some blocks hold no page at all)
    case = C.make_vq_case(101, B=3, H=2, lens=[73, 80, 513])
    assert case.n_pages == [0, 1, 55]
    cache = C.fill_vq_cache(case)
    check_all(case, cache, steps=(1, 4), n_splits=n_splits)


@pytest.mark.parametrize("lens", [[1], [5], [8], [72], [79], [80], [81], [8 + 64 + 8 * 7 + 7]])
def test_short_and_boundary_contexts(lens):
    case = C.make_vq_case(102, B=1, H=1, lens=lens)
    cache = C.fill_vq_cache(case)
    check_all(case, cache, steps=(1, 3))


def test_bf16_output_is_rounded_fp32_output():
    case = C.make_vq_case(103, B=2, H=2, lens=[300, 301])
    cache = C.fill_vq_cache(case)
    o32 = run_attn(case, cache, 2, out_dtype=torch.float32)
    o16 = run_attn(case, cache, 2, out_dtype=torch.bfloat16)
    assert torch.equal(o32.to(torch.bfloat16), o16)
    ref = np.stack([C.oracle_vq(case, b, h, 2) for b in range(2) for h in range(2)])
    got = o16.float().cpu().numpy().reshape(4, 128)
    f32 = o32.cpu().numpy().astype(np.float64).reshape(4, 128)
    # bf16 rounding moves the fp32 result by at most half a bf16 ulp of the rounded value, so
    # the bf16 output is off the fp64 oracle by at most that plus the fp32 result's own error
    half_ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(got), 2.0 ** -126))) - 8)
    assert np.all(np.abs(got - ref) <= half_ulp + np.abs(f32 - ref))
    C.check_close(f32, ref)


def test_quarter_bit_long_context_layout():
    # Tc=4, G=32 (0.25 bit), recent 256: shape of the long-context workload, smaller context
    case = C.make_vq_case(104, B=2, H=2, lens=[8 + 256 + 8 * 300 + 5, 8 + 256 + 8 * 123], T=4, Tc=4, G=32,
                          recent=256, rho=(0.85, 0.85))
    cache = C.fill_vq_cache(case)
    check_all(case, cache, steps=(1, 2, 3, 4), n_splits=64)
    check_all(case, cache, steps=(3,), n_splits=0)


@pytest.mark.parametrize("Tc", [1, 4])
def test_half_bit_loop_grouping_variants(Tc):
    # 0.5 bit (G = 16) with Tc = 1 (c = 16: per-step codewords, 8 index groups per token,
    # 64-byte pages) and Tc = 4 (c = 4: one index serves all four steps, 32 groups, 256-byte
    # pages); ragged batch, every loop step, several split counts
    case = C.make_vq_case(108 + Tc, B=3, H=2, lens=[73, 8 + 64 + 8 * 70 + 3, 513], Tc=Tc, G=16)
    cache = C.fill_vq_cache(case)
    check_all(case, cache, steps=(1, 2, 3, 4))
    check_all(case, cache, steps=(2, 4), n_splits=7)


def test_repeated_calls_reuse_workspace():
    case = C.make_vq_case(105, B=4, H=3, lens=[600, 1000, 999, 1500])
    cache = C.fill_vq_cache(case)
    ws = kvq.make_workspace(case.cfg, len(case.lens), 5)
    outs = [run_attn(case, cache, 1, n_splits=5, ws=ws) for _ in range(3)]
    # the value weights are summed as integers (order-free) and every partial is merged in a
    # fixed order, so repeated calls on one workspace agree bit for bit; the merge counters
    # return to zero after each call
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    cnt = ws[: len(case.lens) * case.cfg.n_heads * 4].view(torch.int32)
    assert int(cnt.abs().sum()) == 0
    check_all(case, cache, steps=(1,), n_splits=5)


@pytest.mark.parametrize("n_splits", [1, 2, 5])
def test_long_segments_and_head_changes(n_splits):
    # 1000 and 460 pages per request: segments run over several sub-pieces of at most 448
    # pages, and a block's share crosses from one head to the next (restaging the key slice)
    case = C.make_vq_case(112, B=2, H=3, lens=[8 + 64 + 8 * 1000 + 3, 8 + 64 + 8 * 460])
    assert case.n_pages == [1000, 460]
    cache = C.fill_vq_cache(case)
    check_all(case, cache, steps=(1, 4), n_splits=n_splits)


def test_windows_only_batch():
    # no request has an index page yet (contexts up to sink + recent + 7): every output comes
    # from the bf16 window alone, spread over the blocks
    case = C.make_vq_case(113, B=5, H=2, lens=[1, 9, 40, 72, 79])
    assert case.n_pages == [0] * 5
    cache = C.fill_vq_cache(case)
    check_all(case, cache, steps=(2,), n_splits=3)
    check_all(case, cache, steps=(3,))


@pytest.mark.parametrize("cfgname", ["b64_ctx6144_half_bit", "b8_ctx32768_quarter_bit", "b64_ctx6144_half_bit_tc1",
                                     "b64_ctx6144_half_bit_tc4"])
def test_full_size_sampled(cfgname):
    # full workload sizes in the launch configuration the bench uses (automatic split);
    # the oracle evaluates a sample of (request, head) pairs one by one
    if cfgname.startswith("b64_ctx6144_half_bit"):
        Tc = {"b64_ctx6144_half_bit": 2, "b64_ctx6144_half_bit_tc1": 1, "b64_ctx6144_half_bit_tc4": 4}[cfgname]
        case = C.make_vq_case(106, B=64, H=16, lens=[6144] * 64, Tc=Tc, G=16)
        steps = (1, 2, 3, 4)
    else:
        case = C.make_vq_case(107, B=8, H=16, lens=[32768] * 8, Tc=4, G=32, recent=256, rho=(0.85, 0.85))
        steps = (1, 4)
    cache = C.fill_vq_cache(case)
    rng = np.random.default_rng(7)
    pairs = [(int(b), int(h)) for b, h in zip(rng.integers(0, len(case.lens), 6), rng.integers(0, 16, 6))]
    pairs += [(0, 0), (len(case.lens) - 1, 15)]
    check_all(case, cache, steps=steps, pairs=pairs)
    if cfgname == "b8_ctx32768_quarter_bit":
        check_all(case, cache, steps=(2,), n_splits=64, pairs=pairs[:3])


def _oracle_encoded_pair(args):
    """Oracle side of one (request, head) of the prefill-encoded full-size case: encode the
    pages of each step's block from the same synthetic K/V, then decode attention (runs in a
    spawned worker)."""
    from oracle import loopvq as olv
    xk, xv, cbk, cbv, q, L, npg, Tc, steps = args
    qpos = np.arange(8, 8 + 8 * npg)
    refs = []
    for t in steps:
        beta, _ = olv.step_to_block(t, Tc)
        ik, _ = olv.encode_block(xk[:, qpos], cbk[beta], beta, Tc)
        iv, _ = olv.encode_block(xv[:, qpos], cbv[beta], beta, Tc)
        refs.append(olv.decode_attention(q, t, Tc, L, npg, ik, iv, cbk[beta], cbv[beta], xk[t - 1, :L], xv[t - 1, :L]))
    return refs


def test_full_size_prefill_encoded():
    # batch 64, 16 heads, context 6144, 0.5 bit (Tc = 2) in the bench's launch configuration,
    # on a cache filled by the library's own prefill encode (the index distribution the bench
    # times); 8 requests of seeded loop-correlated K/V are generated and request b holds the
    # data of request b % 8. 32 (request, head) pairs, one step of each loop block, are
    # checked against the oracle, which encodes the same K/V itself (spawned worker pool).
    import multiprocessing as mp

    import synth
    from oracle import loopvq as olv

    B, H, L, T, Tc, G, NSRC = 64, 16, 6144, 4, 2, 16, 8
    g = synth.rng(120)
    rhos = synth.rho_schedule(T, 0.69, 0.94)
    outl = [synth.outlier_channels(g, D, 4) for _ in range(H)]
    xk = np.empty((NSRC, T, H, L, D), np.float32)
    xv = np.empty_like(xk)
    for r in range(NSRC):
        for h in range(H):
            xk[r, :, h] = synth.bf16_round(synth.scale_channels(synth.loop_correlated(g, T, L, D, rhos), outl[h], 15.0))
            xv[r, :, h] = synth.bf16_round(synth.loop_correlated(g, T, L, D, rhos))
    cbk = np.stack([synth.sample_codebooks(g, xk[:, :, h].transpose(1, 0, 2, 3).reshape(T, NSRC * L, D)[:, ::7], Tc, G)
                    for h in range(H)], axis=1)
    cbv = np.stack([synth.sample_codebooks(g, xv[:, :, h].transpose(1, 0, 2, 3).reshape(T, NSRC * L, D)[:, ::7], Tc, G)
                    for h in range(H)], axis=1)
    npg = olv.prefill_split(L)[1]
    cfg = kvq.VqConfig(T=T, Tc=Tc, G=G, n_heads=H, max_pages=npg, max_batch=B, max_ctx=L + 8)
    cache = kvq.VqCache(cfg)
    C.load_codebooks(cache, cbk, cbv)
    src = [(C.bf16_tensor(np.ascontiguousarray(xk[r][:, None])), C.bf16_tensor(np.ascontiguousarray(xv[r][:, None])))
           for r in range(NSRC)]
    for b in range(B):
        kvq.kvq_prefill_vq(cfg, cache, 0, src[b % NSRC][0], src[b % NSRC][1], b, L)
    del src
    torch.cuda.synchronize()
    assert kvq.device_error() == 0
    assert cache.n_pages.tolist() == [npg] * B
    q = synth.bf16_round(synth.gaussian(g, (B, H, D)))
    rng = np.random.default_rng(8)
    pairs = sorted({(int(b), int(h)) for b, h in zip(rng.integers(0, B, 64), rng.integers(0, H, 64))})[:30]
    pairs += [(0, 0), (B - 1, H - 1)]
    assert len(set(pairs)) >= 32
    steps = (2, 3)  # blocks 0 and 1
    outs = []
    for t in steps:
        out = torch.empty((B, H, D), dtype=torch.float32, device="cuda")
        kvq.kvq_decode_attn(cfg, cache, 0, t, C.bf16_tensor(q), out)
        torch.cuda.synchronize()
        assert kvq.device_error() == 0
        outs.append(out.cpu().numpy().astype(np.float64))
    jobs = [(xk[b % NSRC, :, h].astype(np.float64), xv[b % NSRC, :, h].astype(np.float64), cbk[:, h], cbv[:, h],
             q[b, h], L, npg, Tc, steps) for b, h in pairs]
    with mp.get_context("spawn").Pool(min(16, os.cpu_count() or 1)) as pool:
        refs = pool.map(_oracle_encoded_pair, jobs)
    for k, t in enumerate(steps):
        got = np.stack([outs[k][b, h] for b, h in pairs])
        ref = np.stack([r[k] for r in refs])
        C.check_close(got, ref)
