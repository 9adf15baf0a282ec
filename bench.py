"""Benchmark: LoopVQ 0.5-bit decode attention, Ouro-1.4B-shaped serving step on one GB300.

One step = one generated token through the whole looped stack: 4 loop steps x 24 layers =
96 kvq_decode_attn calls, batch 64, 16 heads, context 6144 (8 sink + 759 index pages + 64
recent per request), each layer with its own cache. Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload loopvq_b64_6k|loopvq_b8_32k|kivi_b16_4k|kivi4_gqa_b16_4k|stream_b64_6k|
                                kivi_stream_b16_4k|encode_32k|kivi_quant_32k]

Under torchrun each rank runs its own replica on its own GPU (requests shard across GPUs
with no collective on the data path); rank 0 prints the max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-KV decode attn: effective HBM GB/s (% of GB300 peak), µs/step @B64 6K"
D = 128


# ------------------------------------------------------------------------------ workloads

WORKLOADS = {
    "loopvq_b64_6k": dict(kind="loopvq", B=64, H=16, L=6144, layers=24, T=4, Tc=2, G=16, recent=64,
                          rho=(0.69, 0.94), n_splits=0,
                          name="LoopVQ 0.5-bit serving decode, Ouro-1.4B-shaped: 24 layers x 4 loop steps, "
                               "16 heads, D=128, Tc=2, G=16, batch 64, context 6144"),
    "loopvq_b64_6k_tc1": dict(kind="loopvq", B=64, H=16, L=6144, layers=24, T=4, Tc=1, G=16, recent=64,
                              rho=(0.69, 0.94), n_splits=0,
                              name="LoopVQ 0.5-bit serving decode without loop coupling (Tc=1, c=16: per-step "
                                   "codewords), Ouro-1.4B-shaped: 24 layers x 4 loop steps, 16 heads, batch 64, "
                                   "context 6144"),
    "loopvq_b64_6k_tc4": dict(kind="loopvq", B=64, H=16, L=6144, layers=24, T=4, Tc=4, G=16, recent=64,
                              rho=(0.69, 0.94), n_splits=0,
                              name="LoopVQ 0.5-bit serving decode, one index for all 4 loop steps (Tc=4, c=4), "
                                   "Ouro-1.4B-shaped: 24 layers x 4 loop steps, 16 heads, batch 64, context 6144"),
    "loopvq_b8_32k": dict(kind="loopvq", B=8, H=16, L=32768, layers=1, T=4, Tc=4, G=32, recent=256,
                          rho=(0.85, 0.85), n_splits=0,
                          name="LoopVQ 0.25-bit long-context decode: 16 heads, D=128, Tc=4, G=32, batch 8, "
                               "context 32768, 4 loop steps"),
    "kivi_b16_4k": dict(kind="kivi", B=16, H=32, n_quant=3968, n_resid=128, layers=32,
                        name="KIVI 2-bit decode attention, Llama-2-7B-shaped: 32 layers, 32 heads, batch 16, "
                             "context 4096 = 3968 quantized + 128 fp16"),
    "kivi4_gqa_b16_4k": dict(kind="kivi", B=16, H=8, Hq=32, k_bits=4, v_bits=4, n_quant=3968, n_resid=128,
                             layers=32,
                             name="KIVI-4 decode attention with GQA, Llama-3-8B-shaped: 32 layers, 32 query heads "
                                  "over 8 KV heads, 4-bit K and V, batch 16, context 4096 = 3968 quantized + 128 fp16"),
    "kivi_stream_b16_4k": dict(kind="kivi_stream", B=16, H=32, n_quant=3968, n_resid=128, layers=32,
                               name="KIVI 2-bit streaming decode, Llama-2-7B-shaped: per generated token 32 layers "
                                    "of fp16 append (a whole key residual quantized every 128 tokens, one value "
                                    "quantized per token) + decode attention, batch 16 from context 4096"),
    "stream_b64_6k": dict(kind="stream", B=64, H=16, L=6144, layers=24, T=4, Tc=2, G=16, recent=64,
                          rho=(0.69, 0.94),
                          name="LoopVQ 0.5-bit streaming decode, Ouro-1.4B-shaped: per generated token 24 layers x "
                               "4 loop steps of bf16 append + decode attention, page roll every 8 tokens, "
                               "batch 64 from context 6144"),
    "encode_32k": dict(kind="encode", H=16, L=32768, T=4, Tc=2, G=16, groups=8,
                       name="LoopVQ prefill encode: 16 heads x 8 groups x 2 loop blocks x 32768 tokens"),
    "kivi_quant_32k": dict(kind="kivi_quant", H=16, L=32768,
                           name="KIVI 2-bit quantize of K and V: 16 heads x 32768 tokens"),
}


def bf16_peak():
    """Measured dense bf16 tensor throughput (TFLOP/s, burst) and where it came from."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.p = None

    def __enter__(self):
        import threading
        self.lines = []
        self.t0 = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
            return self
        first = threading.Event()

        def read():
            for ln in self.p.stdout:
                if ln.strip():
                    if self.t0 is not None:  # only samples taken once the timed region began
                        self.lines.append(ln)
                    first.set()
        self.th = threading.Thread(target=read, daemon=True)
        self.th.start()
        first.wait(5.0)  # sampling is running before the timed region starts
        self.t0 = time.time()
        return self

    def __exit__(self, *a):
        if self.p:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except Exception:
                self.p.kill()
            self.th.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------ CPU oracle leg

def _oracle_vq_job(args):
    seed, n_pairs, L, T, Tc, G, recent = args
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    import numpy as np
    import synth
    from oracle import loopvq as olv
    g = synth.rng(seed)
    _, n_pages, _ = olv.prefill_split(L, 8, recent)
    rhos = synth.rho_schedule(T)
    pool = synth.loop_correlated(g, T, 512, D, rhos)
    NG = D // (G // Tc)
    cb_k = synth.sample_codebooks(g, pool, Tc, G)[0]
    cb_v = synth.sample_codebooks(g, pool, Tc, G)[0]
    inputs = []
    for _ in range(n_pairs):
        wk = np.zeros((L, D))
        wv = np.zeros((L, D))
        bf = olv.cache_positions(L, n_pages)[0]
        wk[bf] = synth.bf16_round(g.standard_normal((len(bf), D)))
        wv[bf] = synth.bf16_round(g.standard_normal((len(bf), D)))
        inputs.append((synth.bf16_round(g.standard_normal(D)), synth.random_indices(g, (8 * n_pages, NG)),
                       synth.random_indices(g, (8 * n_pages, NG)), wk, wv))
    t0 = time.perf_counter()
    for q, ik, iv, wk, wv in inputs:
        olv.decode_attention(q, 1, Tc, L, n_pages, ik, iv, cb_k, cb_v, wk, wv)
    return time.perf_counter() - t0


def _oracle_kivi_job(args):
    seed, n_pairs, nq, nr, kb, vb = args
    import numpy as np
    import synth
    from oracle import kivi as okivi
    g = synth.rng(seed)
    inputs = []
    for _ in range(n_pairs):
        inputs.append((g.standard_normal(D), g.integers(0, 2 ** kb, (nq, D)),
                       (np.abs(g.standard_normal((nq // 32, D))) + 0.05).astype(np.float16),
                       g.standard_normal((nq // 32, D)).astype(np.float16), g.integers(0, 2 ** vb, (nq, D)),
                       (np.abs(g.standard_normal((nq, D // 32))) + 0.05).astype(np.float16),
                       g.standard_normal((nq, D // 32)).astype(np.float16),
                       g.standard_normal((nr, D)).astype(np.float16), g.standard_normal((nr, D)).astype(np.float16)))
    t0 = time.perf_counter()
    for q, kc, ks, kz, vc, vs, vz, kr, vr in inputs:
        okivi.decode_attention(q, kc, ks, kz, vc, vs, vz, kr, vr)
    return time.perf_counter() - t0


def cpu_oracle_single(wl, bytes_per_unit, n_pairs, pool=None):
    """Time the oracle on ``n_pairs`` (request, head) units in one single-threaded process while
    the other cores stay idle. Returns (GB/s, wall seconds)."""
    if wl["kind"] == "loopvq":
        job = (999, n_pairs, wl["L"], wl["T"], wl["Tc"], wl["G"], wl["recent"])
        fn = _oracle_vq_job
    else:
        job = (999, n_pairs, wl["n_quant"], wl["n_resid"], wl.get("k_bits", 2), wl.get("v_bits", 2))
        fn = _oracle_kivi_job
    own = pool is None
    if own:
        pool = mp.get_context("spawn").Pool(1)
    secs = pool.apply(fn, (job,))
    if own:
        pool.close()
    return bytes_per_unit * n_pairs / secs / 1e9, secs


def cpu_oracle(wl, bytes_per_unit, unit_pairs_total, n_pairs, pool=None):
    """Time the oracle on ``n_pairs`` (request, head) units on all host cores, one
    single-threaded process per core. Returns (GB/s, cores, wall seconds)."""
    cores = os.cpu_count() or 1
    per = max(1, math.ceil(n_pairs / cores))
    jobs = []
    done = 0
    k = 0
    while done < n_pairs:
        n = min(per, n_pairs - done)
        if wl["kind"] == "loopvq":
            jobs.append((1000 + k, n, wl["L"], wl["T"], wl["Tc"], wl["G"], wl["recent"]))
        else:
            jobs.append((1000 + k, n, wl["n_quant"], wl["n_resid"], wl.get("k_bits", 2), wl.get("v_bits", 2)))
        done += n
        k += 1
    fn = _oracle_vq_job if wl["kind"] == "loopvq" else _oracle_kivi_job
    own = pool is None
    if own:
        pool = mp.get_context("spawn").Pool(min(cores, len(jobs)))
    secs = pool.map(fn, jobs)
    if own:
        pool.close()
    # the jobs run side by side, one per core: the sample takes as long as the slowest job
    wall = max(secs)
    gbs = bytes_per_unit * n_pairs / wall / 1e9
    return gbs, min(cores, len(jobs)), wall


# ------------------------------------------------------------------------------ GPU legs

def vq_ng(wl):
    """Index groups per token: D / c with c = G / Tc channels per codeword."""
    return D // (wl["G"] // wl["Tc"])


def vq_call_bytes(B, H, n_pages, n_win, NG=16):
    """Algorithmic bytes of one LoopVQ decode-attention call (one layer, one loop step):
    K and V index pages (8 NG bytes each), bf16 window K and V, the fp32 key and fp16 value
    codebook slices, the cos/sin rows the call needs (one per page start and per window
    token), query and bf16 output."""
    idx = B * H * n_pages * 8 * NG * 2
    win = B * H * n_win * D * 2 * 2
    bt = H * 256 * D * (4 + 2)
    rope = (n_pages + n_win) * (D // 2) * 4 * 2
    qo = B * H * D * 2 * 2
    return idx + win + bt + rope + qo


# Shared-memory bytes the decode kernel must move per quantized token and head: every key index
# selects one fp32 codeword row of its channel group (4 B per channel), every value index adds
# the token's 4-byte integer weight into its (group, codeword) bin, and both index bytes are read
# from the ring. On this GPU that on-chip traffic, not HBM, is the binding resource of the
# LoopVQ decode (121 B per SM cycle measured for conflict-free 128-bit shared loads; 128 nominal).
SMEM_BYTES_PER_CLK_SM = 121.0


def vq_smem_bytes(B, H, n_pages, NG=16):
    return B * H * n_pages * 8 * (D * 4 + NG * 4 + 2 * NG)


def setup_loopvq(wl, dev, seed, extra_tokens=0):
    """LoopVQ cache of the workload, prefilled to L tokens per request (room for
    ``extra_tokens`` more, for streaming)."""
    import torch
    import synth
    from sub_bit_quantized_gb300 import kvq
    B, H, L, NL, T, Tc, G, W = wl["B"], wl["H"], wl["L"], wl["layers"], wl["T"], wl["Tc"], wl["G"], wl["recent"]
    n_pages = max(0, (L - 8 - W) // 8)
    cfg = kvq.VqConfig(T=T, Tc=Tc, G=G, n_layers=NL, n_heads=H, recent=W,
                       max_pages=n_pages + (extra_tokens + 7) // 8, max_batch=B, max_ctx=L + extra_tokens)
    cache = kvq.VqCache(cfg, dev)
    gen = torch.Generator(device=dev).manual_seed(seed)
    rhos = synth.rho_schedule(T, *wl["rho"])
    cbk = torch.empty_like(cache.cb_k)
    cbv = torch.empty_like(cache.cb_v)
    chunk = max(1, min(B, (1 << 30) // (T * H * L * D * 4)))
    for layer in range(NL):
        outl = torch.randperm(D, generator=gen, device=dev)[:4]
        # codebooks: sampled from one request's synthetic K/V of this layer, per head
        xk = synth.torch_loop_correlated(gen, T, (H, L, D), rhos, dev)
        xk[..., outl] *= 15.0
        xv = synth.torch_loop_correlated(gen, T, (H, L, D), rhos, dev)
        for h in range(H):
            cbk[layer, :, h] = synth.torch_sample_codebooks(gen, xk[:, h], Tc, G)
            cbv[layer, :, h] = synth.torch_sample_codebooks(gen, xv[:, h], Tc, G)
        del xk, xv
    cache.load_codebooks(cbk, cbv)
    del cbk, cbv
    for layer in range(NL):
        outl = torch.randperm(D, generator=gen, device=dev)[:4]
        for b0 in range(0, B, chunk):
            nb = min(chunk, B - b0)
            xk = synth.torch_loop_correlated(gen, T, (nb, H, L, D), rhos, dev)
            xk[..., outl] *= 15.0
            xk = xk.to(torch.bfloat16).contiguous()
            xv = synth.torch_loop_correlated(gen, T, (nb, H, L, D), rhos, dev).to(torch.bfloat16).contiguous()
            kvq.kvq_prefill_vq(cfg, cache, layer, xk, xv, b0, L)
            del xk, xv
    torch.cuda.synchronize(dev)
    assert kvq.device_error() == 0
    return cfg, cache, n_pages, (L - 8 * n_pages)


def kivi_cfg(wl, extra_tokens=0):
    from sub_bit_quantized_gb300 import kvq
    return kvq.KiviConfig(n_heads=wl["H"], n_q_heads=wl.get("Hq", wl["H"]), k_bits=wl.get("k_bits", 2),
                          v_bits=wl.get("v_bits", 2), residual=wl["n_resid"], max_batch=wl["B"],
                          max_tokens=wl["n_quant"] + extra_tokens)


def setup_kivi(wl, dev, seed, extra_tokens=0):
    """One KIVI cache per layer, filled by the library's prefill from random fp16 K/V
    (keys with 6 outlier channels scaled 20x): n_quant quantized + n_resid fp16 tokens."""
    import torch
    from sub_bit_quantized_gb300 import kvq
    B, H, NQ, NR, NL = wl["B"], wl["H"], wl["n_quant"], wl["n_resid"], wl["layers"]
    cfg = kivi_cfg(wl, extra_tokens)
    gen = torch.Generator(device=dev).manual_seed(seed)
    caches = []
    for layer in range(NL):
        c = kvq.KiviCache(cfg, dev)
        outl = torch.randperm(D, generator=gen, device=dev)[:6]
        K = torch.randn((B, H, NQ + NR, D), generator=gen, device=dev)
        K[..., outl] *= 20.0
        K = K.half()
        V = torch.randn((B, H, NQ + NR, D), generator=gen, device=dev).half()
        kvq.kvq_kivi_prefill(cfg, c, K, V)
        caches.append(c)
    torch.cuda.synchronize(dev)
    assert kvq.device_error() == 0
    assert int(caches[0].n_quant_k[0]) == NQ
    return cfg, caches


def kivi_call_bytes(B, H, NQ, NR, Hq=None, k_bits=2, v_bits=2):
    """Algorithmic bytes of one KIVI attention call: codes, key and value scales and zeros,
    the fp16 residual K and V, the bf16 queries read and outputs written."""
    Hq = Hq or H
    codes = B * H * NQ * D * (k_bits + v_bits) // 8
    ksz = B * H * (NQ // 32) * D * 2 * 2
    vsz = B * H * NQ * (D // 32) * 2 * 2
    res = B * H * NR * D * 2 * 2
    qo = B * Hq * D * 2 * 2
    return codes + ksz + vsz + res + qo


def kivi_wl_bytes(wl):
    return kivi_call_bytes(wl["B"], wl["H"], wl["n_quant"], wl["n_resid"], wl.get("Hq"), wl.get("k_bits", 2),
                           wl.get("v_bits", 2))


# arithmetic of each path (the JSON line's dtype)
DTYPE_LABEL = {
    "loopvq": "f32 (fp32 key codebook; values: fp16 codebook, weights in 2^-20 fixed point)",
    "stream": "f32 (fp32 key codebook; values: fp16 codebook, weights in 2^-20 fixed point)",
    "kivi": "f32 (2/4-bit codes, fp16 scales; fp16-rounded weights when one query head per block)",
    "kivi_stream": "f32 (2-bit codes, fp16 scales; fp16-rounded weights when one query head per block)",
    "encode": "bf16 x 3-part bf16 codebook -> f32 (compensated f32 near-tie decisions)",
    "kivi_quant": "f32->u8",
}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch from an ncu capture,
# valid only for the kernel source it was taken on (profiles/ holds the capture summary)
PROFILED_TRAFFIC = {
    "loopvq_b64_6k:vq_attn_kernel": (
        "sub_bit_quantized_gb300/csrc/vq_attn.cu",
        "0b5678e43e43cf1baab2d5ef0842ea12d8f8b3e2ba305d6d02da53b416c1be28",
        245771008 + 3553280),
    "kivi_b16_4k:kivi_attn_kernel": (
        "sub_bit_quantized_gb300/csrc/kivi.cu",
        "d9212bd30963454ad0bd578eb125492d04f4c19620162fddb05c762924a4ffbd",
        228793344 + 3551488),
    "encode_32k:encode_tc_kernel": (
        "sub_bit_quantized_gb300/csrc/vq_encode_tc.cu",
        "8f4d7c4d56f8e4813997994084beadad628c36cd5447f2bd11be519377daa3e4",
        287095296 + 14688512),
    # both quantize launches (keys per channel, values per token) of one step
    "kivi_quant_32k:kivi_quant_kernel": (
        "sub_bit_quantized_gb300/csrc/kivi.cu",
        "d9212bd30963454ad0bd578eb125492d04f4c19620162fddb05c762924a4ffbd",
        134273792 + 9351936 + 134293760 + 6658560),
    "kivi4_gqa_b16_4k:kivi_attn_kernel": (
        "sub_bit_quantized_gb300/csrc/kivi.cu",
        "d9212bd30963454ad0bd578eb125492d04f4c19620162fddb05c762924a4ffbd",
        89870592 + 2173440),
}


def profiled_traffic(workload, kernel):
    """Per-launch DRAM bytes of ``kernel`` on ``workload`` if its source is unchanged since the
    capture, else None."""
    import hashlib
    entry = PROFILED_TRAFFIC.get(f"{workload}:{kernel}")
    if entry is None:
        return None
    path, digest, nbytes = entry
    if digest is None:
        return None
    try:
        with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), path), "rb") as f:
            ok = hashlib.sha256(f.read()).hexdigest() == digest
    except OSError:
        return None
    return nbytes if ok else None


def time_region(fn, steps, stream, dist, nvtx_name=None):
    """Device time of ``steps`` calls of ``fn`` (CUDA events on ``stream``), max over ranks.
    ``nvtx_name`` marks the launches with an NVTX range so that a profiler can be limited to
    them (ncu --nvtx --nvtx-include "<name>/")."""
    import torch
    if dist:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    if nvtx_name:
        torch.cuda.nvtx.range_push(nvtx_name)
    for _ in range(steps):
        fn()
    if nvtx_name:
        torch.cuda.nvtx.range_pop()
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    if dist:
        ms = max_over_ranks(ms, "cuda")
        torch.distributed.barrier()
    return ms


def max_over_ranks(value: float, device="cpu") -> float:
    """The largest ``value`` over all ranks of the default process group (every rank gets it):
    the whole job takes as long as its slowest replica."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def run_ours(args, wl, rank, world, dist, pool):
    import torch
    from sub_bit_quantized_gb300 import kvq
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    gpu_index = dev.index
    hbm_peak, peak_src = peaks()
    result = {}

    if wl["kind"] in ("loopvq", "kivi"):
        if wl["kind"] == "loopvq":
            cfg, cache, n_pages, n_win = setup_loopvq(wl, dev, 1234 + rank)
            B, H, NL, T = wl["B"], wl["H"], wl["layers"], wl["T"]
            calls = [(l, t) for t in range(1, T + 1) for l in range(NL)]
            call_bytes = vq_call_bytes(B, H, n_pages, n_win, vq_ng(wl))
            caches = None
        else:
            cfg, caches = setup_kivi(wl, dev, 1234 + rank)
            B, H, NL = wl["B"], wl.get("Hq", wl["H"]), wl["layers"]   # H: query heads from here on
            calls = [(l, 1) for l in range(NL)]
            call_bytes = kivi_wl_bytes(wl)
        n_calls = len(calls)
        # one launch per call for either format: the roofline is that kernel's
        launches_per_call = 1
        kernel_name = "vq_attn_kernel" if wl["kind"] == "loopvq" else "kivi_attn_kernel"
        gen = torch.Generator(device=dev).manual_seed(99 + rank)
        q = torch.randn((n_calls, B, H, D), generator=gen, device=dev).to(torch.bfloat16)
        out = torch.empty((n_calls, B, H, D), dtype=torch.bfloat16, device=dev)
        n_splits = kvq.kvq_decode_auto_splits(cfg, B)
        ws = kvq.make_workspace(cfg, B, 0, dev)
        dcalls = [kvq.DecodeCall(cfg, cache if caches is None else caches[l], l, t, q[i], out[i], 0, ws, stream)
                  for i, (l, t) in enumerate(calls)]

        def step():
            for c in dcalls:
                c()

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        assert kvq.device_error() == 0
        with ClockSampler(gpu_index) as cs:
            ms = time_region(step, args.steps, stream, dist, nvtx_name="timed")
        clocks = cs.summary()
        ms_step = ms / args.steps
        step_bytes = call_bytes * n_calls
        gbs = step_bytes / (ms_step * 1e-3) / 1e9 * world
        per_launch_us = ms_step * 1e3 / n_calls
        achieved = call_bytes / (per_launch_us * 1e-6) / 1e9

        # end to end through the public API with host buffers: H2D of the step's queries from
        # pinned memory, the 96 calls, D2H of the outputs
        q_host = q.cpu().pin_memory()
        out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()

        def step_e2e():
            q.copy_(q_host, non_blocking=True)
            step()
            out_host.copy_(out, non_blocking=True)

        for _ in range(2):
            step_e2e()
        e2e_steps = max(3, args.steps // 4)
        ms_e2e = time_region(step_e2e, e2e_steps, stream, dist) / e2e_steps
        e2e = {"value": round(step_bytes / (ms_e2e * 1e-3) / 1e9 * world, 1), "unit": "GB/s",
               "h2d_bytes_per_step": q.numel() * 2, "d2h_bytes_per_step": out.numel() * 2,
               "ms_per_step": round(ms_e2e, 4)}
        result.update(dict(value=round(gbs, 1), unit="GB/s", ms_per_step=round(ms_step, 4),
                           us_per_call=round(per_launch_us, 2), gpu_launches=args.steps * n_calls * launches_per_call,
                           tokens_per_s=round(B * world / (ms_step * 1e-3), 1), e2e=e2e, clocks=clocks,
                           roofline={"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                                     "traffic": profiled_traffic(args.workload, kernel_name),
                                     "peak_source": peak_src,
                                     "kernel": kernel_name,
                                     "bytes_per_launch": call_bytes},
                           n_splits=n_splits))
        # LoopVQ's on-chip bound: codeword-row bytes read from shared memory per call over the
        # same call time, against the shared-memory rate of all SMs at the sampled clock
        if wl["kind"] == "loopvq":
            sm_mhz = clocks.get("sm_mhz") or 2070.0  # the sampled median under load, else the maximum
            smem_peak = torch.cuda.get_device_properties(dev).multi_processor_count * SMEM_BYTES_PER_CLK_SM * sm_mhz * 1e6 / 1e9
            smem_b = vq_smem_bytes(B, H, n_pages, vq_ng(wl))
            smem_ach = smem_b / (per_launch_us * 1e-6) / 1e9
            result["roofline"]["on_chip"] = {"bound": "smem", "achieved": round(smem_ach, 1), "peak": round(smem_peak, 1),
                                             "unit": "GB/s", "frac": round(smem_ach / smem_peak, 4),
                                             "bytes_per_launch": smem_b}
        if rank == 0 and not args.no_cpu_baseline:
            # eight calls' worth of (request, head) units: about 10 s on 16 host cores
            n_pairs = 8 * B * H
            unit_bytes = call_bytes / (B * H)
            cgbs, cores, wall = cpu_oracle(wl, unit_bytes, B * H, n_pairs, pool)
            n1 = 64 if wl["kind"] == "loopvq" else 32
            sgbs, swall = cpu_oracle_single(wl, unit_bytes, n1, pool)
            result["cpu_baseline"] = {"value": round(cgbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                      "nproc": os.cpu_count(),
                                      "sample": f"{n_pairs} (request, head) units (8 calls' worth), fp64 NumPy "
                                                f"oracle, {wall:.1f} s wall on {cores} single-threaded processes",
                                      "single_thread": {"value": round(sgbs, 5), "unit": "GB/s", "cores": 1,
                                                        "sample": f"{n1} (request, head) units in one process, "
                                                                  f"{swall:.1f} s"}}
        return result

    if wl["kind"] == "stream":
        # a step = one generated token: for every (layer, loop step) the new token's K/V is
        # appended in bf16 and the step's decode attention runs; every 8 tokens the append of
        # the token's last (layer, step) also encodes the oldest recent page into index pages
        B, H, NL, T = wl["B"], wl["H"], wl["layers"], wl["T"]
        n_tok = args.warmup + 2 * args.steps + 32
        cfg, cache, _, _ = setup_loopvq(wl, dev, 1234 + rank, extra_tokens=n_tok)
        gen = torch.Generator(device=dev).manual_seed(77 + rank)
        kn = torch.randn((B, H, D), generator=gen, device=dev).to(torch.bfloat16)
        vn = torch.randn((B, H, D), generator=gen, device=dev).to(torch.bfloat16)
        q = torch.randn((B, H, D), generator=gen, device=dev).to(torch.bfloat16)
        out = torch.empty((B, H, D), dtype=torch.bfloat16, device=dev)
        ws = kvq.make_workspace(cfg, B, 0, dev)
        calls = {(l, t): kvq.DecodeCall(cfg, cache, l, t, q, out, 0, ws, stream)
                 for l in range(NL) for t in range(1, T + 1)}

        def token(attend=True):
            for l in range(NL):
                for t in range(1, T + 1):
                    kvq.kvq_append_page(cfg, cache, l, t, kn, vn, stream)
                    if attend:
                        calls[(l, t)]()

        for _ in range(args.warmup):
            token()
        torch.cuda.synchronize()
        with ClockSampler(gpu_index) as cs:
            ms = time_region(token, args.steps, stream, dist, nvtx_name="timed") / args.steps
        # the same 96 attention calls without appends (the cache stops growing), then per-token
        # events over 16 more tokens: tokens whose first append rolls a page vs the others
        ms_attn = time_region(lambda: [c() for c in calls.values()], args.steps, stream, dist) / args.steps
        # per-token events around the token's first append (the call that rolls when a page is
        # due): the roll's cost is that call's time on a rolling token minus its time on the others
        n_meas = 32
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_meas)]
        rolled = []
        for i in range(n_meas):
            Lb = int(cache.seq_len[0].item())  # length before this token
            np_b = int(cache.n_pages[0].item())
            rolled.append(Lb + 1 - 8 - 8 * np_b == wl["recent"] + 8)  # the first append advances, then rolls
            ev[i][0].record(stream)
            kvq.kvq_append_page(cfg, cache, 0, 1, kn, vn, stream)
            ev[i][1].record(stream)
            calls[(0, 1)]()
            for l in range(NL):
                for t in range(1, T + 1):
                    if (l, t) != (0, 1):
                        kvq.kvq_append_page(cfg, cache, l, t, kn, vn, stream)
                        calls[(l, t)]()
        torch.cuda.synchronize()
        assert kvq.device_error() == 0
        tms = [e0.elapsed_time(e1) for e0, e1 in ev]
        plain = statistics.median([t for t, r in zip(tms, rolled) if not r])
        roll_extra = statistics.mean([t - plain for t, r in zip(tms, rolled) if r]) if any(rolled) else 0.0
        L_end = int(cache.seq_len[0].item())
        result.update(dict(value=round(B * world / (ms * 1e-3), 1), unit="tokens/s", ms_per_step=round(ms, 4),
                           attention_only_ms_per_token=round(ms_attn, 4),
                           append_roll_overhead_fraction=round((ms - ms_attn) / ms, 4),
                           roll_ms_per_roll=round(roll_extra, 4),
                           roll_fraction_amortized=round(roll_extra / 8 / ms, 5),
                           # per token: NL*T appends, the roll's 2 launches (at the first append;
                           # they leave at once unless a page is due), 1 launch per attention call
                           higher_is_better=True, gpu_launches=args.steps * (NL * T * 2 + 2),
                           context_end=L_end, clocks=cs.summary(),
                           roofline={"bound": "hbm", "achieved": None, "peak": hbm_peak, "unit": "GB/s",
                                     "frac": None, "traffic": None,
                                     "note": "per-call rooflines: workloads loopvq_b64_6k (attention), encode_32k"}))
        return result

    if wl["kind"] == "kivi_stream":
        # a step = one generated token: for every layer the token's K/V enters the cache
        # (kvq_kivi_append: a whole key residual is quantized every 128 tokens, the value
        # window quantizes its oldest token every token) and the layer's decode attention runs
        B, H, NL, R = wl["B"], wl["H"], wl["layers"], wl["n_resid"]
        n_tok = args.warmup + 2 * args.steps + 2 * R + 16
        cfg, caches = setup_kivi(wl, dev, 1234 + rank, extra_tokens=(n_tok + R - 1) // R * R)
        gen = torch.Generator(device=dev).manual_seed(77 + rank)
        kn = torch.randn((B, H, D), generator=gen, device=dev).half()
        vn = torch.randn((B, H, D), generator=gen, device=dev).half()
        q = torch.randn((B, H, D), generator=gen, device=dev).to(torch.bfloat16)
        out = torch.empty((B, H, D), dtype=torch.bfloat16, device=dev)
        ws = kvq.make_workspace(cfg, B, 0, dev)
        calls = [kvq.DecodeCall(cfg, caches[l], l, 1, q, out, 0, ws, stream) for l in range(NL)]
        appends = [(kvq.lib().kvq_kivi_append, (ctypes.byref(cfg.to_c()), ctypes.byref(caches[l].c_struct()),
                                                 kn.data_ptr(), vn.data_ptr(), B, stream.cuda_stream))
                   for l in range(NL)]
        keep = [a[1] for a in appends]   # the ctypes structs must outlive the calls

        def token():
            for l in range(NL):
                f, a = appends[l]
                if f(*a) != 0:
                    raise RuntimeError("kvq_kivi_append failed")
                calls[l]()

        for _ in range(args.warmup):
            token()
        torch.cuda.synchronize()
        assert kvq.device_error() == 0
        with ClockSampler(gpu_index) as cs:
            ms = time_region(token, args.steps, stream, dist, nvtx_name="timed") / args.steps
        ms_attn = time_region(lambda: [c() for c in calls], args.steps, stream, dist) / args.steps
        # per-token events over the next R + 8 tokens: the token whose append flushes a key
        # residual against the others
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(R + 9)]
        flushed = []
        for i in range(R + 8):
            flushed.append(int(caches[0].n_tok[0]) - int(caches[0].n_quant_k[0]) == R)
            ev[i].record(stream)
            token()
        ev[R + 8].record(stream)
        torch.cuda.synchronize()
        assert kvq.device_error() == 0
        tms = [ev[i].elapsed_time(ev[i + 1]) for i in range(R + 8)]
        plain = statistics.median([t for t, f in zip(tms, flushed) if not f])
        flush_extra = statistics.mean([t - plain for t, f in zip(tms, flushed) if f]) if any(flushed) else 0.0
        del keep
        result.update(dict(value=round(B * world / (ms * 1e-3), 1), unit="tokens/s", ms_per_step=round(ms, 4),
                           attention_only_ms_per_token=round(ms_attn, 4),
                           append_overhead_fraction=round((ms - ms_attn) / ms, 4),
                           key_flush_ms_per_flush=round(flush_extra, 4),
                           key_flush_fraction_amortized=round(flush_extra / R / ms, 5),
                           higher_is_better=True, gpu_launches=args.steps * NL * 2,
                           context_end=int(caches[0].n_tok[0]), clocks=cs.summary(),
                           roofline={"bound": "hbm", "achieved": None, "peak": hbm_peak, "unit": "GB/s",
                                     "frac": None, "traffic": None,
                                     "note": "per-call roofline: workload kivi_b16_4k (attention)"}))
        return result

    if wl["kind"] == "encode":
        import synth
        tc_peak, tc_src = bf16_peak()
        H, L, T, Tc, G = wl["H"], wl["L"], wl["T"], wl["Tc"], wl["G"]
        cfg = kvq.VqConfig(T=T, Tc=Tc, G=G, n_heads=H, max_pages=L // 8, max_batch=1, max_ctx=L + 80)
        gen = torch.Generator(device=dev).manual_seed(5)
        x = synth.torch_loop_correlated(gen, T, (1, H, L, D), synth.rho_schedule(T), dev).to(torch.bfloat16)
        cb = torch.stack([synth.torch_sample_codebooks(gen, x[:, 0, h].float(), Tc, G) for h in range(H)], 1)
        idx = torch.zeros((cfg.NB, 1, H, L // 8, 128), dtype=torch.uint8, device=dev)
        ties = torch.zeros(1, dtype=torch.int32, device=dev)
        strides = (H * L * D, H * L * D, L * D)

        def step():
            kvq.kvq_encode_vq(cfg, x, strides, 0, 1, L, cb, idx, 0, 0, wl["groups"], ties, stream)

        for _ in range(args.warmup):
            step()
        with ClockSampler(gpu_index) as cs:
            ms = time_region(step, args.steps, stream, dist) / args.steps
        n_vec = H * wl["groups"] * (T // Tc) * L
        flops = 2.0 * n_vec * 256 * G
        byts = n_vec * G * 2 + H * (T // Tc) * wl["groups"] * 256 * G * 4 + n_vec
        result.update(dict(value=round(byts / (ms * 1e-3) / 1e9 * world, 1), unit="GB/s", ms_per_step=round(ms, 4),
                           gpu_launches=args.steps, clocks=cs.summary(),
                           vectors_per_s=round(n_vec / (ms * 1e-3), 1),
                           # the distance GEMM runs on the tensor cores (bf16 operands, a 3-part split
                           # of the fp32 codebook); the row argmin on CUDA cores is what binds the time
                           roofline={"bound": "tensor", "achieved": round(flops / (ms * 1e-3) / 1e12, 2),
                                     "peak": tc_peak, "unit": "TFLOP/s",
                                     "frac": round(flops / (ms * 1e-3) / 1e12 / tc_peak, 4),
                                     "traffic": profiled_traffic(args.workload, "encode_tc_kernel"),
                                     "peak_source": tc_src, "kernel": "encode_tc_kernel"}))
        return result

    if wl["kind"] == "kivi_quant":
        H, L = wl["H"], wl["L"]
        cfg = kvq.KiviConfig(n_heads=H, max_batch=1, max_tokens=L)
        gen = torch.Generator(device=dev).manual_seed(6)
        K = torch.randn((1, H, L, D), generator=gen, device=dev).half()
        V = torch.randn((1, H, L, D), generator=gen, device=dev).half()
        c = kvq.KiviCache(cfg, dev)

        def step():
            kvq.kvq_quantize_kivi(cfg, kvq.PER_CHANNEL, K, c.k_codes, c.k_scale, c.k_zero, 0, stream)
            kvq.kvq_quantize_kivi(cfg, kvq.PER_TOKEN, V, c.v_codes, c.v_scale, c.v_zero, 0, stream)

        for _ in range(args.warmup):
            step()
        with ClockSampler(gpu_index) as cs:
            ms = time_region(step, args.steps, stream, dist) / args.steps
        byts = 2 * H * L * D * 2 + 2 * H * L * D // 4 + H * (L // 32) * D * 4 + H * L * (D // 32) * 4
        gbs = byts / (ms * 1e-3) / 1e9
        result.update(dict(value=round(gbs * world, 1), unit="GB/s", ms_per_step=round(ms, 4),
                           gpu_launches=2 * args.steps, clocks=cs.summary(),
                           roofline={"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                                     "frac": round(gbs / hbm_peak, 4),
                                     "traffic": profiled_traffic(args.workload, "kivi_quant_kernel"),
                                     "kernel": "kivi_quant_kernel"}))
        return result
    raise ValueError(wl["kind"])


def run_reference(args, wl, pool):
    """The CPU oracle as the reference arm: each step is a bounded sample of the workload."""
    if wl["kind"] == "loopvq":
        n_pages = max(0, (wl["L"] - 8 - wl["recent"]) // 8)
        call_bytes = vq_call_bytes(wl["B"], wl["H"], n_pages, wl["L"] - 8 * n_pages, vq_ng(wl))
        units = wl["B"] * wl["H"]
    elif wl["kind"] == "kivi":
        call_bytes = kivi_wl_bytes(wl)
        units = wl["B"] * wl.get("Hq", wl["H"])   # (request, query head) units
    else:
        raise SystemExit(json.dumps({"impl": "reference", "unavailable": "the CPU oracle arm covers the decode "
                                     "attention workloads only"}))
    unit_bytes = call_bytes / units
    n_pairs = 64
    for _ in range(args.warmup):
        cpu_oracle(wl, unit_bytes, units, 16, pool)
    total = 0.0
    cores = 1
    for _ in range(args.steps):
        _, cores, wall = cpu_oracle(wl, unit_bytes, units, n_pairs, pool)
        total += wall
    wall = total
    gbs = unit_bytes * n_pairs * args.steps / wall / 1e9
    return dict(value=round(gbs, 4), unit="GB/s", ms_per_step=round(wall / args.steps * 1e3, 3),
                cpu_baseline={"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                              "nproc": os.cpu_count(),
                              "sample": f"{n_pairs} (request, head) units of one call per step, one "
                                        f"single-threaded process per core"},
                e2e={"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                gpu_launches=0)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="loopvq_b64_6k", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    wl = dict(WORKLOADS[args.workload])
    if args.layers > 0 and "layers" in wl:
        wl["layers"] = args.layers
        wl["name"] += f" [profiling subset: {args.layers} layer(s)]"
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    pool = None
    if rank == 0 and (args.impl == "reference" or not args.no_cpu_baseline) and wl["kind"] in ("loopvq", "kivi"):
        # the oracle's process pool starts (spawn) before any GPU work
        pool = mp.get_context("spawn").Pool(os.cpu_count() or 1)
    base = {"metric": METRIC, "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "data": "synthetic"}
    if args.impl == "reference":
        if rank != 0:
            return
        res = run_reference(args, wl, pool)
        line = dict(base, impl="reference", dtype="f64", **res)
        line["config"] = {"workload": wl["name"], "sample_units": "(request, head) pairs"}
        print(json.dumps(line))
        pool.close()
        return
    dist = world > 1
    if dist:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, wl, rank, world, dist, pool)
    if rank == 0:
        cfgd = {"workload": wl["name"], "parallelism": f"replicas x{world} (requests shard, no collective)",
                "l2": "inputs larger than L2: each call reads its own layer's cache (~240 MB)"
                if wl["kind"] == "loopvq" else "inputs larger than L2"}
        for k in ("B", "H", "Hq", "k_bits", "v_bits", "L", "layers", "T", "Tc", "G", "recent", "n_quant", "n_resid"):
            if k in wl:
                cfgd[k] = wl[k]
        if "n_splits" in res:
            cfgd["n_splits"] = res.pop("n_splits")
        line = dict(base, dtype=DTYPE_LABEL.get(wl["kind"], "f32"), config=cfgd, **res)
        print(json.dumps(line))
    if pool is not None:
        pool.close()
    if dist:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
