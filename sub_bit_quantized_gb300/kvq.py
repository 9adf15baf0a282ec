"""Thin ctypes binding of libkvq (include/kvq.h). Argument marshalling only: every step of
the computation runs in the library's CUDA kernels. PyTorch provides device memory and
streams. The binding fails loudly when the library is missing or a call returns an error;
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
from dataclasses import dataclass

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkvq.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "kvq.h")

KVQ_OK = 0
ERR_INVALID_ARG, ERR_CAPACITY, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE, ERR_TIMEOUT = 1, 2, 3, 4, 5, 6
STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_CAPACITY", 3: "KVQ_ERR_UNSUPPORTED",
          4: "KVQ_ERR_CUDA", 5: "KVQ_ERR_WORKSPACE", 6: "KVQ_ERR_TIMEOUT"}
FMT_LOOPVQ, FMT_KIVI = 0, 1
OUT_BF16, OUT_FP32 = 0, 1
PER_CHANNEL, PER_TOKEN = 0, 1
PAGE = 8


class KvqError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}: {detail}")


class VqCfg(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int), ("T", ctypes.c_int), ("Tc", ctypes.c_int), ("G", ctypes.c_int),
                ("K", ctypes.c_int), ("n_layers", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("sink", ctypes.c_int), ("recent", ctypes.c_int), ("max_pages", ctypes.c_int),
                ("max_batch", ctypes.c_int), ("max_ctx", ctypes.c_int), ("rope_base", ctypes.c_float)]


class VqCacheC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("idx_k", "idx_v", "win_k", "win_v", "bt_k", "bt_v", "cb_k", "cb_v",
                 "rope_cos", "rope_sin", "seq_len", "n_pages", "cbp_k", "cbp_v")]


class VqSizes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("idx", "win", "bt", "bt_v", "cb", "rope", "per_request", "cbp")]


class KiviCfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("D", "n_heads", "n_q_heads", "k_bits", "v_bits", "group", "residual", "max_batch",
                 "max_tokens")]


KIVI_CACHE_FIELDS = ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero",
                     "k_resid", "v_resid", "n_tok", "n_quant_k", "n_quant_v", "sync")


class KiviCacheC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in KIVI_CACHE_FIELDS]


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_SIGS = {
    "kvq_version": (_I, []),
    "kvq_status_string": (ctypes.c_char_p, [_I]),
    "kvq_last_error": (ctypes.c_char_p, []),
    "kvq_device_error": (_I, []),
    "kvq_vq_cache_sizes": (_I, [_P, _P]),
    "kvq_rope_table": (_I, [_P, _P, _P, _P]),
    "kvq_slice_codebooks": (_I, [_P, _P, _P, _P]),
    "kvq_slice_codebooks_fp16": (_I, [_P, _P, _P, _P]),
    "kvq_split_codebooks": (_I, [_P, _P, _P, _P]),
    "kvq_encode_vq": (_I, [_P, _P, _I64, _I64, _I64, _I, _I, _I, _P, _P, _I, _I, _I, _P, _P]),
    "kvq_prefill_vq": (_I, [_P, _P, _I, _P, _P, _I64, _I64, _I64, _I, _I, _I, _P, _P]),
    "kvq_append_page": (_I, [_P, _P, _I, _I, _P, _P, _I, _P]),
    "kvq_quantize_kivi": (_I, [_P, _I, _P, _I64, _I64, _I, _I, _P, _P, _P, _I, _P]),
    "kvq_kivi_prefill": (_I, [_P, _P, _P, _P, _I64, _I64, _I, _I, _I, _P]),
    "kvq_kivi_append": (_I, [_P, _P, _P, _P, _I, _P]),
    "kvq_decode_attn": (_I, [_I, _P, _P, _I, _I, _P, _I, _P, _I, _I, _P, _SZ, _P]),
    "kvq_decode_attn_noalloc": (_I, [_I, _P, _P, _I, _I, _P, _I, _P, _I, _I, _P]),
    "kvq_decode_workspace_size": (_SZ, [_I, _P, _I, _I]),
    "kvq_decode_auto_splits": (_I, [_I, _P, _I]),
}

_lib = None


def header_functions() -> list[str]:
    """Names of the functions include/kvq.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", text)))


def lib() -> ctypes.CDLL:
    """The loaded libkvq.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libkvq.so not found at {LIB_PATH}: run __graft_entry__.build() "
                               "(or python sub_bit_quantized_gb300/_build.py) first")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(st: int, where: str):
    if st != KVQ_OK:
        raise KvqError(st, where, lib().kvq_last_error().decode())


def version() -> int:
    return lib().kvq_version()


def device_error() -> int:
    """Read and clear the device error word (synchronizes the device)."""
    return lib().kvq_device_error()


def _bits(t: torch.Tensor, dtypes) -> torch.Tensor:
    if t.dtype not in dtypes:
        raise TypeError(f"expected one of {dtypes}, got {t.dtype}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return t


# ------------------------------------------------------------------------------------------
# LoopVQ
# ------------------------------------------------------------------------------------------

@dataclass
class VqConfig:
    D: int = 128
    T: int = 4
    Tc: int = 2
    G: int = 16
    K: int = 256
    n_layers: int = 1
    n_heads: int = 1
    sink: int = 8
    recent: int = 64
    max_pages: int = 0
    max_batch: int = 1
    max_ctx: int = 2
    rope_base: float = 1.0e4

    @property
    def NB(self) -> int:
        return self.T // self.Tc

    @property
    def c(self) -> int:
        return self.G // self.Tc

    @property
    def NG(self) -> int:
        return self.D // self.c

    @property
    def win_slots(self) -> int:
        return self.sink + self.recent + PAGE

    def to_c(self) -> VqCfg:
        return VqCfg(self.D, self.T, self.Tc, self.G, self.K, self.n_layers, self.n_heads, self.sink,
                     self.recent, self.max_pages, self.max_batch, self.max_ctx, float(self.rope_base))


class VqCache:
    """A LoopVQ cache whose buffers PyTorch allocates on the current device.

    Shapes follow include/kvq.h. ``cb_k`` / ``cb_v`` hold the full codebooks; call
    ``load_codebooks`` to set them (it also cuts the per-step slices on the GPU), and
    ``rope_table`` is filled on construction.
    """

    def __init__(self, cfg: VqConfig, device="cuda"):
        self.cfg = cfg
        c = cfg
        dev = torch.device(device)
        L, NB, B, H, P = c.n_layers, c.NB, c.max_batch, c.n_heads, c.max_pages
        self.idx_k = torch.zeros((L, NB, B, H, P, PAGE * c.NG), dtype=torch.uint8, device=dev)
        self.idx_v = torch.zeros_like(self.idx_k)
        self.win_k = torch.zeros((L, c.T, B, H, c.win_slots, c.D), dtype=torch.bfloat16, device=dev)
        self.win_v = torch.zeros_like(self.win_k)
        self.bt_k = torch.zeros((L, c.T, H, 2, c.K, c.D // 2), dtype=torch.float32, device=dev)
        self.bt_v = torch.zeros((L, c.T, H, c.K, c.D), dtype=torch.float16, device=dev)
        self.cb_k = torch.zeros((L, NB, H, c.NG, c.K, c.G), dtype=torch.float32, device=dev)
        self.cb_v = torch.zeros_like(self.cb_k)
        sizes = vq_cache_sizes(cfg)
        # codebook parts for the tensor-core page roll (kvq_split_codebooks)
        self.cbp_k = torch.zeros(sizes.cbp, dtype=torch.uint8, device=dev)
        self.cbp_v = torch.zeros_like(self.cbp_k)
        self.rope_cos = torch.empty((c.max_ctx, c.D // 2), dtype=torch.float32, device=dev)
        self.rope_sin = torch.empty_like(self.rope_cos)
        self.seq_len = torch.zeros(B, dtype=torch.int32, device=dev)
        self.n_pages = torch.zeros(B, dtype=torch.int32, device=dev)
        self._cfg_c = cfg.to_c()
        sizes = vq_cache_sizes(cfg)
        assert sizes.idx == self.idx_k.numel() and sizes.win == self.win_k.numel() * 2
        assert sizes.bt == self.bt_k.numel() * 4 and sizes.bt_v == self.bt_v.numel() * 2
        assert sizes.cb == self.cb_k.numel() * 4
        kvq_rope_table(cfg, self.rope_cos, self.rope_sin)

    def c_struct(self) -> VqCacheC:
        return VqCacheC(*[_ptr(getattr(self, n)) for n in
                          ("idx_k", "idx_v", "win_k", "win_v", "bt_k", "bt_v", "cb_k", "cb_v",
                           "rope_cos", "rope_sin", "seq_len", "n_pages", "cbp_k", "cbp_v")])

    def load_codebooks(self, cb_k: torch.Tensor, cb_v: torch.Tensor, stream=None):
        self.cb_k.copy_(cb_k)
        self.cb_v.copy_(cb_v)
        kvq_slice_codebooks(self.cfg, self.cb_k, self.bt_k, stream)
        kvq_slice_codebooks_fp16(self.cfg, self.cb_v, self.bt_v, stream)
        kvq_split_codebooks(self.cfg, self.cb_k, self.cbp_k, stream)
        kvq_split_codebooks(self.cfg, self.cb_v, self.cbp_v, stream)


def vq_cache_sizes(cfg: VqConfig) -> VqSizes:
    out = VqSizes()
    c = cfg.to_c()
    _check(lib().kvq_vq_cache_sizes(ctypes.byref(c), ctypes.byref(out)), "kvq_vq_cache_sizes")
    return out


def kvq_rope_table(cfg: VqConfig, rope_cos, rope_sin, stream=None):
    c = cfg.to_c()
    _check(lib().kvq_rope_table(ctypes.byref(c), _ptr(rope_cos), _ptr(rope_sin), _stream(stream)),
           "kvq_rope_table")


def kvq_slice_codebooks(cfg: VqConfig, cb, bt, stream=None):
    c = cfg.to_c()
    _check(lib().kvq_slice_codebooks(ctypes.byref(c), _ptr(cb), _ptr(bt), _stream(stream)),
           "kvq_slice_codebooks")


def kvq_slice_codebooks_fp16(cfg: VqConfig, cb, bt16, stream=None):
    c = cfg.to_c()
    _check(lib().kvq_slice_codebooks_fp16(ctypes.byref(c), _ptr(cb), _ptr(bt16), _stream(stream)),
           "kvq_slice_codebooks_fp16")


def kvq_split_codebooks(cfg: VqConfig, cb, cbp, stream=None):
    c = cfg.to_c()
    _check(lib().kvq_split_codebooks(ctypes.byref(c), _ptr(cb), _ptr(cbp), _stream(stream)), "kvq_split_codebooks")


def kvq_encode_vq(cfg: VqConfig, x, x_strides, seq_begin, n_seq, n_tok, cb, idx, page_begin=0,
                  g_begin=0, g_count=None, n_ties=None, stream=None):
    """x: bf16 tensor (or base pointer with explicit element strides (t, b, h))."""
    c = cfg.to_c()
    g_count = cfg.NG - g_begin if g_count is None else g_count
    st, sb, sh = x_strides
    _check(lib().kvq_encode_vq(ctypes.byref(c), _ptr(x), st, sb, sh, seq_begin, n_seq, n_tok,
                               _ptr(cb), _ptr(idx), page_begin, g_begin, g_count, _ptr(n_ties),
                               _stream(stream)), "kvq_encode_vq")


def kvq_prefill_vq(cfg: VqConfig, cache: VqCache, layer: int, xk, xv, seq_begin: int, L: int,
                   n_ties=None, stream=None):
    """xk, xv: bf16 [T][n_seq][H][L][D] pre-RoPE keys / values of one layer."""
    T, n_seq, H, Lx, D = xk.shape
    assert xv.shape == xk.shape and Lx >= L
    _bits(xk, (torch.bfloat16,))
    _bits(xv, (torch.bfloat16,))
    c = cfg.to_c()
    kc = cache.c_struct()
    st, sb, sh = n_seq * H * Lx * D, H * Lx * D, Lx * D
    _check(lib().kvq_prefill_vq(ctypes.byref(c), ctypes.byref(kc), layer, _ptr(xk), _ptr(xv), st, sb, sh,
                                seq_begin, n_seq, L, _ptr(n_ties), _stream(stream)), "kvq_prefill_vq")


def kvq_append_page(cfg: VqConfig, cache: VqCache, layer: int, loop_step: int, k_new, v_new,
                    stream=None):
    """k_new, v_new: bf16 [n_seq][H][D] pre-RoPE key / value of the newest token at (layer, step)."""
    _bits(k_new, (torch.bfloat16,))
    _bits(v_new, (torch.bfloat16,))
    c = cfg.to_c()
    kc = cache.c_struct()
    _check(lib().kvq_append_page(ctypes.byref(c), ctypes.byref(kc), layer, loop_step, _ptr(k_new),
                                 _ptr(v_new), k_new.shape[0], _stream(stream)), "kvq_append_page")


# ------------------------------------------------------------------------------------------
# KIVI
# ------------------------------------------------------------------------------------------

@dataclass
class KiviConfig:
    """kvq_kivi_cfg. n_q_heads defaults to n_heads (multi-head attention)."""
    D: int = 128
    n_heads: int = 1
    n_q_heads: int | None = None
    k_bits: int = 2
    v_bits: int = 2
    group: int = 32
    residual: int = 128
    max_batch: int = 1
    max_tokens: int = 0

    @property
    def q_heads(self) -> int:
        return self.n_heads if self.n_q_heads is None else self.n_q_heads

    def to_c(self) -> KiviCfg:
        return KiviCfg(self.D, self.n_heads, self.q_heads, self.k_bits, self.v_bits, self.group,
                       self.residual, self.max_batch, self.max_tokens)


class KiviCache:
    """Device buffers of a KIVI cache (layouts of kvq_kivi_cache), zero-filled."""

    def __init__(self, cfg: KiviConfig, device="cuda"):
        self.cfg = cfg
        c = cfg
        dev = torch.device(device)
        B, H, N, D, Gq = c.max_batch, c.n_heads, c.max_tokens, c.D, c.group
        self.k_codes = torch.zeros((B, H, N, D * c.k_bits // 8), dtype=torch.uint8, device=dev)
        self.v_codes = torch.zeros((B, H, N, D * c.v_bits // 8), dtype=torch.uint8, device=dev)
        self.k_scale = torch.zeros((B, H, N // Gq, D), dtype=torch.float16, device=dev)
        self.k_zero = torch.zeros_like(self.k_scale)
        self.v_scale = torch.zeros((B, H, N, D // Gq), dtype=torch.float16, device=dev)
        self.v_zero = torch.zeros_like(self.v_scale)
        self.k_resid = torch.zeros((B, H, max(c.residual, 1), D), dtype=torch.float16, device=dev)
        self.v_resid = torch.zeros_like(self.k_resid)
        self.n_tok = torch.zeros(B, dtype=torch.int32, device=dev)
        self.n_quant_k = torch.zeros(B, dtype=torch.int32, device=dev)
        self.n_quant_v = torch.zeros(B, dtype=torch.int32, device=dev)
        self.sync = torch.zeros(B, dtype=torch.int32, device=dev)

    def c_struct(self) -> KiviCacheC:
        return KiviCacheC(*[_ptr(getattr(self, n)) for n in KIVI_CACHE_FIELDS])


def kvq_quantize_kivi(cfg: KiviConfig, axis: int, x, codes, scale, zero, tok_begin=0, stream=None):
    """x: fp16 [B][H][n_tok][D]."""
    _bits(x, (torch.float16,))
    B, H, n, D = x.shape
    c = cfg.to_c()
    _check(lib().kvq_quantize_kivi(ctypes.byref(c), axis, _ptr(x), H * n * D, n * D, B, n, _ptr(codes),
                                   _ptr(scale), _ptr(zero), tok_begin, _stream(stream)),
           "kvq_quantize_kivi")


def kvq_kivi_prefill(cfg: KiviConfig, cache: KiviCache, k, v, b0: int = 0, stream=None):
    """k, v: fp16 [B][H][n_tok][D] (same strides) for requests b0 .. b0+B-1."""
    _bits(k, (torch.float16,))
    _bits(v, (torch.float16,))
    if k.shape != v.shape or k.stride() != v.stride() or k.stride(3) != 1 or k.stride(2) != k.shape[3]:
        raise ValueError("k and v need one shape and rows of D contiguous channels")
    B, H, n, D = k.shape
    c = cfg.to_c()
    kc = cache.c_struct()
    _check(lib().kvq_kivi_prefill(ctypes.byref(c), ctypes.byref(kc), _ptr(k), _ptr(v), k.stride(0), k.stride(1),
                                  b0, B, n, _stream(stream)), "kvq_kivi_prefill")


def kvq_kivi_append(cfg: KiviConfig, cache: KiviCache, k_new, v_new, stream=None):
    """k_new, v_new: fp16 [n_seq][H][D], contiguous."""
    _bits(k_new, (torch.float16,))
    _bits(v_new, (torch.float16,))
    c = cfg.to_c()
    kc = cache.c_struct()
    _check(lib().kvq_kivi_append(ctypes.byref(c), ctypes.byref(kc), _ptr(k_new), _ptr(v_new), k_new.shape[0],
                                 _stream(stream)), "kvq_kivi_append")


# ------------------------------------------------------------------------------------------
# Decode attention
# ------------------------------------------------------------------------------------------

def _fmt_cfg(cfg):
    if isinstance(cfg, VqConfig):
        return FMT_LOOPVQ, cfg.to_c()
    if isinstance(cfg, KiviConfig):
        return FMT_KIVI, cfg.to_c()
    raise TypeError(type(cfg))


def kvq_decode_workspace_size(cfg, B: int, n_splits: int = 0) -> int:
    fmt, c = _fmt_cfg(cfg)
    return lib().kvq_decode_workspace_size(fmt, ctypes.byref(c), B, n_splits)


def kvq_decode_auto_splits(cfg, B: int) -> int:
    fmt, c = _fmt_cfg(cfg)
    return lib().kvq_decode_auto_splits(fmt, ctypes.byref(c), B)


def make_workspace(cfg, B: int, n_splits: int = 0, device="cuda") -> torch.Tensor | None:
    n = kvq_decode_workspace_size(cfg, B, n_splits)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device)


class DecodeCall:
    """Pre-marshalled arguments of one repeated kvq_decode_attn call (cheap to launch)."""

    def __init__(self, cfg, cache, layer, loop_step, q, out, n_splits=0, ws=None, stream=None):
        self.fmt, self.cfg_c = _fmt_cfg(cfg)
        self.cache_c = cache.c_struct()
        _bits(q, (torch.bfloat16,))
        _bits(out, (torch.bfloat16, torch.float32))
        self.args = (self.fmt, ctypes.byref(self.cfg_c), ctypes.byref(self.cache_c), layer, loop_step,
                     _ptr(q), q.shape[0], _ptr(out), OUT_FP32 if out.dtype == torch.float32 else OUT_BF16,
                     n_splits, _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream))
        self._f = lib().kvq_decode_attn

    def __call__(self):
        st = self._f(*self.args)
        if st != KVQ_OK:
            _check(st, "kvq_decode_attn")


def kvq_decode_attn(cfg, cache, layer: int, loop_step: int, q, out, n_splits: int = 0, ws=None,
                    stream=None):
    """q: bf16 [B][H][D]; out: bf16 or fp32 [B][H][D]. When the split plan needs a workspace
    and none is given, a zero-filled one is allocated for this call (through PyTorch)."""
    if ws is None:
        ws = make_workspace(cfg, q.shape[0], n_splits, q.device)
    DecodeCall(cfg, cache, layer, loop_step, q, out, n_splits, ws, stream)()
