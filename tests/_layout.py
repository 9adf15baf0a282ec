"""Host-side packing of logical cache contents into the byte layouts include/kvq.h documents
(test infrastructure: used to build GPU inputs and to read GPU outputs back)."""
from __future__ import annotations

import numpy as np

PAGE = 8


def page_byte_index(NG: int = 16):
    """(group g, token j) -> byte offset in a page: (s*8 + j)*2 + half, s = g mod NG/2."""
    half = NG // 2
    g = np.arange(NG)[:, None]
    j = np.arange(PAGE)[None, :]
    return ((g % half) * PAGE + j) * 2 + (g // half)          # [NG][8]


def pack_pages(idx: np.ndarray) -> np.ndarray:
    """Logical indices [..., n_pages*8, NG] -> page bytes [..., n_pages, 8*NG]."""
    idx = np.asarray(idx, dtype=np.uint8)
    *lead, n, NG = idx.shape
    assert n % PAGE == 0
    P = n // PAGE
    pages = idx.reshape(*lead, P, PAGE, NG)                   # [..][p][j][g]
    out = np.zeros((*lead, P, PAGE * NG), dtype=np.uint8)
    off = page_byte_index(NG)                                 # [g][j]
    for g in range(NG):
        for j in range(PAGE):
            out[..., off[g, j]] = pages[..., j, g]
    return out


def unpack_pages(pages: np.ndarray, NG: int = 16) -> np.ndarray:
    """Page bytes [..., n_pages, 8*NG] -> logical indices [..., n_pages*8, NG]."""
    pages = np.asarray(pages, dtype=np.uint8)
    *lead, P, nb = pages.shape
    assert nb == PAGE * NG
    off = page_byte_index(NG)
    out = np.empty((*lead, P, PAGE, NG), dtype=np.uint8)
    for g in range(NG):
        for j in range(PAGE):
            out[..., j, g] = pages[..., off[g, j]]
    return out.reshape(*lead, P * PAGE, NG)


def window_slot(p: int, sink: int = 8, recent: int = 64) -> int:
    return p if p < sink else sink + (p - sink) % (recent + PAGE)


def pack_codes(codes: np.ndarray, bits: int = 2) -> np.ndarray:
    """b-bit codes [..., D] -> bytes [..., D*b/8]: channel (8/b)k + i in bits [b i, b i + b) of byte k."""
    c = np.asarray(codes, dtype=np.uint8)
    *lead, D = c.shape
    per = 8 // bits
    c = c.reshape(*lead, D // per, per)
    out = np.zeros((*lead, D // per), dtype=np.uint8)
    for i in range(per):
        out |= (c[..., i] << (bits * i)).astype(np.uint8)
    return out


def unpack_codes(b: np.ndarray, bits: int = 2) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint8)
    per = 8 // bits
    out = np.stack([(b >> (bits * i)) & ((1 << bits) - 1) for i in range(per)], axis=-1)
    return out.reshape(*b.shape[:-1], b.shape[-1] * per)
