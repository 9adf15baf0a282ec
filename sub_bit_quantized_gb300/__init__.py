"""Quantized-KV decode attention for NVIDIA GB300 (sm_103a): LoopVQ and KIVI caches.

The computation lives in libkvq.so (CUDA C++, C ABI declared in include/kvq.h); this
package is its thin ctypes binding plus the in-tree build script.
"""
from . import kvq  # noqa: F401
from .kvq import (KiviCache, KiviConfig, KvqError, VqCache, VqConfig,  # noqa: F401
                  kvq_append_page, kvq_decode_attn, kvq_decode_workspace_size, kvq_encode_vq,
                  kvq_kivi_append, kvq_kivi_prefill, kvq_prefill_vq, kvq_quantize_kivi,
                  kvq_rope_table, kvq_slice_codebooks,
                  kvq_slice_codebooks_fp16)

__version__ = "0.1.0"
