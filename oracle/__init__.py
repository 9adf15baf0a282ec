"""CPU oracle for quantized-KV decode attention (LoopVQ and KIVI formats).

TEST INFRASTRUCTURE ONLY. This package is the plain, slow, obviously-correct statement of
what the CUDA library computes. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it. The CUDA path
(``sub_bit_quantized_gb300``) never imports it, and it never imports the CUDA path: the
two share no code. The one thing they share is the seeded input generator in ``synth/``.

Sources (web pages, cited by title and section throughout):

* "LoopVQ: Sub 1-bit KV Cache Quantization for Looped Transformers" (a digest of the
  paper): background on vector quantization and RoPE, the five method steps, Figure 3,
  Algorithm 1 and Figure 5.
* "KIVI 完全拆解：非对称 2-bit KV Cache 量化" (a walkthrough of KIVI): the KV memory
  formula, the asymmetric quantize/dequantize formula, the grouped + residual cache
  layout (eq. (3), Algorithm 1) and the memory accounting.

Floating point is fp64 except where the method fixes the precision (KIVI's fp16 scale and
zero-point, computed in fp32; the bf16/fp16 storage of cached values).

Each function's pin (what checks it against the pages or the mathematics rather than
against itself) is listed in ``tests/test_oracle_*.py``. Parity unpinned: none of the
functions here; the pages' own kernels ship no code, so how close they come is not known.
"""
from . import accounting, attention, kivi, loopvq  # noqa: F401
