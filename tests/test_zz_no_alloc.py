"""kvq_decode_attn_noalloc: decode attention for callers that cannot allocate device memory
(an engine whose memory pool owns the whole GPU, or code inside another framework's
callback). It takes its workspace (unit prefix and partial softmaxes) from an array the
library reserves per device.
Checked through the C ABI against kvq_decode_attn with a caller workspace, on two calls in
a row (the second call reuses the array the first one left behind). Collected last on
purpose, and self-contained so that it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from sub_bit_quantized_gb300 import kvq
from tests import _cases as C

pytestmark = pytest.mark.gpu


def call_noalloc(case, cache, t, out, n_splits):
    c = case.cfg.to_c()
    kc = cache.c_struct()
    q = C.bf16_tensor(case.q)
    st = kvq.lib().kvq_decode_attn_noalloc(kvq.FMT_LOOPVQ, ctypes.byref(c), ctypes.byref(kc), 0, t,
                                           q.data_ptr(), q.shape[0], out.data_ptr(), kvq.OUT_FP32, n_splits,
                                           torch.cuda.current_stream().cuda_stream)
    assert st == kvq.KVQ_OK, kvq.lib().kvq_last_error()


@pytest.mark.parametrize("n_splits", [3, 0])
def test_noalloc_matches_workspace_call_twice(n_splits):
    case = C.make_vq_case(500, B=5, H=3, lens=[700, 1300, 64, 999, 2000])
    cache = C.fill_vq_cache(case)
    B, H = len(case.lens), case.cfg.n_heads
    need = kvq.kvq_decode_workspace_size(case.cfg, B, n_splits)
    assert 0 < need <= (8 << 20) or n_splits == 0
    ref = torch.empty((B, H, 128), dtype=torch.float32, device="cuda")
    kvq.kvq_decode_attn(case.cfg, cache, 0, 2, C.bf16_tensor(case.q), ref, n_splits)
    for _ in range(2):
        out = torch.full((B, H, 128), float("nan"), dtype=torch.float32, device="cuda")
        call_noalloc(case, cache, 2, out, n_splits)
        torch.cuda.synchronize()
        assert kvq.device_error() == 0
        C.check_close(out.cpu().numpy(), ref.cpu().numpy())
        assert torch.allclose(out, ref, rtol=1e-5, atol=1e-6)


def test_noalloc_rejects_calls_beyond_the_reserved_scratch():
    # 4096 page-kernel blocks keep two piece slots each (2 x 8320 B): 68 MB, over the
    # reserved array, so the call is refused before anything launches
    cfg = kvq.VqConfig(n_heads=16, max_pages=4063, max_batch=64, max_ctx=32768, recent=256, Tc=4, G=32)
    need = kvq.kvq_decode_workspace_size(cfg, 64, 4096)
    assert need > (8 << 20)
    c = cfg.to_c()
    kc = kvq.VqCacheC(*([0x10000] * 12))
    st = kvq.lib().kvq_decode_attn_noalloc(kvq.FMT_LOOPVQ, ctypes.byref(c), ctypes.byref(kc), 0, 1, 0x10000, 64,
                                           0x10000, kvq.OUT_FP32, 4096, None)
    assert st == 5 and b"reserves" in kvq.lib().kvq_last_error()
