"""kvq_decode_attn_noalloc: decode attention for callers that cannot allocate device memory
(an engine whose memory pool owns the whole GPU, or code inside another framework's
callback). It takes its workspace (merge counters and partial softmaxes) from an array
inside the library, one per device.
Checked through the C ABI against kvq_decode_attn with a caller workspace, on two calls in
a row (the second call reuses the array the first one left behind), for both cache formats.
The array is set aside when the library's device code loads on the device, at its first
call there: a test makes that call first and then checks that later calls, made after
other device memory has been taken, still succeed. Collected last on purpose, and
self-contained so that it also passes alone in a fresh process."""
import ctypes

import pytest
import torch

from sub_bit_quantized_gb300 import kvq
from tests import _cases as C

pytestmark = pytest.mark.gpu


def call_noalloc(fmt, cfg, cache, t, q, out, n_splits):
    c = cfg.to_c()
    kc = cache.c_struct()
    return kvq.lib().kvq_decode_attn_noalloc(fmt, ctypes.byref(c), ctypes.byref(kc), 0, t, q.data_ptr(),
                                             q.shape[0], out.data_ptr(), kvq.OUT_FP32, n_splits,
                                             torch.cuda.current_stream().cuda_stream)


def test_first_call_then_later_calls_after_other_allocations():
    case = C.make_vq_case(501, B=2, H=2, lens=[300, 900])
    cache = C.fill_vq_cache(case)
    q = C.bf16_tensor(case.q)
    out = torch.empty((2, 2, 128), dtype=torch.float32, device="cuda")
    # the first call on the device: looks the array up (its device code is loaded by now)
    assert call_noalloc(kvq.FMT_LOOPVQ, case.cfg, cache, 1, q, out, 0) == kvq.KVQ_OK, kvq.lib().kvq_last_error()
    torch.cuda.synchronize()
    first = out.clone()
    # other device memory taken afterwards (a pool, say) does not affect later calls
    hold = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        out.fill_(float("nan"))
        assert call_noalloc(kvq.FMT_LOOPVQ, case.cfg, cache, 1, q, out, 0) == kvq.KVQ_OK
        torch.cuda.synchronize()
        assert kvq.device_error() == 0
        assert torch.equal(out, first)
    del hold


@pytest.mark.parametrize("n_splits", [3, 0])
def test_noalloc_matches_workspace_call_twice(n_splits):
    case = C.make_vq_case(500, B=5, H=3, lens=[700, 1300, 64, 999, 2000])
    cache = C.fill_vq_cache(case)
    B, H = len(case.lens), case.cfg.n_heads
    need = kvq.kvq_decode_workspace_size(case.cfg, B, n_splits)
    assert 0 < need <= (8 << 20)
    q = C.bf16_tensor(case.q)
    ref = torch.empty((B, H, 128), dtype=torch.float32, device="cuda")
    kvq.kvq_decode_attn(case.cfg, cache, 0, 2, q, ref, n_splits)
    for _ in range(2):
        out = torch.full((B, H, 128), float("nan"), dtype=torch.float32, device="cuda")
        st = call_noalloc(kvq.FMT_LOOPVQ, case.cfg, cache, 2, q, out, n_splits)
        assert st == kvq.KVQ_OK, kvq.lib().kvq_last_error()
        torch.cuda.synchronize()
        assert kvq.device_error() == 0
        # integer value sums and a fixed merge order: the same bits as with a caller workspace
        assert torch.equal(out, ref)


@pytest.mark.parametrize("n_splits", [3, 0])
def test_noalloc_kivi_split_counters_twice(n_splits):
    # the KIVI split merge counts arriving blocks in the workspace and the last one resets the
    # count: two calls in a row on the shared array must both merge correctly
    case = C.make_kivi_case(502, B=3, H=2, n_quant=[32 * 40, 96, 32 * 70], n_resid=[17, 128, 5])
    cache = C.fill_kivi_cache(case)
    B, Hq = len(case.n_tok), case.cfg.q_heads
    q = C.bf16_tensor(case.q)
    ref = torch.empty((B, Hq, 128), dtype=torch.float32, device="cuda")
    kvq.kvq_decode_attn(case.cfg, cache, 0, 1, q, ref, n_splits, kvq.make_workspace(case.cfg, B, n_splits))
    for _ in range(2):
        out = torch.full((B, Hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        st = call_noalloc(kvq.FMT_KIVI, case.cfg, cache, 1, q, out, n_splits)
        assert st == kvq.KVQ_OK, kvq.lib().kvq_last_error()
        torch.cuda.synchronize()
        assert kvq.device_error() == 0
        assert torch.allclose(out, ref, rtol=1e-5, atol=1e-6)


def test_noalloc_rejects_calls_beyond_the_reserved_scratch():
    # 8191 requests x 256 heads of merge counters (8.4 MB) plus 4096 blocks' partial slots:
    # over the array, so the call is refused before anything launches
    cfg = kvq.VqConfig(n_heads=256, max_pages=8, max_batch=8191, max_ctx=512)
    need = kvq.kvq_decode_workspace_size(cfg, 8191, 4096)
    assert need > (8 << 20)
    c = cfg.to_c()
    kc = kvq.VqCacheC(*([0x10000] * 12))
    st = kvq.lib().kvq_decode_attn_noalloc(kvq.FMT_LOOPVQ, ctypes.byref(c), ctypes.byref(kc), 0, 1, 0x10000, 8191,
                                           0x10000, kvq.OUT_FP32, 4096, None)
    assert st == 5 and b"reserves" in kvq.lib().kvq_last_error()


def test_noalloc_refuses_what_the_workspace_call_refuses():
    # argument errors come first, with kvq_decode_attn's status, before the scratch check
    cfg = kvq.VqConfig(n_heads=16, max_pages=760, max_batch=64, max_ctx=6144)
    c = cfg.to_c()
    kc = kvq.VqCacheC(*([0x10000] * 12))
    f = kvq.lib().kvq_decode_attn_noalloc
    assert f(kvq.FMT_LOOPVQ, ctypes.byref(c), ctypes.byref(kc), 0, 1, 0x10000, 64, 0x10000, kvq.OUT_FP32, 5000,
             None) == 1   # n_splits out of range
    assert f(kvq.FMT_LOOPVQ, ctypes.byref(c), ctypes.byref(kc), 0, 1, 0x10000, 65, 0x10000, kvq.OUT_FP32, 0,
             None) == 2   # B > max_batch
    assert f(kvq.FMT_LOOPVQ, ctypes.byref(c), ctypes.byref(kc), 0, 1, 0x10000, 64, 0x10000, 7, 0,
             None) == 1   # out_dtype
