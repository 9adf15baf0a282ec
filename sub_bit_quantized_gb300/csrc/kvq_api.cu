// C ABI of libkvq: argument validation, split planning and kernel launches.
// Every entry point checks its arguments on the host before it launches anything.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/kvq.h"
#include "kvq_internal.h"

#define KVQ_API extern "C" __attribute__((visibility("default")))

namespace {

thread_local char g_last_error[512] = "";

kvq_status fail(kvq_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

kvq_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return KVQ_OK;
  return fail(KVQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define CHECK_PTR(p)                                                                          \
  do {                                                                                        \
    if (!aligned16(p)) return fail(KVQ_ERR_INVALID_ARG, "%s: pointer " #p " is null or not " \
                                                        "16-byte aligned", __func__);         \
  } while (0)

// ---- per-device error word ------------------------------------------------------------
__device__ int g_device_error;
std::mutex g_err_mu;
int* g_err_ptr[64] = {nullptr};

int* device_error_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

// ---- LoopVQ config ---------------------------------------------------------------------
kvq_status check_vq_cfg(const kvq_vq_cfg* c, const char* fn) {
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "%s: cfg is null", fn);
  if (c->D <= 0 || c->T <= 0 || c->Tc <= 0 || c->G <= 0 || c->K <= 0 || c->n_layers <= 0 || c->n_heads <= 0 ||
      c->sink < 0 || c->recent < 0 || c->max_pages < 0 || c->max_batch <= 0 || c->max_ctx < 2 ||
      !(c->rope_base > 0.f))
    return fail(KVQ_ERR_INVALID_ARG, "%s: cfg has a non-positive field (max_ctx needs >= 2)", fn);
  if (c->T % c->Tc != 0 || c->G % c->Tc != 0)
    return fail(KVQ_ERR_INVALID_ARG, "%s: Tc=%d must divide T=%d and G=%d", fn, c->Tc, c->T, c->G);
  const int cc = c->G / c->Tc;
  if (c->D % cc != 0) return fail(KVQ_ERR_INVALID_ARG, "%s: c=G/Tc=%d must divide D=%d", fn, cc, c->D);
  if (c->D != kvq::kD) return fail(KVQ_ERR_UNSUPPORTED, "%s: D=%d (this build supports 128)", fn, c->D);
  // (Tc, c): c = 8 at Tc = 1, 2, 4 (G = 8, 16, 32); at G = 16 also Tc = 1 (c = 16, the
  // per-step special case) and Tc = 4 (c = 4)
  const bool built = (cc == 8 && (c->Tc == 1 || c->Tc == 2 || c->Tc == 4)) || (cc == 16 && c->Tc == 1) ||
                     (cc == 4 && c->Tc == 4);
  if (!built)
    return fail(KVQ_ERR_UNSUPPORTED, "%s: Tc=%d with c=G/Tc=%d (this build: c=8 with Tc=1,2,4; c=16 with Tc=1; "
                "c=4 with Tc=4)", fn, c->Tc, cc);
  if (c->K != kvq::kCB) return fail(KVQ_ERR_UNSUPPORTED, "%s: K=%d (8-bit indices need 256)", fn, c->K);
  return KVQ_OK;
}

int win_slots(const kvq_vq_cfg* c) { return c->sink + c->recent + kvq::kPage; }

// Blocks of the LoopVQ decode kernel: one per SM unless the caller names a count (every block
// takes an equal contiguous share of the page positions, so any count is correct).
int plan_vq_blocks(int n_splits) { return n_splits > 0 ? n_splits : sm_count(); }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t vq_ws_bytes(const kvq_vq_cfg* c, int B, int blocks) { return kvq::vq_attn_ws_bytes(B, c->n_heads, blocks); }

// ---- KIVI config -----------------------------------------------------------------------
kvq_status check_kivi_cfg(const kvq_kivi_cfg* c, const char* fn) {
  if (!c) return fail(KVQ_ERR_INVALID_ARG, "%s: cfg is null", fn);
  if (c->D <= 0 || c->n_heads <= 0 || c->n_q_heads <= 0 || c->k_bits <= 0 || c->v_bits <= 0 || c->group <= 0 ||
      c->residual < 0 || c->max_batch <= 0 || c->max_tokens < 0)
    return fail(KVQ_ERR_INVALID_ARG, "%s: cfg has a non-positive field", fn);
  if (c->max_tokens % c->group != 0 || c->D % c->group != 0 || c->residual % c->group != 0)
    return fail(KVQ_ERR_INVALID_ARG, "%s: group=%d must divide D=%d, max_tokens=%d and residual=%d", fn, c->group,
                c->D, c->max_tokens, c->residual);
  if (c->n_q_heads % c->n_heads != 0)
    return fail(KVQ_ERR_INVALID_ARG, "%s: n_q_heads=%d is not a multiple of n_heads=%d", fn, c->n_q_heads,
                c->n_heads);
  if (c->D != kvq::kD) return fail(KVQ_ERR_UNSUPPORTED, "%s: D=%d (this build supports 128)", fn, c->D);
  if ((c->k_bits != 2 && c->k_bits != 4) || (c->v_bits != 2 && c->v_bits != 4))
    return fail(KVQ_ERR_UNSUPPORTED, "%s: k_bits=%d v_bits=%d (this build supports 2 and 4)", fn, c->k_bits,
                c->v_bits);
  if (c->group != 32) return fail(KVQ_ERR_UNSUPPORTED, "%s: group=%d (this build supports 32)", fn, c->group);
  if (c->n_heads > 65535 || c->max_batch > 65535)
    return fail(KVQ_ERR_UNSUPPORTED, "%s: n_heads and max_batch must be at most 65535", fn);
  return KVQ_OK;
}

kvq_status check_kivi_cache(const kvq_kivi_cache* k, const char* fn) {
  if (!k) return fail(KVQ_ERR_INVALID_ARG, "%s: cache is null", fn);
  const void* ptrs[] = {k->k_codes, k->k_scale, k->k_zero, k->v_codes, k->v_scale, k->v_zero,
                        k->k_resid, k->v_resid, k->n_tok,  k->n_quant_k, k->n_quant_v, k->sync};
  for (const void* pp : ptrs)
    if (!aligned16(pp)) return fail(KVQ_ERR_INVALID_ARG, "%s: a cache pointer is null or misaligned", fn);
  return KVQ_OK;
}

struct KiviPlan {
  int n_split, tps;
};

// Token splits of the KIVI kernel per (request, KV head, head subgroup): split k takes
// quantized tokens [k tps, (k + 1) tps), and the last split also attends the fp16 residual.
// The residual's 512 B per token count as quantized tokens of the same bytes, so tps divides
// the quantized tokens plus that share evenly. A block's time is taken as tps plus a per-block
// cost. The GPU starts a block whenever a slot frees (slots = resident blocks per SM x SMs),
// so the call lasts about blocks / slots block times plus a tail in which the last blocks
// finish on a partly idle GPU, 0.83 of a block time. The plan minimises that over plans of at
// least 1.5 rounds. Measured split sweeps on this GPU (us per call): one head at 2 bits,
// batch 16 x 32 heads, 4K: 2: 97.2, 3: 94.4, 4: 93.6 (picked), 5: 94.2, 6: 98.1. 4-bit GQA,
// 32 over 8 heads: 5: 82.4, 6: 79.1, 7: 75.0 (picked), 8: 81.4, 9: 78.8. Whole rounds (the
// earlier model) picked 2 splits for the first; a tail of half a block time picked 6 for the
// second. Tails between 0.78 and 0.875 pick both optima.
KiviPlan plan_kivi(const kvq_kivi_cfg* c, int B, int n_splits) {
  const double q_bytes = (c->k_bits + c->v_bits) * 16.0 + 24.0;  // codes + per-token share of scales
  const double resid_cost = c->residual * (512.0 / q_bytes);
  auto tps_for = [&](int n) {
    const int t = (int)std::ceil((c->max_tokens + resid_cost) / n);
    return std::max(c->group, (t + c->group - 1) / c->group * c->group);
  };
  if (n_splits > 0) return KiviPlan{n_splits, tps_for(n_splits)};
  if (c->max_tokens == 0) return KiviPlan{1, c->group};
  const int rh = kvq::kivi_heads_per_block(c->n_q_heads / c->n_heads);
  const long long slots = (long long)kvq::kivi_attn_blocks_per_sm(c->k_bits, c->v_bits, rh) * sm_count();
  KiviPlan p{1, tps_for(1)};
  double best = 1e300;
  for (int n = 1; n <= std::min(64, c->max_tokens / c->group); ++n) {
    const int tps = tps_for(n);
    const long long blocks = (long long)B * (c->n_q_heads / rh) * n;
    if (2 * blocks < 3 * slots && n < std::min(64, c->max_tokens / c->group)) continue;  // under 1.5 rounds
    const double cost = ((double)blocks / (double)slots + 0.83) * (tps + 200.0);
    if (cost < best * 0.999) {
      best = cost;
      p = KiviPlan{n, tps};
    }
  }
  return p;
}

size_t kivi_ws_bytes(const kvq_kivi_cfg* c, int B, const KiviPlan& p) {
  const int total = p.n_split;
  if (total <= 1) return 0;
  return align256((size_t)B * c->n_q_heads * total * (kvq::kD + 2) * sizeof(float)) +
         align256((size_t)B * c->n_q_heads * sizeof(int));
}

}  // namespace

void kvq::set_last_error(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }

// ======================================================================================
// Exported entry points
// ======================================================================================

KVQ_API int kvq_version(void) { return 100; }

KVQ_API const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_CAPACITY: return "capacity exceeded";
    case KVQ_ERR_UNSUPPORTED: return "unsupported shape";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_WORKSPACE: return "workspace too small";
    case KVQ_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

KVQ_API const char* kvq_last_error(void) { return g_last_error; }

KVQ_API int kvq_device_error(void) {
  int* p = device_error_ptr();
  if (!p) return KVQ_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return KVQ_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return KVQ_ERR_CUDA;
  if (v != 0 && cudaMemset(p, 0, sizeof(int)) != cudaSuccess) return KVQ_ERR_CUDA;
  return v;
}

KVQ_API kvq_status kvq_vq_cache_sizes(const kvq_vq_cfg* c, kvq_vq_sizes* out) {
  kvq_status st = check_vq_cfg(c, __func__);
  if (st != KVQ_OK) return st;
  if (!out) return fail(KVQ_ERR_INVALID_ARG, "%s: out is null", __func__);
  const size_t NB = c->T / c->Tc, NG = c->D / (c->G / c->Tc);
  out->idx = (size_t)c->n_layers * NB * c->max_batch * c->n_heads * c->max_pages * (8 * NG);
  out->win = (size_t)c->n_layers * c->T * c->max_batch * c->n_heads * win_slots(c) * c->D * 2;
  out->bt = (size_t)c->n_layers * c->T * c->n_heads * c->K * c->D * 4;
  out->bt_v = (size_t)c->n_layers * c->T * c->n_heads * c->K * c->D * 2;
  out->cb = (size_t)c->n_layers * NB * c->n_heads * NG * c->K * c->G * 4;
  out->rope = (size_t)c->max_ctx * (c->D / 2) * 4;
  out->per_request = (size_t)c->max_batch * 4;
  out->cbp = (size_t)c->n_layers * NB * c->n_heads * NG * kvq::split_codebook_bytes(c->G);
  return KVQ_OK;
}

KVQ_API kvq_status kvq_rope_table(const kvq_vq_cfg* c, float* rc, float* rs, kvq_stream stream) {
  kvq_status st = check_vq_cfg(c, __func__);
  if (st != KVQ_OK) return st;
  CHECK_PTR(rc);
  CHECK_PTR(rs);
  return cuda_status(kvq::launch_rope_table(rc, rs, c->max_ctx, c->D, c->rope_base, (cudaStream_t)stream),
                     __func__);
}

KVQ_API kvq_status kvq_slice_codebooks(const kvq_vq_cfg* c, const float* cb, float* bt, kvq_stream stream) {
  kvq_status st = check_vq_cfg(c, __func__);
  if (st != KVQ_OK) return st;
  CHECK_PTR(cb);
  CHECK_PTR(bt);
  return cuda_status(
      kvq::launch_slice_codebooks(cb, bt, c->n_layers, c->T, c->Tc, c->G, c->n_heads, (cudaStream_t)stream),
      __func__);
}

KVQ_API kvq_status kvq_slice_codebooks_fp16(const kvq_vq_cfg* c, const float* cb, uint16_t* bt16,
                                            kvq_stream stream) {
  kvq_status st = check_vq_cfg(c, __func__);
  if (st != KVQ_OK) return st;
  CHECK_PTR(cb);
  CHECK_PTR(bt16);
  return cuda_status(kvq::launch_slice_codebooks_fp16(cb, bt16, c->n_layers, c->T, c->Tc, c->G, c->n_heads,
                                                      (cudaStream_t)stream),
                     __func__);
}

KVQ_API kvq_status kvq_split_codebooks(const kvq_vq_cfg* c, const float* cb, uint8_t* cbp, kvq_stream stream) {
  kvq_status st = check_vq_cfg(c, __func__);
  if (st != KVQ_OK) return st;
  CHECK_PTR(cb);
  CHECK_PTR(cbp);
  const long long n = (long long)c->n_layers * (c->T / c->Tc) * c->n_heads * (c->D / (c->G / c->Tc));
  return cuda_status(kvq::launch_split_codebooks(cb, cbp, n, c->Tc, c->G, (cudaStream_t)stream), __func__);
}

static kvq_status check_x_strides(const char* fn, int64_t st, int64_t sb, int64_t sh) {
  if (st < 0 || sb < 0 || sh < 0 || (st % 8) || (sb % 8) || (sh % 8))
    return fail(KVQ_ERR_INVALID_ARG, "%s: strides must be non-negative multiples of 8 elements", fn);
  return KVQ_OK;
}

KVQ_API kvq_status kvq_encode_vq(const kvq_vq_cfg* c, const uint16_t* x, int64_t st_t, int64_t st_b, int64_t st_h,
                                 int seq_begin, int n_seq, int n_tok, const float* cb, uint8_t* idx,
                                 int page_begin, int g_begin, int g_count, int32_t* n_ties, kvq_stream stream) {
  kvq_status st = check_vq_cfg(c, __func__);
  if (st != KVQ_OK) return st;
  if ((st = check_x_strides(__func__, st_t, st_b, st_h)) != KVQ_OK) return st;
  CHECK_PTR(x);
  CHECK_PTR(cb);
  CHECK_PTR(idx);
  if (n_ties && (reinterpret_cast<uintptr_t>(n_ties) & 3u)) return fail(KVQ_ERR_INVALID_ARG, "%s: n_ties misaligned", __func__);
  const int NG = c->D / (c->G / c->Tc);
  if (n_seq < 0 || n_tok < 0 || n_tok % kvq::kPage || seq_begin < 0 || page_begin < 0)
    return fail(KVQ_ERR_INVALID_ARG, "%s: n_seq/n_tok/seq_begin/page_begin invalid (n_tok multiple of 8)", __func__);
  if (g_begin < 0 || g_count < 0 || g_begin + g_count > NG)
    return fail(KVQ_ERR_INVALID_ARG, "%s: groups [%d, %d) outside [0, %d)", __func__, g_begin, g_begin + g_count, NG);
  if (seq_begin + n_seq > c->max_batch || page_begin + n_tok / kvq::kPage > c->max_pages)
    return fail(KVQ_ERR_CAPACITY, "%s: requests or pages exceed max_batch / max_pages", __func__);
  kvq::VqEncodeArgs a{};
  a.x = x; a.st = st_t; a.sb = st_b; a.sh = st_h;
  a.cb = cb; a.idx = idx; a.n_ties = n_ties; a.err = device_error_ptr();
  a.T = c->T; a.Tc = c->Tc; a.G = c->G; a.NB = c->T / c->Tc; a.H = c->n_heads;
  a.max_batch = c->max_batch; a.max_pages = c->max_pages;
  a.seq_begin = seq_begin; a.n_seq = n_seq; a.n_tok = n_tok; a.page_begin = page_begin;
  a.g_begin = g_begin; a.g_count = g_count;
  return cuda_status(kvq::launch_vq_encode(a, (cudaStream_t)stream), __func__);
}

static kvq_status check_vq_cache(const kvq_vq_cache* k, const char* fn) {
  if (!k) return fail(KVQ_ERR_INVALID_ARG, "%s: cache is null", fn);
  const void* ptrs[] = {k->idx_k, k->idx_v, k->win_k, k->win_v, k->bt_k, k->bt_v,
                        k->cb_k, k->cb_v, k->rope_cos, k->rope_sin, k->seq_len, k->n_pages};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(KVQ_ERR_INVALID_ARG, "%s: a cache pointer is null or not 16-byte aligned", fn);
  for (const void* p : {static_cast<const void*>(k->cbp_k), static_cast<const void*>(k->cbp_v)})
    if (p && !aligned16(p)) return fail(KVQ_ERR_INVALID_ARG, "%s: cbp_k / cbp_v not 16-byte aligned", fn);
  return KVQ_OK;
}

KVQ_API kvq_status kvq_prefill_vq(const kvq_vq_cfg* c, const kvq_vq_cache* k, int layer, const uint16_t* xk,
                                  const uint16_t* xv, int64_t st_t, int64_t st_b, int64_t st_h, int seq_begin,
                                  int n_seq, int L, int32_t* n_ties, kvq_stream stream) {
  kvq_status st = check_vq_cfg(c, __func__);
  if (st != KVQ_OK) return st;
  if ((st = check_vq_cache(k, __func__)) != KVQ_OK) return st;
  if ((st = check_x_strides(__func__, st_t, st_b, st_h)) != KVQ_OK) return st;
  CHECK_PTR(xk);
  CHECK_PTR(xv);
  if (layer < 0 || layer >= c->n_layers || seq_begin < 0 || n_seq < 0 || L < 1)
    return fail(KVQ_ERR_INVALID_ARG, "%s: layer/seq_begin/n_seq/L out of range", __func__);
  if (seq_begin + n_seq > c->max_batch || L > c->max_ctx)
    return fail(KVQ_ERR_CAPACITY, "%s: requests exceed max_batch or L exceeds max_ctx", __func__);
  const int n_pages = std::max(0, (L - c->sink - c->recent) / kvq::kPage);
  if (n_pages > c->max_pages)
    return fail(KVQ_ERR_CAPACITY, "%s: L=%d needs %d pages > max_pages=%d", __func__, L, n_pages, c->max_pages);
  if (n_seq == 0) return KVQ_OK;
  const int NB = c->T / c->Tc, NG = c->D / (c->G / c->Tc);
  const size_t idx_layer = (size_t)NB * c->max_batch * c->n_heads * c->max_pages * (8 * NG);
  const size_t cb_layer = (size_t)NB * c->n_heads * NG * c->K * c->G;
  const size_t win_layer = (size_t)c->T * c->max_batch * c->n_heads * win_slots(c) * c->D;
  cudaStream_t s = (cudaStream_t)stream;
  if (n_pages > 0) {
    for (int kv = 0; kv < 2; ++kv) {
      kvq::VqEncodeArgs a{};
      a.x = (kv ? xv : xk) + (size_t)c->sink * c->D;
      a.st = st_t; a.sb = st_b; a.sh = st_h;
      a.cb = (kv ? k->cb_v : k->cb_k) + layer * cb_layer;
      a.idx = (kv ? k->idx_v : k->idx_k) + layer * idx_layer;
      a.n_ties = n_ties; a.err = device_error_ptr();
      a.T = c->T; a.Tc = c->Tc; a.G = c->G; a.NB = NB; a.H = c->n_heads;
      a.max_batch = c->max_batch; a.max_pages = c->max_pages;
      a.seq_begin = seq_begin; a.n_seq = n_seq; a.n_tok = n_pages * kvq::kPage; a.page_begin = 0;
      a.g_begin = 0; a.g_count = NG;
      if ((st = cuda_status(kvq::launch_vq_encode(a, s), __func__)) != KVQ_OK) return st;
    }
  }
  kvq::VqWindowArgs w{};
  w.xk = xk; w.xv = xv; w.st = st_t; w.sb = st_b; w.sh = st_h;
  w.win_k = k->win_k + layer * win_layer; w.win_v = k->win_v + layer * win_layer;
  w.seq_len = (layer == 0) ? k->seq_len : nullptr; w.n_pages = k->n_pages;
  w.T = c->T; w.H = c->n_heads; w.max_batch = c->max_batch; w.win_slots = win_slots(c);
  w.sink = c->sink; w.recent = c->recent;
  w.seq_begin = seq_begin; w.n_seq = n_seq; w.L = L; w.n_pages_val = n_pages;
  return cuda_status(kvq::launch_vq_prefill_window(w, s), __func__);
}

KVQ_API kvq_status kvq_append_page(const kvq_vq_cfg* c, const kvq_vq_cache* k, int layer, int loop_step,
                                   const uint16_t* k_new, const uint16_t* v_new, int n_seq, kvq_stream stream) {
  kvq_status st = check_vq_cfg(c, __func__);
  if (st != KVQ_OK) return st;
  if ((st = check_vq_cache(k, __func__)) != KVQ_OK) return st;
  CHECK_PTR(k_new);
  CHECK_PTR(v_new);
  if (layer < 0 || layer >= c->n_layers || loop_step < 1 || loop_step > c->T || n_seq < 0)
    return fail(KVQ_ERR_INVALID_ARG, "%s: layer/loop_step/n_seq out of range", __func__);
  if (n_seq > c->max_batch) return fail(KVQ_ERR_CAPACITY, "%s: n_seq > max_batch", __func__);
  if (n_seq == 0) return KVQ_OK;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t win_step = (size_t)c->max_batch * c->n_heads * win_slots(c) * c->D;
  const size_t off = ((size_t)layer * c->T + (loop_step - 1)) * win_step;
  kvq::VqAppendArgs a{};
  a.k_new = k_new; a.v_new = v_new;
  a.win_k = k->win_k + off; a.win_v = k->win_v + off;
  a.seq_len = k->seq_len; a.n_pages = k->n_pages; a.err = device_error_ptr();
  a.H = c->n_heads; a.n_seq = n_seq; a.win_slots = win_slots(c); a.sink = c->sink; a.recent = c->recent;
  a.max_pages = c->max_pages; a.max_ctx = c->max_ctx;
  a.advance = (layer == 0 && loop_step == 1);
  if ((st = cuda_status(kvq::launch_vq_append(a, s), __func__)) != KVQ_OK) return st;
  if (!a.advance) return KVQ_OK;
  kvq::VqRollArgs r{};
  r.win_k = k->win_k; r.win_v = k->win_v; r.cb_k = k->cb_k; r.cb_v = k->cb_v;
  r.idx_k = k->idx_k; r.idx_v = k->idx_v; r.seq_len = k->seq_len; r.n_pages = k->n_pages;
  r.cbp_k = k->cbp_k; r.cbp_v = k->cbp_v;
  r.err = device_error_ptr();
  r.L = c->n_layers; r.T = c->T; r.Tc = c->Tc; r.G = c->G; r.NB = c->T / c->Tc; r.H = c->n_heads;
  r.n_seq = n_seq; r.max_batch = c->max_batch; r.max_pages = c->max_pages; r.win_slots = win_slots(c);
  r.sink = c->sink; r.recent = c->recent;
  return cuda_status(kvq::launch_vq_roll(r, s), __func__);
}

KVQ_API kvq_status kvq_quantize_kivi(const kvq_kivi_cfg* c, int axis, const uint16_t* x, int64_t st_b,
                                     int64_t st_h, int B, int n_tok, uint8_t* codes, uint16_t* scale,
                                     uint16_t* zero, int tok_begin, kvq_stream stream) {
  kvq_status st = check_kivi_cfg(c, __func__);
  if (st != KVQ_OK) return st;
  if ((st = check_x_strides(__func__, 0, st_b, st_h)) != KVQ_OK) return st;
  CHECK_PTR(x);
  CHECK_PTR(codes);
  CHECK_PTR(scale);
  CHECK_PTR(zero);
  if (axis != KVQ_PER_CHANNEL && axis != KVQ_PER_TOKEN)
    return fail(KVQ_ERR_INVALID_ARG, "%s: axis must be KVQ_PER_CHANNEL or KVQ_PER_TOKEN", __func__);
  if (B < 0 || n_tok < 0 || tok_begin < 0) return fail(KVQ_ERR_INVALID_ARG, "%s: negative size", __func__);
  if (axis == KVQ_PER_CHANNEL && (n_tok % c->group || tok_begin % c->group))
    return fail(KVQ_ERR_INVALID_ARG, "%s: per-channel groups need n_tok and tok_begin multiples of %d", __func__,
                c->group);
  if (B > c->max_batch || tok_begin + n_tok > c->max_tokens)
    return fail(KVQ_ERR_CAPACITY, "%s: B or tokens exceed the cache capacity", __func__);
  if (B == 0 || n_tok == 0) return KVQ_OK;
  kvq::KiviQuantArgs a{};
  a.x = x; a.sb = st_b; a.sh = st_h; a.codes = codes; a.scale = scale; a.zero = zero;
  a.axis = axis; a.bits = (axis == KVQ_PER_CHANNEL) ? c->k_bits : c->v_bits;
  a.B = B; a.H = c->n_heads; a.n_tok = n_tok; a.tok_begin = tok_begin;
  a.max_tokens = c->max_tokens; a.group = c->group; a.err = device_error_ptr();
  return cuda_status(kvq::launch_kivi_quantize(a, (cudaStream_t)stream), __func__);
}

KVQ_API kvq_status kvq_kivi_prefill(const kvq_kivi_cfg* c, const kvq_kivi_cache* k, const uint16_t* xk,
                                    const uint16_t* xv, int64_t st_b, int64_t st_h, int b0, int B, int n_tok,
                                    kvq_stream stream) {
  kvq_status st = check_kivi_cfg(c, __func__);
  if (st != KVQ_OK) return st;
  if ((st = check_kivi_cache(k, __func__)) != KVQ_OK) return st;
  if ((st = check_x_strides(__func__, 0, st_b, st_h)) != KVQ_OK) return st;
  CHECK_PTR(xk);
  CHECK_PTR(xv);
  if (c->residual <= 0) return fail(KVQ_ERR_INVALID_ARG, "%s: the streaming cache needs residual > 0", __func__);
  if (b0 < 0 || B < 0 || n_tok < 0) return fail(KVQ_ERR_INVALID_ARG, "%s: negative size", __func__);
  const int R = c->residual, G = c->group;
  const int nq = n_tok <= R ? 0 : (n_tok - R + G - 1) / G * G;
  if (b0 + B > c->max_batch || nq > c->max_tokens)
    return fail(KVQ_ERR_CAPACITY, "%s: requests or quantized tokens exceed the cache capacity", __func__);
  if (B == 0) return KVQ_OK;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t H = c->n_heads, N = c->max_tokens, D = c->D;
  if (nq > 0) {
    kvq::KiviQuantArgs a{};
    a.sb = st_b; a.sh = st_h; a.B = B; a.H = c->n_heads; a.n_tok = nq; a.tok_begin = 0;
    a.max_tokens = c->max_tokens; a.group = G; a.err = device_error_ptr();
    a.x = xk; a.axis = KVQ_PER_CHANNEL; a.bits = c->k_bits;
    a.codes = k->k_codes + (size_t)b0 * H * N * (D * c->k_bits / 8);
    a.scale = k->k_scale + (size_t)b0 * H * (N / G) * D;
    a.zero = k->k_zero + (size_t)b0 * H * (N / G) * D;
    if ((st = cuda_status(kvq::launch_kivi_quantize(a, s), __func__)) != KVQ_OK) return st;
    a.x = xv; a.axis = KVQ_PER_TOKEN; a.bits = c->v_bits;
    a.codes = k->v_codes + (size_t)b0 * H * N * (D * c->v_bits / 8);
    a.scale = k->v_scale + (size_t)b0 * H * N * (D / G);
    a.zero = k->v_zero + (size_t)b0 * H * N * (D / G);
    if ((st = cuda_status(kvq::launch_kivi_quantize(a, s), __func__)) != KVQ_OK) return st;
  }
  kvq::KiviTailArgs t{};
  t.k = xk; t.v = xv; t.sb = st_b; t.sh = st_h; t.k_resid = k->k_resid; t.v_resid = k->v_resid;
  t.n_tok = k->n_tok; t.n_quant_k = k->n_quant_k; t.n_quant_v = k->n_quant_v;
  t.b0 = b0; t.B = B; t.H = c->n_heads; t.n_tok_new = n_tok; t.nq = nq; t.residual = R;
  return cuda_status(kvq::launch_kivi_prefill_tail(t, s), __func__);
}

KVQ_API kvq_status kvq_kivi_append(const kvq_kivi_cfg* c, const kvq_kivi_cache* k, const uint16_t* k_new,
                                   const uint16_t* v_new, int n_seq, kvq_stream stream) {
  kvq_status st = check_kivi_cfg(c, __func__);
  if (st != KVQ_OK) return st;
  if ((st = check_kivi_cache(k, __func__)) != KVQ_OK) return st;
  CHECK_PTR(k_new);
  CHECK_PTR(v_new);
  if (c->residual <= 0) return fail(KVQ_ERR_INVALID_ARG, "%s: the streaming cache needs residual > 0", __func__);
  if (n_seq < 0) return fail(KVQ_ERR_INVALID_ARG, "%s: n_seq < 0", __func__);
  if (n_seq > c->max_batch) return fail(KVQ_ERR_CAPACITY, "%s: n_seq > max_batch", __func__);
  if (n_seq == 0) return KVQ_OK;
  kvq::KiviAppendArgs a{};
  a.k_new = k_new; a.v_new = v_new;
  a.k_codes = k->k_codes; a.k_scale = k->k_scale; a.k_zero = k->k_zero;
  a.v_codes = k->v_codes; a.v_scale = k->v_scale; a.v_zero = k->v_zero;
  a.k_resid = k->k_resid; a.v_resid = k->v_resid;
  a.n_tok = k->n_tok; a.n_quant_k = k->n_quant_k; a.n_quant_v = k->n_quant_v; a.sync = k->sync;
  a.err = device_error_ptr();
  a.n_seq = n_seq; a.H = c->n_heads; a.k_bits = c->k_bits; a.v_bits = c->v_bits; a.residual = c->residual;
  a.max_tokens = c->max_tokens;
  return cuda_status(kvq::launch_kivi_append(a, (cudaStream_t)stream), __func__);
}

KVQ_API size_t kvq_decode_workspace_size(int format, const void* cfg, int B, int n_splits) {
  if (B <= 0 || !cfg) return 0;
  if (format == KVQ_FMT_LOOPVQ) {
    const kvq_vq_cfg* c = static_cast<const kvq_vq_cfg*>(cfg);
    if (check_vq_cfg(c, __func__) != KVQ_OK) return 0;
    return vq_ws_bytes(c, B, plan_vq_blocks(n_splits));
  }
  if (format == KVQ_FMT_KIVI) {
    const kvq_kivi_cfg* c = static_cast<const kvq_kivi_cfg*>(cfg);
    if (check_kivi_cfg(c, __func__) != KVQ_OK) return 0;
    return kivi_ws_bytes(c, B, plan_kivi(c, B, n_splits));
  }
  return 0;
}

KVQ_API int kvq_decode_auto_splits(int format, const void* cfg, int B) {
  if (B <= 0 || !cfg) return 0;
  if (format == KVQ_FMT_LOOPVQ) {
    const kvq_vq_cfg* c = static_cast<const kvq_vq_cfg*>(cfg);
    if (check_vq_cfg(c, __func__) != KVQ_OK) return 0;
    return plan_vq_blocks(0);
  }
  if (format == KVQ_FMT_KIVI) {
    const kvq_kivi_cfg* c = static_cast<const kvq_kivi_cfg*>(cfg);
    if (check_kivi_cfg(c, __func__) != KVQ_OK) return 0;
    return plan_kivi(c, B, 0).n_split;
  }
  return 0;
}

namespace kvq {
// Every host-side check of kvq_decode_attn except the workspace (shared with the no-allocation
// entry point, so that both refuse the same calls with the same status before touching memory).
kvq_status check_decode_args(int format, const void* cfg, const void* cache, int layer, int loop_step,
                             const uint16_t* q, int B, const void* out, int out_dtype, int n_splits, const char* fn) {
  if (out_dtype != KVQ_OUT_BF16 && out_dtype != KVQ_OUT_FP32)
    return fail(KVQ_ERR_INVALID_ARG, "%s: out_dtype must be KVQ_OUT_BF16 or KVQ_OUT_FP32", fn);
  if (n_splits < 0 || n_splits > 4096) return fail(KVQ_ERR_INVALID_ARG, "%s: n_splits out of range", fn);
  if (!aligned16(q) || !aligned16(out))
    return fail(KVQ_ERR_INVALID_ARG, "%s: q or out is null or not 16-byte aligned", fn);
  if (format == KVQ_FMT_LOOPVQ) {
    const kvq_vq_cfg* c = static_cast<const kvq_vq_cfg*>(cfg);
    kvq_status st = check_vq_cfg(c, fn);
    if (st != KVQ_OK) return st;
    if ((st = check_vq_cache(static_cast<const kvq_vq_cache*>(cache), fn)) != KVQ_OK) return st;
    if (layer < 0 || layer >= c->n_layers || loop_step < 1 || loop_step > c->T || B < 1)
      return fail(KVQ_ERR_INVALID_ARG, "%s: layer/loop_step/B out of range", fn);
    if (B > c->max_batch) return fail(KVQ_ERR_CAPACITY, "%s: B=%d > max_batch=%d", fn, B, c->max_batch);
    if (B > kvq::kVqMaxBatch)
      return fail(KVQ_ERR_UNSUPPORTED, "%s: B=%d exceeds %d requests", fn, B, kvq::kVqMaxBatch);
    if ((long long)B * c->max_pages >= (1ll << 31))
      return fail(KVQ_ERR_UNSUPPORTED, "%s: too many index pages for one call", fn);
    return KVQ_OK;
  }
  if (format == KVQ_FMT_KIVI) {
    const kvq_kivi_cfg* c = static_cast<const kvq_kivi_cfg*>(cfg);
    kvq_status st = check_kivi_cfg(c, fn);
    if (st != KVQ_OK) return st;
    if ((st = check_kivi_cache(static_cast<const kvq_kivi_cache*>(cache), fn)) != KVQ_OK) return st;
    if (B < 1) return fail(KVQ_ERR_INVALID_ARG, "%s: B < 1", fn);
    if (B > c->max_batch) return fail(KVQ_ERR_CAPACITY, "%s: B > max_batch", fn);
    return KVQ_OK;
  }
  return fail(KVQ_ERR_INVALID_ARG, "%s: unknown format %d", fn, format);
}
}  // namespace kvq

KVQ_API kvq_status kvq_decode_attn(int format, const void* cfg, const void* cache, int layer, int loop_step,
                                   const uint16_t* q, int B, void* out, int out_dtype, int n_splits, void* ws,
                                   size_t ws_bytes, kvq_stream stream) {
  kvq_status st0 = kvq::check_decode_args(format, cfg, cache, layer, loop_step, q, B, out, out_dtype, n_splits,
                                          __func__);
  if (st0 != KVQ_OK) return st0;
  cudaStream_t s = (cudaStream_t)stream;
  if (format == KVQ_FMT_LOOPVQ) {
    const kvq_vq_cfg* c = static_cast<const kvq_vq_cfg*>(cfg);
    const kvq_vq_cache* k = static_cast<const kvq_vq_cache*>(cache);
    const int blocks = plan_vq_blocks(n_splits);
    const size_t need = vq_ws_bytes(c, B, blocks);
    if (!ws || ws_bytes < need || !aligned16(ws))
      return fail(KVQ_ERR_WORKSPACE, "%s: workspace needs %zu bytes (got %zu)", __func__, need, ws_bytes);
    const int NB = c->T / c->Tc, NG = c->D / (c->G / c->Tc);
    const int beta = (loop_step - 1) / c->Tc;
    const size_t idx_blk = (size_t)c->max_batch * c->n_heads * c->max_pages * (8 * NG);
    const size_t win_step = (size_t)c->max_batch * c->n_heads * win_slots(c) * c->D;
    const size_t bt_step = (size_t)c->n_heads * c->K * c->D;
    const size_t ls = (size_t)layer * c->T + (loop_step - 1);
    kvq::VqAttnArgs a{};
    a.idx_k = k->idx_k + ((size_t)layer * NB + beta) * idx_blk;
    a.idx_v = k->idx_v + ((size_t)layer * NB + beta) * idx_blk;
    a.win_k = k->win_k + ls * win_step;
    a.win_v = k->win_v + ls * win_step;
    a.bt_k = k->bt_k + ls * bt_step;
    a.bt_v = k->bt_v + ls * bt_step;
    a.rope_cos = k->rope_cos; a.rope_sin = k->rope_sin;
    a.seq_len = k->seq_len; a.n_pages = k->n_pages;
    a.q = q; a.out = out; a.out_fp32 = (out_dtype == KVQ_OUT_FP32);
    a.err = device_error_ptr();
    a.B = B; a.H = c->n_heads; a.max_pages = c->max_pages; a.max_ctx = c->max_ctx; a.sink = c->sink;
    a.recent = c->recent; a.win_slots = win_slots(c); a.G = blocks; a.NG = NG;
    return cuda_status(kvq::launch_vq_attn(a, ws, s), __func__);
  }
  if (format == KVQ_FMT_KIVI) {
    const kvq_kivi_cfg* c = static_cast<const kvq_kivi_cfg*>(cfg);
    const kvq_kivi_cache* k = static_cast<const kvq_kivi_cache*>(cache);
    const int rh = kvq::kivi_heads_per_block(c->n_q_heads / c->n_heads);
    if (kvq::kivi_attn_smem_bytes(c->k_bits, c->v_bits, rh, c->residual) > 232448)
      return fail(KVQ_ERR_UNSUPPORTED, "%s: residual=%d needs more shared memory than a block has", __func__,
                  c->residual);
    const KiviPlan p = plan_kivi(c, B, n_splits);
    if (p.tps > kvq::kivi_attn_max_tok_per_split(c->residual))
      return fail(KVQ_ERR_UNSUPPORTED, "%s: tokens per split exceed the shared-memory limit; use more splits",
                  __func__);
    const int total = p.n_split;  // blocks per (request, head subgroup); the last takes the residual
    if ((long long)total * (c->n_q_heads / c->n_heads / rh) >= (1ll << 31))
      return fail(KVQ_ERR_UNSUPPORTED, "%s: too many splits", __func__);
    const size_t need = kivi_ws_bytes(c, B, p);
    if (need > 0 && (!ws || ws_bytes < need || !aligned16(ws)))
      return fail(KVQ_ERR_WORKSPACE, "%s: workspace needs %zu bytes (got %zu)", __func__, need, ws_bytes);
    kvq::KiviAttnArgs a{};
    a.k_codes = k->k_codes; a.k_scale = k->k_scale; a.k_zero = k->k_zero;
    a.v_codes = k->v_codes; a.v_scale = k->v_scale; a.v_zero = k->v_zero;
    a.k_resid = k->k_resid; a.v_resid = k->v_resid;
    a.n_tok = k->n_tok; a.n_quant_k = k->n_quant_k; a.n_quant_v = k->n_quant_v;
    a.q = q; a.out = out; a.out_fp32 = (out_dtype == KVQ_OUT_FP32);
    if (total > 1) {
      a.part = static_cast<float*>(ws);
      a.counters = reinterpret_cast<int*>(static_cast<char*>(ws) +
                                          align256((size_t)B * c->n_q_heads * total * (kvq::kD + 2) * sizeof(float)));
    }
    a.err = device_error_ptr();
    a.B = B; a.H = c->n_heads; a.Hq = c->n_q_heads; a.k_bits = c->k_bits; a.v_bits = c->v_bits;
    a.max_tokens = c->max_tokens; a.residual = c->residual; a.group = c->group;
    a.n_split = p.n_split; a.tok_per_split = p.tps;
    return cuda_status(kvq::launch_kivi_attn(a, s), __func__);
  }
  return fail(KVQ_ERR_INVALID_ARG, "%s: unknown format %d", __func__, format);
}
