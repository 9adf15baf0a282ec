// kvq_decode_attn_noalloc: decode attention for callers that cannot allocate device memory.
//
// Some callers own no allocator: a serving engine that reserves all device memory for its
// own pool at start-up and refuses any further cudaMalloc, or code running inside a host
// framework's callback that is handed only the tensors it works on. They cannot provide the
// split-K workspace that kvq_decode_attn asks for. This entry point keeps that workspace in
// a fixed array inside the library instead (KVQ_NOALLOC_SCRATCH_BYTES per device) and
// otherwise runs exactly kvq_decode_attn.
//
// When the array takes device memory: CUDA loads the library's device code on a device
// lazily, at the first kernel launch or symbol lookup there, and sets the array aside then;
// from that point it is held until the process exits. A caller whose pool takes all device
// memory must therefore make its first call on each device (which looks the address up)
// before the pool is created. The address is looked up once per device and kept: after a
// cudaDeviceReset the array may move, so the library must not be used across a reset.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/kvq.h"
#include "kvq_internal.h"

#define KVQ_API extern "C" __attribute__((visibility("default")))

namespace {

// The shared scratch. In host code this name is only a stand-in for the device array; the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of the scratch array on the current device, looked up once per device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

KVQ_API kvq_status kvq_decode_attn_noalloc(int format, const void* cfg, const void* cache, int layer,
                                           int loop_step, const uint16_t* q, int B, void* out, int out_dtype,
                                           int n_splits, kvq_stream stream) {
  // the same argument checks as kvq_decode_attn first, so a call it would refuse is refused
  // here with the same status, before the scratch array is touched
  const kvq_status st = kvq::check_decode_args(format, cfg, cache, layer, loop_step, q, B, out, out_dtype, n_splits,
                                               __func__);
  if (st != KVQ_OK) return st;
  const size_t need = kvq_decode_workspace_size(format, cfg, B, n_splits);
  if (need > KVQ_NOALLOC_SCRATCH_BYTES) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "kvq_decode_attn_noalloc: this call needs %zu bytes of scratch, more than the %u the library "
             "reserves; use kvq_decode_attn with a workspace",
             need, (unsigned)KVQ_NOALLOC_SCRATCH_BYTES);
    kvq::set_last_error(msg);
    return KVQ_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  size_t ws_bytes = 0;
  if (need > 0) {
    cudaError_t e = scratch_address(&ws);
    if (e != cudaSuccess) {
      char msg[256];
      snprintf(msg, sizeof(msg), "kvq_decode_attn_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      kvq::set_last_error(msg);
      return KVQ_ERR_CUDA;
    }
    // the array keeps whatever the previous call left: clear the part this call uses
    e = cudaMemsetAsync(ws, 0, need, (cudaStream_t)stream);
    if (e != cudaSuccess) {
      char msg[256];
      snprintf(msg, sizeof(msg), "kvq_decode_attn_noalloc: cudaMemsetAsync: %s", cudaGetErrorString(e));
      kvq::set_last_error(msg);
      return KVQ_ERR_CUDA;
    }
    ws_bytes = KVQ_NOALLOC_SCRATCH_BYTES;
  }
  return kvq_decode_attn(format, cfg, cache, layer, loop_step, q, B, out, out_dtype, n_splits, ws, ws_bytes,
                         stream);
}
