// Device helpers shared by the libkvq kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

// ---- error word -----------------------------------------------------------------------
// Kernels never trap. A failed device-side check or a timed-out wait stores a KVQ_ERR_*
// code in a per-device word (first error wins); kvq_device_error() reads and clears it.
__device__ __forceinline__ void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ---- number formats -----------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}
// low / high bf16 of a packed pair
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// round-to-nearest-even fp32 -> bf16 bits (finite inputs)
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

// ---- shared-memory addresses ---------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier + bulk (TMA) copies ------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// orders this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses of the same memory
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// 1-D bulk copy global -> shared; dst, src 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// shared-memory atomic add with acquire-release ordering at block scope; returns the old value
__device__ __forceinline__ int atom_add_acq_rel_shared(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_u32(p)), "r"(v) : "memory");
  return old;
}
// prefetch [src, src + bytes) into L2 (src 16-byte aligned, bytes a multiple of 16)
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for phase `parity` of `bar` to complete, for at most `limit_ns` nanoseconds.
// Returns false on timeout (the caller records an error and leaves).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = 1000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// As mbar_wait_bounded, but each retry lets the hardware suspend the warp for up to
// `hint_ns` until the phase completes, instead of spinning: a warp that waits long (a
// producer or consumer of a pipeline) then takes few issue slots from the warps that work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded_sleep(uint64_t* bar, uint32_t parity,
                                                        uint64_t limit_ns = 1000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// ---- exact-enough distances without fp64 -----------------------------------------------
// hi + lo += (z - e)^2 with error-free steps: z - e = s + t exactly (two-sum), s^2 = p + q
// exactly (fma), hi + p = h + err exactly (two-sum); the low parts gather in lo. The sum of
// 8..32 such terms keeps a relative error near one fp32 rounding (~1e-7), far below the 1e-6
// tie threshold, without fp64 arithmetic (slow on this GPU).
__device__ __forceinline__ void add_sq_diff(float z, float e, float& hi, float& lo) {
  const float s = __fsub_rn(z, e);
  const float bb = __fsub_rn(s, z);
  const float t = __fadd_rn(__fsub_rn(z, __fsub_rn(s, bb)), __fsub_rn(-e, bb));
  const float p = __fmul_rn(s, s);
  const float q = __fmaf_rn(s, s, -p);
  const float r = __fmaf_rn(__fmul_rn(2.f, s), t, q);
  const float h = __fadd_rn(hi, p);
  const float b2 = __fsub_rn(h, hi);
  const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(h, b2)), __fsub_rn(p, b2));
  hi = h;
  lo = __fadd_rn(lo, __fadd_rn(err, r));
}

// ---- streaming loads (read-once data: do not keep in L1) -------------------------------
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

}  // namespace kvq
