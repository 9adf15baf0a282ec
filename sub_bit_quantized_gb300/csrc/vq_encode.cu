// LoopVQ cache maintenance: RoPE table, codebook slicing, prefill window copy, decode-time
// append and page roll (the prefill encode itself runs on the tensor cores, vq_encode_tc.cu).
//
// "LoopVQ: Sub 1-bit KV Cache Quantization for Looped Transformers":
//  * background "vector quantization and codebooks": a(z) = argmin_r ||z - e_r||^2;
//  * method step 1 / Figure 3: coordinate i*Tc + m of the coupled vector of group g in loop
//    block beta is channel g*c + i at loop step beta*Tc + m + 1;
//  * method step 4 / Figure 5: sink + recent tokens stay bf16, the rest is encoded into
//    8-token index pages; during decode the oldest recent page is encoded every 8 tokens;
//  * method step 5: the per-loop-step codebook slice B_t is cut once at load time.
//
// Roll encode arithmetic (one page of 8 tokens per (layer, block, head), on CUDA cores):
// fp32 distances sum_k (z_k - e_k)^2 screen the 256 codewords (relative error below 1.1e-6
// for nonnegative sums of 16..32 fp32 terms); every candidate within 4e-6 (relative) of the
// fp32 minimum is re-evaluated in fp64, where bf16 inputs and fp32 entries subtract and
// square exactly. The result is the exact-arithmetic argmin with the lowest index on ties; a
// second-best fp64 distance within 1e-6 of the best counts as a tie.
#include <cuda_fp16.h>

#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "../../include/kvq.h"

namespace kvq {
namespace {

// ---------------------------------------------------------------- RoPE table
__global__ void rope_table_kernel(float* cos_t, float* sin_t, int max_ctx, int D, double base) {
  const int half = D / 2;
  const long long n = (long long)max_ctx * half;
  for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < n; k += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(k / half), i = (int)(k % half);
    const double theta = pow(base, -2.0 * i / D);
    double sv, cv;
    sincos((double)p * theta, &sv, &cv);
    cos_t[k] = (float)cv;
    sin_t[k] = (float)sv;
  }
}

// ---------------------------------------------------------------- B_t slices
// bt[l][t][h][ch / 64][r][ch % 64] = cb[l][beta][h][g][r][i*Tc + m], ch = g*c + i
__global__ void slice_kernel(const float* __restrict__ cb, float* __restrict__ bt, int L, int T, int Tc,
                             int G, int H) {
  const int c = G / Tc, NG = kD / c, NB = T / Tc;
  const long long n = (long long)L * T * H * kCB * kD;
  for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < n; k += (long long)gridDim.x * blockDim.x) {
    long long q = k;
    const int col = (int)(q % (kD / 2)); q /= (kD / 2);
    const int r = (int)(q % kCB); q /= kCB;
    const int half = (int)(q % 2); q /= 2;
    const int h = (int)(q % H); q /= H;
    const int t0 = (int)(q % T); q /= T;  // 0-based step
    const int l = (int)q;
    const int ch = half * (kD / 2) + col;
    const int beta = t0 / Tc, m = t0 % Tc, g = ch / c, i = ch % c;
    bt[k] = cb[((((size_t)l * NB + beta) * H + h) * NG + g) * (size_t)kCB * G + (size_t)r * G + i * Tc + m];
  }
}

// value slices in fp16 codeword rows: bt16[l][t][h][r][ch]
__global__ void slice_fp16_kernel(const float* __restrict__ cb, __half* __restrict__ bt16, int L, int T, int Tc,
                                  int G, int H) {
  const int c = G / Tc, NG = kD / c, NB = T / Tc;
  const long long n = (long long)L * T * H * kCB * kD;
  for (long long k = blockIdx.x * (long long)blockDim.x + threadIdx.x; k < n; k += (long long)gridDim.x * blockDim.x) {
    long long q = k;
    const int ch = (int)(q % kD); q /= kD;
    const int r = (int)(q % kCB); q /= kCB;
    const int h = (int)(q % H); q /= H;
    const int t0 = (int)(q % T); q /= T;  // 0-based step
    const int l = (int)q;
    const int beta = t0 / Tc, m = t0 % Tc, g = ch / c, i = ch % c;
    bt16[k] = __float2half_rn(cb[((((size_t)l * NB + beta) * H + h) * NG + g) * (size_t)kCB * G + (size_t)r * G + i * Tc + m]);
  }
}

// ---------------------------------------------------------------- exact nearest codeword
// z: G floats (bf16 values, exact in fp32); e: codebook [256][G] (global or shared).
// Returns the index; *tie set when the runner-up is within 1e-6 (relative) in fp64.
template <int G>
__device__ __forceinline__ int nearest_exact(const float (&z)[G], const float* __restrict__ e, bool* tie) {
  float best = INFINITY, second = INFINITY;
  int bi = 0;
  for (int r = 0; r < kCB; ++r) {
    const float* er = e + r * G;
    float d = 0.f;
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const float df = z[k] - er[k];
      d = fmaf(df, df, d);
    }
    if (d < best) {
      second = best;
      best = d;
      bi = r;
    } else if (d < second) {
      second = d;
    }
  }
  *tie = false;
  const float band = best * 4e-6f + 1e-30f;
  if (second > best + band) return bi;  // unique winner, no candidate near it
  // refine every candidate inside the band in fp64
  double b64 = INFINITY, s64 = INFINITY;
  int b64i = kCB;
  for (int r = 0; r < kCB; ++r) {
    const float* er = e + r * G;
    float d = 0.f;
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const float df = z[k] - er[k];
      d = fmaf(df, df, d);
    }
    if (d > best + band) continue;
    double dd = 0.0;
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const double df = (double)z[k] - (double)er[k];
      dd = fma(df, df, dd);
    }
    if (dd < b64) {  // strict: the lowest index wins exact ties
      s64 = b64;
      b64 = dd;
      b64i = r;
    } else if (dd < s64) {
      s64 = dd;
    }
  }
  *tie = (s64 <= b64 * (1.0 + 1e-6));
  return b64i;
}

__device__ __forceinline__ size_t page_byte(int g, int j) {  // in-page byte of (group, token)
  return (size_t)(((g & 7) * kPage + (j & 7)) * 2 + (g >> 3));
}

// ---------------------------------------------------------------- prefill window copy
// One block per (step, sequence, head); copies sink + recent tokens to their slots.
__global__ void prefill_window_kernel(const VqWindowArgs a) {
  const int h = blockIdx.x % a.H;
  const int b = (blockIdx.x / a.H) % a.n_seq;
  const int t0 = blockIdx.x / (a.H * a.n_seq);
  const int n_sink = min(a.sink, a.L);
  const int q1 = a.sink + kPage * a.n_pages_val;
  const int n_rec = max(0, a.L - q1);
  const int n = n_sink + n_rec;
  const size_t src0 = (size_t)t0 * a.st + (size_t)b * a.sb + (size_t)h * a.sh;
  const size_t dst0 = ((((size_t)t0 * a.max_batch) + a.seq_begin + b) * a.H + h) * (size_t)a.win_slots * kD;
  for (int k = threadIdx.x; k < n * (kD / 8); k += blockDim.x) {
    const int w = k / (kD / 8), q8 = k % (kD / 8);
    const int p = (w < n_sink) ? w : q1 + (w - n_sink);
    const int slot = (p < a.sink) ? p : a.sink + (p - a.sink) % (a.recent + kPage);
    const uint4 kv = __ldg(reinterpret_cast<const uint4*>(a.xk + src0 + (size_t)p * kD) + q8);
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(a.xv + src0 + (size_t)p * kD) + q8);
    reinterpret_cast<uint4*>(a.win_k + dst0 + (size_t)slot * kD)[q8] = kv;
    reinterpret_cast<uint4*>(a.win_v + dst0 + (size_t)slot * kD)[q8] = vv;
  }
  if (blockIdx.x == 0 && a.seq_len) {
    for (int i = threadIdx.x; i < a.n_seq; i += blockDim.x) {
      a.seq_len[a.seq_begin + i] = a.L;
      a.n_pages[a.seq_begin + i] = a.n_pages_val;
    }
  }
}

// ---------------------------------------------------------------- decode append
// One block per sequence. On the first (layer, step) of a token the block advances
// seq_len; every call writes the new token's K and V into its ring slot.
__global__ void append_kernel(const VqAppendArgs a) {
  const int b = blockIdx.x;
  __shared__ int pos;
  if (threadIdx.x == 0) {
    int L = a.seq_len[b];
    const int np = a.n_pages[b];
    if (a.advance) {
      // a request whose next token would overflow its buffers is left untouched
      const bool ok = (L + 1 <= a.max_ctx) && (L + 1 - a.sink - kPage * np <= a.recent + kPage) &&
                      (L + 1 - a.sink - kPage * np < a.recent + kPage || np < a.max_pages);
      if (ok) {
        L += 1;
        a.seq_len[b] = L;
      } else {
        set_error(a.err, KVQ_ERR_CAPACITY);
        L = -1;
      }
    }
    pos = (L > 0) ? L - 1 : -1;
  }
  __syncthreads();
  const int p = pos;
  if (p < 0) return;
  const int slot = (p < a.sink) ? p : a.sink + (p - a.sink) % (a.recent + kPage);
  for (int k = threadIdx.x; k < a.H * (kD / 8); k += blockDim.x) {
    const int h = k / (kD / 8), q8 = k % (kD / 8);
    const size_t dst = (((size_t)b * a.H + h) * a.win_slots + slot) * kD;
    const size_t src = ((size_t)b * a.H + h) * kD;
    reinterpret_cast<uint4*>(a.win_k + dst)[q8] = __ldg(reinterpret_cast<const uint4*>(a.k_new + src) + q8);
    reinterpret_cast<uint4*>(a.win_v + dst)[q8] = __ldg(reinterpret_cast<const uint4*>(a.v_new + src) + q8);
  }
}

__device__ __forceinline__ bool roll_due(const int32_t* seq_len, const int32_t* n_pages, int b, int sink,
                                         int recent, int max_pages) {
  const int L = seq_len[b], np = n_pages[b];
  return (L - sink - kPage * np == recent + kPage) && (np < max_pages);
}

// Roll: one block per (layer, block beta, head, K/V, sequence); 8 tokens x 16 groups.
template <int TC>
__global__ void __launch_bounds__(128) roll_kernel(const VqRollArgs a) {
  constexpr int G = TC * kC;
  const int b = blockIdx.y;
  if (!roll_due(a.seq_len, a.n_pages, b, a.sink, a.recent, a.max_pages)) return;
  int q = blockIdx.x;
  const int kv = q % 2; q /= 2;
  const int h = q % a.H; q /= a.H;
  const int beta = q % a.NB; q /= a.NB;
  const int l = q;
  const int np = a.n_pages[b];
  const int j = threadIdx.x / kNG, g = threadIdx.x % kNG;  // token in page, group
  const int p = a.sink + kPage * np + j;                   // position of the token
  const int slot = a.sink + (p - a.sink) % (a.recent + kPage);
  const uint16_t* win = kv ? a.win_v : a.win_k;
  float z[G];
#pragma unroll
  for (int m = 0; m < TC; ++m) {
    const int t0 = beta * TC + m;
    const uint16_t* xp =
        win + (((((size_t)l * a.T + t0) * a.max_batch + b) * a.H + h) * a.win_slots + slot) * kD + g * kC;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(xp));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < kC; ++i) {
      const uint32_t bits = (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu);
      z[i * TC + m] = bf16_to_f32(bits);
    }
  }
  const float* cb = (kv ? a.cb_v : a.cb_k) + ((((size_t)l * a.NB + beta) * a.H + h) * kNG + g) * (size_t)kCB * G;
  bool tie;
  const int r = nearest_exact<G>(z, cb, &tie);
  uint8_t* idx = (kv ? a.idx_v : a.idx_k) +
                 ((((size_t)l * a.NB + beta) * a.max_batch + b) * a.H + h) * (size_t)a.max_pages * kPageBytes;
  idx[(size_t)np * kPageBytes + page_byte(g, j)] = (uint8_t)r;
}

__global__ void roll_commit_kernel(const VqRollArgs a) {
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < a.n_seq; b += gridDim.x * blockDim.x)
    if (roll_due(a.seq_len, a.n_pages, b, a.sink, a.recent, a.max_pages)) a.n_pages[b] += 1;
}

int grid_for(long long n, int threads) {
  long long blocks = (n + threads - 1) / threads;
  if (blocks > 152 * 32) blocks = 152 * 32;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

}  // namespace

cudaError_t launch_rope_table(float* cos_t, float* sin_t, int max_ctx, int D, float base, cudaStream_t s) {
  rope_table_kernel<<<grid_for((long long)max_ctx * D / 2, 256), 256, 0, s>>>(cos_t, sin_t, max_ctx, D,
                                                                                (double)base);
  return cudaGetLastError();
}

cudaError_t launch_slice_codebooks(const float* cb, float* bt, int L, int T, int Tc, int G, int H,
                                   cudaStream_t s) {
  slice_kernel<<<grid_for((long long)L * T * H * kCB * kD, 256), 256, 0, s>>>(cb, bt, L, T, Tc, G, H);
  return cudaGetLastError();
}

cudaError_t launch_slice_codebooks_fp16(const float* cb, uint16_t* bt16, int L, int T, int Tc, int G, int H,
                                        cudaStream_t s) {
  slice_fp16_kernel<<<grid_for((long long)L * T * H * kCB * kD, 256), 256, 0, s>>>(
      cb, reinterpret_cast<__half*>(bt16), L, T, Tc, G, H);
  return cudaGetLastError();
}

cudaError_t launch_vq_prefill_window(const VqWindowArgs& a, cudaStream_t s) {
  prefill_window_kernel<<<a.T * a.n_seq * a.H, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_vq_append(const VqAppendArgs& a, cudaStream_t s) {
  append_kernel<<<a.n_seq, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_vq_roll(const VqRollArgs& a, cudaStream_t s) {
  dim3 grid(a.L * a.NB * a.H * 2, a.n_seq);
  switch (a.Tc) {
    case 1: roll_kernel<1><<<grid, 128, 0, s>>>(a); break;
    case 2: roll_kernel<2><<<grid, 128, 0, s>>>(a); break;
    case 4: roll_kernel<4><<<grid, 128, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  roll_commit_kernel<<<1, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
