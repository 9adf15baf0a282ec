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
// Roll encode: with the split codebook parts in the cache it runs on the tensor cores (the
// prefill encode kernel's roll instantiation, vq_encode_tc.cu); without them on CUDA cores
// (roll_kernel below) with the same decision rule: fp32 screening of z.e - |e|^2 / 2, every
// vector whose runner-up is inside the error band decided on distances summed with
// error-free fp32 steps, the lowest index winning exact ties.
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

// Roll: one block per (layer, block beta, head, K/V, group). The block stages that group's
// codebook (and each codeword's |e|^2 / 2) in shared memory once, codewords 2i and 2i + 1
// side by side per coordinate, and encodes the oldest recent page (8 tokens) of every due
// sequence against it, two vectors per thread: every codeword read (a broadcast: all threads
// of a warp read the same pair) serves both, and one packed FMA advances two codewords. Screening uses
// acc_r = z.e_r - |e_r|^2 / 2 (one FMA per coordinate; larger is nearer); a vector whose
// runner-up lies within the error band of its best (8x the fp32 accumulation bound of the
// codewords that can compete, plus the 1e-6 tie threshold) is decided on distances summed
// with error-free fp32 steps, the lowest index winning exact ties.
template <int TC, int C>
__global__ void __launch_bounds__(256) roll_kernel(const VqRollArgs a) {
  constexpr int G = TC * C, kNG = kD / C, kPageBytes = kPage * kNG;
  __shared__ __align__(16) float2 cbp[kCB / 2 * G];  // codewords 2i and 2i + 1 side by side per coordinate
  __shared__ __align__(8) float2 nhp[kCB / 2];
  int q = blockIdx.x;
  const int g = q % kNG; q /= kNG;
  const int kv = q % 2; q /= 2;
  const int h = q % a.H; q /= a.H;
  const int beta = q % a.NB; q /= a.NB;
  const int l = q;
  // between rolls no sequence is due: leave before staging anything
  int any = 0;
  for (int b = threadIdx.x; b < a.n_seq; b += blockDim.x)
    any |= roll_due(a.seq_len, a.n_pages, b, a.sink, a.recent, a.max_pages) ? 1 : 0;
  if (!__syncthreads_or(any)) return;
  const float* cb = (kv ? a.cb_v : a.cb_k) + ((((size_t)l * a.NB + beta) * a.H + h) * kNG + g) * (size_t)kCB * G;
  for (int r = threadIdx.x; r < kCB; r += blockDim.x) {
    float n_hi = 0.f, n_lo = 0.f;
#pragma unroll 4
    for (int k = 0; k < G; ++k) {
      const float e = __ldg(cb + (size_t)r * G + k);
      add_sq_diff(e, 0.f, n_hi, n_lo);
      reinterpret_cast<float*>(cbp)[((r >> 1) * G + k) * 2 + (r & 1)] = e;
    }
    reinterpret_cast<float*>(nhp)[r] = 0.5f * __fadd_rn(n_hi, n_lo);
  }
  __syncthreads();
  const float* nh = reinterpret_cast<const float*>(nhp);
  const uint16_t* win = kv ? a.win_v : a.win_k;
  uint8_t* idx_base = (kv ? a.idx_v : a.idx_k) + (((size_t)l * a.NB + beta) * a.max_batch) * a.H * (size_t)a.max_pages * kPageBytes;
  const int n_vec = a.n_seq * kPage;
  for (int v0 = threadIdx.x; v0 < n_vec; v0 += 2 * blockDim.x) {
    // ---- the two vectors (sequence, token in page) of this thread ------------------------
    float z[2][G];
    bool live[2];
    int b_of[2], np_of[2], j_of[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int v = v0 + u * blockDim.x;
      const int b = min(v, n_vec - 1) / kPage, j = v % kPage;
      live[u] = v < n_vec && roll_due(a.seq_len, a.n_pages, b, a.sink, a.recent, a.max_pages);
      const int np = a.n_pages[b];
      b_of[u] = b;
      np_of[u] = np;
      j_of[u] = j;
      const int p = a.sink + kPage * np + j;  // position of the token
      const int slot = a.sink + (p - a.sink) % (a.recent + kPage);
#pragma unroll
      for (int m = 0; m < TC; ++m) {  // channels g C .. g C + C - 1 of loop step beta TC + m
        uint32_t w[C / 2];
#pragma unroll
        for (int k = 0; k < C / 2; ++k) w[k] = 0;
        if (live[u]) {
          const int t0 = beta * TC + m;
          const uint16_t* xp =
              win + (((((size_t)l * a.T + t0) * a.max_batch + b) * a.H + h) * a.win_slots + slot) * kD + g * C;
          if constexpr (C == 4) {
            const uint2 w2 = __ldg(reinterpret_cast<const uint2*>(xp));
            w[0] = w2.x;
            w[1] = w2.y;
          } else {
#pragma unroll
            for (int k4 = 0; k4 < C / 8; ++k4) {
              const uint4 w4 = __ldg(reinterpret_cast<const uint4*>(xp) + k4);
              w[4 * k4] = w4.x;
              w[4 * k4 + 1] = w4.y;
              w[4 * k4 + 2] = w4.z;
              w[4 * k4 + 3] = w4.w;
            }
          }
        }
#pragma unroll
        for (int i = 0; i < C; ++i) z[u][i * TC + m] = (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
      }
    }
    // ---- screening: best two of acc_r = z.e_r - |e_r|^2/2 for both vectors, codewords two
    //      at a time with packed FMAs (each lane the same fma sequence as a scalar loop) ----
    float best[2] = {-INFINITY, -INFINITY}, second[2] = {-INFINITY, -INFINITY};
    int bi[2] = {0, 0};
    float2 zz[2][G];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int k = 0; k < G; ++k) zz[u][k] = make_float2(z[u][k], z[u][k]);
#pragma unroll 2
    for (int rp = 0; rp < kCB / 2; ++rp) {
      const float4* er = reinterpret_cast<const float4*>(cbp + rp * G);
      const float2 n2 = nhp[rp];
      float2 acc[2] = {make_float2(-n2.x, -n2.y), make_float2(-n2.x, -n2.y)};
#pragma unroll
      for (int k2 = 0; k2 < G / 2; ++k2) {
        const float4 e = er[k2];  // (e_r, e_r+1) at coordinates 2 k2 and 2 k2 + 1
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          acc[u] = __ffma2_rn(zz[u][2 * k2], make_float2(e.x, e.y), acc[u]);
          acc[u] = __ffma2_rn(zz[u][2 * k2 + 1], make_float2(e.z, e.w), acc[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {  // codeword 2 rp, then 2 rp + 1
          const float av = h2 ? acc[u].y : acc[u].x;
          second[u] = fmaxf(second[u], fminf(av, best[u]));
          bi[u] = (av > best[u]) ? 2 * rp + h2 : bi[u];
          best[u] = fmaxf(best[u], av);
        }
      }
    }
    // ---- band check; exact decision of near-ties; index out ----------------------------------
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (!live[u]) continue;
      float z2 = 0.f;
#pragma unroll
      for (int k = 0; k < G; ++k) z2 = fmaf(z[u][k], z[u][k], z2);
      const float znorm = sqrtf(z2);
      const float dbest = fmaxf(0.f, z2 - 2.f * best[u]);
      const float enear = znorm + 1.01f * sqrtf(dbest) + 1e-3f * znorm + 1e-6f;
      const float band = 8.f * (G + 2) * 5.97e-8f * (znorm * enear + 0.5f * enear * enear) + 1e-6f * dbest + 1e-30f;
      int result = bi[u];
      if (second[u] >= best[u] - band) {
        float bd = INFINITY;
        for (int r = 0; r < kCB; ++r) {
          const float* er = reinterpret_cast<const float*>(cbp + (r >> 1) * G) + (r & 1);  // stride 2
          float acc = -nh[r];  // the screening value again, computed the same way
#pragma unroll
          for (int k = 0; k < G; ++k) acc = fmaf(z[u][k], er[2 * k], acc);
          if (acc < best[u] - band) continue;
          float dh = 0.f, dl = 0.f;
#pragma unroll
          for (int k = 0; k < G; ++k) add_sq_diff(z[u][k], er[2 * k], dh, dl);
          const float dd = __fadd_rn(dh, dl);
          if (dd < bd) {  // increasing r: the lowest index wins exact ties
            bd = dd;
            result = r;
          }
        }
      }
      idx_base[((size_t)b_of[u] * a.H + h) * (size_t)a.max_pages * kPageBytes + (size_t)np_of[u] * kPageBytes +
               page_byte(g, j_of[u], kNG)] = (uint8_t)result;
    }
  }
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
  const int C = a.G / a.Tc;
  if (a.cbp_k && a.cbp_v) {
    // on the tensor cores: every (layer, K/V, beta, head, group) codebook against the oldest
    // recent page of every due request, the (request, token) rows of one plane sharing it
    const int NG = kD / C;
    const int64_t st = (int64_t)a.max_batch * a.H * a.win_slots * kD;  // loop-step stride of a window
    VqEncodeArgs e{};
    e.x = a.win_k; e.x2 = a.win_v;
    e.cb = a.cb_k;
    e.cbp = a.cbp_k; e.cbp2 = a.cbp_v;
    e.idx = a.idx_k; e.idx2 = a.idx_v;
    e.st = st; e.sb = (int64_t)a.H * a.win_slots * kD; e.sh = (int64_t)a.win_slots * kD;
    e.x_layer = (int64_t)a.T * st;
    e.cbp_layer = (int64_t)a.NB * a.H * NG * (int64_t)split_codebook_bytes(a.G);
    e.idx_layer = (int64_t)a.NB * a.max_batch * a.H * a.max_pages * kPage * NG;
    e.seq_len = a.seq_len; e.n_pages = a.n_pages;
    e.sink = a.sink; e.recent = a.recent; e.n_req = a.n_seq;
    e.n_ties = nullptr; e.err = a.err;
    e.T = a.T; e.Tc = a.Tc; e.G = a.G; e.NB = a.NB; e.H = a.H; e.max_batch = a.max_batch; e.max_pages = a.max_pages;
    e.seq_begin = 0; e.n_seq = 2 * a.L; e.n_tok = kPage * a.n_seq; e.page_begin = 0; e.g_begin = 0; e.g_count = NG;
    cudaError_t err = launch_vq_roll_tc(e, s);
    if (err != cudaSuccess) return err;
    roll_commit_kernel<<<1, 256, 0, s>>>(a);
    return cudaGetLastError();
  }
  dim3 grid(a.L * a.NB * a.H * 2 * (kD / C));
  if (a.Tc == 1 && C == 8) roll_kernel<1, 8><<<grid, 256, 0, s>>>(a);
  else if (a.Tc == 2 && C == 8) roll_kernel<2, 8><<<grid, 256, 0, s>>>(a);
  else if (a.Tc == 4 && C == 8) roll_kernel<4, 8><<<grid, 256, 0, s>>>(a);
  else if (a.Tc == 1 && C == 16) roll_kernel<1, 16><<<grid, 256, 0, s>>>(a);
  else if (a.Tc == 4 && C == 4) roll_kernel<4, 4><<<grid, 256, 0, s>>>(a);
  else return cudaErrorInvalidValue;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  roll_commit_kernel<<<1, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
