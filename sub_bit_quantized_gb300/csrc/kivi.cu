// KIVI 2-bit KV cache: group quantization and decode attention.
//
// "KIVI 完全拆解：非对称 2-bit KV Cache 量化":
//  * quantization-direction section: q = clamp(round(X/s + z), 0, 2^b - 1), X_hat = s(q - z),
//    [min, max] split evenly by s; keys per channel, values per token (core design);
//  * core design, eq. (3) and Algorithm 1: grouped (quantized) + fp16 residual segments,
//    logits of both concatenated before one softmax;
//  * implementation section: the Q_MatMul kernel fuses dequantization into the product.
//
// Quantize: one fp32 sequence (IEEE division, separate rounding of every step, round half
// to even) so codes, scales and zero-points match a reference that follows the same steps
// bit for bit. Attention: keys dequantize into the query instead of the cache -
// sum_ch q_ch s_ch (code - z_ch) = sum_ch (q_ch s_ch) code + bias - so each 32-token group
// folds its per-channel scale into the query once; values accumulate
// sum_j p_j s_jg code_j,ch and subtract sum_j p_j s_jg z_jg per channel group at the end.
#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "../../include/kvq.h"

#include <cuda_fp16.h>

namespace kvq {
namespace {

struct GroupQ {
  float s16f, z16f;
  uint16_t s_bits, z_bits;
};

__device__ __forceinline__ GroupQ group_params(float mn, float mx) {
  const float s = __fdiv_rn(__fsub_rn(mx, mn), 3.0f);
  __half s16 = __float2half_rn(s);
  if (__half2float(s16) == 0.0f) s16 = __float2half_rn(1.0f);
  const float s16f = __half2float(s16);
  const __half z16 = __float2half_rn(__fdiv_rn(-mn, s16f));
  GroupQ g;
  g.s16f = s16f;
  g.z16f = __half2float(z16);
  g.s_bits = __half_as_ushort(s16);
  g.z_bits = __half_as_ushort(z16);
  return g;
}

__device__ __forceinline__ uint32_t quant_code(float x, const GroupQ& g) {
  const float t = __fadd_rn(__fdiv_rn(x, g.s16f), g.z16f);
  const float r = fminf(fmaxf(rintf(t), 0.0f), 3.0f);
  return (uint32_t)r;
}

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// keys: one warp per (b, h, 32-token group); lane l owns channels 4l..4l+3, so each of the 32
// token rows is one coalesced 256-byte read (8 bytes per lane), all 32 in flight at once
__global__ void __launch_bounds__(256) kivi_quant_channel_kernel(const KiviQuantArgs a) {
  constexpr int kG = 32;  // tokens per key group (checked by the caller)
  const int lane = threadIdx.x & 31;
  const int n_groups = a.n_tok / kG;
  const long long total = (long long)a.B * a.H * n_groups;
  for (long long w = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; w < total;
       w += ((long long)gridDim.x * blockDim.x) >> 5) {
    const int gi = (int)(w % n_groups);
    const long long q = w / n_groups;
    const int h = (int)(q % a.H);
    const int b = (int)(q / a.H);
    const uint16_t* xp = a.x + (size_t)b * a.sb + (size_t)h * a.sh + (size_t)gi * kG * kD + 4 * lane;
    uint2 raw[kG];
#pragma unroll
    for (int j = 0; j < kG; ++j) raw[j] = __ldg(reinterpret_cast<const uint2*>(xp + (size_t)j * kD));
    float mn[4], mx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mn[i] = INFINITY;
      mx[i] = -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < kG; ++j) {
      const float v[4] = {h2f(raw[j].x & 0xFFFFu), h2f(raw[j].x >> 16), h2f(raw[j].y & 0xFFFFu), h2f(raw[j].y >> 16)};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        mn[i] = fminf(mn[i], v[i]);
        mx[i] = fmaxf(mx[i], v[i]);
      }
    }
    GroupQ g[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) g[i] = group_params(mn[i], mx[i]);
    const int tg = a.tok_begin / kG + gi;  // global token group
    const size_t sz = (((size_t)b * a.H + h) * (a.max_tokens / kG) + tg) * kD + 4 * lane;
    *reinterpret_cast<uint2*>(a.scale + sz) =
        make_uint2(g[0].s_bits | ((uint32_t)g[1].s_bits << 16), g[2].s_bits | ((uint32_t)g[3].s_bits << 16));
    *reinterpret_cast<uint2*>(a.zero + sz) =
        make_uint2(g[0].z_bits | ((uint32_t)g[1].z_bits << 16), g[2].z_bits | ((uint32_t)g[3].z_bits << 16));
    uint8_t* cp = a.codes + (((size_t)b * a.H + h) * a.max_tokens + a.tok_begin + (size_t)gi * kG) * (kD / 4) + lane;
#pragma unroll
    for (int j = 0; j < kG; ++j) {
      const float v[4] = {h2f(raw[j].x & 0xFFFFu), h2f(raw[j].x >> 16), h2f(raw[j].y & 0xFFFFu), h2f(raw[j].y >> 16)};
      uint32_t byte = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) byte |= quant_code(v[i], g[i]) << (2 * i);
      cp[(size_t)j * (kD / 4)] = (uint8_t)byte;
    }
  }
}

// values: a group is 32 channels of one token; 8 lanes per group (lane l owns channels
// 4l..4l+3), so a warp covers one 256-byte token row per step; 4 rows are loaded per step
__global__ void __launch_bounds__(256) kivi_quant_token_kernel(const KiviQuantArgs a) {
  constexpr int kRows = 4;
  const int lane = threadIdx.x & 31;
  const int gi = lane >> 3;  // channel group of this lane (32 channels = 8 lanes)
  const long long rows = (long long)a.B * a.H * a.n_tok;
  const long long n_steps = (rows + kRows - 1) / kRows;
  for (long long w = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5; w < n_steps;
       w += ((long long)gridDim.x * blockDim.x) >> 5) {
    uint2 raw[kRows];
    size_t tok[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const long long r = min(w * kRows + u, rows - 1);
      const int j = (int)(r % a.n_tok);
      const long long q = r / a.n_tok;
      const int h = (int)(q % a.H);
      const int b = (int)(q / a.H);
      raw[u] = __ldg(reinterpret_cast<const uint2*>(a.x + (size_t)b * a.sb + (size_t)h * a.sh + (size_t)j * kD + 4 * lane));
      tok[u] = ((size_t)b * a.H + h) * a.max_tokens + a.tok_begin + j;
    }
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      if (w * kRows + u >= rows) break;  // uniform across the warp
      const float v[4] = {h2f(raw[u].x & 0xFFFFu), h2f(raw[u].x >> 16), h2f(raw[u].y & 0xFFFFu), h2f(raw[u].y >> 16)};
      float mn = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
      float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
#pragma unroll
      for (int off = 4; off >= 1; off >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, off));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
      }
      const GroupQ g = group_params(mn, mx);
      if ((lane & 7) == 0) {
        a.scale[tok[u] * (kD / 32) + gi] = g.s_bits;
        a.zero[tok[u] * (kD / 32) + gi] = g.z_bits;
      }
      uint32_t byte = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) byte |= quant_code(v[i], g) << (2 * i);
      a.codes[tok[u] * (kD / 4) + lane] = (uint8_t)byte;
    }
  }
}

// ---------------------------------------------------------------- attention
constexpr int kAThreads = 256;
constexpr int kAWarps = kAThreads / 32;
constexpr int kKiviSmemLimit = 100 * 1024;
// shared layout (floats): q[128] | qf[kAWarps][128] | ored[kAWarps][128] | red[64] | flag | scores
constexpr int kOffQf = kD;
constexpr int kOffOred = kOffQf + kAWarps * kD;
constexpr int kOffRed = kOffOred + kAWarps * kD;
constexpr int kOffFlag = kOffRed + 64;
constexpr int kOffSc = kOffFlag + 4;

__global__ void __launch_bounds__(kAThreads, 2) kivi_attn_kernel(const KiviAttnArgs a, const float scale_log2) {
  extern __shared__ __align__(16) float sm[];
  float* qs = sm;
  float* qf = sm + kOffQf;
  float* ored = sm + kOffOred;
  float* red = sm + kOffRed;
  int* flag = reinterpret_cast<int*>(sm + kOffFlag);
  float* sc = sm + kOffSc;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, b = blockIdx.y, h = blockIdx.z, H = a.H;
  const int NQ = a.n_quant[b];
  const int NR = (split == 0) ? a.n_resid[b] : 0;
  const int t0 = split * a.tok_per_split;
  const int t1 = min(NQ, t0 + a.tok_per_split);
  const int nq = max(0, t1 - t0);
  const size_t bh = (size_t)b * H + h;
  if (tid < kD) qs[tid] = bf16_to_f32(a.q[bh * kD + tid]);
  __syncthreads();

  float mloc = -INFINITY;
  // ---- quantized keys: a warp per 32-token group, lane = token ------------------------
  const int G = a.group;
  for (int gl = warp; gl < nq / G; gl += kAWarps) {
    const int tg = t0 / G + gl;  // token group index
    const uint16_t* ks = a.k_scale + (bh * (a.max_tokens / G) + tg) * kD;
    const uint16_t* kz = a.k_zero + (bh * (a.max_tokens / G) + tg) * kD;
    float bias = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int ch = lane * 4 + i;
      const float qv = qs[ch] * h2f(__ldg(ks + ch));
      qf[warp * kD + ch] = qv;
      bias = fmaf(-qv, h2f(__ldg(kz + ch)), bias);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) bias += __shfl_xor_sync(0xFFFFFFFFu, bias, off);
    __syncwarp();
    const int j = tg * G + lane;
    const uint4* cr = reinterpret_cast<const uint4*>(a.k_codes + (bh * a.max_tokens + j) * (kD / 4));
    const uint4 c0 = ld_stream_u4(cr), c1 = ld_stream_u4(cr + 1);
    const uint32_t wds[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float4* qf4 = reinterpret_cast<const float4*>(qf + warp * kD);
    float acc = 0.f;
#pragma unroll
    for (int wi = 0; wi < 8; ++wi) {
#pragma unroll
      for (int bi = 0; bi < 4; ++bi) {
        const uint32_t byte = (wds[wi] >> (8 * bi)) & 0xFFu;
        const float4 qq = qf4[wi * 4 + bi];
        acc = fmaf(qq.x, (float)(byte & 3u), acc);
        acc = fmaf(qq.y, (float)((byte >> 2) & 3u), acc);
        acc = fmaf(qq.z, (float)((byte >> 4) & 3u), acc);
        acc = fmaf(qq.w, (float)(byte >> 6), acc);
      }
    }
    const float v = (acc + bias) * scale_log2;
    sc[gl * G + lane] = v;
    mloc = fmaxf(mloc, v);
    __syncwarp();
  }
  // ---- residual keys (fp16): lane = token ---------------------------------------------
  for (int r = tid; r < NR; r += kAThreads) {
    const uint4* kr = reinterpret_cast<const uint4*>(a.k_resid + (bh * a.residual + r) * kD);
    float acc = 0.f;
#pragma unroll 4
    for (int k8 = 0; k8 < kD / 8; ++k8) {
      const uint4 v = __ldg(kr + k8);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        acc = fmaf(qs[k8 * 8 + 2 * i], f.x, acc);
        acc = fmaf(qs[k8 * 8 + 2 * i + 1], f.y, acc);
      }
    }
    const float v = acc * scale_log2;
    sc[nq + r] = v;
    mloc = fmaxf(mloc, v);
  }
  // ---- softmax statistics ---------------------------------------------------------------
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xFFFFFFFFu, mloc, off));
  if (lane == 0) red[warp] = mloc;
  __syncthreads();
  float M = -INFINITY;
  for (int w = 0; w < kAWarps; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  float ls = 0.f;
  if (M != -INFINITY) {
    for (int i = tid; i < nq + NR; i += kAThreads) {
      const float e = exp2f(sc[i] - M);
      sc[i] = e;
      ls += e;
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) ls += __shfl_xor_sync(0xFFFFFFFFu, ls, off);
  if (lane == 0) red[warp] = ls;
  __syncthreads();
  float Ls = 0.f;
  for (int w = 0; w < kAWarps; ++w) Ls += red[w];

  // ---- values: warp per token (strided), lane = channels 4 lane .. 4 lane + 3 -----------
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  float oz = 0.f;
  const int gch = (lane * 4) / G;  // value channel group of this lane
  const int ngv = kD / G;
  for (int jl = warp; jl < nq; jl += kAWarps) {
    const size_t j = bh * a.max_tokens + t0 + jl;
    const float p = sc[jl];
    const float wgt = p * h2f(__ldg(a.v_scale + j * ngv + gch));
    const uint32_t byte = __ldg(a.v_codes + j * (kD / 4) + lane);
    o[0] = fmaf(wgt, (float)(byte & 3u), o[0]);
    o[1] = fmaf(wgt, (float)((byte >> 2) & 3u), o[1]);
    o[2] = fmaf(wgt, (float)((byte >> 4) & 3u), o[2]);
    o[3] = fmaf(wgt, (float)(byte >> 6), o[3]);
    oz = fmaf(wgt, h2f(__ldg(a.v_zero + j * ngv + gch)), oz);
  }
  for (int r = warp; r < NR; r += kAWarps) {
    const float p = sc[nq + r];
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(a.v_resid + (bh * a.residual + r) * kD + lane * 4));
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
    o[0] = fmaf(p, f0.x, o[0]);
    o[1] = fmaf(p, f0.y, o[1]);
    o[2] = fmaf(p, f1.x, o[2]);
    o[3] = fmaf(p, f1.y, o[3]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) ored[warp * kD + lane * 4 + i] = o[i] - oz;
  __syncthreads();
  float ov = 0.f;
  if (tid < kD) {
    for (int w = 0; w < kAWarps; ++w) ov += ored[w * kD + tid];
  }

  if (a.n_split == 1) {
    if (tid < kD) {
      const float val = (Ls > 0.f) ? ov / Ls : 0.f;
      if (a.out_fp32) reinterpret_cast<float*>(a.out)[bh * kD + tid] = val;
      else reinterpret_cast<uint16_t*>(a.out)[bh * kD + tid] = f32_to_bf16(val);
    }
    return;
  }
  float* pp = a.part + (bh * a.n_split + split) * (kD + 2);
  if (tid < kD) pp[2 + tid] = ov;
  if (tid == 0) {
    pp[0] = M;
    pp[1] = Ls;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) *flag = (atomicAdd(&a.counters[bh], 1) == a.n_split - 1);
  __syncthreads();
  if (!*flag) return;
  __threadfence();
  if (tid < kD) {
    const float* base = a.part + bh * a.n_split * (kD + 2);
    float Mx = -INFINITY;
    for (int s = 0; s < a.n_split; ++s) Mx = fmaxf(Mx, __ldcg(base + s * (kD + 2)));
    float Lt = 0.f, acc = 0.f;
    if (Mx != -INFINITY) {
      for (int s = 0; s < a.n_split; ++s) {
        const float ms = __ldcg(base + s * (kD + 2));
        if (ms == -INFINITY) continue;
        const float w = exp2f(ms - Mx);
        Lt = fmaf(w, __ldcg(base + s * (kD + 2) + 1), Lt);
        acc = fmaf(w, __ldcg(base + s * (kD + 2) + 2 + tid), acc);
      }
    }
    const float val = (Lt > 0.f) ? acc / Lt : 0.f;
    if (a.out_fp32) reinterpret_cast<float*>(a.out)[bh * kD + tid] = val;
    else reinterpret_cast<uint16_t*>(a.out)[bh * kD + tid] = f32_to_bf16(val);
  }
  if (tid == 0) a.counters[bh] = 0;
}

}  // namespace

int kivi_attn_max_tok_per_split(int residual) {
  return (kKiviSmemLimit / 4 - kOffSc) - residual;
}

size_t kivi_attn_smem_bytes(int tok_per_split, int residual) {
  return (size_t)(kOffSc + tok_per_split + residual) * 4;
}

cudaError_t launch_kivi_quantize(const KiviQuantArgs& a, cudaStream_t s) {
  // grid-stride warps; 8 blocks of 256 threads per SM keep enough rows in flight
  const long long warps = (a.axis == KVQ_PER_CHANNEL) ? (long long)a.B * a.H * (a.n_tok / a.group)
                                                      : ((long long)a.B * a.H * a.n_tok + 3) / 4;
  if (warps <= 0) return cudaSuccess;
  long long blocks = (warps + 7) / 8;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (blocks > (long long)sms * 8) blocks = (long long)sms * 8;
  if (a.axis == KVQ_PER_CHANNEL) kivi_quant_channel_kernel<<<(int)blocks, 256, 0, s>>>(a);
  else kivi_quant_token_kernel<<<(int)blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_kivi_attn(const KiviAttnArgs& a, cudaStream_t st) {
  const size_t smem = kivi_attn_smem_bytes(a.tok_per_split, a.residual);
  cudaError_t e = cudaFuncSetAttribute(kivi_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)kD);
  dim3 grid(a.n_split, a.B, a.H);
  kivi_attn_kernel<<<grid, kAThreads, smem, st>>>(a, scale_log2);
  return cudaGetLastError();
}

}  // namespace kvq
