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
// One block per (split, request, head); splits 0 .. n_split-1 take equal token ranges of the
// quantized segment, the last block the fp16 residual segment. A quantized split streams its
// tokens through a 4-stage shared-memory ring of 128-token chunks (TMA bulk copies of the
// chunk's key codes, key scales and zeros, value codes, value scales and zeros: 12 KB), with a
// block-wide online softmax across chunks. Partials of all splits merge exactly in the last
// block of a (request, head) to finish (arrival counter, no spin-wait).
constexpr int kAThreads = 256;
constexpr int kAWarps = kAThreads / 32;
constexpr int kAChunk = 128;                      // tokens per ring stage (4 key groups of 32)
constexpr int kAStages = 4;
constexpr int kCKc = 0;                           // stage layout (bytes)
constexpr int kCKs = kCKc + kAChunk * 32;         // key scales [4 groups][128] fp16
constexpr int kCKz = kCKs + 4 * kD * 2;
constexpr int kCVc = kCKz + 4 * kD * 2;
constexpr int kCVs = kCVc + kAChunk * 32;         // value scales [128 tokens][4 groups] fp16
constexpr int kCVz = kCVs + kAChunk * 4 * 2;
constexpr int kAStageBytes = kCVz + kAChunk * 4 * 2;  // 12 KB
// shared layout (bytes)
constexpr int kAOffRing = 0;
constexpr int kAOffQ = kAOffRing + kAStages * kAStageBytes;  // float q[128]
constexpr int kAOffQf = kAOffQ + kD * 4;                      // float q' [4 groups][128]
constexpr int kAOffBias = kAOffQf + 4 * kD * 4;               // float [4 groups][2 halves]
constexpr int kAOffRed = kAOffBias + 32;                      // float [8 warps] + flag
constexpr int kAOffBar = kAOffRed + 64;                       // mbarriers [4] + failed
constexpr int kAOffSc = kAOffBar + 64;                        // float scores [max(128, residual)]
static_assert(kAStageBytes % 128 == 0 && kAOffBar % 8 == 0, "alignment");

// Codes j and j + 8 (j < 8) of a 16-code word, each as (code * 4^j) in fp32: the code is
// masked in place (bits 2j, 2j+1 of each half word), placed in the mantissa of 2^23 and 2^23
// is subtracted, all exact. One integer op per code and one packed add per pair instead of
// shift + int-to-float conversion; the 4^-j scale is folded into the other operand.
__device__ __forceinline__ float2 code_pair(uint32_t w, uint32_t w_hi, int j) {
  const uint32_t m = 3u << (2 * j);
  const float2 f = make_float2(__uint_as_float((w & m) | 0x4B000000u), __uint_as_float((w_hi & m) | 0x4B000000u));
  return __fadd2_rn(f, make_float2(-8388608.f, -8388608.f));
}
__device__ __forceinline__ float pow4_neg(int j) { return __uint_as_float((uint32_t)(127 - 2 * j) << 23); }

__device__ __forceinline__ bool kivi_wait(uint64_t* bar, uint32_t parity, volatile int* failed, int* err) {
  if (*failed) return false;
  if (mbar_wait_bounded(bar, parity)) return true;
  *failed = 1;
  set_error(err, KVQ_ERR_TIMEOUT);
  return false;
}

__global__ void __launch_bounds__(kAThreads) kivi_attn_kernel(const KiviAttnArgs a, const float scale_log2) {
  extern __shared__ __align__(128) unsigned char sma[];
  float* qs = reinterpret_cast<float*>(sma + kAOffQ);
  float* qf = reinterpret_cast<float*>(sma + kAOffQf);
  float* bias = reinterpret_cast<float*>(sma + kAOffBias);
  float* red = reinterpret_cast<float*>(sma + kAOffRed);
  int* flag = reinterpret_cast<int*>(sma + kAOffRed + 8 * 4);
  uint64_t* full = reinterpret_cast<uint64_t*>(sma + kAOffBar);
  volatile int* failed = reinterpret_cast<volatile int*>(sma + kAOffBar + kAStages * 8);
  float* sc = reinterpret_cast<float*>(sma + kAOffSc);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, b = blockIdx.y, h = blockIdx.z, H = a.H;
  const int n_total = gridDim.x;                 // quantized splits + the residual block
  const bool resid_block = (a.residual > 0) && (split == n_total - 1);
  const size_t bh = (size_t)b * H + h;
  const int NQ = min(a.n_quant[b], a.max_tokens) / a.group * a.group;
  if (tid < kD) qs[tid] = bf16_to_f32(a.q[bh * kD + tid]);
  if (tid == 0) {
    for (int s = 0; s < kAStages; ++s) mbar_init(&full[s], 1);
    *failed = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // running softmax state; the max is block-wide
  // quantized blocks: lane holds channels 16 (lane % 8) .. + 15 of its token slot (lane / 8);
  // the residual block: channels 4 lane .. 4 lane + 3 in o[0..3]
  float M = -INFINITY, l = 0.f, oz = 0.f;
  float o[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i] = 0.f;
  auto rescale_to = [&](float Mn) {
    const float f = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i] *= f;
    oz *= f;
    l *= f;
    M = Mn;
  };
  // block max of sc[0, n) (every warp computes it)
  auto scores_max = [&](int n) {
    float m = -INFINITY;
    for (int i = lane; i < n; i += 32) m = fmaxf(m, sc[i]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    return m;
  };

  if (!resid_block) {
    // ================================ quantized tokens ======================================
    const int t0 = split * a.tok_per_split;
    const int t1 = min(NQ, t0 + a.tok_per_split);
    const int n_tok = max(0, t1 - t0);
    const int n_chunks = (n_tok + kAChunk - 1) / kAChunk;
    const size_t tok0 = bh * a.max_tokens;         // token row base of (b, h)
    const size_t grp0 = bh * (a.max_tokens / 32);  // key group row base of (b, h)
    auto produce = [&](int c) {                    // thread 0
      const int st = c % kAStages;
      unsigned char* dst = sma + kAOffRing + st * kAStageBytes;
      const int t = t0 + c * kAChunk;
      const int n = min(kAChunk, t1 - t), ng = n / 32;
      mbar_arrive_expect_tx(&full[st], (uint32_t)(n * 32 * 2 + ng * kD * 2 * 2 + n * 8 * 2));
      bulk_g2s(dst + kCKc, a.k_codes + (tok0 + t) * 32, n * 32, &full[st]);
      bulk_g2s(dst + kCVc, a.v_codes + (tok0 + t) * 32, n * 32, &full[st]);
      bulk_g2s(dst + kCKs, a.k_scale + (grp0 + t / 32) * kD, ng * kD * 2, &full[st]);
      bulk_g2s(dst + kCKz, a.k_zero + (grp0 + t / 32) * kD, ng * kD * 2, &full[st]);
      bulk_g2s(dst + kCVs, a.v_scale + (tok0 + t) * 4, n * 8, &full[st]);
      bulk_g2s(dst + kCVz, a.v_zero + (tok0 + t) * 4, n * 8, &full[st]);
    };
    int issued = 0;  // thread 0
    if (tid == 0)
      for (int c = 0; c < min(kAStages, n_chunks); ++c) {
        produce(c);
        ++issued;
      }

    for (int c = 0; c < n_chunks; ++c) {
      const int st = c % kAStages;
      kivi_wait(&full[st], (c / kAStages) & 1, failed, a.err);
      const unsigned char* stage = sma + kAOffRing + st * kAStageBytes;
      const int n = min(kAChunk, t1 - (t0 + c * kAChunk)), ng = n / 32;
      // ---- q' = q s per key group (the scale folds into the query) and bias = -sum q' z ----
      {
        const int g = warp >> 1, hf = warp & 1;
        if (g < ng) {
          const int ch = 64 * hf + 2 * lane;
          const uint32_t s2 = *reinterpret_cast<const uint32_t*>(stage + kCKs + (g * kD + ch) * 2);
          const uint32_t z2 = *reinterpret_cast<const uint32_t*>(stage + kCKz + (g * kD + ch) * 2);
          const float qa = qs[ch] * h2f(s2 & 0xFFFFu), qb = qs[ch + 1] * h2f(s2 >> 16);
          // pair layout: [group][half][word m][j] = (channel 16m + j, channel 16m + 8 + j) of the
          // half, scaled by 4^-j to match code_pair
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = ch + e, k = c & 15, j = k & 7;
            qf[g * kD + 64 * hf + 2 * (8 * ((c & 63) >> 4) + j) + (k >> 3)] = (e ? qb : qa) * pow4_neg(j);
          }
          float pb = -(qa * h2f(z2 & 0xFFFFu) + qb * h2f(z2 >> 16));
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) pb += __shfl_xor_sync(0xFFFFFFFFu, pb, off);
          if (lane == 0) bias[g * 2 + hf] = pb;
        }
      }
      __syncthreads();
      // ---- scores: warp (group, 16 tokens), lanes 0-15 channels 0-63, lanes 16-31 64-127 ----
      {
        const int g = warp >> 1;
        if (g < ng) {
          const int tk = 32 * g + 16 * (warp & 1) + (lane & 15), chh = lane >> 4;
          const uint4 cw = *reinterpret_cast<const uint4*>(stage + kCKc + tk * 32 + 16 * chh);
          const uint32_t wds[4] = {cw.x, cw.y, cw.z, cw.w};
          const float2* q2 = reinterpret_cast<const float2*>(qf + g * kD + 64 * chh);
          float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t w_hi = wds[k] >> 16;
#pragma unroll
            for (int j = 0; j < 8; ++j) acc2 = __ffma2_rn(q2[8 * k + j], code_pair(wds[k], w_hi, j), acc2);
          }
          float acc = acc2.x + acc2.y;
          acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 16);
          if (chh == 0) sc[tk] = (acc + bias[g * 2] + bias[g * 2 + 1]) * scale_log2;
        }
      }
      __syncthreads();
      // ---- online softmax, then values: warp w takes tokens 16w .. 16w + 15, four at a time;
      //      lane: token 4 step + lane / 8, code word lane % 8 (channels 16 (lane % 8) .. + 15,
      //      value group (lane % 8) / 2) ----
      const float Mn = fmaxf(M, scores_max(n));
      if (Mn > M) rescale_to(Mn);
      {
        const int tb = 16 * warp;
        const float pk = (tb + (lane & 15) < n) ? exp2f(sc[tb + (lane & 15)] - M) : 0.f;
        float ls = (lane < 16) ? pk : 0.f;
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) ls += __shfl_xor_sync(0xFFFFFFFFu, ls, off);
        l += __shfl_sync(0xFFFFFFFFu, ls, 0);
        const int lw = lane & 7, ts = lane >> 3, gv = lw >> 1;
#pragma unroll
        for (int step = 0; step < 4; ++step) {
          const float p = __shfl_sync(0xFFFFFFFFu, pk, 4 * step + ts);
          const int tk = tb + 4 * step + ts;
          if (tk < n) {
            const uint32_t wv = *reinterpret_cast<const uint32_t*>(stage + kCVc + tk * 32 + 4 * lw);
            const float wgt = p * h2f(*reinterpret_cast<const uint16_t*>(stage + kCVs + (tk * 4 + gv) * 2));
            oz = fmaf(wgt, h2f(*reinterpret_cast<const uint16_t*>(stage + kCVz + (tk * 4 + gv) * 2)), oz);
            const uint32_t wv_hi = wv >> 16;
            const float2 w2 = make_float2(wgt, wgt);
#pragma unroll
            for (int j = 0; j < 8; ++j) {  // o2[j] = (channel j, channel 8 + j) of the word, x 4^j
              const float2 acc = __ffma2_rn(w2, code_pair(wv, wv_hi, j), make_float2(o[2 * j], o[2 * j + 1]));
              o[2 * j] = acc.x;
              o[2 * j + 1] = acc.y;
            }
          }
        }
      }
      __syncthreads();  // every thread is done with this stage
      if (tid == 0 && c + kAStages < n_chunks && !*failed) {
        produce(c + kAStages);
        ++issued;
      }
    }
    // after a timed-out wait, let this block's copies still in flight land first
    if (tid == 0 && *failed)
      for (int c = max(0, issued - kAStages); c < issued; ++c) mbar_wait_bounded(&full[c % kAStages], (c / kAStages) & 1);
  } else {
    // ================================ fp16 residual tokens ==================================
    const int NR = min(a.n_resid[b], a.residual);
    for (int r = tid; r < NR; r += kAThreads) {  // keys: a thread per token
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
      sc[r] = acc * scale_log2;
    }
    __syncthreads();
    rescale_to(scores_max(NR));
    for (int r = warp; r < NR; r += kAWarps) {  // values: a warp per token, lane 4 channels
      const float p = exp2f(sc[r] - M);
      l += p;
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(a.v_resid + (bh * a.residual + r) * kD + lane * 4));
      const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
      const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
      o[0] = fmaf(p, f0.x, o[0]);
      o[1] = fmaf(p, f0.y, o[1]);
      o[2] = fmaf(p, f1.x, o[2]);
      o[3] = fmaf(p, f1.y, o[3]);
    }
  }

  // ---- warps -> block: sum o - oz and l over the warps (one max for the block) -----------
  __syncthreads();  // the ring is idle
  float* ored = reinterpret_cast<float*>(sma + kAOffRing);  // [warp][128]
  if (!resid_block) {  // the four token slots of a code word meet, then 8 lanes hold 128 channels
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i] += __shfl_xor_sync(0xFFFFFFFFu, o[i], 8);
      o[i] += __shfl_xor_sync(0xFFFFFFFFu, o[i], 16);
    }
    oz += __shfl_xor_sync(0xFFFFFFFFu, oz, 8);
    oz += __shfl_xor_sync(0xFFFFFFFFu, oz, 16);
    if (lane < 8) {  // o[2j] is channel j of the word, o[2j + 1] channel 8 + j, both x 4^j
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        ored[warp * kD + 16 * lane + j] = o[2 * j] * pow4_neg(j) - oz;
        ored[warp * kD + 16 * lane + 8 + j] = o[2 * j + 1] * pow4_neg(j) - oz;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) ored[warp * kD + lane * 4 + i] = o[i];
  }
  if (lane == 0) red[warp] = l;
  __syncthreads();
  if (*failed) return;  // uniform after the barrier
  float ov = 0.f, Ls = 0.f;
  if (tid < kD) {
    for (int w = 0; w < kAWarps; ++w) {
      ov += ored[w * kD + tid];
      Ls += red[w];
    }
  }

  if (n_total == 1) {
    if (tid < kD) {
      const float val = (Ls > 0.f) ? ov / Ls : 0.f;
      if (a.out_fp32) reinterpret_cast<float*>(a.out)[bh * kD + tid] = val;
      else reinterpret_cast<uint16_t*>(a.out)[bh * kD + tid] = f32_to_bf16(val);
    }
    return;
  }
  float* pp = a.part + (bh * n_total + split) * (kD + 2);
  if (tid < kD) pp[2 + tid] = ov;
  if (tid == 0) {
    pp[0] = M;
    pp[1] = Ls;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) *flag = (atomicAdd(&a.counters[bh], 1) == n_total - 1);
  __syncthreads();
  if (!*flag) return;
  __threadfence();
  if (tid < kD) {
    const float* base = a.part + bh * n_total * (kD + 2);
    float Mx = -INFINITY;
    for (int s = 0; s < n_total; ++s) Mx = fmaxf(Mx, __ldcg(base + s * (kD + 2)));
    float Lt = 0.f, acc = 0.f;
    if (Mx != -INFINITY) {
      for (int s = 0; s < n_total; ++s) {
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

int kivi_attn_max_tok_per_split(int) { return 1 << 30; }  // tokens stream through the ring

size_t kivi_attn_smem_bytes(int, int residual) { return (size_t)kAOffSc + 4 * (size_t)max(kAChunk, residual); }

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
  // quantized splits, plus one block for the fp16 residual segment
  dim3 grid(a.n_split + (a.residual > 0 ? 1 : 0), a.B, a.H);
  kivi_attn_kernel<<<grid, kAThreads, smem, st>>>(a, scale_log2);
  return cudaGetLastError();
}

}  // namespace kvq
