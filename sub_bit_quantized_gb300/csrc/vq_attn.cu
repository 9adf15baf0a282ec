// LoopVQ decode attention over the bf16 window and the 8-token index pages of one
// (layer, loop step), split-K over pages with an exact logsumexp merge.
//
// Follows "LoopVQ: Sub 1-bit KV Cache Quantization for Looped Transformers", method
// step 5, Algorithm 1 and Figure 5: the step's codebook slice B_t is staged in shared
// memory once per thread block, keys are rebuilt from D/c = 16 indices per token, rotated
// by RoPE and dotted with the query; the bf16 sink/recent tokens are attended directly and
// the partials of every split are merged exactly. Two requests of the same head share a
// thread block and its B_t load.
//
// GB300 design (differs from the page's Triton kernel):
//  * B_t is copied into shared memory with TMA bulk copies (one mbarrier, bounded wait).
//  * Keys: 8 lanes per 8-token page, lane s owns the RoPE partner groups s and s+8. Its
//    rotated-query slice u = R(p_q - p) q is built once per page from the cos/sin table and
//    advanced one position per token by a fixed rotation (exact within a few ulp over the
//    7 steps), so no cos/sin load per token. Codeword rows are read with 128-bit shared
//    loads in a lane-dependent half order that makes the 8 lanes of a phase hit 8
//    distinct bank quads. Per-token partial dot products are combined by a transposing
//    shuffle reduction (7 shuffles per 8 tokens).
//  * Values: scores are kept in shared memory (two-pass softmax), and instead of rebuilding
//    every value vector the kernel accumulates the softmax weight of each codeword per
//    group (w[g][r] += p_j) and forms o_g = sum_r w[g][r] * B_t,V[g][r] once per split.
//    This is the same sum re-associated. The histogram is laid out [codeword][request*16
//    + group] so the 32 lanes of a warp (2 requests x 16 groups) hit 32 distinct banks.
//  * The last thread block of a (request pair, head) to finish merges the split partials
//    (arrival counter, no spin-wait) and resets the counter for the next call.
#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "../../include/kvq.h"

namespace kvq {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kLaneGroups = kThreads / 8;
constexpr uint32_t kSliceBytes = kCB * kD * 4;  // 128 KB fp32 B_t slice

// shared-memory layout (bytes)
constexpr int kOffCb = 0;
constexpr int kOffHist = kOffCb + kSliceBytes;         // float [256][32]
constexpr int kOffQ = kOffHist + kCB * 32 * 4;         // float [2][128]
constexpr int kOffOw = kOffQ + 2 * kD * 4;             // float [2][128] bf16-window V sums
constexpr int kOffComb = kOffOw + 2 * kD * 4;          // float [2][128]
constexpr int kOffRed = kOffComb + 2 * kD * 4;         // float [2][kWarps] + [4]
constexpr int kOffBar = kOffRed + 256;                 // uint64 mbarrier, int flag
constexpr int kOffScores = kOffBar + 64;               // float [2][sc_stride]
constexpr int kSmemLimit = 232448;                     // 227 KB opt-in per block

__device__ __forceinline__ void load8_perm(const float* p, int o0, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p + o0);
  const float4 b = *reinterpret_cast<const float4*>(p + (4 - o0));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void ldg8_perm(const float* p, int o0, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p + o0));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p + (4 - o0)));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void ldg8_bf16_perm(const uint16_t* p, int o0, float (&v)[8]) {
  const uint2 a = __ldg(reinterpret_cast<const uint2*>(p + o0));
  const uint2 b = __ldg(reinterpret_cast<const uint2*>(p + (4 - o0)));
  v[0] = bf16_lo(a.x); v[1] = bf16_hi(a.x); v[2] = bf16_lo(a.y); v[3] = bf16_hi(a.y);
  v[4] = bf16_lo(b.x); v[5] = bf16_hi(b.x); v[6] = bf16_lo(b.y); v[7] = bf16_hi(b.y);
}

__device__ __forceinline__ void transpose_reduce8(float (&p)[8], int s, unsigned mask) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const bool up = (s & 4) != 0;
    const float send = up ? p[k] : p[k + 4];
    const float keep = up ? p[k + 4] : p[k];
    p[k] = keep + __shfl_xor_sync(mask, send, 4);
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const bool up = (s & 2) != 0;
    const float send = up ? p[k] : p[k + 2];
    const float keep = up ? p[k + 2] : p[k];
    p[k] = keep + __shfl_xor_sync(mask, send, 2);
  }
  {
    const bool up = (s & 1) != 0;
    const float send = up ? p[0] : p[1];
    const float keep = up ? p[1] : p[0];
    p[0] = keep + __shfl_xor_sync(mask, send, 1);
  }
}

__global__ void __launch_bounds__(kThreads, 1) vq_attn_kernel(const VqAttnArgs a, const float scale_log2,
                                                                const int sc_stride) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* cbs = reinterpret_cast<float*>(smem + kOffCb);
  float* hist = reinterpret_cast<float*>(smem + kOffHist);
  float* qs = reinterpret_cast<float*>(smem + kOffQ);
  float* ow = reinterpret_cast<float*>(smem + kOffOw);
  float* comb = reinterpret_cast<float*>(smem + kOffComb);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  int* flag = reinterpret_cast<int*>(smem + kOffBar + 8);
  float* sc = reinterpret_cast<float*>(smem + kOffScores);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, pair = blockIdx.y, h = blockIdx.z;
  const int H = a.H;
  const int b0 = pair * 2;
  const int nreq = min(2, a.B - b0);

  // ---- lengths of the two requests; pages of this split -------------------------------
  int L[2], NP[2], pend[2], nq[2], nsink[2], nwin[2];
  const int pg0 = split * a.pages_per_split;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (r < nreq) {
      L[r] = a.seq_len[b0 + r];
      NP[r] = a.n_pages[b0 + r];
      // lengths that do not describe a valid cache are reported and attended as empty
      const bool bad = L[r] < 0 || L[r] > a.max_ctx || NP[r] < 0 || NP[r] > a.max_pages ||
                       (NP[r] > 0 && a.sink + kPage * NP[r] > L[r]) ||
                       L[r] - a.sink - kPage * NP[r] > a.recent + kPage;
      if (bad) {
        if (split == 0 && threadIdx.x == 0) set_error(a.err, KVQ_ERR_CAPACITY);
        L[r] = 0;
        NP[r] = 0;
      }
    } else {
      L[r] = 0;
      NP[r] = 0;
    }
    pend[r] = min(NP[r], pg0 + a.pages_per_split);
    nq[r] = max(0, pend[r] - pg0) * kPage;
    nsink[r] = min(a.sink, L[r]);
    nwin[r] = (split == 0 && L[r] > 0) ? (nsink[r] + max(0, L[r] - a.sink - kPage * NP[r])) : 0;
  }
  const int n_items = max(nq[0], nq[1]) / kPage;  // pages processed by this block

  // ---- stage the key slice B_t (TMA bulk) and set up ----------------------------------
  const float* btk = a.bt_k + (size_t)h * kCB * kD;
  const float* btv = a.bt_v + (size_t)h * kCB * kD;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0 && n_items > 0) {
    mbar_arrive_expect_tx(bar, kSliceBytes);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      bulk_g2s(cbs + k * (kSliceBytes / 16), btk + k * (kSliceBytes / 16), kSliceBytes / 4, bar);
  }
  for (int i = tid; i < kCB * 32 / 4; i += kThreads)
    reinterpret_cast<float4*>(hist)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid < 2 * kD) {
    const int r = tid >> 7;
    const uint16_t* qp = a.q + ((size_t)(b0 + min(r, nreq - 1)) * H + h) * kD;
    qs[tid] = bf16_to_f32(qp[tid & 127]);
    ow[tid] = 0.f;
  }
  __syncthreads();

  const int s = tid & 7;                 // slot: groups s and s + 8
  const int o0 = (s & 4) ? 4 : 0;        // half order (bank-quad spreading)
  const unsigned gmask = 0xFFu << (lane & 24);

  float qlo[2][8], qhi[2][8];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    load8_perm(qs + r * kD + 8 * s, o0, qlo[r]);
    load8_perm(qs + r * kD + 64 + 8 * s, o0, qhi[r]);
  }
  float cth[8], sth[8];  // cos/sin(theta_i) of this lane's 8 frequencies (table row 1)
  ldg8_perm(a.rope_cos + (kD / 2) + 8 * s, o0, cth);
  ldg8_perm(a.rope_sin + (kD / 2) + 8 * s, o0, sth);

  float mloc[2] = {-INFINITY, -INFINITY};

  // ---- bf16 window scores (split 0 only) ------------------------------------------------
  const int lg = tid >> 3;
  for (int wi = lg; wi < nwin[0] + nwin[1]; wi += kLaneGroups) {
    const bool r1 = wi >= nwin[0];
    const int r = r1 ? 1 : 0;
    const int w = r1 ? wi - nwin[0] : wi;
    const int ns = r1 ? nsink[1] : nsink[0];
    const int np = r1 ? NP[1] : NP[0];
    const int Lr = r1 ? L[1] : L[0];
    const int nqr = r1 ? nq[1] : nq[0];
    const int p = (w < ns) ? w : a.sink + kPage * np + (w - ns);
    const int slot = (p < a.sink) ? p : a.sink + (p - a.sink) % (a.recent + kPage);
    const uint16_t* kr = a.win_k + (((size_t)(b0 + r) * H + h) * a.win_slots + slot) * kD;
    float klo[8], khi[8], c[8], sn[8];
    ldg8_bf16_perm(kr + 8 * s, o0, klo);
    ldg8_bf16_perm(kr + 64 + 8 * s, o0, khi);
    const int dl = Lr - 1 - p;
    ldg8_perm(a.rope_cos + (size_t)dl * (kD / 2) + 8 * s, o0, c);
    ldg8_perm(a.rope_sin + (size_t)dl * (kD / 2) + 8 * s, o0, sn);
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float ql = r1 ? qlo[1][k] : qlo[0][k];
      const float qh = r1 ? qhi[1][k] : qhi[0][k];
      const float ul = ql * c[k] - qh * sn[k];
      const float uh = qh * c[k] + ql * sn[k];
      acc = fmaf(ul, klo[k], acc);
      acc = fmaf(uh, khi[k], acc);
    }
    acc += __shfl_xor_sync(gmask, acc, 4);
    acc += __shfl_xor_sync(gmask, acc, 2);
    acc += __shfl_xor_sync(gmask, acc, 1);
    if (s == 0) {
      const float v = acc * scale_log2;
      sc[r * sc_stride + nqr + w] = v;
      if (r1) mloc[1] = fmaxf(mloc[1], v);
      else mloc[0] = fmaxf(mloc[0], v);
    }
  }

  // ---- wait for B_t(K) ----------------------------------------------------------------
  bool failed = false;
  if (n_items > 0) failed = !mbar_wait_bounded(bar, 0);
  if (__syncthreads_or(failed)) {
    if (tid == 0) set_error(a.err, KVQ_ERR_TIMEOUT);
    mbar_wait_bounded(bar, 0);  // let an in-flight copy land before the block exits
    return;
  }

  // ---- quantized key scores -------------------------------------------------------------
  const uint8_t* ik[2];
#pragma unroll
  for (int r = 0; r < 2; ++r)
    ik[r] = a.idx_k + ((size_t)(b0 + min(r, nreq - 1)) * H + h) * (size_t)a.max_pages * kPageBytes;

  for (int pi = lg; pi < n_items; pi += kLaneGroups) {
    const int pg = pg0 + pi;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (pg >= pend[r]) continue;  // uniform within the 8-lane group
      const uint4 row = ld_stream_u4(ik[r] + (size_t)pg * kPageBytes + 16 * s);
      const int d0 = L[r] - 1 - (a.sink + kPage * pg);
      float c[8], sn[8];
      ldg8_perm(a.rope_cos + (size_t)d0 * (kD / 2) + 8 * s, o0, c);
      ldg8_perm(a.rope_sin + (size_t)d0 * (kD / 2) + 8 * s, o0, sn);
      float ul[8], uh[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        ul[k] = qlo[r][k] * c[k] - qhi[r][k] * sn[k];
        uh[k] = qhi[r][k] * c[k] + qlo[r][k] * sn[k];
      }
      float part[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t wd = (j < 2) ? row.x : (j < 4) ? row.y : (j < 6) ? row.z : row.w;
        const uint32_t sh = (j & 1) * 16;
        const uint32_t rlo = (wd >> sh) & 0xFFu;
        const uint32_t rhi = (wd >> (sh + 8)) & 0xFFu;
        float klo[8], khi[8];
        load8_perm(cbs + rlo * kD + 8 * s, o0, klo);
        load8_perm(cbs + rhi * kD + 64 + 8 * s, o0, khi);
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          acc0 = fmaf(ul[k], klo[k], acc0);
          acc1 = fmaf(uh[k], khi[k], acc1);
        }
        part[j] = acc0 + acc1;
        if (j < 7) {  // next token is one position later: u <- R(-1) u
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float t0 = fmaf(ul[k], cth[k], uh[k] * sth[k]);
            uh[k] = fmaf(uh[k], cth[k], -(ul[k] * sth[k]));
            ul[k] = t0;
          }
        }
      }
      // transposing reduction: lane s ends with the full score of token s
      transpose_reduce8(part, s, gmask);
      const float v = part[0] * scale_log2;
      sc[r * sc_stride + pi * kPage + s] = v;
      mloc[r] = fmaxf(mloc[r], v);
    }
  }

  // ---- B_t(K) no longer read: start loading B_t(V) into the same buffer -----------------
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0 && n_items > 0) {
    mbar_arrive_expect_tx(bar, kSliceBytes);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      bulk_g2s(cbs + k * (kSliceBytes / 16), btv + k * (kSliceBytes / 16), kSliceBytes / 4, bar);
  }

  // ---- softmax statistics per request ---------------------------------------------------
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float m = mloc[r];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    if (lane == 0) red[r * kWarps + warp] = m;
  }
  __syncthreads();
  float M[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float m = -INFINITY;
    for (int w = 0; w < kWarps; ++w) m = fmaxf(m, red[r * kWarps + w]);
    M[r] = m;
  }
  __syncthreads();  // red is reused below
  float lsum[2] = {0.f, 0.f};
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int n = nq[r] + nwin[r];
    if (M[r] == -INFINITY) continue;
    for (int i = tid; i < n; i += kThreads) {
      const float e = exp2f(sc[r * sc_stride + i] - M[r]);
      sc[r * sc_stride + i] = e;
      lsum[r] += e;
    }
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float v = lsum[r];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    if (lane == 0) red[r * kWarps + warp] = v;
  }
  __syncthreads();  // weights in sc are final
  float Ls[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float v = 0.f;
    for (int w = 0; w < kWarps; ++w) v += red[r * kWarps + w];
    Ls[r] = v;
  }

  // ---- value histogram over the quantized tokens --------------------------------------
  {
    const int r = lane >> 4, g = lane & 15;
    const int sl = g & 7, hb = (g >> 3) * 8;
    const uint8_t* iv = a.idx_v + ((size_t)(b0 + min(r, nreq - 1)) * H + h) * (size_t)a.max_pages * kPageBytes;
    for (int pi = warp; pi < n_items; pi += kWarps) {
      const int pg = pg0 + pi;
      if (pg < (r ? pend[1] : pend[0])) {
        const uint4 row = ld_stream_u4(iv + (size_t)pg * kPageBytes + 16 * sl);
        const float* pw = sc + r * sc_stride + pi * kPage;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t wd = (j < 2) ? row.x : (j < 4) ? row.y : (j < 6) ? row.z : row.w;
          const uint32_t bin = (wd >> ((j & 1) * 16 + hb)) & 0xFFu;
          atomicAdd(&hist[bin * 32 + lane], pw[j]);
        }
      }
    }
  }
  // ---- bf16 window values (direct) ------------------------------------------------------
  if (tid < 2 * kD) {
    const bool r1 = (tid >> 7) != 0;
    const int r = r1 ? 1 : 0, ch = tid & 127;
    const int nw = r1 ? nwin[1] : nwin[0];
    const int ns = r1 ? nsink[1] : nsink[0];
    const int np = r1 ? NP[1] : NP[0];
    const int nqr = r1 ? nq[1] : nq[0];
    float acc = 0.f;
    for (int w = 0; w < nw; ++w) {
      const int p = (w < ns) ? w : a.sink + kPage * np + (w - ns);
      const int slot = (p < a.sink) ? p : a.sink + (p - a.sink) % (a.recent + kPage);
      const uint16_t* vr = a.win_v + (((size_t)(b0 + r) * H + h) * a.win_slots + slot) * kD;
      acc = fmaf(sc[r * sc_stride + nqr + w], bf16_to_f32(__ldg(vr + ch)), acc);
    }
    ow[tid] = acc;
  }

  // ---- wait for B_t(V), then o_g = sum_r w[g][r] * B_t,V[g][r] ------------------------
  failed = false;
  if (n_items > 0) failed = !mbar_wait_bounded(bar, 1);
  if (__syncthreads_or(failed)) {
    if (tid == 0) set_error(a.err, KVQ_ERR_TIMEOUT);
    mbar_wait_bounded(bar, 1);
    return;
  }
  float o = 0.f;
  const int rr = (tid >> 7) & 1, ch = tid & 127, half = tid >> 8;
  if (n_items > 0) {
    const int col = rr * 16 + (ch >> 3);
    const int b_lo = half * 128;
#pragma unroll 8
    for (int bin = b_lo; bin < b_lo + 128; ++bin) o = fmaf(hist[bin * 32 + col], cbs[bin * kD + ch], o);
  }
  if (half) comb[rr * kD + ch] = o;
  __syncthreads();

  if (a.n_split == 1) {
    if (!half && rr < nreq) {
      const int b = b0 + rr;
      o += comb[rr * kD + ch] + ow[rr * kD + ch];
      const float lr = rr ? Ls[1] : Ls[0];
      const float val = (lr > 0.f) ? o / lr : 0.f;
      const size_t oi = ((size_t)b * H + h) * kD + ch;
      if (a.out_fp32) reinterpret_cast<float*>(a.out)[oi] = val;
      else reinterpret_cast<uint16_t*>(a.out)[oi] = f32_to_bf16(val);
    }
    return;
  }

  // ---- split partial, then the last block of this (pair, head) merges -------------------
  if (!half && rr < nreq) {
    const int b = b0 + rr;
    float* pp = a.part + (((size_t)b * H + h) * a.n_split + split) * (kD + 2);
    pp[2 + ch] = o + comb[rr * kD + ch] + ow[rr * kD + ch];
    if (ch == 0) {
      pp[0] = rr ? M[1] : M[0];
      pp[1] = rr ? Ls[1] : Ls[0];
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&a.counters[pair * H + h], 1);
    *flag = (prev == a.n_split - 1);
  }
  __syncthreads();
  if (!*flag) return;
  __threadfence();
  if (!half && rr < nreq) {
    const int b = b0 + rr;
    const float* pp = a.part + ((size_t)b * H + h) * a.n_split * (kD + 2);
    float Mx = -INFINITY;
    for (int sp = 0; sp < a.n_split; ++sp) Mx = fmaxf(Mx, __ldcg(pp + sp * (kD + 2)));
    float Lt = 0.f, acc = 0.f;
    if (Mx != -INFINITY) {
      for (int sp = 0; sp < a.n_split; ++sp) {
        const float ms = __ldcg(pp + sp * (kD + 2));
        if (ms == -INFINITY) continue;
        const float wgt = exp2f(ms - Mx);
        Lt = fmaf(wgt, __ldcg(pp + sp * (kD + 2) + 1), Lt);
        acc = fmaf(wgt, __ldcg(pp + sp * (kD + 2) + 2 + ch), acc);
      }
    }
    const float val = (Lt > 0.f) ? acc / Lt : 0.f;
    const size_t oi = ((size_t)b * H + h) * kD + ch;
    if (a.out_fp32) reinterpret_cast<float*>(a.out)[oi] = val;
    else reinterpret_cast<uint16_t*>(a.out)[oi] = f32_to_bf16(val);
  }
  if (tid == 0) a.counters[pair * H + h] = 0;
}

}  // namespace

int vq_attn_max_pages_per_split(int win_slots) {
  const int per_req = (kSmemLimit - kOffScores) / (2 * 4);
  return (per_req - win_slots) / kPage;
}

size_t vq_attn_smem_bytes(int pages_per_split, int win_slots) {
  return kOffScores + (size_t)2 * 4 * (pages_per_split * kPage + win_slots);
}

cudaError_t launch_vq_attn(const VqAttnArgs& a, cudaStream_t st) {
  const int sc_stride = a.pages_per_split * kPage + a.win_slots;
  const size_t smem = vq_attn_smem_bytes(a.pages_per_split, a.win_slots);
  cudaError_t e = cudaFuncSetAttribute(vq_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)kD);
  dim3 grid(a.n_split, (a.B + 1) / 2, a.H);
  vq_attn_kernel<<<grid, kThreads, smem, st>>>(a, scale_log2, sc_stride);
  return cudaGetLastError();
}

}  // namespace kvq
