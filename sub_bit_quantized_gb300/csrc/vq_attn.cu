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
//  * B_t is copied into shared memory with TMA bulk copies; the index pages stream through
//    a 4-stage shared-memory ring (32 pages of each request per stage) filled by TMA bulk
//    copies, with full/empty mbarriers, so no warp waits on HBM latency per page. Every
//    wait is bounded and reports a timeout through the device error word.
//  * Keys: 8 lanes per page, lane s owns the RoPE partner groups s and s+8 (channels
//    8s..8s+7 and 64+8s..64+8s+7). The rotated query u = R(p_q - p) q satisfies
//    <R(p_q) q, R(p) k> = <u, k>, so the key is never rotated: u is built once from the
//    cos/sin table at the lane-group's first page, advanced one position per token by a
//    fixed rotation R(-theta) and 256 positions per chunk by R(-256 theta), and re-read
//    from the table every 16 chunks (a few ulp of drift at most). Rotation and dot
//    product use packed fp32x2 FMAs. Codeword rows are read with 128-bit shared loads in a
//    lane-dependent half order so the 8 lanes of a phase hit 8 distinct bank quads, and a
//    transposing shuffle reduction (7 shuffles per 8 tokens) leaves lane s with token s.
//  * Values: scores stay in shared memory (two-pass softmax) and, instead of rebuilding
//    value vectors, each token adds its softmax weight to w[g][r] for its 16 codewords;
//    o_g = sum_r w[g][r] B_t,V[g][r] is formed once per split (the same sum,
//    re-associated), reading B_t,V from L2. The histogram is laid out
//    [codeword][request*16 + group] so the 32 lanes of a warp (2 requests x 16 groups) hit
//    32 distinct banks. Once the key pass is done, the value pages of the whole split are
//    fetched by one bulk copy per request into the (then free) codebook buffer, and the
//    bf16 window values are read by all warps at once.
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
constexpr int kChunk = 32;                               // pages of each request per ring stage
constexpr int kStages = 4;
constexpr int kResync = 16;                              // chunks between cos/sin table reloads
constexpr uint32_t kSliceBytes = kCB * kD * 4;           // 128 KB fp32 B_t slice
constexpr uint32_t kStageBytes = 2 * kChunk * kPageBytes;  // 8 KB

// shared-memory layout (bytes)
constexpr int kOffCb = 0;
constexpr int kOffHist = kOffCb + kSliceBytes;           // float [256][32]
constexpr int kOffRing = kOffHist + kCB * 32 * 4;        // kStages x [2][kChunk][128] bytes
constexpr int kOffQ = kOffRing + kStages * kStageBytes;  // float [2][128]
constexpr int kOffOw = kOffQ + 2 * kD * 4;               // float [2][128] bf16-window V sums
constexpr int kOffComb = kOffOw + 2 * kD * 4;            // float [2][128]
constexpr int kOffRed = kOffComb + 2 * kD * 4;           // float [2][kWarps]
constexpr int kOffBar = kOffRed + 256;                   // mbarriers + flags
constexpr int kOffScores = kOffBar + 128;                // float [2][sc_stride]
constexpr int kSmemLimit = 232448;                       // 227 KB opt-in per block

static_assert(kOffBar % 8 == 0 && kOffRing % 128 == 0, "alignment");

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

// u <- R(-a) u for 8 channel pairs held as 4 float2 (pairs k, k+1) per half:
//   lo' = lo cos(a) + hi sin(a),  hi' = hi cos(a) - lo sin(a)
__device__ __forceinline__ void rotate8(float2 (&ul)[4], float2 (&uh)[4], const float2 (&c)[4],
                                        const float2 (&sn)[4], const float2 (&nsn)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 l = ul[k], hh = uh[k];
    ul[k] = __ffma2_rn(l, c[k], __fmul2_rn(hh, sn[k]));
    uh[k] = __ffma2_rn(l, nsn[k], __fmul2_rn(hh, c[k]));
  }
}

// A timed-out wait marks the block as failed; every later wait then returns at once so
// that all threads reach the same barriers and leave together.
__device__ __forceinline__ bool wait_stage(uint64_t* bar, uint32_t parity, volatile int* failed, int* err) {
  if (*failed) return false;
  if (mbar_wait_bounded(bar, parity)) return true;
  *failed = 1;
  set_error(err, KVQ_ERR_TIMEOUT);
  return false;
}

struct Req {
  int L, NP, pend, nq, nsink, nwin;
};

__global__ void __launch_bounds__(kThreads, 1) vq_attn_kernel(const VqAttnArgs a, const float scale_log2,
                                                                const int sc_stride) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* cbs = reinterpret_cast<float*>(smem + kOffCb);
  float* hist = reinterpret_cast<float*>(smem + kOffHist);
  unsigned char* ring = smem + kOffRing;
  float* qs = reinterpret_cast<float*>(smem + kOffQ);
  float* ow = reinterpret_cast<float*>(smem + kOffOw);
  float* comb = reinterpret_cast<float*>(smem + kOffComb);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  uint64_t* cbar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = cbar + 1;
  uint64_t* empty = full + kStages;
  int* sflag = reinterpret_cast<int*>(empty + kStages);  // [0] merge, [1] failed
  volatile int* failed = sflag + 1;
  float* sc = reinterpret_cast<float*>(smem + kOffScores);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, pair = blockIdx.y, h = blockIdx.z;
  const int H = a.H;
  const int b0 = pair * 2;
  const int nreq = min(2, a.B - b0);

  // ---- lengths of the two requests; pages of this split -------------------------------
  Req rq[2];
  const int pg0 = split * a.pages_per_split;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    int L = 0, NP = 0;
    if (r < nreq) {
      L = a.seq_len[b0 + r];
      NP = a.n_pages[b0 + r];
      // lengths that do not describe a valid cache are reported and attended as empty
      const bool bad = L < 0 || L > a.max_ctx || NP < 0 || NP > a.max_pages ||
                       (NP > 0 && a.sink + kPage * NP > L) || L - a.sink - kPage * NP > a.recent + kPage;
      if (bad) {
        if (split == 0 && tid == 0) set_error(a.err, KVQ_ERR_CAPACITY);
        L = 0;
        NP = 0;
      }
    }
    rq[r].L = L;
    rq[r].NP = NP;
    rq[r].pend = min(NP, pg0 + a.pages_per_split);
    rq[r].nq = max(0, rq[r].pend - pg0) * kPage;
    rq[r].nsink = min(a.sink, L);
    rq[r].nwin = (split == 0 && L > 0) ? (rq[r].nsink + max(0, L - a.sink - kPage * NP)) : 0;
  }
  const int n_items = max(rq[0].nq, rq[1].nq) / kPage;  // pages of the longer request
  const int n_chunks = (n_items + kChunk - 1) / kChunk;
  const int total_chunks = n_chunks;                     // key pages through the ring

  const size_t bh0 = ((size_t)b0 * H + h) * (size_t)a.max_pages * kPageBytes;
  const size_t bh1 = ((size_t)(b0 + (nreq > 1 ? 1 : 0)) * H + h) * (size_t)a.max_pages * kPageBytes;

  // producer (thread 0): chunk c of the key pages into ring stage c % kStages
  auto produce = [&](int c) {
    const int st = c % kStages;
    const uint8_t* base = a.idx_k;
    const int p_first = pg0 + c * kChunk;
    const int n0 = min(kChunk, max(0, rq[0].pend - p_first));
    const int n1 = min(kChunk, max(0, rq[1].pend - p_first));
    mbar_arrive_expect_tx(&full[st], (uint32_t)(n0 + n1) * kPageBytes);
    unsigned char* dst = ring + st * kStageBytes;
    if (n0 > 0) bulk_g2s(dst, base + bh0 + (size_t)p_first * kPageBytes, n0 * kPageBytes, &full[st]);
    if (n1 > 0)
      bulk_g2s(dst + kChunk * kPageBytes, base + bh1 + (size_t)p_first * kPageBytes, n1 * kPageBytes, &full[st]);
  };

  if (tid == 0) {
    mbar_init(cbar, 1);
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    sflag[0] = 0;
    sflag[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const float* btk = a.bt_k + (size_t)h * kCB * kD;
  const float* btv = a.bt_v + (size_t)h * kCB * kD;
  if (tid == 0 && n_items > 0) {
    mbar_arrive_expect_tx(cbar, kSliceBytes);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      bulk_g2s(cbs + k * (kSliceBytes / 16), btk + k * (kSliceBytes / 16), kSliceBytes / 4, cbar);
    for (int gc = 0; gc < min(kStages, total_chunks); ++gc) produce(gc);
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
  const int lg = tid >> 3;

  float mloc0 = -INFINITY, mloc1 = -INFINITY;

  // ---- bf16 window scores (split 0 only) ------------------------------------------------
  for (int wi = lg; wi < rq[0].nwin + rq[1].nwin; wi += kLaneGroups) {
    const bool r1 = wi >= rq[0].nwin;
    const Req R = r1 ? rq[1] : rq[0];
    const int r = r1 ? 1 : 0;
    const int w = r1 ? wi - rq[0].nwin : wi;
    const int p = (w < R.nsink) ? w : a.sink + kPage * R.NP + (w - R.nsink);
    const int slot = (p < a.sink) ? p : a.sink + (p - a.sink) % (a.recent + kPage);
    const uint16_t* kr = a.win_k + (((size_t)(b0 + r) * H + h) * a.win_slots + slot) * kD;
    float klo[8], khi[8], c[8], sn[8], ql[8], qh[8];
    ldg8_bf16_perm(kr + 8 * s, o0, klo);
    ldg8_bf16_perm(kr + 64 + 8 * s, o0, khi);
    const int dl = R.L - 1 - p;
    ldg8_perm(a.rope_cos + (size_t)dl * (kD / 2) + 8 * s, o0, c);
    ldg8_perm(a.rope_sin + (size_t)dl * (kD / 2) + 8 * s, o0, sn);
    load8_perm(qs + r * kD + 8 * s, o0, ql);
    load8_perm(qs + r * kD + 64 + 8 * s, o0, qh);
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float ul = ql[k] * c[k] - qh[k] * sn[k];
      const float uh = qh[k] * c[k] + ql[k] * sn[k];
      acc = fmaf(ul, klo[k], acc);
      acc = fmaf(uh, khi[k], acc);
    }
    acc += __shfl_xor_sync(gmask, acc, 4);
    acc += __shfl_xor_sync(gmask, acc, 2);
    acc += __shfl_xor_sync(gmask, acc, 1);
    if (s == 0) {
      const float v = acc * scale_log2;
      sc[r * sc_stride + R.nq + w] = v;
      if (r1) mloc1 = fmaxf(mloc1, v);
      else mloc0 = fmaxf(mloc0, v);
    }
  }

  // ---- key pages: lane-group lg takes request lg/32, page lg%32 of every chunk ----------
  {
    const int r = lg >> 5, po = lg & 31;
    const Req R = (r == 0) ? rq[0] : rq[1];
    float2 cth[4], sth[4], nsth[4], cj[4], sj[4], nsj[4];
    {
      float c8[8], s8[8];
      ldg8_perm(a.rope_cos + (kD / 2) + 8 * s, o0, c8);
      ldg8_perm(a.rope_sin + (kD / 2) + 8 * s, o0, s8);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        cth[k] = make_float2(c8[2 * k], c8[2 * k + 1]);
        sth[k] = make_float2(s8[2 * k], s8[2 * k + 1]);
        nsth[k] = make_float2(-s8[2 * k], -s8[2 * k + 1]);
      }
      const int jrow = kChunk * kPage;  // one chunk further: 256 positions
      if (n_chunks > 1 && jrow < a.max_ctx) {
        ldg8_perm(a.rope_cos + (size_t)jrow * (kD / 2) + 8 * s, o0, c8);
        ldg8_perm(a.rope_sin + (size_t)jrow * (kD / 2) + 8 * s, o0, s8);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        cj[k] = make_float2(c8[2 * k], c8[2 * k + 1]);
        sj[k] = make_float2(s8[2 * k], s8[2 * k + 1]);
        nsj[k] = make_float2(-s8[2 * k], -s8[2 * k + 1]);
      }
    }
    float ql8[8], qh8[8];
    load8_perm(qs + r * kD + 8 * s, o0, ql8);
    load8_perm(qs + r * kD + 64 + 8 * s, o0, qh8);
    float2 u0l[4], u0h[4];  // rotated query at this lane-group's current page start
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      u0l[k] = make_float2(0.f, 0.f);
      u0h[k] = make_float2(0.f, 0.f);
    }

    if (n_items > 0) wait_stage(cbar, 0, failed, a.err);
    for (int c = 0; c < n_chunks; ++c) {
      const int st = c % kStages;
      wait_stage(&full[st], (c / kStages) & 1, failed, a.err);
      const int pg = pg0 + c * kChunk + po;
      if (!*failed && pg < R.pend) {
        if (c % kResync == 0) {
          const int d0 = R.L - 1 - (a.sink + kPage * pg);
          float c8[8], s8[8];
          ldg8_perm(a.rope_cos + (size_t)d0 * (kD / 2) + 8 * s, o0, c8);
          ldg8_perm(a.rope_sin + (size_t)d0 * (kD / 2) + 8 * s, o0, s8);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            u0l[k] = make_float2(ql8[2 * k] * c8[2 * k] - qh8[2 * k] * s8[2 * k],
                                 ql8[2 * k + 1] * c8[2 * k + 1] - qh8[2 * k + 1] * s8[2 * k + 1]);
            u0h[k] = make_float2(qh8[2 * k] * c8[2 * k] + ql8[2 * k] * s8[2 * k],
                                 qh8[2 * k + 1] * c8[2 * k + 1] + ql8[2 * k + 1] * s8[2 * k + 1]);
          }
        } else {
          rotate8(u0l, u0h, cj, sj, nsj);  // 256 positions later
        }
        const uint4 row =
            *reinterpret_cast<const uint4*>(ring + st * kStageBytes + (r * kChunk + po) * kPageBytes + 16 * s);
        float2 ul[4], uh[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ul[k] = u0l[k];
          uh[k] = u0h[k];
        }
        float part[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t wd = (j < 2) ? row.x : (j < 4) ? row.y : (j < 6) ? row.z : row.w;
          const uint32_t sh = (j & 1) * 16;
          const uint32_t rlo = (wd >> sh) & 0xFFu;
          const uint32_t rhi = (wd >> (sh + 8)) & 0xFFu;
          const float* pl = cbs + rlo * kD + 8 * s;
          const float* ph = cbs + rhi * kD + 64 + 8 * s;
          const float4 la = *reinterpret_cast<const float4*>(pl + o0);
          const float4 lb = *reinterpret_cast<const float4*>(pl + (4 - o0));
          const float4 ha = *reinterpret_cast<const float4*>(ph + o0);
          const float4 hb = *reinterpret_cast<const float4*>(ph + (4 - o0));
          float2 acc = __fmul2_rn(ul[0], make_float2(la.x, la.y));
          acc = __ffma2_rn(ul[1], make_float2(la.z, la.w), acc);
          acc = __ffma2_rn(ul[2], make_float2(lb.x, lb.y), acc);
          acc = __ffma2_rn(ul[3], make_float2(lb.z, lb.w), acc);
          acc = __ffma2_rn(uh[0], make_float2(ha.x, ha.y), acc);
          acc = __ffma2_rn(uh[1], make_float2(ha.z, ha.w), acc);
          acc = __ffma2_rn(uh[2], make_float2(hb.x, hb.y), acc);
          acc = __ffma2_rn(uh[3], make_float2(hb.z, hb.w), acc);
          part[j] = acc.x + acc.y;
          if (j < 7) rotate8(ul, uh, cth, sth, nsth);  // next token: one position later
        }
        transpose_reduce8(part, s, gmask);
        const float v = part[0] * scale_log2;
        sc[r * sc_stride + (c * kChunk + po) * kPage + s] = v;
        if (r) mloc1 = fmaxf(mloc1, v);
        else mloc0 = fmaxf(mloc0, v);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (tid == 0 && c + kStages < total_chunks) {
        if (wait_stage(&empty[st], (c / kStages) & 1, failed, a.err)) produce(c + kStages);
      }
    }
  }

  // ---- B_t(K) no longer read: fetch this split's value pages into the same buffer -------
  // (request r's pages at byte offset r * pages_per_split * 128; at most 128 KB in all)
  unsigned char* vpages = reinterpret_cast<unsigned char*>(cbs);
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0 && n_items > 0 && !*failed) {
    const int n0 = max(0, rq[0].pend - pg0), n1 = max(0, rq[1].pend - pg0);
    mbar_arrive_expect_tx(cbar, (uint32_t)(n0 + n1) * kPageBytes);
    if (n0 > 0) bulk_g2s(vpages, a.idx_v + bh0 + (size_t)pg0 * kPageBytes, n0 * kPageBytes, cbar);
    if (n1 > 0)
      bulk_g2s(vpages + (size_t)a.pages_per_split * kPageBytes, a.idx_v + bh1 + (size_t)pg0 * kPageBytes,
               n1 * kPageBytes, cbar);
  }

  // ---- softmax statistics per request ---------------------------------------------------
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    mloc0 = fmaxf(mloc0, __shfl_xor_sync(0xFFFFFFFFu, mloc0, off));
    mloc1 = fmaxf(mloc1, __shfl_xor_sync(0xFFFFFFFFu, mloc1, off));
  }
  if (lane == 0) {
    red[warp] = mloc0;
    red[kWarps + warp] = mloc1;
  }
  __syncthreads();
  float M0 = -INFINITY, M1 = -INFINITY;
  for (int w = 0; w < kWarps; ++w) {
    M0 = fmaxf(M0, red[w]);
    M1 = fmaxf(M1, red[kWarps + w]);
  }
  __syncthreads();  // red is reused below
  float ls0 = 0.f, ls1 = 0.f;
  if (M0 != -INFINITY) {
    for (int i = tid; i < rq[0].nq + rq[0].nwin; i += kThreads) {
      const float e = exp2f(sc[i] - M0);
      sc[i] = e;
      ls0 += e;
    }
  }
  if (M1 != -INFINITY) {
    for (int i = tid; i < rq[1].nq + rq[1].nwin; i += kThreads) {
      const float e = exp2f(sc[sc_stride + i] - M1);
      sc[sc_stride + i] = e;
      ls1 += e;
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    ls0 += __shfl_xor_sync(0xFFFFFFFFu, ls0, off);
    ls1 += __shfl_xor_sync(0xFFFFFFFFu, ls1, off);
  }
  if (lane == 0) {
    red[warp] = ls0;
    red[kWarps + warp] = ls1;
  }
  __syncthreads();  // weights in sc are final
  float L0s = 0.f, L1s = 0.f;
  for (int w = 0; w < kWarps; ++w) {
    L0s += red[w];
    L1s += red[kWarps + w];
  }

  // ---- bf16 window values: warp w takes window tokens w, w+16, ...; lane = 4 channels ----
  {
    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
    const int nw = rq[0].nwin + rq[1].nwin;
#pragma unroll 4
    for (int wi = warp; wi < nw; wi += kWarps) {
      const bool r1 = wi >= rq[0].nwin;
      const Req R = r1 ? rq[1] : rq[0];
      const int r = r1 ? 1 : 0;
      const int w = r1 ? wi - rq[0].nwin : wi;
      const int p = (w < R.nsink) ? w : a.sink + kPage * R.NP + (w - R.nsink);
      const int slot = (p < a.sink) ? p : a.sink + (p - a.sink) % (a.recent + kPage);
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(
          a.win_v + (((size_t)(b0 + r) * H + h) * a.win_slots + slot) * kD + 4 * lane));
      const float pw = sc[r * sc_stride + R.nq + w];
      const float p0 = r1 ? 0.f : pw, p1 = r1 ? pw : 0.f;
      const float v0 = bf16_lo(v.x), v1 = bf16_hi(v.x), v2 = bf16_lo(v.y), v3 = bf16_hi(v.y);
      acc0.x = fmaf(p0, v0, acc0.x); acc0.y = fmaf(p0, v1, acc0.y);
      acc0.z = fmaf(p0, v2, acc0.z); acc0.w = fmaf(p0, v3, acc0.w);
      acc1.x = fmaf(p1, v0, acc1.x); acc1.y = fmaf(p1, v1, acc1.y);
      acc1.z = fmaf(p1, v2, acc1.z); acc1.w = fmaf(p1, v3, acc1.w);
    }
    // per-warp partial sums into the ring buffer (free now): [warp][request][128]
    float* wpart = reinterpret_cast<float*>(ring);
    reinterpret_cast<float4*>(wpart + (warp * 2 + 0) * kD)[lane] = acc0;
    reinterpret_cast<float4*>(wpart + (warp * 2 + 1) * kD)[lane] = acc1;
  }

  // ---- value pages (now in shared memory): warp w takes pages w, w+16, ...; lane =
  //      (request, group) column of the histogram ----------------------------------------
  if (n_items > 0) wait_stage(cbar, 1, failed, a.err);
  {
    const int r = lane >> 4, g = lane & 15;
    const int sl = g & 7, hb = (g >> 3) * 8;
    const int np_r = max(0, (r ? rq[1].pend : rq[0].pend) - pg0);
    const unsigned char* vp = vpages + (size_t)r * a.pages_per_split * kPageBytes + 16 * sl;
    if (!*failed) {
      for (int pi = warp; pi < np_r; pi += kWarps) {
        const uint4 row = *reinterpret_cast<const uint4*>(vp + (size_t)pi * kPageBytes);
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
  __syncthreads();
  if (tid < 2 * kD) {  // window value sums of the 16 warps
    const float* wpart = reinterpret_cast<const float*>(ring);
    const int r = tid >> 7, ch = tid & 127;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) acc += wpart[(w * 2 + r) * kD + ch];
    ow[tid] = acc;
  }

  // ---- o_g = sum_r w[g][r] * B_t,V[g][r], B_t,V read from L2 ---------------------------
  if (*failed) return;  // uniform: every thread read the flag after the last barrier
  float o = 0.f;
  const int rr = (tid >> 7) & 1, ch = tid & 127, half = tid >> 8;
  if (n_items > 0) {
    const int col = rr * 16 + (ch >> 3);
    const int b_lo = half * 128;
    float o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll 4
    for (int bin = b_lo; bin < b_lo + 128; bin += 4) {
      o = fmaf(hist[bin * 32 + col], __ldg(btv + bin * kD + ch), o);
      o1 = fmaf(hist[(bin + 1) * 32 + col], __ldg(btv + (bin + 1) * kD + ch), o1);
      o2 = fmaf(hist[(bin + 2) * 32 + col], __ldg(btv + (bin + 2) * kD + ch), o2);
      o3 = fmaf(hist[(bin + 3) * 32 + col], __ldg(btv + (bin + 3) * kD + ch), o3);
    }
    o = (o + o1) + (o2 + o3);
  }
  if (half) comb[rr * kD + ch] = o;
  __syncthreads();

  const float Mr = rr ? M1 : M0;
  const float Lr = rr ? L1s : L0s;
  if (a.n_split == 1) {
    if (!half && rr < nreq) {
      const int b = b0 + rr;
      o += comb[rr * kD + ch] + ow[rr * kD + ch];
      const float val = (Lr > 0.f) ? o / Lr : 0.f;
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
      pp[0] = Mr;
      pp[1] = Lr;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&a.counters[pair * H + h], 1);
    sflag[0] = (prev == a.n_split - 1);
  }
  __syncthreads();
  if (!sflag[0]) return;
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
