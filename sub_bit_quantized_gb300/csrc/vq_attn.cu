// LoopVQ decode attention over the bf16 window and the 8-token index pages of one
// (layer, loop step), split-K over pages with an exact logsumexp merge.
//
// Follows "LoopVQ: Sub 1-bit KV Cache Quantization for Looped Transformers", method
// step 5, Algorithm 1 and Figure 5: the step's codebook slice B_t is staged in shared
// memory once per thread block, keys and values are rebuilt from D/c = 16 indices per
// token, keys are rotated by RoPE and dotted with the query, the bf16 sink/recent tokens are
// attended directly, and the partials of every split are merged exactly. Two requests of
// the same head share a thread block and its B_t load.
//
// GB300 design (differs from the page's Triton kernel). On this GPU each codeword lookup
// costs shared-memory bandwidth (32 B per fp32 group), and that, not HBM, bounds the
// kernel; the structure keeps every lookup a conflict-free 128-bit shared load and moves
// no other data through shared memory per token:
//  * Both slices stay resident: keys in fp32 (128 KB, TMA bulk copy; channels 0..63 and
//    64..127 as two [256][64] tables), values in fp16 ([256][128], converted while
//    staging; value rounding error ~1e-4 of the output). A codeword's shared-memory address
//    is one byte permute: (index << 8) | lane offset.
//  * Index pages stream through a 2-stage shared-memory ring (32 key and 32 value pages of
//    each request per stage) filled by TMA bulk copies with full/empty mbarriers. Every
//    wait is bounded and reports a timeout through the device error word.
//  * 8 lanes per page, lane s owns the RoPE partner groups s and s+8 (channels 8s..8s+7 and
//    64+8s..64+8s+7). The rotated query u = R(p_q - p) q satisfies <R(p_q) q, R(p) k> =
//    <u, k>, so keys are never rotated: u is built from the cos/sin table at a lane-group's
//    first page, advanced one position per token by R(-theta) and one chunk (256
//    positions) by R(-256 theta), and re-read from the table every 16 chunks. Packed fp32x2
//    FMAs. A transposing shuffle reduction leaves lane s with the score of token s.
//  * One pass with an online softmax per lane-group (running max, rescale on increase):
//    the 8 softmax weights of a page are broadcast by shuffles and each lane accumulates
//    its 16 value channels directly from the fp16 value table.
//  * Lane-groups merge in registers (shuffles), warps through shared memory, splits in the
//    last block of a (request pair, head) to finish (arrival counter, no spin-wait).
#include <cuda_fp16.h>

#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "../../include/kvq.h"

namespace kvq {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kLaneGroups = kThreads / 8;
constexpr int kChunk = 32;                                // pages of each request per ring stage
constexpr int kStages = 2;
constexpr int kResync = 16;                               // chunks between cos/sin table reloads
constexpr uint32_t kKSliceBytes = kCB * kD * 4;           // fp32 key codebook slice
constexpr uint32_t kVSliceBytes = kCB * kD * 2;           // fp16 value codebook slice
constexpr uint32_t kPart = kChunk * kPageBytes;           // 4 KB: one request's pages of one kind
constexpr uint32_t kStageBytes = 4 * kPart;               // [K r0 | K r1 | V r0 | V r1]

// shared-memory layout (bytes)
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKSliceBytes;
constexpr int kOffRing = kOffV + kVSliceBytes;
constexpr int kOffQ = kOffRing + kStages * kStageBytes;    // float [2][128]
constexpr int kOffJ = kOffQ + 2 * kD * 4;                  // float [8 slots][16]: cos, sin(256 theta)
constexpr int kOffBar = kOffJ + 8 * 16 * 4;                // mbarriers + flags
constexpr int kSmemBytes = kOffBar + 128;
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kOffBar % 8 == 0 && kOffRing % 128 == 0, "alignment");

__device__ __forceinline__ void ldg8_perm(const float* p, int o0, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p + o0));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p + (4 - o0)));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8_perm(const float* p, int o0, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p + o0);
  const float4 b = *reinterpret_cast<const float4*>(p + (4 - o0));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
// 8 consecutive bf16 values in the lane's half order
__device__ __forceinline__ void ldg8_bf16_perm(const uint16_t* p, int o0, float (&v)[8]) {
  const uint2 a = __ldg(reinterpret_cast<const uint2*>(p + o0));
  const uint2 b = __ldg(reinterpret_cast<const uint2*>(p + (4 - o0)));
  v[0] = bf16_lo(a.x); v[1] = bf16_hi(a.x); v[2] = bf16_lo(a.y); v[3] = bf16_hi(a.y);
  v[4] = bf16_lo(b.x); v[5] = bf16_hi(b.x); v[6] = bf16_lo(b.y); v[7] = bf16_hi(b.y);
}
// 8 consecutive fp16 values (one 128-bit shared load), natural order
__device__ __forceinline__ void lds8_fp16(const unsigned char* p, float2 (&v)[4]) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  v[0] = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
  v[1] = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
  v[2] = __half22float2(*reinterpret_cast<const __half2*>(&w.z));
  v[3] = __half22float2(*reinterpret_cast<const __half2*>(&w.w));
}
// byte offset (index << 8) | lane_byte, the index being byte k of w (lane_byte < 256)
template <int K>
__device__ __forceinline__ uint32_t row_off(uint32_t w, uint32_t lane_byte) {
  return __byte_perm(w, lane_byte, 0x5504u | (K << 4));
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

// rotated query u = R(d) q for the lane's 8 pairs (lane half order), q from shared memory
__device__ __forceinline__ void rotated_query(const float* rc, const float* rs, int d, int s, int o0,
                                              const float* q, float2 (&ul)[4], float2 (&uh)[4]) {
  float c8[8], s8[8], ql[8], qh[8];
  ldg8_perm(rc + (size_t)d * (kD / 2) + 8 * s, o0, c8);
  ldg8_perm(rs + (size_t)d * (kD / 2) + 8 * s, o0, s8);
  load8_perm(q + 8 * s, o0, ql);
  load8_perm(q + 64 + 8 * s, o0, qh);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ul[k] = make_float2(ql[2 * k] * c8[2 * k] - qh[2 * k] * s8[2 * k],
                        ql[2 * k + 1] * c8[2 * k + 1] - qh[2 * k + 1] * s8[2 * k + 1]);
    uh[k] = make_float2(qh[2 * k] * c8[2 * k] + ql[2 * k] * s8[2 * k],
                        qh[2 * k + 1] * c8[2 * k + 1] + ql[2 * k + 1] * s8[2 * k + 1]);
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

// running softmax state of one lane (the max is shared by its lane-group)
struct Acc {
  float M, l;
  float2 ol[4], oh[4];
};

// Fold the 8 scores of a page (lane s holds token s; -inf for a missing token) into the
// running state: raise the shared max if needed (rescaling the sums), return this lane's
// token weight.
__device__ __forceinline__ float online_weights(Acc& A, float sc, unsigned mask) {
  float mp = sc;
  mp = fmaxf(mp, __shfl_xor_sync(mask, mp, 4));
  mp = fmaxf(mp, __shfl_xor_sync(mask, mp, 2));
  mp = fmaxf(mp, __shfl_xor_sync(mask, mp, 1));
  if (mp > A.M) {  // uniform within the lane-group
    const float f = (A.M == -INFINITY) ? 0.f : exp2f(A.M - mp);
    const float2 f2 = make_float2(f, f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      A.ol[k] = __fmul2_rn(A.ol[k], f2);
      A.oh[k] = __fmul2_rn(A.oh[k], f2);
    }
    A.l *= f;
    A.M = mp;
  }
  const float p = (sc == -INFINITY) ? 0.f : exp2f(sc - A.M);
  A.l += p;
  return p;
}

struct Req {
  int L, NP, pend, nsink, nwin;
};

__global__ void __launch_bounds__(kThreads, 1) vq_attn_kernel(const VqAttnArgs a, const float scale_log2) {
  extern __shared__ __align__(128) unsigned char smem[];
  float* ks = reinterpret_cast<float*>(smem + kOffK);
  __half* vs = reinterpret_cast<__half*>(smem + kOffV);
  unsigned char* ring = smem + kOffRing;
  float* qs = reinterpret_cast<float*>(smem + kOffQ);
  uint64_t* kbar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = kbar + 1;
  uint64_t* empty = full + kStages;
  int* sflag = reinterpret_cast<int*>(empty + kStages);  // [0] merge, [1] failed
  volatile int* failed = sflag + 1;

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
    rq[r].nsink = min(a.sink, L);
    rq[r].nwin = (split == 0 && L > 0) ? (rq[r].nsink + max(0, L - a.sink - kPage * NP)) : 0;
  }
  const int n_items = max(max(0, rq[0].pend - pg0), max(0, rq[1].pend - pg0));
  const int n_chunks = (n_items + kChunk - 1) / kChunk;
  const size_t bh0 = ((size_t)b0 * H + h) * (size_t)a.max_pages * kPageBytes;
  const size_t bh1 = ((size_t)(b0 + (nreq > 1 ? 1 : 0)) * H + h) * (size_t)a.max_pages * kPageBytes;

  // producer (thread 0): key and value pages of chunk c into ring stage c % kStages
  auto produce = [&](int c) {
    const int st = c % kStages;
    const int p_first = pg0 + c * kChunk;
    const int n0 = min(kChunk, max(0, rq[0].pend - p_first));
    const int n1 = min(kChunk, max(0, rq[1].pend - p_first));
    mbar_arrive_expect_tx(&full[st], (uint32_t)(n0 + n1) * 2 * kPageBytes);
    unsigned char* dst = ring + st * kStageBytes;
    const size_t off = (size_t)p_first * kPageBytes;
    if (n0 > 0) {
      bulk_g2s(dst, a.idx_k + bh0 + off, n0 * kPageBytes, &full[st]);
      bulk_g2s(dst + 2 * kPart, a.idx_v + bh0 + off, n0 * kPageBytes, &full[st]);
    }
    if (n1 > 0) {
      bulk_g2s(dst + kPart, a.idx_k + bh1 + off, n1 * kPageBytes, &full[st]);
      bulk_g2s(dst + 3 * kPart, a.idx_v + bh1 + off, n1 * kPageBytes, &full[st]);
    }
  };

  if (tid == 0) {
    mbar_init(kbar, 1);
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
  if (tid == 0 && n_items > 0) {
    const float* btk = a.bt_k + (size_t)h * kCB * kD;
    mbar_arrive_expect_tx(kbar, kKSliceBytes);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      bulk_g2s(ks + k * (kKSliceBytes / 16), btk + k * (kKSliceBytes / 16), kKSliceBytes / 4, kbar);
    for (int c = 0; c < min(kStages, n_chunks); ++c) produce(c);
  }
  if (n_items > 0) {  // value slice: fp32 [2][256][64] in L2 -> fp16 [256][128] in shared memory
    const float4* src = reinterpret_cast<const float4*>(a.bt_v + (size_t)h * kCB * kD);
    for (int i = tid; i < kCB * kD / 4; i += kThreads) {
      const float4 v = __ldg(src + i);
      const int half = i / (kCB * kD / 8), rem = i % (kCB * kD / 8);
      const int row = rem / (kD / 8), c4 = rem % (kD / 8);
      __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
      uint2 w;
      w.x = *reinterpret_cast<uint32_t*>(&lo);
      w.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(vs + row * kD + half * (kD / 2))[c4] = w;
    }
  }
  if (tid < 2 * kD) {
    const int r = tid >> 7;
    qs[tid] = bf16_to_f32(a.q[((size_t)(b0 + min(r, nreq - 1)) * H + h) * kD + (tid & 127)]);
  }
  if (tid < 8 && n_chunks > 1) {  // cos/sin(256 theta_i) for slot tid, in that slot's half order
    float* jt = reinterpret_cast<float*>(smem + kOffJ) + tid * 16;
    const int jo0 = (tid & 4) ? 4 : 0;
    float c8[8], s8[8];
    ldg8_perm(a.rope_cos + (size_t)(kChunk * kPage) * (kD / 2) + 8 * tid, jo0, c8);
    ldg8_perm(a.rope_sin + (size_t)(kChunk * kPage) * (kD / 2) + 8 * tid, jo0, s8);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      jt[k] = c8[k];
      jt[8 + k] = s8[k];
    }
  }
  __syncthreads();

  const int s = tid & 7;                 // slot: groups s and s + 8
  const int o0 = (s & 4) ? 4 : 0;        // key half order (bank-quad spreading)
  const unsigned gmask = 0xFFu << (lane & 24);
  const int lg = tid >> 3;
  const int r = lg >> 5, po = lg & 31;   // this lane-group's request and page slot
  const Req R = r ? rq[1] : rq[0];
  const float* qr = qs + r * kD;

  // value accumulators in natural channel order: ol = channels 8s..8s+7, oh = 64+8s..
  Acc A;
  A.M = -INFINITY;
  A.l = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    A.ol[k] = make_float2(0.f, 0.f);
    A.oh[k] = make_float2(0.f, 0.f);
  }
  const uint16_t* wk = a.win_k + ((size_t)(b0 + r) * H + h) * a.win_slots * kD;
  const uint16_t* wv = a.win_v + ((size_t)(b0 + r) * H + h) * a.win_slots * kD;

  // ---- bf16 window (split 0): lane-group po takes window tokens [8 wp, 8 wp + 8) ----------
  for (int wp = po; wp * kPage < R.nwin; wp += kLaneGroups / 2) {
    float part[8];
    int slots[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int w = wp * kPage + j;
      part[j] = 0.f;
      slots[j] = 0;
      if (w < R.nwin) {
        const int p = (w < R.nsink) ? w : a.sink + kPage * R.NP + (w - R.nsink);
        const int slot = (p < a.sink) ? p : a.sink + (p - a.sink) % (a.recent + kPage);
        slots[j] = slot;
        float kl[8], kh[8];
        ldg8_bf16_perm(wk + (size_t)slot * kD + 8 * s, o0, kl);
        ldg8_bf16_perm(wk + (size_t)slot * kD + 64 + 8 * s, o0, kh);
        float2 ul[4], uh[4];
        rotated_query(a.rope_cos, a.rope_sin, R.L - 1 - p, s, o0, qr, ul, uh);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc = __ffma2_rn(ul[k], make_float2(kl[2 * k], kl[2 * k + 1]), acc);
          acc = __ffma2_rn(uh[k], make_float2(kh[2 * k], kh[2 * k + 1]), acc);
        }
        part[j] = acc.x + acc.y;
      }
    }
    transpose_reduce8(part, s, gmask);
    const float sc = (wp * kPage + s < R.nwin) ? part[0] * scale_log2 : -INFINITY;
    const float p = online_weights(A, sc, gmask);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float pj = __shfl_sync(gmask, p, (lane & 24) + j);
      if (wp * kPage + j < R.nwin) {
        float vl[8], vh[8];
        ldg8_bf16_perm(wv + (size_t)slots[j] * kD + 8 * s, 0, vl);
        ldg8_bf16_perm(wv + (size_t)slots[j] * kD + 64 + 8 * s, 0, vh);
        const float2 p2 = make_float2(pj, pj);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          A.ol[k] = __ffma2_rn(p2, make_float2(vl[2 * k], vl[2 * k + 1]), A.ol[k]);
          A.oh[k] = __ffma2_rn(p2, make_float2(vh[2 * k], vh[2 * k + 1]), A.oh[k]);
        }
      }
    }
  }

  // ---- quantized pages -------------------------------------------------------------------
  {
    float2 cth[4], sth[4], nsth[4];
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
    }
    float2 u0l[4], u0h[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      u0l[k] = make_float2(0.f, 0.f);
      u0h[k] = make_float2(0.f, 0.f);
    }
    // lane byte offsets inside a 256-byte table row: key halves swapped for s >= 4 so the 8
    // lanes of a phase hit 8 bank quads; value lanes read 16 natural bytes each
    const uint32_t kb0 = 32 * s + 4 * o0, kb1 = kb0 ^ 16u;
    const uint32_t vb0 = 16 * s, vb1 = 128 + 16 * s;
    const unsigned char* ksb = reinterpret_cast<const unsigned char*>(ks);
    const unsigned char* vsb = reinterpret_cast<const unsigned char*>(vs);
    const float* jt = reinterpret_cast<const float*>(smem + kOffJ) + s * 16;

    if (n_items > 0) wait_stage(kbar, 0, failed, a.err);
    for (int c = 0; c < n_chunks; ++c) {
      const int st = c % kStages;
      wait_stage(&full[st], (c / kStages) & 1, failed, a.err);
      const int pg = pg0 + c * kChunk + po;
      if (!*failed && pg < R.pend) {
        if (c % kResync == 0) {
          rotated_query(a.rope_cos, a.rope_sin, R.L - 1 - (a.sink + kPage * pg), s, o0, qr, u0l, u0h);
        } else {  // 256 positions later
          const float4 c0 = *reinterpret_cast<const float4*>(jt), c1 = *reinterpret_cast<const float4*>(jt + 4);
          const float4 s0 = *reinterpret_cast<const float4*>(jt + 8), s1 = *reinterpret_cast<const float4*>(jt + 12);
          const float2 cj[4] = {make_float2(c0.x, c0.y), make_float2(c0.z, c0.w), make_float2(c1.x, c1.y),
                                make_float2(c1.z, c1.w)};
          const float2 sj[4] = {make_float2(s0.x, s0.y), make_float2(s0.z, s0.w), make_float2(s1.x, s1.y),
                                make_float2(s1.z, s1.w)};
          const float2 nsj[4] = {make_float2(-s0.x, -s0.y), make_float2(-s0.z, -s0.w), make_float2(-s1.x, -s1.y),
                                 make_float2(-s1.z, -s1.w)};
          rotate8(u0l, u0h, cj, sj, nsj);
        }
        const unsigned char* stage = ring + st * kStageBytes;
        const uint4 rowk = *reinterpret_cast<const uint4*>(stage + r * kPart + po * kPageBytes + 16 * s);
        float2 ul[4], uh[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ul[k] = u0l[k];
          uh[k] = u0h[k];
        }
        float part[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t wd = (j < 2) ? rowk.x : (j < 4) ? rowk.y : (j < 6) ? rowk.z : rowk.w;
          uint32_t al0, al1, ah0, ah1;
          if (j & 1) {
            al0 = row_off<2>(wd, kb0); al1 = row_off<2>(wd, kb1);
            ah0 = row_off<3>(wd, kb0); ah1 = row_off<3>(wd, kb1);
          } else {
            al0 = row_off<0>(wd, kb0); al1 = row_off<0>(wd, kb1);
            ah0 = row_off<1>(wd, kb0); ah1 = row_off<1>(wd, kb1);
          }
          const float4 la = *reinterpret_cast<const float4*>(ksb + al0);
          const float4 lb = *reinterpret_cast<const float4*>(ksb + al1);
          const float4 ha = *reinterpret_cast<const float4*>(ksb + kKSliceBytes / 2 + ah0);
          const float4 hb = *reinterpret_cast<const float4*>(ksb + kKSliceBytes / 2 + ah1);
          float2 acc0 = __fmul2_rn(ul[0], make_float2(la.x, la.y));
          float2 acc1 = __fmul2_rn(uh[0], make_float2(ha.x, ha.y));
          acc0 = __ffma2_rn(ul[1], make_float2(la.z, la.w), acc0);
          acc1 = __ffma2_rn(uh[1], make_float2(ha.z, ha.w), acc1);
          acc0 = __ffma2_rn(ul[2], make_float2(lb.x, lb.y), acc0);
          acc1 = __ffma2_rn(uh[2], make_float2(hb.x, hb.y), acc1);
          acc0 = __ffma2_rn(ul[3], make_float2(lb.z, lb.w), acc0);
          acc1 = __ffma2_rn(uh[3], make_float2(hb.z, hb.w), acc1);
          const float2 acc = __fadd2_rn(acc0, acc1);
          part[j] = acc.x + acc.y;
          if (j < 7) rotate8(ul, uh, cth, sth, nsth);  // next token: one position later
        }
        transpose_reduce8(part, s, gmask);
        const float p = online_weights(A, part[0] * scale_log2, gmask);
        const uint4 rowv = *reinterpret_cast<const uint4*>(stage + (2 + r) * kPart + po * kPageBytes + 16 * s);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float pj = __shfl_sync(gmask, p, (lane & 24) + j);
          const uint32_t wd = (j < 2) ? rowv.x : (j < 4) ? rowv.y : (j < 6) ? rowv.z : rowv.w;
          const uint32_t avl = (j & 1) ? row_off<2>(wd, vb0) : row_off<0>(wd, vb0);
          const uint32_t avh = (j & 1) ? row_off<3>(wd, vb1) : row_off<1>(wd, vb1);
          float2 vl[4], vh[4];
          lds8_fp16(vsb + avl, vl);
          lds8_fp16(vsb + avh, vh);
          const float2 p2 = make_float2(pj, pj);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            A.ol[k] = __ffma2_rn(p2, vl[k], A.ol[k]);
            A.oh[k] = __ffma2_rn(p2, vh[k], A.oh[k]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      if (tid == 0 && c + kStages < n_chunks) {
        if (wait_stage(&empty[st], (c / kStages) & 1, failed, a.err)) produce(c + kStages);
      }
    }
  }

  // ---- merge: lanes of a group (l), lane-groups of a warp (shuffles), warps (smem) -------
  A.l += __shfl_xor_sync(0xFFFFFFFFu, A.l, 1);
  A.l += __shfl_xor_sync(0xFFFFFFFFu, A.l, 2);
  A.l += __shfl_xor_sync(0xFFFFFFFFu, A.l, 4);
#pragma unroll
  for (int off = 8; off <= 16; off <<= 1) {
    const float Mo = __shfl_xor_sync(0xFFFFFFFFu, A.M, off);
    const float lo = __shfl_xor_sync(0xFFFFFFFFu, A.l, off);
    const float Mn = fmaxf(A.M, Mo);
    const float f = (A.M == -INFINITY) ? 0.f : exp2f(A.M - Mn);
    const float fo = (Mo == -INFINITY) ? 0.f : exp2f(Mo - Mn);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 xl = make_float2(__shfl_xor_sync(0xFFFFFFFFu, A.ol[k].x, off),
                                    __shfl_xor_sync(0xFFFFFFFFu, A.ol[k].y, off));
      const float2 xh = make_float2(__shfl_xor_sync(0xFFFFFFFFu, A.oh[k].x, off),
                                    __shfl_xor_sync(0xFFFFFFFFu, A.oh[k].y, off));
      A.ol[k] = __ffma2_rn(A.ol[k], make_float2(f, f), __fmul2_rn(xl, make_float2(fo, fo)));
      A.oh[k] = __ffma2_rn(A.oh[k], make_float2(f, f), __fmul2_rn(xh, make_float2(fo, fo)));
    }
    A.l = A.l * f + lo * fo;
    A.M = Mn;
  }
  // per-warp partials in the (now idle) ring: [warp][130] = o[128], M, l
  __syncthreads();  // every warp is done with the ring
  float* wpart = reinterpret_cast<float*>(ring);
  if (lane < 8) {
    float* wp = wpart + warp * (kD + 2);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      reinterpret_cast<float2*>(wp + 8 * s)[k] = A.ol[k];
      reinterpret_cast<float2*>(wp + 64 + 8 * s)[k] = A.oh[k];
    }
    if (lane == 0) {
      wp[kD] = A.M;
      wp[kD + 1] = A.l;
    }
  }
  __syncthreads();
  if (*failed) return;  // uniform: every thread read the flag after the barrier

  // threads (request rr, channel ch) merge the 8 warps of their request
  const int rr = tid >> 7, ch = tid & 127;
  float Mr = -INFINITY, Lr = 0.f, o = 0.f;
  if (tid < 2 * kD) {
    for (int w = rr * 8; w < rr * 8 + 8; ++w) Mr = fmaxf(Mr, wpart[w * (kD + 2) + kD]);
    if (Mr != -INFINITY) {
      for (int w = rr * 8; w < rr * 8 + 8; ++w) {
        const float mw = wpart[w * (kD + 2) + kD];
        if (mw == -INFINITY) continue;
        const float f = exp2f(mw - Mr);
        Lr = fmaf(f, wpart[w * (kD + 2) + kD + 1], Lr);
        o = fmaf(f, wpart[w * (kD + 2) + ch], o);
      }
    }
  }

  if (a.n_split == 1) {
    if (tid < 2 * kD && rr < nreq) {
      const float val = (Lr > 0.f) ? o / Lr : 0.f;
      const size_t oi = ((size_t)(b0 + rr) * H + h) * kD + ch;
      if (a.out_fp32) reinterpret_cast<float*>(a.out)[oi] = val;
      else reinterpret_cast<uint16_t*>(a.out)[oi] = f32_to_bf16(val);
    }
    return;
  }

  // ---- split partial, then the last block of this (pair, head) merges -------------------
  if (tid < 2 * kD && rr < nreq) {
    float* pp = a.part + (((size_t)(b0 + rr) * H + h) * a.n_split + split) * (kD + 2);
    pp[2 + ch] = o;
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
  if (tid < 2 * kD && rr < nreq) {
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

int vq_attn_max_pages_per_split(int) { return 1 << 20; }  // one pass: no per-split storage

size_t vq_attn_smem_bytes(int, int) { return kSmemBytes; }

cudaError_t launch_vq_attn(const VqAttnArgs& a, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(vq_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)kD);
  dim3 grid(a.n_split, (a.B + 1) / 2, a.H);
  vq_attn_kernel<<<grid, kThreads, kSmemBytes, st>>>(a, scale_log2);
  return cudaGetLastError();
}

}  // namespace kvq
