// LoopVQ decode attention over the bf16 window and the 8-token index pages of one
// (layer, loop step), with an exact logsumexp merge of partial softmaxes.
//
// Follows "LoopVQ: Sub 1-bit KV Cache Quantization for Looped Transformers", method
// step 5, Algorithm 1 and Figure 5: the step's codebook slice B_t is staged in shared
// memory, keys and values are rebuilt from D/c indices per token, keys are rotated by
// RoPE and dotted with the query, the bf16 sink/recent tokens are attended directly, and
// the partial results are merged exactly (the Flash-Decoding merge the page builds on).
//
// GB300 design (differs from the page's Triton kernel, which gives every (request, head,
// split) its own program). On this GPU a codeword lookup costs shared-memory bandwidth and
// every key 6 FMAs per channel pair, so the work is bound on chip, not by HBM. Two kernels:
//
// vq_pages_kernel: persistent, one 512-thread block per SM. The work units (head, request
// pair, chunk of kVqChunk = 32 index pages), head-major, are cut into G equal contiguous
// shares, one per block, so every SM gets the same number of pages whatever the batch mix,
// and a block restages the codebook slices only when its share crosses into the next head
// (at most twice for the usual shapes).
//  * Both slices stay resident, staged by TMA bulk copies: keys in fp32 (128 KB; channels
//    0..63 and 64..127 as two [256][64] tables), values in fp16 as the cache stores them
//    ([256][128]; value rounding error ~1e-4 of the output). A codeword's shared-memory address
//    is one byte permute: (index << 8) | lane offset, and every lookup is a 128-bit load.
//  * The units stream through a 2-stage ring with TMA bulk copies: 32 key and 32 value
//    pages of each request, the two bf16 queries and a header naming the unit. A full
//    mbarrier per stage; the last warp to finish with a stage (a shared-memory arrival
//    counter) issues its refill. Every wait is bounded and reports a timeout through the
//    device error word instead of hanging.
//  * 8 lanes per page, lane s owns the RoPE partner groups s and s+8 (channels 8s..8s+7 and
//    64+8s..64+8s+7). The rotated query u = R(p_q - p) q satisfies <R(p_q) q, R(p) k> =
//    <u, k>, so keys are never rotated: u is built from the cos/sin table at a lane-group's
//    first page of a piece, advanced one position per token by R(-theta) and, from the last
//    token of a page to the first of the lane-group's next page (one unit, 256 positions,
//    later), by R(-249 theta), so a lane keeps a single copy of u; it is re-read from the
//    table every 64 units. Every score is one chain of packed FMAs. A transposing shuffle
//    reduction leaves lane s with the score of token s.
//  * One pass with an online softmax per lane-group; the 8 weights of a page are broadcast
//    by shuffles (as fp16) and each lane accumulates its 16 value channels from the fp16
//    table with the mixed-precision FMA (fp16 operands, fp32 sums: no conversions).
//  * At the end of each piece of a (pair, head) segment the lane-groups of a warp merge by
//    shuffles and every warp writes its partial (M, l, o) to the workspace (eight per
//    request), with no block-wide barrier.
//
// vq_window_kernel: one block (128 threads, or 512 for few long windows) per (request, head)
// attends the bf16 sink and recent tokens (one token per lane-group step, online softmax) and
// merges the result with the warp partials of every page piece of its segment, found from
// the same share arithmetic.
#include <cuda_fp16.h>

#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "../../include/kvq.h"

namespace kvq {
namespace {

constexpr int kThreads = kVqThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = kVqChunk;                          // pages of each request per unit
constexpr int kResync = 64;                               // units between cos/sin table reloads
constexpr int kJump = kChunk * kPage;                     // positions between a lane-group's pages
constexpr uint32_t kKSliceBytes = kCB * kD * 4;           // fp32 key codebook slice
constexpr uint32_t kVSliceBytes = kCB * kD * 2;           // fp16 value codebook slice
constexpr int kOffK = 0;                                  // shared-memory layout (bytes)
constexpr int kOffV = kOffK + kKSliceBytes;

// Ring and shared-memory layout for NG index groups per token (c = 128 / NG channels per
// codeword): a page is 8 NG bytes. NG = 32 (c = 4) keeps a single ring stage so that its
// 256-byte pages fit beside the two codebook slices; its refill still overlaps the unit's work
// because every thread copies what it needs from the stage to registers first.
template <int NG>
struct PageLay {
  static constexpr int kPageB = kPage * NG;
  static constexpr int kStg = (NG == 32) ? 1 : 2;
  static constexpr uint32_t kPart = kChunk * kPageB;           // one request's pages of one kind
  static constexpr uint32_t kOffHdr = 4 * kPart;               // unit header within a stage
  static constexpr uint32_t kOffQs = kOffHdr + 64;             // bf16 queries [2][128] within a stage
  static constexpr uint32_t kStageBytes = kOffQs + 2 * kD * 2 + 64;  // [K r0|K r1|V r0|V r1|hdr|q r0|q r1]
  static constexpr int kOffRing = kOffV + kVSliceBytes;
  static constexpr int kOffJ = kOffRing + kStg * kStageBytes;  // float4 [4][8 slots]: cos, sin(256 theta)
  static constexpr int kOffProd = kOffJ + 8 * 16 * 4;          // producer state (thread 0)
  static constexpr int kOffBar = kOffProd + 64;                // mbarriers + flags
  static constexpr int kSmemBytes = kOffBar + 128;
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kOffBar % 8 == 0 && kOffRing % 128 == 0 && kStageBytes % 128 == 0, "alignment");
};
constexpr int kMaxPairs = (int)(kVSliceBytes / 4) - 1;    // unit scan runs in the value-slice area

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
// acc += p * v for the two fp16 values of w (low half -> acc.x), p an fp16 in the low 16 bits
// of ph: the mixed-precision FMA takes fp16 operands and accumulates in fp32 (the product of
// two fp16 is exact in fp32), so a value row needs no separate conversion to fp32
__device__ __forceinline__ void fma_f16x2(float2& acc, uint32_t w, uint32_t ph) {
  asm("{\n\t.reg .b16 l, h, p;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.u16.u32 p, %3;\n\t"
      "fma.rn.f32.f16 %0, l, p, %0;\n\t"
      "fma.rn.f32.f16 %1, h, p, %1;\n\t}"
      : "+f"(acc.x), "+f"(acc.y)
      : "r"(w), "r"(ph));
}
// 8 consecutive fp16 values (one 128-bit shared load) into acc[0..3]
__device__ __forceinline__ void lds8_fp16_fma(const unsigned char* p, uint32_t ph, float2 (&acc)[4]) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  fma_f16x2(acc[0], w.x, ph);
  fma_f16x2(acc[1], w.y, ph);
  fma_f16x2(acc[2], w.z, ph);
  fma_f16x2(acc[3], w.w, ph);
}
// 4 consecutive fp16 values (one 64-bit shared load) into a0, a1
__device__ __forceinline__ void lds4_fp16_fma(const unsigned char* p, uint32_t ph, float2& a0, float2& a1) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  fma_f16x2(a0, w.x, ph);
  fma_f16x2(a1, w.y, ph);
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
                                        const float2 (&sn)[4]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 l = ul[k], hh = uh[k];
    ul[k] = __ffma2_rn(l, c[k], __fmul2_rn(hh, sn[k]));
    uh[k] = __ffma2_rn(make_float2(-l.x, -l.y), sn[k], __fmul2_rn(hh, c[k]));
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

// 8 consecutive bf16 values from shared memory in the lane's half order
__device__ __forceinline__ void lds8_bf16_perm(const uint16_t* p, int o0, float (&v)[8]) {
  const uint2 a = *reinterpret_cast<const uint2*>(p + o0);
  const uint2 b = *reinterpret_cast<const uint2*>(p + (4 - o0));
  v[0] = bf16_lo(a.x); v[1] = bf16_hi(a.x); v[2] = bf16_lo(a.y); v[3] = bf16_hi(a.y);
  v[4] = bf16_lo(b.x); v[5] = bf16_hi(b.x); v[6] = bf16_lo(b.y); v[7] = bf16_hi(b.y);
}

// A timed-out wait marks the block as failed; every later wait then returns at once, so a
// block that lost a copy finishes (with the error word set) instead of hanging.
__device__ __forceinline__ bool wait_stage(uint64_t* bar, uint32_t parity, volatile int* failed, int* err) {
  if (*failed) return false;
  if (mbar_wait_bounded(bar, parity)) return true;
  *failed = 1;
  set_error(err, KVQ_ERR_TIMEOUT);
  return false;
}

// Block-wide barrier on an mbarrier that every thread arrives on, with a bounded wait. Used
// inside the unit loop instead of __syncthreads so that a failed wait elsewhere can never
// leave threads parked at a barrier.
__device__ __forceinline__ void block_sync(uint64_t* bar, uint32_t& phase, volatile int* failed, int* err) {
  mbar_arrive(bar);
  wait_stage(bar, phase, failed, err);
  phase ^= 1u;
}

// running softmax state of one lane (the max is shared by its lane-group)
struct Acc {
  float M, l;
  float2 ol[4], oh[4];
};

__device__ __forceinline__ void acc_reset(Acc& A) {
  A.M = -INFINITY;
  A.l = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    A.ol[k] = make_float2(0.f, 0.f);
    A.oh[k] = make_float2(0.f, 0.f);
  }
}

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

// Merge the running states of the lane-groups 8 and 16 lanes apart (all lanes end with the
// merged state of their warp half pair, i.e. of the whole warp after both steps).
__device__ __forceinline__ void merge_lane_groups(Acc& A) {
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
}

// Lengths of request b, or zeros when b >= B or when they do not describe a valid cache
// (returns false then; the window kernel reports it).
__device__ __forceinline__ bool req_len(const VqAttnArgs& a, int b, int& L, int& NP) {
  L = 0;
  NP = 0;
  if (b >= a.B) return true;
  const int l = a.seq_len[b], np = a.n_pages[b];
  const bool ok = !(l < 0 || l > a.max_ctx || np < 0 || np > a.max_pages || (np > 0 && a.sink + kPage * np > l) ||
                    l - a.sink - kPage * np > a.recent + kPage);
  if (ok) {
    L = l;
    NP = np;
  }
  return ok;
}

__device__ __forceinline__ int pair_units(int NP0, int NP1) { return (max(NP0, NP1) + kChunk - 1) / kChunk; }

// share k of U units among G blocks starts at unit floor(k U / G)
__device__ __forceinline__ long long share_lo(long long U, int k, int G) { return U * k / G; }
// the block whose share holds unit u (0 <= u < U)
__device__ __forceinline__ int share_of(long long u, long long U, int G) { return (int)(((u + 1) * G - 1) / U); }

// header of a unit in its ring stage
struct UnitHdr {
  int h, pair, c, flags;   // flags: 1 first unit of a piece, 2 last unit, (dest << 2)
  int L0, NP0, L1, NP1;    // dest: 0 whole segment, 1 block's first piece, 2 block's last piece
};

// a position in a block's share of units
struct Walker {
  long long i;  // unit index
  int h, pair, c, nu;
  int L0, NP0, L1, NP1;
};

// producer state (used by whichever warp refills a stage), in shared memory so it costs the
// consumers no registers
struct ProdState {
  Walker cur;   // next unit to issue
  int issued;   // units issued by this block
  int k_loads;  // key-slice copies issued
  long long lo, hi;  // the block's share: read here by the refilling warp, so the consumers
                     // keep no registers for it
};
static_assert(sizeof(ProdState) <= 64, "producer state fits its shared-memory slot");

__device__ __forceinline__ void walker_load_pair(const VqAttnArgs& a, Walker& P) {
  req_len(a, 2 * P.pair, P.L0, P.NP0);
  req_len(a, 2 * P.pair + 1, P.L1, P.NP1);
  P.nu = pair_units(P.NP0, P.NP1);
}

// step to the next unit (the caller checks that one is left in the share), skipping request
// pairs without pages
__device__ __forceinline__ void walker_next(const VqAttnArgs& a, Walker& P, int n_pairs) {
  ++P.i;
  if (++P.c < P.nu) return;
  P.c = 0;
  do {
    if (++P.pair == n_pairs) {
      P.pair = 0;
      ++P.h;
    }
    walker_load_pair(a, P);
  } while (P.nu == 0 && P.h < a.H);
}

// Issue the next unit into its ring stage (header, index pages, queries) and step to the one
// after it.
template <int NG>
__device__ void prod_next(const VqAttnArgs& a, ProdState& S, unsigned char* ring, uint64_t* full, long long lo,
                          long long hi, int n_pairs) {
  using Ly = PageLay<NG>;
  Walker& P = S.cur;
  const int st = S.issued % Ly::kStg;
  unsigned char* dst = ring + st * Ly::kStageBytes;
  UnitHdr* hd = reinterpret_cast<UnitHdr*>(dst + Ly::kOffHdr);
  const long long seg0 = P.i - P.c, seg1 = seg0 + P.nu;
  int flags = 0;
  if (P.i == lo || P.c == 0) flags |= 1;
  if (P.i == hi - 1 || P.c == P.nu - 1) flags |= 2;
  const int dest = (seg0 >= lo && seg1 <= hi) ? 0 : (seg0 <= lo ? 1 : 2);
  hd->h = P.h;
  hd->pair = P.pair;
  hd->c = P.c;
  hd->flags = flags | (dest << 2);
  hd->L0 = P.L0;
  hd->NP0 = P.NP0;
  hd->L1 = P.L1;
  hd->NP1 = P.NP1;
  const int p_first = P.c * kChunk;
  const int n0 = min(kChunk, max(0, P.NP0 - p_first));
  const int n1 = min(kChunk, max(0, P.NP1 - p_first));
  const int b0 = 2 * P.pair;
  const bool two = b0 + 1 < a.B;
  // the header stores above are released to the consumers by this arrive
  mbar_arrive_expect_tx(&full[st], (uint32_t)(n0 + n1) * 2 * Ly::kPageB + (two ? 2u : 1u) * kD * 2);
  const size_t off = (size_t)p_first * Ly::kPageB;
  const size_t bh0 = ((size_t)b0 * a.H + P.h) * (size_t)a.max_pages * Ly::kPageB;
  if (n0 > 0) {
    bulk_g2s(dst, a.idx_k + bh0 + off, n0 * Ly::kPageB, &full[st]);
    bulk_g2s(dst + 2 * Ly::kPart, a.idx_v + bh0 + off, n0 * Ly::kPageB, &full[st]);
  }
  if (n1 > 0) {
    const size_t bh1 = ((size_t)(b0 + 1) * a.H + P.h) * (size_t)a.max_pages * Ly::kPageB;
    bulk_g2s(dst + Ly::kPart, a.idx_k + bh1 + off, n1 * Ly::kPageB, &full[st]);
    bulk_g2s(dst + 3 * Ly::kPart, a.idx_v + bh1 + off, n1 * Ly::kPageB, &full[st]);
  }
  bulk_g2s(dst + Ly::kOffQs, a.q + ((size_t)b0 * a.H + P.h) * kD, kD * 2, &full[st]);
  if (two) bulk_g2s(dst + Ly::kOffQs + kD * 2, a.q + ((size_t)(b0 + 1) * a.H + P.h) * kD, kD * 2, &full[st]);
  ++S.issued;
  if (P.i + 1 < hi) walker_next(a, P, n_pairs);
  else ++P.i;
}

template <int NG>
__global__ void __launch_bounds__(kThreads, 1) vq_pages_kernel(const VqAttnArgs a, const float scale_log2) {
  using Ly = PageLay<NG>;
  extern __shared__ __align__(128) unsigned char smem[];
  float* ks = reinterpret_cast<float*>(smem + kOffK);
  __half* vs = reinterpret_cast<__half*>(smem + kOffV);
  unsigned char* ring = smem + Ly::kOffRing;
  ProdState* ps = reinterpret_cast<ProdState*>(smem + Ly::kOffProd);
  uint64_t* kbar = reinterpret_cast<uint64_t*>(smem + Ly::kOffBar);
  uint64_t* full = kbar + 1;
  uint64_t* bsync = full + Ly::kStg;
  int* iflags = reinterpret_cast<int*>(bsync + 1);
  volatile int* failed = iflags;
  int* released = iflags + 1;  // [Ly::kStg]: warps done with the stage's current unit

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, blk = blockIdx.x;
  // let the window kernel launch now: its blocks take SMs as page blocks finish, attend
  // their window tokens and wait for this grid before they read the partials
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int n_pairs = (a.B + 1) / 2;

  // ---- units per request pair and their exclusive prefix (every block; block 0 publishes
  //      it for the window kernel). Runs in the value-slice area before the slice is staged.
  int* scan = reinterpret_cast<int*>(smem + kOffV);
  {
    int* wsum = reinterpret_cast<int*>(ring);
    for (int p = tid; p < n_pairs; p += kThreads) {
      int L0, NP0, L1, NP1;
      req_len(a, 2 * p, L0, NP0);
      req_len(a, 2 * p + 1, L1, NP1);
      scan[p] = pair_units(NP0, NP1);
    }
    __syncthreads();
    const int per = (n_pairs + kThreads - 1) / kThreads;
    const int beg = min(n_pairs, tid * per), end = min(n_pairs, beg + per);
    int local = 0;
    for (int p = beg; p < end; ++p) local += scan[p];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int run = incl - local;
    for (int w = 0; w < warp; ++w) run += wsum[w];
    for (int p = beg; p < end; ++p) {
      const int u = scan[p];
      scan[p] = run;
      run += u;
    }
    if (tid == kThreads - 1) scan[n_pairs] = run;  // the last thread ends on the total
    __syncthreads();
  }
  if (blk == 0)
    for (int p = tid; p <= n_pairs; p += kThreads) a.pref[p] = scan[p];
  const int Up = scan[n_pairs];
  const long long U = (long long)a.H * Up;
  const long long lo = share_lo(U, blk, G), hi = share_lo(U, blk + 1, G);
  if (lo >= hi) return;  // uniform: an empty share

  if (tid == 0) {
    mbar_init(kbar, 1);
#pragma unroll
    for (int s = 0; s < Ly::kStg; ++s) {
      mbar_init(&full[s], 1);
      released[s] = 0;
    }
    mbar_init(bsync, kThreads);
    *failed = 0;
    fence_mbar_init();
    // first unit of the share: head, then the last pair whose prefix is <= the remainder
    Walker& P = ps->cur;
    ps->issued = 0;
    ps->k_loads = 0;
    ps->lo = lo;
    ps->hi = hi;
    P.i = lo;
    P.h = (int)(lo / Up);
    const int rem = (int)(lo - (long long)P.h * Up);
    int pl = 0, ph = n_pairs - 1;
    while (pl < ph) {
      const int mid = (pl + ph + 1) >> 1;
      if (scan[mid] <= rem) pl = mid;
      else ph = mid - 1;
    }
    P.pair = pl;
    P.c = rem - scan[pl];
    walker_load_pair(a, P);
    // codebook slices of the (at most 4 first) heads of the share: HBM -> L2 now
    const int h_last = min((int)((hi - 1) / Up), P.h + 3);
    for (int hh = P.h; hh <= h_last; ++hh)
      for (int k = 0; k < 4; ++k) {
        bulk_prefetch_l2(a.bt_k + (size_t)hh * kCB * kD + k * (kCB * kD / 4), kKSliceBytes / 4);
        bulk_prefetch_l2(a.bt_v + (size_t)hh * kCB * kD + k * (kCB * kD / 4), kVSliceBytes / 4);
      }
  }
  if (tid < 8 && a.max_ctx > kJump) {
    // cos/sin((kJump - 7) theta_i) for slot tid in that slot's half order, stored [chunk][slot]
    // so that the 8 slots of a lane-group read 8 consecutive float4s (no bank conflicts): the
    // step from the last token of one of a lane-group's pages to the first of its next
    float4* jt = reinterpret_cast<float4*>(smem + Ly::kOffJ);
    const int jo0 = (tid & 4) ? 4 : 0;
    float c8[8], s8[8];
    ldg8_perm(a.rope_cos + (size_t)(kJump - 7) * (kD / 2) + 8 * tid, jo0, c8);
    ldg8_perm(a.rope_sin + (size_t)(kJump - 7) * (kD / 2) + 8 * tid, jo0, s8);
    jt[0 * 8 + tid] = make_float4(c8[0], c8[1], c8[2], c8[3]);
    jt[1 * 8 + tid] = make_float4(c8[4], c8[5], c8[6], c8[7]);
    jt[2 * 8 + tid] = make_float4(s8[0], s8[1], s8[2], s8[3]);
    jt[3 * 8 + tid] = make_float4(s8[4], s8[5], s8[6], s8[7]);
  }
  __syncthreads();  // barriers initialised, scan read by thread 0: the value area is free
  if (tid == 0)
    for (int s = 0; s < Ly::kStg && ps->cur.i < hi; ++s) prod_next<NG>(a, *ps, ring, full, lo, hi, n_pairs);

  const int s = tid & 7;                 // slot: groups s and s + 8
  const int o0 = (s & 4) ? 4 : 0;        // key half order (bank-quad spreading)
  const unsigned gmask = 0xFFu << (lane & 24);
  const int lg = tid >> 3;
  const int r = lg / kChunk, po = lg % kChunk;  // this lane-group's request and page slot

  float2 cth[4], sth[4];
  {
    float c8[8], s8[8];
    const int row = (a.max_ctx > 1) ? 1 : 0;
    ldg8_perm(a.rope_cos + (size_t)row * (kD / 2) + 8 * s, o0, c8);
    ldg8_perm(a.rope_sin + (size_t)row * (kD / 2) + 8 * s, o0, s8);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      cth[k] = make_float2(c8[2 * k], c8[2 * k + 1]);
      sth[k] = make_float2(s8[2 * k], s8[2 * k + 1]);
    }
  }
  // the lane-group's rotated query, advanced token by token through its pages
  float2 ulo[4], uhi[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    ulo[k] = make_float2(0.f, 0.f);
    uhi[k] = make_float2(0.f, 0.f);
  }
  Acc A;
  acc_reset(A);
  // lane byte offsets inside a 256-byte table row: key halves swapped for s >= 4 so the 8
  // lanes of a phase hit 8 bank quads; value lanes read 16 natural bytes each
  const uint32_t kb0 = 32 * s + 4 * o0, kb1 = kb0 ^ 16u;
  const uint32_t vb0 = 16 * s, vb1 = 128 + 16 * s;
  const unsigned char* ksb = reinterpret_cast<const unsigned char*>(ks);
  const unsigned char* vsb = reinterpret_cast<const unsigned char*>(vs);
  const float4* jt = reinterpret_cast<const float4*>(smem + Ly::kOffJ) + s;

  const int n_units = (int)(hi - lo);
  int cur_head = -1;
  uint32_t kphase = 0, sphase = 0;
  for (int i = 0; i < n_units; ++i) {
    const int st = i % Ly::kStg;
    wait_stage(&full[st], (i / Ly::kStg) & 1, failed, a.err);
    // ---- everything this thread needs from the stage goes to registers, then the stage is
    //      released: its refill overlaps this unit's work
    const unsigned char* stage = ring + st * Ly::kStageBytes;
    const int4 hv0 = *reinterpret_cast<const int4*>(stage + Ly::kOffHdr);
    const int4 hv1 = *reinterpret_cast<const int4*>(stage + Ly::kOffHdr + 16);
    const int uh = hv0.x, upair = hv0.y, uc = hv0.z, uflags = hv0.w;
    const int L = r ? hv1.z : hv1.x, NP = r ? hv1.w : hv1.y;
    const int pg = uc * kChunk + po;
    const bool active = !*failed && pg < NP;
    const bool resync = (uflags & 1) || uc % kResync == 0;
    // the lane's index words: 16 bytes (tokens 0..7 x lo/hi group) of its slot's row; with
    // c = 4 two slots (groups 2s and 2s + 1 of each half), the key row serving la first
    uint4 rowk = make_uint4(0, 0, 0, 0), rowv = rowk, rowk2 = rowk, rowv2 = rowk;
    float ql[8], qh[8];
    if (active) {
      const unsigned char* pk = stage + r * Ly::kPart + po * Ly::kPageB;
      const unsigned char* pv = stage + (2 + r) * Ly::kPart + po * Ly::kPageB;
      if constexpr (NG == 32) {
        rowk = *reinterpret_cast<const uint4*>(pk + 32 * s + 4 * o0);
        rowk2 = *reinterpret_cast<const uint4*>(pk + 32 * s + 16 - 4 * o0);
        rowv = *reinterpret_cast<const uint4*>(pv + 32 * s);
        rowv2 = *reinterpret_cast<const uint4*>(pv + 32 * s + 16);
      } else {
        constexpr int kSlotShift = (NG == 8) ? 1 : 0;  // c = 16: lanes 2p and 2p + 1 share slot p
        rowk = *reinterpret_cast<const uint4*>(pk + 16 * (s >> kSlotShift));
        rowv = *reinterpret_cast<const uint4*>(pv + 16 * (s >> kSlotShift));
      }
      if (resync) {
        const uint16_t* qr = reinterpret_cast<const uint16_t*>(stage + Ly::kOffQs) + r * kD;
        lds8_bf16_perm(qr + 8 * s, o0, ql);
        lds8_bf16_perm(qr + 64 + 8 * s, o0, qh);
      }
    }
    __syncwarp();
    if (lane == 0) {
      // the last warp done with this stage refills it with the unit Ly::kStg ahead: no warp
      // waits to produce, and the copy starts as soon as the stage is free
      if (atom_add_acq_rel_shared(&released[st], 1) == kWarps - 1) {
        released[st] = 0;
        if (!*failed && ps->cur.i < ps->hi) {
          fence_proxy_async_smem();
          prod_next<NG>(a, *ps, ring, full, ps->lo, ps->hi, n_pairs);
        }
      }
    }

    if (uh != cur_head) {  // uniform: every thread read the same header
      // ---- stage the codebook slices of head uh ----
      block_sync(bsync, sphase, failed, a.err);  // every warp is done with the old slices
      if (tid == 0 && !*failed) {  // both slices by TMA: fp32 keys 128 KB, fp16 values 64 KB
        const float* btk = a.bt_k + (size_t)uh * kCB * kD;
        const uint16_t* btv = a.bt_v + (size_t)uh * kCB * kD;
        mbar_arrive_expect_tx(kbar, kKSliceBytes + kVSliceBytes);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          bulk_g2s(ks + k * (kKSliceBytes / 16), btk + k * (kKSliceBytes / 16), kKSliceBytes / 4, kbar);
          bulk_g2s(vs + k * (kVSliceBytes / 8), btv + k * (kVSliceBytes / 8), kVSliceBytes / 4, kbar);
        }
        ++ps->k_loads;
      }
      wait_stage(kbar, kphase, failed, a.err);
      kphase ^= 1u;
      cur_head = uh;
    }
    if (uflags & 1) acc_reset(A);  // a new piece

    if (active) {
      if (resync) {  // u = R(p_q - p) q from the cos/sin table
        const int d = L - 1 - (a.sink + kPage * pg);
        float c8[8], s8[8];
        ldg8_perm(a.rope_cos + (size_t)d * (kD / 2) + 8 * s, o0, c8);
        ldg8_perm(a.rope_sin + (size_t)d * (kD / 2) + 8 * s, o0, s8);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          ulo[k] = make_float2(ql[2 * k] * c8[2 * k] - qh[2 * k] * s8[2 * k],
                                ql[2 * k + 1] * c8[2 * k + 1] - qh[2 * k + 1] * s8[2 * k + 1]);
          uhi[k] = make_float2(qh[2 * k] * c8[2 * k] + ql[2 * k] * s8[2 * k],
                                qh[2 * k + 1] * c8[2 * k + 1] + ql[2 * k + 1] * s8[2 * k + 1]);
        }
      } else {  // the next page: kJump - 7 positions after this lane-group's last token
        const float4 c0 = jt[0], c1 = jt[8], s0 = jt[16], s1 = jt[24];
        const float2 cj[4] = {make_float2(c0.x, c0.y), make_float2(c0.z, c0.w), make_float2(c1.x, c1.y),
                              make_float2(c1.z, c1.w)};
        const float2 sj[4] = {make_float2(s0.x, s0.y), make_float2(s0.z, s0.w), make_float2(s1.x, s1.y),
                              make_float2(s1.z, s1.w)};
        rotate8(ulo, uhi, cj, sj);
      }
      float part[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t wd = (j < 2) ? rowk.x : (j < 4) ? rowk.y : (j < 6) ? rowk.z : rowk.w;
        uint32_t wd2 = wd;  // c = 4: the index of the other 4 channels of each half
        if constexpr (NG == 32) wd2 = (j < 2) ? rowk2.x : (j < 4) ? rowk2.y : (j < 6) ? rowk2.z : rowk2.w;
        uint32_t al0, al1, ah0, ah1;
        if (j & 1) {
          al0 = row_off<2>(wd, kb0); al1 = row_off<2>(wd2, kb1);
          ah0 = row_off<3>(wd, kb0); ah1 = row_off<3>(wd2, kb1);
        } else {
          al0 = row_off<0>(wd, kb0); al1 = row_off<0>(wd2, kb1);
          ah0 = row_off<1>(wd, kb0); ah1 = row_off<1>(wd2, kb1);
        }
        const float4 la = *reinterpret_cast<const float4*>(ksb + al0);
        const float4 lb = *reinterpret_cast<const float4*>(ksb + al1);
        const float4 ha = *reinterpret_cast<const float4*>(ksb + kKSliceBytes / 2 + ah0);
        const float4 hb = *reinterpret_cast<const float4*>(ksb + kKSliceBytes / 2 + ah1);
        float2 acc = __fmul2_rn(ulo[0], make_float2(la.x, la.y));  // one chain: fewer live registers
        acc = __ffma2_rn(uhi[0], make_float2(ha.x, ha.y), acc);
        acc = __ffma2_rn(ulo[1], make_float2(la.z, la.w), acc);
        acc = __ffma2_rn(uhi[1], make_float2(ha.z, ha.w), acc);
        acc = __ffma2_rn(ulo[2], make_float2(lb.x, lb.y), acc);
        acc = __ffma2_rn(uhi[2], make_float2(hb.x, hb.y), acc);
        acc = __ffma2_rn(ulo[3], make_float2(lb.z, lb.w), acc);
        acc = __ffma2_rn(uhi[3], make_float2(hb.z, hb.w), acc);
        part[j] = acc.x + acc.y;
        if (j < 7) rotate8(ulo, uhi, cth, sth);  // next token: one position later
      }
      transpose_reduce8(part, s, gmask);
      const float p = online_weights(A, part[0] * scale_log2, gmask);
      // the weights enter the value sums rounded to fp16 (relative error 2^-12; the
      // normaliser l keeps the fp32 weights)
      const uint32_t ph = __half_as_ushort(__float2half_rn(p));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t pj = __shfl_sync(gmask, ph, (lane & 24) + j);
        const uint32_t wd = (j < 2) ? rowv.x : (j < 4) ? rowv.y : (j < 6) ? rowv.z : rowv.w;
        const uint32_t avl = (j & 1) ? row_off<2>(wd, vb0) : row_off<0>(wd, vb0);
        const uint32_t avh = (j & 1) ? row_off<3>(wd, vb1) : row_off<1>(wd, vb1);
        if constexpr (NG == 32) {  // channels 8s .. 8s + 3 and 8s + 4 .. 8s + 7 from two codewords
          const uint32_t wd2 = (j < 2) ? rowv2.x : (j < 4) ? rowv2.y : (j < 6) ? rowv2.z : rowv2.w;
          const uint32_t avl2 = (j & 1) ? row_off<2>(wd2, vb0 + 8) : row_off<0>(wd2, vb0 + 8);
          const uint32_t avh2 = (j & 1) ? row_off<3>(wd2, vb1 + 8) : row_off<1>(wd2, vb1 + 8);
          lds4_fp16_fma(vsb + avl, pj, A.ol[0], A.ol[1]);
          lds4_fp16_fma(vsb + avl2, pj, A.ol[2], A.ol[3]);
          lds4_fp16_fma(vsb + avh, pj, A.oh[0], A.oh[1]);
          lds4_fp16_fma(vsb + avh2, pj, A.oh[2], A.oh[3]);
        } else {
          lds8_fp16_fma(vsb + avl, pj, A.ol);
          lds8_fp16_fma(vsb + avh, pj, A.oh);
        }
      }
    }

    if (uflags & 2) {
      // ---- end of a piece: lanes of a group (l), lane-groups (shuffles); each warp writes
      //      its partial (M, l, o[128]) for the window kernel to merge
      A.l += __shfl_xor_sync(0xFFFFFFFFu, A.l, 1);
      A.l += __shfl_xor_sync(0xFFFFFFFFu, A.l, 2);
      A.l += __shfl_xor_sync(0xFFFFFFFFu, A.l, 4);
      merge_lane_groups(A);
      if (lane < 8 && 2 * upair + r < a.B) {
        const int dest = uflags >> 2;
        float* pp = (dest == 0) ? a.part_whole + ((size_t)uh * n_pairs + upair) * kVqPartFloats
                                : a.part_slot + ((size_t)blk * 2 + (dest - 1)) * kVqPartFloats;
        pp += (r * kVqWarpsPerReq + (warp - r * kVqWarpsPerReq)) * (kD + 2);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          reinterpret_cast<float2*>(pp + 2 + 8 * s)[k] = A.ol[k];
          reinterpret_cast<float2*>(pp + 2 + 64 + 8 * s)[k] = A.oh[k];
        }
        if (lane == 0) {
          pp[0] = A.M;
          pp[1] = A.l;
        }
      }
    }
  }

  __syncthreads();  // every producer step is done
  // after a timeout, let the block's own copies in flight land before it exits
  if (tid == 0 && *failed) {
    const int issued = ps->issued;
    for (int j = max(0, issued - Ly::kStg); j < issued; ++j) mbar_wait_bounded(&full[j % Ly::kStg], (j / Ly::kStg) & 1);
    if (ps->k_loads > 0) mbar_wait_bounded(kbar, (ps->k_loads - 1) & 1);
  }
}

// ------------------------------------------------------------------ window + merge kernel
// WT threads per block: 128 when the (request, head) blocks fill the GPU (7 resident per SM),
// 512 when there are no more blocks than SMs (long windows of few requests: 4 times the
// lane-groups per window, so a window's tokens take a quarter of the serial steps)
template <int WT>
__global__ void __launch_bounds__(WT, (WT == 128) ? 7 : 1) vq_window_kernel(const VqAttnArgs a, const float scale_log2) {
  __shared__ __align__(16) float qs[kD];
  __shared__ __align__(16) float wpart[WT / 32][kD + 2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / a.H, h = blockIdx.x - b * a.H;
  int L, NP;
  if (!req_len(a, b, L, NP) && h == 0 && tid == 0) set_error(a.err, KVQ_ERR_CAPACITY);
  if (tid < kD) qs[tid] = bf16_to_f32(a.q[((size_t)b * a.H + h) * kD + tid]);
  __syncthreads();

  // ---- bf16 window: lane-group g takes tokens g, g + 16, ... ----------------------------
  const int nsink = min(a.sink, L);
  const int nwin = (L > 0) ? nsink + max(0, L - a.sink - kPage * NP) : 0;
  const int s = lane & 7, g = tid >> 3;
  const unsigned gmask = 0xFFu << (lane & 24);
  const uint16_t* wk = a.win_k + ((size_t)b * a.H + h) * a.win_slots * kD;
  const uint16_t* wv = a.win_v + ((size_t)b * a.H + h) * a.win_slots * kD;
  Acc A;  // here l is the same in every lane of a lane-group
  acc_reset(A);
  for (int w = g; w < nwin; w += WT / 8) {
    const int p = (w < nsink) ? w : a.sink + kPage * NP + (w - nsink);
    const int slot = (p < a.sink) ? p : a.sink + (p - a.sink) % (a.recent + kPage);
    float kl[8], kh[8], vl[8], vh[8];
    ldg8_bf16_perm(wk + (size_t)slot * kD + 8 * s, 0, kl);
    ldg8_bf16_perm(wk + (size_t)slot * kD + 64 + 8 * s, 0, kh);
    ldg8_bf16_perm(wv + (size_t)slot * kD + 8 * s, 0, vl);
    ldg8_bf16_perm(wv + (size_t)slot * kD + 64 + 8 * s, 0, vh);
    float2 ul[4], uh[4];
    rotated_query(a.rope_cos, a.rope_sin, L - 1 - p, s, 0, qs, ul, uh);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      acc = __ffma2_rn(ul[k], make_float2(kl[2 * k], kl[2 * k + 1]), acc);
      acc = __ffma2_rn(uh[k], make_float2(kh[2 * k], kh[2 * k + 1]), acc);
    }
    float sc = acc.x + acc.y;
    sc += __shfl_xor_sync(gmask, sc, 4);
    sc += __shfl_xor_sync(gmask, sc, 2);
    sc += __shfl_xor_sync(gmask, sc, 1);
    sc *= scale_log2;
    if (sc > A.M) {
      const float f = (A.M == -INFINITY) ? 0.f : exp2f(A.M - sc);
      const float2 f2 = make_float2(f, f);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        A.ol[k] = __fmul2_rn(A.ol[k], f2);
        A.oh[k] = __fmul2_rn(A.oh[k], f2);
      }
      A.l *= f;
      A.M = sc;
    }
    const float pw = exp2f(sc - A.M);
    A.l += pw;
    const float2 p2 = make_float2(pw, pw);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      A.ol[k] = __ffma2_rn(p2, make_float2(vl[2 * k], vl[2 * k + 1]), A.ol[k]);
      A.oh[k] = __ffma2_rn(p2, make_float2(vh[2 * k], vh[2 * k + 1]), A.oh[k]);
    }
  }
  merge_lane_groups(A);
  if (lane < 8) {
    float* wp = wpart[warp];
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

  // ---- merge: window warps, then every page piece of the (pair, head) segment; a thread per
  //      channel ----------
  // the page kernel's prefix and partials: wait for that grid (a no-op without a
  // programmatic dependency)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid >= kD) return;
  const int ch = tid;
  float Mx = -INFINITY, Lt = 0.f, o = 0.f;
  auto fold = [&](float Mp, float lp, float op) {
    if (Mp == -INFINITY) return;
    const float Mn = fmaxf(Mx, Mp);
    const float f = (Mx == -INFINITY) ? 0.f : exp2f(Mx - Mn);
    const float fp = exp2f(Mp - Mn);
    Lt = Lt * f + lp * fp;
    o = o * f + op * fp;
    Mx = Mn;
  };
#pragma unroll
  for (int w = 0; w < WT / 32; ++w) fold(wpart[w][kD], wpart[w][kD + 1], wpart[w][ch]);
  const int n_pairs = (a.B + 1) / 2, pair = b >> 1, rr = b & 1;
  const int p0 = a.pref[pair], nu = a.pref[pair + 1] - p0;
  if (nu > 0) {
    const int Up = a.pref[n_pairs];
    const long long U = (long long)a.H * Up;
    const long long s0 = (long long)h * Up + p0, s1 = s0 + nu;
    const int k0 = share_of(s0, U, a.G), k1 = share_of(s1 - 1, U, a.G);
    auto fold_piece = [&](const float* pp) {  // the 8 warp partials of this request
      pp += rr * kVqWarpsPerReq * (kD + 2);
#pragma unroll
      for (int w = 0; w < kVqWarpsPerReq; ++w) fold(pp[w * (kD + 2)], pp[w * (kD + 2) + 1], pp[w * (kD + 2) + 2 + ch]);
    };
    if (k0 == k1) {
      fold_piece(a.part_whole + ((size_t)h * n_pairs + pair) * kVqPartFloats);
    } else {
      for (int kk = k0; kk <= k1; ++kk) {
        const long long lk = share_lo(U, kk, a.G);
        if (lk == share_lo(U, kk + 1, a.G)) continue;  // an empty share
        fold_piece(a.part_slot + ((size_t)kk * 2 + (lk >= s0 ? 0 : 1)) * kVqPartFloats);
      }
    }
  }
  const float val = (Lt > 0.f) ? o / Lt : 0.f;
  const size_t oi = ((size_t)b * a.H + h) * kD + ch;
  if (a.out_fp32) reinterpret_cast<float*>(a.out)[oi] = val;
  else reinterpret_cast<uint16_t*>(a.out)[oi] = f32_to_bf16(val);
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int device_sms() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

template <int NG>
cudaError_t launch_pages(const VqAttnArgs& a, float scale_log2, cudaStream_t st) {
  using Ly = PageLay<NG>;
  cudaError_t e = cudaFuncSetAttribute(vq_pages_kernel<NG>, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kSmemBytes);
  if (e != cudaSuccess) return e;
  vq_pages_kernel<NG><<<a.G, kThreads, Ly::kSmemBytes, st>>>(a, scale_log2);
  return cudaGetLastError();
}

}  // namespace

size_t vq_attn_ws_bytes(int B, int H, int G) {
  const size_t n_pairs = (size_t)(B + 1) / 2;
  return align256((n_pairs + 1) * sizeof(int32_t)) + align256((size_t)H * n_pairs * kVqPartFloats * sizeof(float)) +
         align256((size_t)G * 2 * kVqPartFloats * sizeof(float));
}

int vq_attn_max_pairs() { return kMaxPairs; }

cudaError_t launch_vq_attn(const VqAttnArgs& args, void* ws, cudaStream_t st) {
  VqAttnArgs a = args;
  const size_t n_pairs = (size_t)(a.B + 1) / 2;
  char* w = static_cast<char*>(ws);
  a.pref = reinterpret_cast<int32_t*>(w);
  w += align256((n_pairs + 1) * sizeof(int32_t));
  a.part_whole = reinterpret_cast<float*>(w);
  w += align256((size_t)a.H * n_pairs * kVqPartFloats * sizeof(float));
  a.part_slot = reinterpret_cast<float*>(w);
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)kD);
  cudaError_t e = cudaSuccess;
  switch (a.NG) {
    case 16: e = launch_pages<16>(a, scale_log2, st); break;
    case 8: e = launch_pages<8>(a, scale_log2, st); break;
    case 32: e = launch_pages<32>(a, scale_log2, st); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the window kernel may start before the page kernel ends
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)(a.B * a.H));
  const bool wide = a.B * a.H <= device_sms();
  lc.blockDim = dim3(wide ? 512 : 128);
  lc.dynamicSmemBytes = 0;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return wide ? cudaLaunchKernelEx(&lc, vq_window_kernel<512>, a, scale_log2)
              : cudaLaunchKernelEx(&lc, vq_window_kernel<128>, a, scale_log2);
}

}  // namespace kvq
