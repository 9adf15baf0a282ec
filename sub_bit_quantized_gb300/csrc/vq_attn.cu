// LoopVQ decode attention over the index pages and the bf16 window of one (layer, loop step),
// with an exact logsumexp merge of partial softmaxes.
//
// Follows "LoopVQ: Sub 1-bit KV Cache Quantization for Looped Transformers", method step 5,
// Algorithm 1 and Figure 5: keys and values are rebuilt from D/c indices per token through the
// step's codebook slice B_t, keys are rotated by RoPE and dotted with the query, the bf16
// sink/recent tokens are attended directly, and the partial results are merged exactly (the
// Flash-Decoding merge the page builds on).
//
// GB300 design (the page's kernel gives every (request, head, split) its own program and
// rebuilds value rows token by token). Here a codeword lookup costs shared-memory bandwidth
// and every key 4 FMAs per channel pair, so the work is bound on chip, not by HBM. One
// persistent launch, one block per SM; block k takes the k-th of G equal contiguous shares
// of all index pages (head-major segments of (head, request)). Warp roles:
//
//  * 16 compute warps, 16 lanes per index page (lane = RoPE slot s, channel quarter m:
//    channels 8s+4m..8s+4m+3 and their partners 64+8s+4m..), PPL consecutive pages per
//    16-lane group per work unit (4 with c = 8 or 16, 2 with c = 4). Pages are taken in
//    sub-pieces of at most 384 pages of one segment, in two passes:
//      pass 1 (keys): the key slice B_t stays resident in shared memory (fp32, two [256][64]
//      tables for the two RoPE halves); each lookup is one 128-bit load at (index << 8) | lane
//      offset. The rotated query u = R(p_q - p) q satisfies <R(p_q) q, R(p) k> = <u, k>, so
//      keys are never rotated: u is built from the cos/sin table at a sub-piece's first page,
//      advanced token by token with the three-term recurrence u' = 2 cos(theta) u - u_prev
//      (one FMA per component) and moved between units by one exact rotation. Scores go to a
//      shared buffer; the warps then agree on the sub-piece maximum M.
//      pass 2 (values): the re-association o_g = sum_j p_j B_V[g][idx_jg] = sum_r w[g][r]
//      B_V[g][r] with w[g][r] = sum of p_j over the tokens whose group-g index is r. Each
//      weight p_j = exp2(s_j - M) <= 1 is added as a fixed-point integer (2^-20 units) into a
//      per-(group, codeword) histogram with shared-memory integer atomics (native on this
//      GPU; float atomics are not), laid out [256][32 columns] so that the 32 lanes of every
//      atomic hit 32 different banks. A page's 8 weights reach its lanes through the score
//      buffer (two broadcast loads, not shuffles). No value row is read per token.
//  * 4 aux warps: for each sub-piece, w . B_V (the fp16 value slice, read from L2) gives the
//    sub-piece's partial (M, l, o); they merge it, and the window warps' partial of the
//    segment's bf16 window when the piece starts the segment, and write the output. A segment
//    shared with other blocks is merged by the last block to finish its part (a per-segment
//    counter in the workspace). Segments without index pages are attended by the aux warps
//    themselves, spread over the blocks.
//  * 3 window warps: they walk the block's pieces like the aux warps and attend the bf16
//    window (sink + recent tokens) of every segment whose first page this block holds, three
//    tokens per warp step, rotated query from the table, online softmax, in parallel with the
//    other roles; each window's rows go to the aux warps through a pair of mbarriers.
//  * 1 producer warp (one lane): TMA bulk copies of each unit's index pages (and the query)
//    into a ring of stages, and of the key slice whenever the share enters a new head; an L2
//    prefetch of each owned window's bf16 rows when the share reaches that segment.
//
// Every wait is an mbarrier wait with a time limit (the waiting warp suspends between polls);
// a timeout sets the device error word and a block-wide flag, after which every role leaves
// its loop.
#include <cuda_fp16.h>

#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "../../include/kvq.h"

namespace kvq {
namespace {

constexpr int kCW = kVqComputeWarps;                 // compute warps
constexpr int kAW = 4;                               // aux warps
constexpr int kWW = 3;                               // window warps
constexpr int kThreads = (kCW + kAW + 1 + kWW) * 32; // + one producer warp and the window warps
constexpr int kAuxT0 = kCW * 32;                     // first aux thread
constexpr int kAuxN = kAW * 32;
constexpr int kProdWarp = kCW + kAW;
constexpr int kWinW0 = kProdWarp + 1;                // first window warp
constexpr int kSubP = kVqSubPages;                   // pages per sub-piece
constexpr int kFixBits = 20;                         // fixed-point weight resolution 2^-20
// capacity: a bin sums at most kSubP * 8 weights of at most 2^20 each
static_assert((long long)kSubP * kPage * (1ll << kFixBits) < (1ll << 32), "fixed-point histogram fits 32 bits");
constexpr uint32_t kKSliceBytes = kCB * kD * 4;      // fp32 key slice (two [256][64] tables)
constexpr int kBinCols = 32;                         // histogram columns: copies x groups
constexpr int kBinBytes = kCB * kBinCols * 4;        // 32 KB
constexpr int kSbufBytes = kSubP * kPage * 4;        // scores of one sub-piece
static_assert(kVqMaxBatch + 1 <= kBinBytes / 4, "request prefix scan fits the histogram area");

// unit header flags
constexpr int kFV = 1;       // a value unit (pass 2), else a key unit (pass 1)
constexpr int kFFirst = 2;   // first unit of its sub-piece (of its kind)
constexpr int kFLast = 4;    // last unit of its sub-piece (of its kind)
constexpr int kFHeadEnd = 8; // last key unit of its head in this block's share
constexpr int kFPar = 16;    // sub-piece parity
constexpr int kFEnd = 32;    // no more units

template <int NG>
struct Lay {
  static constexpr int kPageB = kPage * NG;
  static constexpr int kPPL = (NG == 32) ? 2 : 4;              // consecutive pages per 16-lane group per unit
  static constexpr int kUP = 2 * kCW * kPPL;                   // pages per unit
  static constexpr int kJump = (kUP - kPPL) * kPage;           // a group's last token + 1 -> its first of the next unit
  static constexpr int kStg = (NG == 8) ? 4 : 2;
  static_assert(kSubP % kUP == 0, "a sub-piece is a whole number of units");
  static constexpr int kOffHdr = kUP * kPageB;                 // unit header within a stage
  static constexpr int kOffQ = kOffHdr + 64;                   // bf16 query within a stage
  static constexpr int kStageB = ((kOffQ + kD * 2) + 127) / 128 * 128;
  static constexpr int kOffK = 0;
  static constexpr int kOffBins = kOffK + (int)kKSliceBytes;
  static constexpr int kOffSbuf = kOffBins + kBinBytes;
  static constexpr int kOffRing = kOffSbuf + kSbufBytes;
  static constexpr int kOffJ = kOffRing + kStg * kStageB;       // cos, sin(kJump theta), cos, sin(theta) [4][64]
  static constexpr int kOffWm = kOffJ + 4 * 64 * 4;            // sub-piece maxima [2 parities][kCW]
  static constexpr int kOffWp = kOffWm + 2 * kCW * 4;          // aux window partials [kAW][132]
  static constexpr int kOffWw = kOffWp + kAW * 132 * 4;        // window-warp partials [kWW][132]
  static constexpr int kOffRed = kOffWw + kWW * 132 * 4;       // aux reduction [4][128] + [4] + flag
  static constexpr int kOffWalk = kOffRed + (4 * 128 + 8) * 4; // the share's first piece
  static constexpr int kOffBar = kOffWalk + 64;
  // full[kStg], empty[kStg], kbar, ktfree, maxbar, hfull, hfree, wfull, wfree, then flags
  static constexpr int kSmemBytes = kOffBar + (2 * kStg + 7) * 8 + 16;
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kOffRing % 128 == 0 && kStageB % 128 == 0 && kOffBar % 8 == 0 && kOffWalk % 16 == 0, "alignment");
};

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ void red_add_u32(uint32_t saddr, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(saddr), "r"(v) : "memory");
}

// byte offset (index << 8) | lane_byte, the index being byte K of w (lane_byte < 256)
template <int K>
__device__ __forceinline__ uint32_t row_off(uint32_t w, uint32_t lane_byte) {
  return __byte_perm(w, lane_byte, 0x5504u | (K << 4));
}

// u <- R(-a) u for 4 channel pairs held as 2 float2 per half: lo' = lo c + hi s, hi' = hi c - lo s
__device__ __forceinline__ void rotate4(float2 (&ul)[2], float2 (&uh)[2], const float2 (&c)[2], const float2 (&sn)[2]) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float2 l = ul[k], hh = uh[k];
    ul[k] = __ffma2_rn(l, c[k], __fmul2_rn(hh, sn[k]));
    uh[k] = __ffma2_rn(make_float2(-l.x, -l.y), sn[k], __fmul2_rn(hh, c[k]));
  }
}

__device__ __forceinline__ float4 ldg_f4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

// 4 bf16 (8 bytes) -> 4 floats
__device__ __forceinline__ void bf16x4(uint2 w, float (&v)[4]) {
  v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
}

// A timed-out wait marks the block as failed; every later wait then returns at once, so a
// block that lost a copy finishes (with the error word set) instead of hanging. Between polls
// the hardware may suspend the waiting warp.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* failed, int* err) {
  if (*failed) return false;
  if (mbar_wait_bounded_sleep(bar, parity)) return true;
  *failed = 1;
  set_error(err, KVQ_ERR_TIMEOUT);
  return false;
}

// true in every aux thread when it is true in any (a barrier over the aux warps): the aux warps
// take their exit decisions together, so none is left waiting at a named barrier
__device__ __forceinline__ bool aux_any(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p), "n"(kAuxN)
      : "memory");
  return r != 0;
}

// Lengths of request b, or zeros when b >= B or when they do not describe a valid cache
// (returns false then; block 0 reports it).
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

// share k of P page positions among G blocks starts at floor(k P / G)
__device__ __forceinline__ long long share_lo(long long P, int k, int G) { return P * k / G; }
// the block whose share holds position u (0 <= u < P)
__device__ __forceinline__ int share_of(long long u, long long P, int G) { return (int)(((u + 1) * G - 1) / P); }

// A position in a block's share, one (head, request) segment at a time.
struct Walk {
  long long pos;   // global page position of the piece's first page
  int h, b;        // segment
  int pa, pb;      // its pages [pa, pb) inside the share
  int L, np;       // request lengths
  int valid;
};
static_assert(sizeof(Walk) <= 64, "walk fits its shared-memory slot");

__device__ __forceinline__ void walk_next(const VqAttnArgs& a, Walk& W, long long hi) {
  W.pos += W.pb - W.pa;
  if (W.pos >= hi) {
    W.valid = 0;
    return;
  }
  do {
    if (++W.b == a.B) {
      W.b = 0;
      ++W.h;
    }
    req_len(a, W.b, W.L, W.np);
  } while (W.np == 0 && W.h < a.H);
  if (W.h >= a.H) {
    W.valid = 0;
    return;
  }
  W.pa = 0;
  W.pb = (int)min((long long)W.np, hi - W.pos);
}

// ------------------------------------------------------------------ pass 1: scores of one page
// Lane (s, m) of a 16-lane group: row = the 16-byte index row holding the lane's two groups for
// the page's 8 tokens (byte 2t: lo-half group, 2t + 1: hi-half group). (u, up) = the rotated
// query at the page's first token and one position earlier; each token advances them by the
// three-term recurrence u' = 2 cos(theta) u - up, one FMA per component (a rotation by -theta
// is a linear map whose two eigenvalues exp(-+i theta) sum to 2 cos theta). Returns the score of
// token s in lanes 2s and 2s + 1.
__device__ __forceinline__ float page_scores(const unsigned char* ksb, const uint4 row, const uint32_t lb,
                                             float2 (&ul)[2], float2 (&uh)[2], float2 (&pl)[2], float2 (&ph)[2],
                                             const float2 (&c2)[2], const int j, const unsigned gmask) {
  float part[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const uint32_t wd = (t < 2) ? row.x : (t < 4) ? row.y : (t < 6) ? row.z : row.w;
    const uint32_t al = (t & 1) ? row_off<2>(wd, lb) : row_off<0>(wd, lb);
    const uint32_t ah = (t & 1) ? row_off<3>(wd, lb) : row_off<1>(wd, lb);
    const float4 lo = *reinterpret_cast<const float4*>(ksb + al);
    const float4 hi = *reinterpret_cast<const float4*>(ksb + kKSliceBytes / 2 + ah);
    float2 acc = __fmul2_rn(ul[0], make_float2(lo.x, lo.y));
    acc = __ffma2_rn(uh[0], make_float2(hi.x, hi.y), acc);
    acc = __ffma2_rn(ul[1], make_float2(lo.z, lo.w), acc);
    acc = __ffma2_rn(uh[1], make_float2(hi.z, hi.w), acc);
    part[t] = acc.x + acc.y;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float2 nl = __ffma2_rn(c2[k], ul[k], make_float2(-pl[k].x, -pl[k].y));
      const float2 nh = __ffma2_rn(c2[k], uh[k], make_float2(-ph[k].x, -ph[k].y));
      pl[k] = ul[k];
      ph[k] = uh[k];
      ul[k] = nl;
      uh[k] = nh;
    }
  }
  // transposing reduction over the 16 lanes: after the xor-8/4/2 steps lane j holds token
  // j >> 1 summed over 8 lanes, the xor-1 step adds the other channel quarter
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const bool up = (j & 8) != 0;
    const float send = up ? part[k] : part[k + 4];
    const float keep = up ? part[k + 4] : part[k];
    part[k] = keep + __shfl_xor_sync(gmask, send, 8);
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const bool up = (j & 4) != 0;
    const float send = up ? part[k] : part[k + 2];
    const float keep = up ? part[k + 2] : part[k];
    part[k] = keep + __shfl_xor_sync(gmask, send, 4);
  }
  {
    const bool up = (j & 2) != 0;
    const float send = up ? part[0] : part[1];
    const float keep = up ? part[1] : part[0];
    part[0] = keep + __shfl_xor_sync(gmask, send, 2);
  }
  part[0] += __shfl_xor_sync(gmask, part[0], 1);
  return part[0];
}

// (x, y) -> R(a) (x, y) for the lane's 4 pairs: lo' = lo c - hi s, hi' = hi c + lo s
__device__ __forceinline__ void rotate_fwd(const float2 (&ul)[2], const float2 (&uh)[2], const float2 (&c)[2],
                                           const float2 (&sn)[2], float2 (&ol)[2], float2 (&oh)[2]) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    ol[k] = __ffma2_rn(ul[k], c[k], make_float2(-uh[k].x * sn[k].x, -uh[k].y * sn[k].y));
    oh[k] = __ffma2_rn(uh[k], c[k], __fmul2_rn(ul[k], sn[k]));
  }
}

// ------------------------------------------------------------------ pass 2: histogram of one page
// wt: the fixed-point weights of the page's 8 tokens. bins: shared address of the [256][32]
// u32 histogram. The lanes' columns make every red hit 32 distinct banks.
template <int NG>
__device__ __forceinline__ void page_hist(const uint4 row, const uint32_t (&wt)[8], const uint32_t bins, const int lane) {
  const int j = lane & 15, s = j >> 1, m = j & 1, half = lane >> 4;
  if constexpr (NG == 16) {
    // group s + 8m, column 16 half + s + 8m; token t's index: byte 2t + m of the row
    const uint32_t b0 = bins + (uint32_t)(16 * half + s + 8 * m) * 4;
    const uint32_t sh = 8u * m;
    const uint32_t rw[4] = {row.x >> sh, row.y >> sh, row.z >> sh, row.w >> sh};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint32_t r = (rw[t >> 1] >> (16 * (t & 1))) & 0xFFu;
      red_add_u32(b0 + (r << 7), wt[t]);
    }
  } else if constexpr (NG == 8) {
    // row s >> 1 holds groups s >> 1 (byte 2t) and (s >> 1) + 4 (byte 2t + 1); the lane takes
    // group (s >> 1) + 4m for tokens 4 (s & 1) .. 4 (s & 1) + 3; copy 2 half + (s & 1)
    const uint32_t b0 = bins + (uint32_t)(8 * (2 * half + (s & 1)) + (s >> 1) + 4 * m) * 4;
    const uint32_t sh = 8u * m;
    const uint32_t w0 = ((s & 1) ? row.z : row.x) >> sh, w1 = ((s & 1) ? row.w : row.y) >> sh;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const uint32_t r = (((t < 2) ? w0 : w1) >> (16 * (t & 1))) & 0xFFu;
      red_add_u32(b0 + (r << 7), (s & 1) ? wt[4 + t] : wt[t]);
    }
  } else {
    // NG == 32: row j holds groups j (byte 2t) and j + 16 (byte 2t + 1); page half 0 takes the
    // lo group first, half 1 the hi group first, so the two halves never share a column
    const uint32_t ga = (uint32_t)(j + 16 * half), gb = (uint32_t)(j + 16 * (1 - half));
    const uint32_t sa = 8u * half, sb = 8u * (1 - half);
    const uint32_t ra[4] = {row.x >> sa, row.y >> sa, row.z >> sa, row.w >> sa};
    const uint32_t rb[4] = {row.x >> sb, row.y >> sb, row.z >> sb, row.w >> sb};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint32_t r0 = (ra[t >> 1] >> (16 * (t & 1))) & 0xFFu;
      const uint32_t r1 = (rb[t >> 1] >> (16 * (t & 1))) & 0xFFu;
      red_add_u32(bins + ga * 4 + (r0 << 7), wt[t]);
      red_add_u32(bins + gb * 4 + (r1 << 7), wt[t]);
    }
  }
}

struct Bars {
  uint64_t *full, *empty, *kbar, *ktfree, *maxbar, *hfull, *hfree, *wfull, *wfree;
  volatile int* failed;
  int* flag;  // aux: last-contributor flag
};

// ------------------------------------------------------------------ compute warps
template <int NG>
__device__ void compute_role(const VqAttnArgs& a, unsigned char* smem, const Bars& B, const float scale_log2) {
  using Ly = Lay<NG>;
  constexpr int PPL = Ly::kPPL;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int half = lane >> 4, j = lane & 15, s = j >> 1, m = j & 1;
  const int pg0 = (warp * 2 + half) * PPL;  // this 16-lane group's first page of each unit
  const unsigned gmask = 0xFFFFu << (lane & 16);
  const int rowsel = (NG == 8) ? (s >> 1) : (NG == 16) ? s : j;
  const uint32_t lb = 32u * s + 16u * m;  // the lane's 4 channels in a 256-byte key-table row
  const int k0 = 8 * s + 4 * m;           // its first RoPE pair
  const unsigned char* ksb = smem + Ly::kOffK;
  float* sbuf = reinterpret_cast<float*>(smem + Ly::kOffSbuf);
  float* wm = reinterpret_cast<float*>(smem + Ly::kOffWm);
  const float* jt = reinterpret_cast<const float*>(smem + Ly::kOffJ);
  const unsigned char* ring = smem + Ly::kOffRing;
  const uint32_t bins = smem_u32(smem + Ly::kOffBins);

  float2 c2[2];  // 2 cos(theta) of the lane's pairs
  {
    const float4 c4 = *reinterpret_cast<const float4*>(jt + 128 + k0);
    c2[0] = make_float2(2.f * c4.x, 2.f * c4.y);
    c2[1] = make_float2(2.f * c4.z, 2.f * c4.w);
  }
  // rotated query at the group's current token (u) and one position earlier (p)
  float2 ul[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)}, uh[2] = {ul[0], ul[1]};
  float2 pl[2] = {ul[0], ul[1]}, ph[2] = {ul[0], ul[1]};
  float wmax = -INFINITY, M = 0.f;
  int cur_h = -1;
  uint32_t kph = 0, mph = 0, hfph = 1;

  for (int i = 0;; ++i) {
    const int st = i % Ly::kStg;
    if (!__all_sync(0xFFFFFFFFu, wait_bar(&B.full[st], (i / Ly::kStg) & 1, B.failed, a.err))) break;
    const unsigned char* stage = ring + st * Ly::kStageB;
    const int4 h0 = *reinterpret_cast<const int4*>(stage + Ly::kOffHdr);
    const int4 h1 = *reinterpret_cast<const int4*>(stage + Ly::kOffHdr + 16);
    const int flags = h0.x;
    if (flags & kFEnd) break;
    const int uh_ = h0.y, p0 = h0.w, npg = h1.x, L = h1.y, usub = h1.z;
    uint4 rows[PPL];
#pragma unroll
    for (int pp = 0; pp < PPL; ++pp)
      rows[pp] = (pg0 + pp < npg) ? *reinterpret_cast<const uint4*>(stage + (pg0 + pp) * Ly::kPageB + 16 * rowsel)
                                  : make_uint4(0, 0, 0, 0);
    const bool kunit = !(flags & kFV);
    const bool act = pg0 < npg;
    float ql[4], qh[4];
    if (kunit && (flags & kFFirst) && act) {
      const uint16_t* qs = reinterpret_cast<const uint16_t*>(stage + Ly::kOffQ);
      bf16x4(*reinterpret_cast<const uint2*>(qs + k0), ql);
      bf16x4(*reinterpret_cast<const uint2*>(qs + 64 + k0), qh);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&B.empty[st]);  // the stage is no longer needed: refill it
    const int par = (flags & kFPar) ? 1 : 0;
    float* sp = sbuf + (usub * Ly::kUP + pg0) * kPage;

    if (kunit) {
      if (uh_ != cur_h) {  // the producer staged this head's key slice
        if (!__all_sync(0xFFFFFFFFu, wait_bar(B.kbar, kph, B.failed, a.err))) break;
        kph ^= 1u;
        cur_h = uh_;
      }
      if (flags & kFFirst) wmax = -INFINITY;
      if (act) {
        if (flags & kFFirst) {  // u = R(p_q - p) q from the cos/sin table at the group's first token
          const int d = L - 1 - (a.sink + kPage * (p0 + pg0));
          const float4 c4 = ldg_f4(a.rope_cos + (size_t)d * (kD / 2) + k0);
          const float4 s4 = ldg_f4(a.rope_sin + (size_t)d * (kD / 2) + k0);
          const float c[4] = {c4.x, c4.y, c4.z, c4.w}, sn[4] = {s4.x, s4.y, s4.z, s4.w};
          ul[0] = make_float2(ql[0] * c[0] - qh[0] * sn[0], ql[1] * c[1] - qh[1] * sn[1]);
          ul[1] = make_float2(ql[2] * c[2] - qh[2] * sn[2], ql[3] * c[3] - qh[3] * sn[3]);
          uh[0] = make_float2(qh[0] * c[0] + ql[0] * sn[0], qh[1] * c[1] + ql[1] * sn[1]);
          uh[1] = make_float2(qh[2] * c[2] + ql[2] * sn[2], qh[3] * c[3] + ql[3] * sn[3]);
        } else {  // one exact rotation over the other groups' pages of the last unit
          const float4 jc = *reinterpret_cast<const float4*>(jt + k0);
          const float4 js = *reinterpret_cast<const float4*>(jt + 64 + k0);
          const float2 cj[2] = {make_float2(jc.x, jc.y), make_float2(jc.z, jc.w)};
          const float2 sj[2] = {make_float2(js.x, js.y), make_float2(js.z, js.w)};
          rotate4(ul, uh, cj, sj);
        }
        {  // the recurrence restarts from an exact pair: p = R(theta) u
          const float4 tc = *reinterpret_cast<const float4*>(jt + 128 + k0);
          const float4 ts = *reinterpret_cast<const float4*>(jt + 192 + k0);
          const float2 cth[2] = {make_float2(tc.x, tc.y), make_float2(tc.z, tc.w)};
          const float2 sth[2] = {make_float2(ts.x, ts.y), make_float2(ts.z, ts.w)};
          rotate_fwd(ul, uh, cth, sth, pl, ph);
        }
#pragma unroll
        for (int pp = 0; pp < PPL; ++pp) {
          if (pg0 + pp < npg) {
            const float sc = page_scores(ksb, rows[pp], lb, ul, uh, pl, ph, c2, j, gmask) * scale_log2;
            if (m == 0) sp[pp * kPage + s] = sc;
            wmax = fmaxf(wmax, sc);
          }
        }
      }
      if (flags & kFLast) {  // the warp's maximum over the sub-piece
        float x = wmax;
        x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, 16));
        x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, 8));
        x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, 4));
        x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, 2));
        x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, 1));
        if (lane == 0) {
          wm[par * kCW + warp] = x;
          mbar_arrive(B.maxbar);
        }
      }
      if (flags & kFHeadEnd) {
        __syncwarp();
        if (lane == 0) mbar_arrive(B.ktfree);  // done with this head's key slice
      }
    } else {
      if (flags & kFFirst) {
        if (!__all_sync(0xFFFFFFFFu, wait_bar(B.maxbar, mph, B.failed, a.err))) break;
        mph ^= 1u;
        const float4* w4 = reinterpret_cast<const float4*>(wm + par * kCW);
        float x = -INFINITY;
#pragma unroll
        for (int k = 0; k < kCW / 4; ++k) {
          const float4 v = w4[k];
          x = fmaxf(fmaxf(x, v.x), fmaxf(v.y, fmaxf(v.z, v.w)));
        }
        M = x;
        // the aux warps cleared the histogram
        if (!__all_sync(0xFFFFFFFFu, wait_bar(B.hfree, hfph, B.failed, a.err))) break;
        hfph ^= 1u;
      }
      // p = exp2(s - M) <= 1 in units of 2^-20: p + 8 has an ulp of 2^-20, so its mantissa is
      // round(p 2^20) (nearest, ties to even); lanes 2t write token t's weight over its score
#pragma unroll
      for (int pp = 0; pp < PPL; ++pp) {
        if (pg0 + pp < npg && m == 0) {
          const float p = exp2f(sp[pp * kPage + s] - M);
          reinterpret_cast<uint32_t*>(sp)[pp * kPage + s] = __float_as_uint(p + 8.0f) - 0x41000000u;
        }
      }
      __syncwarp();
#pragma unroll
      for (int pp = 0; pp < PPL; ++pp) {
        if (pg0 + pp < npg) {  // the page's 8 weights: two 16-byte reads every lane of the page shares
          const uint4 w03 = *reinterpret_cast<const uint4*>(sp + pp * kPage);
          const uint4 w47 = *reinterpret_cast<const uint4*>(sp + pp * kPage + 4);
          const uint32_t wt[8] = {w03.x, w03.y, w03.z, w03.w, w47.x, w47.y, w47.z, w47.w};
          page_hist<NG>(rows[pp], wt, bins, lane);
        }
      }
      if (flags & kFLast) {
        __syncwarp();
        if (lane == 0) mbar_arrive(B.hfull);
      }
    }
  }
}

// ------------------------------------------------------------------ producer (one lane)
template <int NG>
__device__ void producer_role(const VqAttnArgs& a, unsigned char* smem, const Bars& B, Walk W, const long long hi,
                              int& issued, int& k_loads) {
  using Ly = Lay<NG>;
  unsigned char* ring = smem + Ly::kOffRing;
  int cur_h = -1, sub_par = 0;
  uint32_t ktf = 0;
  while (W.valid) {
    Walk nx = W;
    walk_next(a, nx, hi);
    if (W.h != cur_h) {
      if (cur_h >= 0) {  // every compute warp is done with the previous head's slice
        if (!wait_bar(B.ktfree, ktf, B.failed, a.err)) return;
        ktf ^= 1u;
      }
      fence_proxy_async_smem();
      const float* btk = a.bt_k + (size_t)W.h * kCB * kD;
      mbar_arrive_expect_tx(B.kbar, kKSliceBytes);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        bulk_g2s(smem + Ly::kOffK + k * (kKSliceBytes / 4), btk + k * (kKSliceBytes / 16), kKSliceBytes / 4, B.kbar);
      ++k_loads;
      cur_h = W.h;
    }
    const size_t seg = ((size_t)W.b * a.H + W.h) * (size_t)a.max_pages;
    if (W.pa == 0) {  // this block attends the segment's bf16 window (aux warps): HBM -> L2 now
      const size_t wo = ((size_t)W.b * a.H + W.h) * a.win_slots * kD;
      bulk_prefetch_l2(a.win_k + wo, (uint32_t)a.win_slots * kD * 2);
      bulk_prefetch_l2(a.win_v + wo, (uint32_t)a.win_slots * kD * 2);
    }
    for (int sa = W.pa; sa < W.pb; sa += kSubP) {
      const int sb = min(sa + kSubP, W.pb), nu = (sb - sa + Ly::kUP - 1) / Ly::kUP;
      const bool head_end = (sb == W.pb) && (!nx.valid || nx.h != W.h);
      for (int kind = 0; kind < 2; ++kind)
        for (int u = 0; u < nu; ++u) {
          const int st = issued % Ly::kStg;
          if (!wait_bar(&B.empty[st], ((issued / Ly::kStg) & 1) ^ 1, B.failed, a.err)) return;
          fence_proxy_async_smem();
          unsigned char* dst = ring + st * Ly::kStageB;
          const int p0 = sa + u * Ly::kUP, npg = min(Ly::kUP, sb - p0);
          int flags = (kind ? kFV : 0) | (u == 0 ? kFFirst : 0) | (u == nu - 1 ? kFLast : 0) | (sub_par ? kFPar : 0);
          if (!kind && u == nu - 1 && head_end) flags |= kFHeadEnd;
          int4* hd = reinterpret_cast<int4*>(dst + Ly::kOffHdr);
          hd[0] = make_int4(flags, W.h, W.b, p0);
          hd[1] = make_int4(npg, W.L, u, 0);
          const uint32_t pb = (uint32_t)npg * Ly::kPageB;
          mbar_arrive_expect_tx(&B.full[st], pb + (kind ? 0u : (uint32_t)kD * 2));
          bulk_g2s(dst, (kind ? a.idx_v : a.idx_k) + (seg + p0) * Ly::kPageB, pb, &B.full[st]);
          if (!kind) bulk_g2s(dst + Ly::kOffQ, a.q + ((size_t)W.b * a.H + W.h) * kD, kD * 2, &B.full[st]);
          ++issued;
        }
      sub_par ^= 1;
    }
    W = nx;
  }
  const int st = issued % Ly::kStg;  // end marker: a header only
  if (!wait_bar(&B.empty[st], ((issued / Ly::kStg) & 1) ^ 1, B.failed, a.err)) return;
  int4* hd = reinterpret_cast<int4*>(ring + st * Ly::kStageB + Ly::kOffHdr);
  hd[0] = make_int4(kFEnd, 0, 0, 0);
  mbar_arrive(&B.full[st]);
  ++issued;
}

// ------------------------------------------------------------------ aux warps
__device__ __forceinline__ void aux_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kAuxN) : "memory"); }

// merge (Mp, lp, op) into (M, l, o) (log2 domain)
__device__ __forceinline__ void merge_part(float& M, float& l, float& o, float Mp, float lp, float op) {
  if (Mp == -INFINITY) return;
  const float Mn = fmaxf(M, Mp);
  const float f = (M == -INFINITY) ? 0.f : exp2f(M - Mn);
  const float fp = exp2f(Mp - Mn);
  l = l * f + lp * fp;
  o = o * f + op * fp;
  M = Mn;
}

// bf16 sink and recent tokens of segment (h, b): NW warps, warp wi taking every NW-th token
// from wi, kTW tokens per step; lane l holds channels 2l, 2l+1 and their RoPE partners.
// Writes the warp's partial to its row of `rows` ([0] M, [1] l, [4 + ch] channel ch; 132
// floats a row).
template <int NW, int kTW>
__device__ void win_attend(const VqAttnArgs& a, int h, int b, int L, int NP, float scale_log2, float* rows, int wi,
                           int lane) {
  const int nsink = min(a.sink, L);
  const int nwin = (L > 0) ? nsink + max(0, L - a.sink - kPage * NP) : 0;
  const size_t bh = (size_t)b * a.H + h;
  const uint32_t qa = __ldg(reinterpret_cast<const uint32_t*>(a.q + bh * kD + 2 * lane));
  const uint32_t qb = __ldg(reinterpret_cast<const uint32_t*>(a.q + bh * kD + 64 + 2 * lane));
  const float q0 = bf16_lo(qa), q1 = bf16_hi(qa), q2 = bf16_lo(qb), q3 = bf16_hi(qb);
  const uint16_t* wk = a.win_k + bh * a.win_slots * kD;
  const uint16_t* wv = a.win_v + bh * a.win_slots * kD;
  float M = -INFINITY, l = 0.f, o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
  // kTW tokens per step (w, w + NW, ...): their key and RoPE loads issued together, the
  // value loads issued after the dot products (in flight during the interleaved reductions),
  // one running-maximum update per step
  for (int w = wi; w < nwin; w += kTW * NW) {
    int slot[kTW];
    float sc[kTW];
    {
      uint32_t ka[kTW], kb[kTW];
      float2 c[kTW], sn[kTW];
#pragma unroll
      for (int e = 0; e < kTW; ++e) {
        const int we = min(w + e * NW, nwin - 1);  // a missing token reloads the last one
        const int p = (we < nsink) ? we : a.sink + kPage * NP + (we - nsink);
        slot[e] = (p < a.sink) ? p : a.sink + (p - a.sink) % (a.recent + kPage);
        ka[e] = __ldg(reinterpret_cast<const uint32_t*>(wk + (size_t)slot[e] * kD + 2 * lane));
        kb[e] = __ldg(reinterpret_cast<const uint32_t*>(wk + (size_t)slot[e] * kD + 64 + 2 * lane));
        const int d = L - 1 - p;
        c[e] = __ldg(reinterpret_cast<const float2*>(a.rope_cos + (size_t)d * (kD / 2) + 2 * lane));
        sn[e] = __ldg(reinterpret_cast<const float2*>(a.rope_sin + (size_t)d * (kD / 2) + 2 * lane));
      }
#pragma unroll
      for (int e = 0; e < kTW; ++e) {
        const float u0 = q0 * c[e].x - q2 * sn[e].x, u2 = q2 * c[e].x + q0 * sn[e].x;
        const float u1 = q1 * c[e].y - q3 * sn[e].y, u3 = q3 * c[e].y + q1 * sn[e].y;
        sc[e] = u0 * bf16_lo(ka[e]) + u1 * bf16_hi(ka[e]) + u2 * bf16_lo(kb[e]) + u3 * bf16_hi(kb[e]);
      }
    }
    uint32_t va[kTW], vb[kTW];
#pragma unroll
    for (int e = 0; e < kTW; ++e) {
      va[e] = __ldg(reinterpret_cast<const uint32_t*>(wv + (size_t)slot[e] * kD + 2 * lane));
      vb[e] = __ldg(reinterpret_cast<const uint32_t*>(wv + (size_t)slot[e] * kD + 64 + 2 * lane));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int e = 0; e < kTW; ++e) sc[e] += __shfl_xor_sync(0xFFFFFFFFu, sc[e], o);
    float mx = -INFINITY;
#pragma unroll
    for (int e = 0; e < kTW; ++e) {  // tokens past the window's end drop out (uniform across the warp)
      sc[e] = (w + e * NW < nwin) ? sc[e] * scale_log2 : -INFINITY;
      mx = fmaxf(mx, sc[e]);
    }
    if (mx > M) {
      const float f = (M == -INFINITY) ? 0.f : exp2f(M - mx);
      l *= f; o0 *= f; o1 *= f; o2 *= f; o3 *= f;
      M = mx;
    }
#pragma unroll
    for (int e = 0; e < kTW; ++e) {
      const float pw = exp2f(sc[e] - M);  // 0 for a dropped token
      l += pw;
      o0 += pw * bf16_lo(va[e]); o1 += pw * bf16_hi(va[e]); o2 += pw * bf16_lo(vb[e]); o3 += pw * bf16_hi(vb[e]);
    }
  }
  float* mine = rows + wi * 132;
  mine[4 + 2 * lane] = o0; mine[5 + 2 * lane] = o1; mine[68 + 2 * lane] = o2; mine[69 + 2 * lane] = o3;
  if (lane == 0) { mine[0] = M; mine[1] = l; }
}

// the NW rows' partials merged for channel ch
template <int NW>
__device__ __forceinline__ void win_merge(const float* rows, int ch, float& Mo, float& lo_, float& oo) {
  Mo = -INFINITY; lo_ = 0.f; oo = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) merge_part(Mo, lo_, oo, rows[w * 132], rows[w * 132 + 1], rows[w * 132 + 4 + ch]);
}

// the window of a segment without index pages, attended by the 4 aux warps themselves
__device__ void aux_window(const VqAttnArgs& a, int h, int b, int L, int NP, float scale_log2, float* wp, int at,
                           float& Mo, float& lo_, float& oo) {
  win_attend<kAW, 3>(a, h, b, L, NP, scale_log2, wp, at >> 5, at & 31);
  aux_sync();
  win_merge<kAW>(wp, at, Mo, lo_, oo);
  aux_sync();  // before the partial area is reused
}

// histogram of a finished sub-piece -> its partial (Ms, ls, os[at]); clears the histogram
template <int NG>
__device__ void aux_finalize(const VqAttnArgs& a, unsigned char* smem, int h, int par, int at, float& Ms, float& ls,
                             float& os) {
  using Ly = Lay<NG>;
  constexpr int kCopies = kBinCols / NG, kCh = kD / NG;  // histogram copies, channels per group
  const uint32_t* bins = reinterpret_cast<const uint32_t*>(smem + Ly::kOffBins);
  float* red = reinterpret_cast<float*>(smem + Ly::kOffRed);
  uint32_t* lred = reinterpret_cast<uint32_t*>(red + 4 * 128);
  const float* wm = reinterpret_cast<const float*>(smem + Ly::kOffWm) + par * kCW;
  Ms = wm[0];
#pragma unroll
  for (int w = 1; w < kCW; ++w) Ms = fmaxf(Ms, wm[w]);
  const int cq = at & 31, rq = at >> 5;  // channels 4 cq .. 4 cq + 3, codewords 64 rq .. 64 rq + 63
  const int g = (4 * cq) / kCh;
  const uint16_t* E = a.bt_v + (size_t)h * kCB * kD + 4 * cq;
  float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
  uint32_t lsum = 0;
#pragma unroll 16
  for (int r = 64 * rq; r < 64 * rq + 64; ++r) {
    uint32_t bs = 0;
#pragma unroll
    for (int c = 0; c < kCopies; ++c) bs += bins[r * kBinCols + c * NG + g];
    const uint2 e = __ldg(reinterpret_cast<const uint2*>(E + (size_t)r * kD));
    const float f = (float)bs;
    const float2 e01 = __half22float2(*reinterpret_cast<const __half2*>(&e.x));
    const float2 e23 = __half22float2(*reinterpret_cast<const __half2*>(&e.y));
    acc0 = fmaf(f, e01.x, acc0); acc1 = fmaf(f, e01.y, acc1); acc2 = fmaf(f, e23.x, acc2); acc3 = fmaf(f, e23.y, acc3);
    lsum += bs;
  }
  *reinterpret_cast<float4*>(red + rq * 128 + 4 * cq) = make_float4(acc0, acc1, acc2, acc3);
  if (cq == 0) lred[rq] = lsum;  // group 0: every token once
  aux_sync();
  const float inv = 1.f / (float)(1u << kFixBits);
  os = (red[at] + red[128 + at] + red[256 + at] + red[384 + at]) * inv;
  ls = (float)(lred[0] + lred[1] + lred[2] + lred[3]) * inv;
  uint4* bz = reinterpret_cast<uint4*>(smem + Ly::kOffBins) + at;
#pragma unroll
  for (int k = 0; k < kBinBytes / 16 / kAuxN; ++k) bz[k * kAuxN] = make_uint4(0, 0, 0, 0);
}

// the segment's result from this block: the output itself when no other block holds part of
// the segment, else a slot partial (and the merge, by the last contributor)
__device__ void aux_emit(const VqAttnArgs& a, unsigned char* flag_smem, int h, int b, long long Ps, int np,
                         long long Ptot, int blk, int at, float M, float l, float o) {
  int k0 = 0, k1 = 0, count = 1;
  if (np > 0) {
    k0 = share_of(Ps, Ptot, a.G);
    k1 = share_of(Ps + np - 1, Ptot, a.G);
    count = 0;
    for (int k = k0; k <= k1; ++k) count += share_lo(Ptot, k + 1, a.G) > share_lo(Ptot, k, a.G);
  }
  const size_t oi = ((size_t)b * a.H + h) * kD + at;
  if (count <= 1) {
    const float val = (l > 0.f) ? o / l : 0.f;
    if (a.out_fp32) reinterpret_cast<float*>(a.out)[oi] = val;
    else reinterpret_cast<uint16_t*>(a.out)[oi] = f32_to_bf16(val);
    return;
  }
  volatile int* flag = reinterpret_cast<volatile int*>(flag_smem);
  float* sp = a.slots + ((size_t)blk * 2 + (blk == k0 ? 1 : 0)) * kVqSlotFloats;
  sp[4 + at] = o;
  if (at == 0) { sp[0] = M; sp[1] = l; }
  __threadfence();
  aux_sync();
  if (at == 0) {
    const int old = atomicAdd(a.cnt + (size_t)h * a.B + b, 1);
    *flag = (old == count - 1);
  }
  aux_sync();
  if (*flag) {
    __threadfence();
    float Mx = -INFINITY, Lt = 0.f, ox = 0.f;
    for (int k = k0; k <= k1; ++k) {
      if (share_lo(Ptot, k + 1, a.G) == share_lo(Ptot, k, a.G)) continue;
      const float* pp = a.slots + ((size_t)k * 2 + (k == k0 ? 1 : 0)) * kVqSlotFloats;
      merge_part(Mx, Lt, ox, __ldcg(pp), __ldcg(pp + 1), __ldcg(pp + 4 + at));
    }
    const float val = (Lt > 0.f) ? ox / Lt : 0.f;
    if (a.out_fp32) reinterpret_cast<float*>(a.out)[oi] = val;
    else reinterpret_cast<uint16_t*>(a.out)[oi] = f32_to_bf16(val);
    if (at == 0) a.cnt[(size_t)h * a.B + b] = 0;  // ready for the next call
  }
  aux_sync();  // before the flag is reused
}

template <int NG>
__device__ void aux_role(const VqAttnArgs& a, unsigned char* smem, const Bars& B, Walk W, const long long hi,
                         const long long Ptot, const float scale_log2) {
  using Ly = Lay<NG>;
  const int at = threadIdx.x - kAuxT0;
  float* wp = reinterpret_cast<float*>(smem + Ly::kOffWp);
  unsigned char* flag = reinterpret_cast<unsigned char*>(B.flag);
  const int blk = blockIdx.x, G = a.G;
  // segments without index pages: window only, spread over the blocks
  for (long long sg = blk; sg < (long long)a.B * a.H; sg += G) {
    const int h = (int)(sg / a.B), b = (int)(sg - (long long)h * a.B);
    int L, NP;
    req_len(a, b, L, NP);
    if (NP != 0) continue;
    float M, l, o;
    aux_window(a, h, b, L, NP, scale_log2, wp, at, M, l, o);
    aux_emit(a, flag, h, b, 0, 0, Ptot, blk, at, M, l, o);
  }
  uint32_t hfull_ph = 0, wfull_ph = 0;
  int par = 0;
  while (W.valid) {
    float M = -INFINITY, l = 0.f, o = 0.f;
    for (int sa = W.pa; sa < W.pb; sa += kSubP) {
      if (aux_any(!wait_bar(B.hfull, hfull_ph, B.failed, a.err))) return;
      hfull_ph ^= 1u;
      float Ms, ls, os;
      aux_finalize<NG>(a, smem, W.h, par, at, Ms, ls, os);
      mbar_arrive(B.hfree);  // this thread's reads and clears are done
      merge_part(M, l, o, Ms, ls, os);
      par ^= 1;
    }
    if (W.pa == 0) {  // the piece starts its segment: the window warps' partial of its window
      if (aux_any(!wait_bar(B.wfull, wfull_ph, B.failed, a.err))) return;
      wfull_ph ^= 1u;
      float Mw, lw, ow;
      win_merge<kWW>(reinterpret_cast<const float*>(smem + Ly::kOffWw), at, Mw, lw, ow);
      __syncwarp();
      if ((at & 31) == 0) mbar_arrive(B.wfree);  // this warp has read the rows
      merge_part(M, l, o, Mw, lw, ow);
    }
    aux_emit(a, flag, W.h, W.b, W.pos - W.pa, W.np, Ptot, blk, at, M, l, o);
    walk_next(a, W, hi);
  }
}

// ------------------------------------------------------------------ window warps
// They walk the block's pieces like the aux warps and attend the bf16 window of every piece
// that starts its segment, in parallel with the compute warps and the aux warps' sub-piece
// sums, handing each window's rows to the aux warps: wfull (kWW arrivals) when written,
// wfree (kAW arrivals) when read.
template <int NG>
__device__ void window_role(const VqAttnArgs& a, unsigned char* smem, const Bars& B, Walk W, const long long hi,
                            const float scale_log2) {
  using Ly = Lay<NG>;
  const int wi = (threadIdx.x >> 5) - kWinW0, lane = threadIdx.x & 31;
  float* rows = reinterpret_cast<float*>(smem + Ly::kOffWw);
  uint32_t wfree_ph = 1;  // the rows start free
  while (W.valid) {
    if (W.pa == 0) {
      if (!__all_sync(0xFFFFFFFFu, wait_bar(B.wfree, wfree_ph, B.failed, a.err))) return;
      wfree_ph ^= 1u;
      win_attend<kWW, 3>(a, W.h, W.b, W.L, W.np, scale_log2, rows, wi, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(B.wfull);
    }
    walk_next(a, W, hi);
  }
}

// ------------------------------------------------------------------ the kernel
template <int NG>
__global__ void __launch_bounds__(kThreads, 1) vq_attn_kernel(const VqAttnArgs a, const float scale_log2) {
  using Ly = Lay<NG>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.G, blk = blockIdx.x;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Ly::kOffBar);
  Bars B;
  B.full = bar;
  B.empty = bar + Ly::kStg;
  B.kbar = bar + 2 * Ly::kStg;
  B.ktfree = B.kbar + 1;
  B.maxbar = B.kbar + 2;
  B.hfull = B.kbar + 3;
  B.hfree = B.kbar + 4;
  B.wfull = B.kbar + 5;
  B.wfree = B.kbar + 6;
  int* iflags = reinterpret_cast<int*>(B.kbar + 7);
  B.failed = iflags;
  B.flag = iflags + 1;
  Walk* wstart = reinterpret_cast<Walk*>(smem + Ly::kOffWalk);

  // ---- pages per request and their exclusive prefix (in the histogram area, cleared after)
  int* pre = reinterpret_cast<int*>(smem + Ly::kOffBins);
  {
    int* wsum = reinterpret_cast<int*>(smem + Ly::kOffSbuf);
    for (int b = tid; b < a.B; b += kThreads) {
      int L, NP;
      if (!req_len(a, b, L, NP) && blk == 0) set_error(a.err, KVQ_ERR_CAPACITY);
      pre[b] = NP;
    }
    __syncthreads();
    const int per = (a.B + kThreads - 1) / kThreads;
    const int beg = min(a.B, tid * per), end = min(a.B, beg + per);
    int local = 0;
    for (int b = beg; b < end; ++b) local += pre[b];
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
    for (int b = beg; b < end; ++b) {
      const int u = pre[b];
      pre[b] = run;
      run += u;
    }
    if (tid == kThreads - 1) pre[a.B] = run;  // the last thread ends on the total
    __syncthreads();
  }
  const long long Pb = pre[a.B];
  const long long Ptot = (long long)a.H * Pb;
  const long long lo = share_lo(Ptot, blk, G), hi = share_lo(Ptot, blk + 1, G);

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < Ly::kStg; ++s) {
      mbar_init(&B.full[s], 1);
      mbar_init(&B.empty[s], kCW);
    }
    mbar_init(B.kbar, 1);
    mbar_init(B.ktfree, kCW);
    mbar_init(B.maxbar, kCW);
    mbar_init(B.hfull, kCW);
    mbar_init(B.hfree, kAuxN);
    mbar_init(B.wfull, kWW);
    mbar_init(B.wfree, kAW);
    *B.failed = 0;
    fence_mbar_init();
    Walk W;
    W.valid = 0;
    if (lo < hi) {  // the first piece: head, then the last request whose prefix is <= the remainder
      W.valid = 1;
      W.pos = lo;
      W.h = (int)(lo / Pb);
      const int rem = (int)(lo - (long long)W.h * Pb);
      int bl = 0, bh = a.B - 1;
      while (bl < bh) {
        const int mid = (bl + bh + 1) >> 1;
        if (pre[mid] <= rem) bl = mid;
        else bh = mid - 1;
      }
      W.b = bl;
      W.pa = rem - pre[bl];
      req_len(a, W.b, W.L, W.np);
      W.pb = (int)min((long long)W.np, W.pa + (hi - lo));
      // the share's later key slices: HBM -> L2 now (a share spans few heads)
      const int h_last = min((int)((hi - 1) / Pb), W.h + 3);
      for (int hh = W.h + 1; hh <= h_last; ++hh) bulk_prefetch_l2(a.bt_k + (size_t)hh * kCB * kD, kKSliceBytes);
    }
    *wstart = W;
  }
  if (tid < 64) {  // cos, sin(kJump theta_i): from one past a group's last token of a unit to its next
    float* jt = reinterpret_cast<float*>(smem + Ly::kOffJ);
    const bool have = a.max_ctx > Ly::kJump;
    jt[tid] = have ? __ldg(a.rope_cos + (size_t)Ly::kJump * (kD / 2) + tid) : 1.f;
    jt[64 + tid] = have ? __ldg(a.rope_sin + (size_t)Ly::kJump * (kD / 2) + tid) : 0.f;
    const int row = (a.max_ctx > 1) ? 1 : 0;  // one position: the per-token step
    jt[128 + tid] = __ldg(a.rope_cos + (size_t)row * (kD / 2) + tid);
    jt[192 + tid] = __ldg(a.rope_sin + (size_t)row * (kD / 2) + tid);
  }
  __syncthreads();  // barriers initialised, prefix read: the histogram area is free
  {
    uint4* bz = reinterpret_cast<uint4*>(smem + Ly::kOffBins);
    for (int k = tid; k < kBinBytes / 16; k += kThreads) bz[k] = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();

  int issued = 0, k_loads = 0;
  if (warp < kCW) {
    compute_role<NG>(a, smem, B, scale_log2);
  } else if (warp < kCW + kAW) {
    aux_role<NG>(a, smem, B, *wstart, hi, Ptot, scale_log2);
  } else if (warp == kProdWarp) {
    if (lane == 0) producer_role<NG>(a, smem, B, *wstart, hi, issued, k_loads);
  } else {
    window_role<NG>(a, smem, B, *wstart, hi, scale_log2);
  }
  __syncthreads();
  // after a timeout, let the block's own copies in flight land before it exits
  if (warp == kProdWarp && lane == 0 && *B.failed) {
    for (int k = max(0, issued - Ly::kStg); k < issued; ++k) mbar_wait_bounded(&B.full[k % Ly::kStg], (k / Ly::kStg) & 1);
    if (k_loads > 0) mbar_wait_bounded(B.kbar, (k_loads - 1) & 1);
  }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <int NG>
cudaError_t launch(const VqAttnArgs& a, float scale_log2, cudaStream_t st) {
  using Ly = Lay<NG>;
  cudaError_t e = cudaFuncSetAttribute(vq_attn_kernel<NG>, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kSmemBytes);
  if (e != cudaSuccess) return e;
  vq_attn_kernel<NG><<<a.G, kThreads, Ly::kSmemBytes, st>>>(a, scale_log2);
  return cudaGetLastError();
}

}  // namespace

size_t vq_attn_ws_bytes(int B, int H, int G) {
  return align256((size_t)B * H * sizeof(int32_t)) + align256((size_t)G * 2 * kVqSlotFloats * sizeof(float));
}

cudaError_t launch_vq_attn(const VqAttnArgs& args, void* ws, cudaStream_t st) {
  VqAttnArgs a = args;
  char* w = static_cast<char*>(ws);
  a.cnt = reinterpret_cast<int32_t*>(w);
  w += align256((size_t)a.B * a.H * sizeof(int32_t));
  a.slots = reinterpret_cast<float*>(w);
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)kD);
  switch (a.NG) {
    case 16: return launch<16>(a, scale_log2, st);
    case 8: return launch<8>(a, scale_log2, st);
    case 32: return launch<32>(a, scale_log2, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
