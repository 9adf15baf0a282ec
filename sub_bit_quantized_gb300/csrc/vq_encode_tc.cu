// Prefill encode on the 5th-generation tensor cores: nearest codeword of every coupled vector
// as a distance GEMM plus a row argmin.
//
// "LoopVQ: Sub 1-bit KV Cache Quantization for Looped Transformers", background (vector
// quantization: a(z) = argmin_r ||z - e_r||^2) and method steps 1 and 4 (coupled vectors of
// G = c T_c coordinates, one 256-entry codebook per (block, layer, head, group), prefill
// encode on tensor cores). ||z - e_r||^2 = ||z||^2 - 2 (z.e_r - ||e_r||^2 / 2), so the best
// codeword maximises z.e_r - ||e_r||^2 / 2: one GEMM row per vector, one column per codeword.
//
// Precision. z is bf16 data, exact in bf16. Each fp32 codebook entry is split into three
// bf16 parts hi + mid + lo (each the bf16 rounding of what the previous parts leave), so the
// three bf16 x bf16 products accumulated in fp32 reproduce z.e to about 2^-24 of |z||e|; the
// -||e||^2 / 2 column is split the same way and multiplies an augmented A column of ones.
// The tensor cores screen; every row whose runner-up lies within a conservative error band
// of the best (far above the accumulation error, and above the 1e-6 tie threshold) is
// decided again over the candidates in the band on distances summed with error-free fp32
// steps (relative error ~1e-7): the result is the argmin with the lowest index on exact ties,
// and candidates closer than 1e-6 (relative) are reported as a tie, where either index is a
// valid answer.
//
// GB300 mapping. One persistent block per SM over an equal contiguous share of the (plane,
// 128-vector tile) units, a plane being one (sequence, head, block beta, group) with its
// codebook, whose three bf16 parts sit in shared memory (K-major, no swizzle: 8-row x 16-byte
// core matrices). The block is a warp-specialised pipeline synchronised only by mbarriers:
//  * a loader warp copies each tile's vector rows into a 4-stage ring with cp.async (zero
//    fill past the last token), two tiles in flight;
//  * an MMA warp issues, from one thread, the tcgen05.mma chain of a tile (3 parts x K steps
//    of 16) into one of two 128 x 256 fp32 TMEM accumulators and commits to that
//    accumulator's barrier; at a plane change it restages the codebook once the earlier
//    tiles are done with it;
//  * two epilogue warpgroups take alternate tiles, one accumulator each: a thread owns a row
//    and reads its 256 columns twice (tcgen05.ld): the best acc (3-input max), then how many
//    columns lie in the error band below it and, when one does, which (a weighted sum on the
//    FMA pipe, so the half-rate ALU pipe is not the limit); it releases the accumulator, decides
//    near-ties as above from shared memory, writes the index and releases the ring stage.
// So the MMAs of one tile run while the other accumulator's epilogue works. Every wait is
// bounded; a timeout sets the device error word and every warp leaves its loop.
//
// Page-roll instantiation (kRoll; method step 4 / Figure 5: during decode the oldest recent
// page is encoded every 8 tokens): a plane is (layer, K/V, head, beta, group) and its rows are
// the 8 tokens of the oldest recent page of every request, read from the bf16 windows, so all
// requests' rows share one staged codebook. A plane then has few tiles, so the three bf16
// parts are cut once at load time (kvq_split_codebooks, the same arithmetic as the staging
// below) and the loader copies each plane's parts with one bulk copy into one of two
// buffers while the previous plane's tiles run. Rows of requests that are not due are
// zero-filled and not written; a launch with no request due returns at once.
#include <cuda_fp16.h>

#include <algorithm>

#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "../../include/kvq.h"

namespace kvq {
namespace {

constexpr int kTcM = 128;            // vectors per tile (MMA M)
constexpr int kTcN = 256;            // codewords (MMA N)
constexpr int kParts = 3;            // hi, mid, lo bf16 parts of the fp32 codebook
constexpr int kEpiWarps = 8;         // two epilogue warpgroups, one accumulator each
constexpr int kLoadWarp = 8;         // cp.async loader
constexpr int kMmaWarp = 9;          // MMA issue (lane 0) and codebook restaging
constexpr int kEncThreads = 320;
constexpr int kAStages = 4;          // vector-row ring
constexpr int kLoadDepth = 2;        // tiles whose row copies the loader keeps in flight
constexpr uint32_t kTmemCols = 512;  // two 128 x 256 fp32 accumulators
constexpr int kNearCap = 64;         // near-tie (row, candidate) pairs an epilogue warp decides together
static_assert(kEpiWarps == 8 && kLoadWarp == kEpiWarps && kMmaWarp == kLoadWarp + 1 &&
              kEncThreads == 32 * (kMmaWarp + 1), "warp roles");

// 16-byte K chunks per row: G/8 chunks of data (row coordinate k' = m c + i holds channel
// g c + i of loop step m, i.e. coupled coordinate i Tc + m), one augmented chunk (A: 1, 0..;
// B: -||e||^2 / 2, 0..), padded to whole MMA K steps of 32 bytes
__host__ __device__ constexpr int tc_chunks(int DC) { return 2 * ((DC + 2) / 2); }

template <int TC, int C, bool kRoll = false>
struct TcLayout {
  static constexpr int G = TC * C;
  static constexpr int DC = G / 8;                          // data chunks per row
  static constexpr int NG = kD / C;                         // groups per token
  static constexpr int kPageBytes = kPage * NG;
  static constexpr int KC = tc_chunks(DC);
  static constexpr int kRowBytes = KC * 16;
  static constexpr int kABytes = kTcM * kRowBytes;          // one tile of vectors
  static constexpr int kBPartBytes = kTcN * kRowBytes;      // one codebook part
  static constexpr int kOffA = 0;                           // kAStages tile buffers
  static constexpr int kOffB = kOffA + kAStages * kABytes;  // the three codebook parts (two buffers: roll)
  static constexpr int kBufBytes = kParts * kBPartBytes;
  static constexpr int kOffBar = kOffB + (kRoll ? 2 : 1) * kBufBytes;  // mbarriers, TMEM address, flags
  static constexpr int kOffNear = kOffBar + 160;            // per epilogue warp: near-tie pairs, distances
  static constexpr int kSmem = kOffNear + kEpiWarps * kNearCap * 8;
  // requested per block so that a second block cannot share the SM (and its 512 TMEM columns)
  static constexpr int kSmemLaunch = kSmem > 120 * 1024 ? kSmem : 120 * 1024;
  static_assert(kSmemLaunch <= 232448, "shared memory");
};

// byte offset of (row, chunk) in a K-major, no-swizzle operand: core matrices of 8 rows x 16
// bytes (128 contiguous bytes); chunks of a row group 128 bytes apart (LBO), row groups
// KC x 128 bytes apart (SBO)
__device__ __forceinline__ uint32_t op_off(int row, int chunk, int KC) {
  return (uint32_t)((row >> 3) * (KC * 128) + chunk * 128 + (row & 7) * 16);
}

// shared-memory matrix descriptor: K-major, no swizzle
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version of this architecture
  return d;                // base offset 0, absolute LBO mode off, layout: no swizzle
}

// instruction descriptor, kind::f16: fp32 D, bf16 A and B, both K-major, M = 128, N = 256
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kTcN >> 3) << 17) |
                            ((uint32_t)(kTcM >> 4) << 24);

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// N (a multiple of 32) consecutive fp32 columns of this thread's TMEM lane: N / 32 loads,
// one wait
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[N]) {
  uint32_t r[N];
#pragma unroll
  for (int h = 0; h < N / 32; ++h)
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[32 * h + 0]), "=r"(r[32 * h + 1]), "=r"(r[32 * h + 2]), "=r"(r[32 * h + 3]), "=r"(r[32 * h + 4]),
          "=r"(r[32 * h + 5]), "=r"(r[32 * h + 6]), "=r"(r[32 * h + 7]), "=r"(r[32 * h + 8]), "=r"(r[32 * h + 9]),
          "=r"(r[32 * h + 10]), "=r"(r[32 * h + 11]), "=r"(r[32 * h + 12]), "=r"(r[32 * h + 13]),
          "=r"(r[32 * h + 14]), "=r"(r[32 * h + 15]), "=r"(r[32 * h + 16]), "=r"(r[32 * h + 17]),
          "=r"(r[32 * h + 18]), "=r"(r[32 * h + 19]), "=r"(r[32 * h + 20]), "=r"(r[32 * h + 21]),
          "=r"(r[32 * h + 22]), "=r"(r[32 * h + 23]), "=r"(r[32 * h + 24]), "=r"(r[32 * h + 25]),
          "=r"(r[32 * h + 26]), "=r"(r[32 * h + 27]), "=r"(r[32 * h + 28]), "=r"(r[32 * h + 29]),
          "=r"(r[32 * h + 30]), "=r"(r[32 * h + 31])
        : "r"(taddr + 32 * h)
        : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
}

// cp.async of 16 (or 8) bytes, zero-filled when `fill` is false (src is then not read)
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool fill) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(fill ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src, bool fill) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(fill ? 8 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint16_t bf16_rn_bits(float f) { return f32_to_bf16(f); }

// Error band in acc units for a row with |z|^2 = z2 whose best acc is `best`. A codeword that
// can compete with the best lies within |z| + sqrt(d_best) of the origin, and its
// acc = z.e - |e|^2/2 is accumulated over 3 x KC/2 MMAs of exact bf16 products: its error is
// below about 3 (KC/2) 17 2^-24 (|z||e| + |e|^2/2) plus the 2^-24 |z||e| of the split. The
// band takes 4 times that (the difference of two candidates, each accumulated with rounding
// that may go toward zero), plus the 1e-6 tie threshold of the best distance. A larger `best`
// (a better candidate) never widens it.
template <int KC>
__device__ __forceinline__ float acc_band(float z2, float best) {
  const float znorm = sqrtf(z2);
  const float dbest = fmaxf(0.f, z2 - 2.f * best);
  const float enear = znorm + 1.01f * sqrtf(dbest) + 1e-3f * znorm + 1e-6f;
  return 4.f * 3.f * (KC / 2) * 18.f * 5.97e-8f * (znorm * enear + 0.5f * enear * enear) + 1e-6f * dbest + 1e-30f;
}

// plane p of the encode: (sequence b, head h, block beta, group index gi)
struct Plane {
  int b, h, beta, gi;
};
__device__ __forceinline__ Plane plane_of(const VqEncodeArgs& a, int p) {
  Plane q;
  q.gi = p % a.g_count;
  q.beta = (p / a.g_count) % a.NB;
  q.h = (p / (a.g_count * a.NB)) % a.H;
  q.b = p / (a.g_count * a.NB * a.H);
  return q;
}

// Roll rows: row q of a plane is token j = q mod 8 of request b = q / 8's oldest recent page;
// true when q is a row and b is due (its recent window holds W + 8 tokens and a page is free)
__device__ __forceinline__ bool roll_row(const VqEncodeArgs& a, int q, int& b, int& jj, int& np) {
  b = q >> 3;
  jj = q & 7;
  np = 0;
  if (q >= a.n_tok) return false;
  const int L = a.seq_len[b];
  np = a.n_pages[b];
  return (L - a.sink - kPage * np == a.recent + kPage) && (np < a.max_pages);
}

// three bf16 parts of the plane's codebook (and its -||e||^2/2 column), rows r0, r0 + nt, ..
// cb: a [256][G] fp32 codebook; sb: the three parts' destination (shared or global memory)
template <int TC, int C>
__device__ void split_codebook(const float* cb, unsigned char* sb, int r0, int nt) {
  using Lay = TcLayout<TC, C>;
  constexpr int G = Lay::G, KC = Lay::KC, DC = Lay::DC;
#pragma unroll 1
  for (int r = r0; r < kTcN; r += nt) {
    float ev[G];  // the row's coordinates, all loads in flight together
#pragma unroll
    for (int k = 0; k < G; k += 4) {
      const float4 q4 = __ldg(reinterpret_cast<const float4*>(cb + (size_t)r * G + k));
      ev[k] = q4.x;
      ev[k + 1] = q4.y;
      ev[k + 2] = q4.z;
      ev[k + 3] = q4.w;
    }
    float nh_hi = 0.f, nh_lo = 0.f;  // |e|^2, compensated
#pragma unroll
    for (int k = 0; k < G; ++k) add_sq_diff(ev[k], 0.f, nh_hi, nh_lo);
    const float nh = -0.5f * __fadd_rn(nh_hi, nh_lo);
    // row coordinate k' = 8 c + i (chunk c < DC, i < 8) = m C + i2 is coupled coordinate i2 TC + m;
    // one 16-byte chunk at a time; parts: hi = bf16(v), mid = bf16(v - hi), lo = bf16(v - hi - mid)
#pragma unroll
    for (int c = 0; c < KC; ++c) {
      uint32_t w[kParts][4];
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) {
        uint16_t pb[kParts][2];
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int i = 2 * i2 + e2, kk = 8 * c + i;
          float v = 0.f;
          if (c < DC) v = ev[(kk % C) * TC + kk / C];
          else if (c == DC && i == 0) v = nh;
#pragma unroll
          for (int p = 0; p < kParts; ++p) {
            const uint16_t bits = bf16_rn_bits(v);
            pb[p][e2] = bits;
            v = v - bf16_to_f32(bits);  // exact: v and its bf16 rounding are within 2^-8 |v|
          }
        }
#pragma unroll
        for (int p = 0; p < kParts; ++p) w[p][i2] = pb[p][0] | ((uint32_t)pb[p][1] << 16);
      }
#pragma unroll
      for (int p = 0; p < kParts; ++p)
        *reinterpret_cast<uint4*>(sb + p * Lay::kBPartBytes + op_off(r, c, KC)) =
            make_uint4(w[p][0], w[p][1], w[p][2], w[p][3]);
    }
  }
}

template <int TC, int C>
__device__ __forceinline__ void stage_codebook(const VqEncodeArgs& a, int plane, unsigned char* sb, int r0, int nt) {
  using Lay = TcLayout<TC, C>;
  const Plane P = plane_of(a, plane);
  split_codebook<TC, C>(a.cb + (((size_t)P.beta * a.H + P.h) * Lay::NG + a.g_begin + P.gi) * (size_t)kCB * Lay::G, sb,
                        r0, nt);
}

// kvq_split_codebooks: one block per codebook, a thread per row
template <int TC, int C>
__global__ void __launch_bounds__(256) split_codebooks_kernel(const float* cb, uint8_t* cbp) {
  using Lay = TcLayout<TC, C>;
  split_codebook<TC, C>(cb + (size_t)blockIdx.x * kCB * Lay::G, cbp + (size_t)blockIdx.x * Lay::kBufBytes, threadIdx.x,
                        blockDim.x);
}

__device__ __forceinline__ bool enc_wait(uint64_t* bar, uint32_t parity, volatile int* failed, int* err) {
  if (*failed) return false;
  if (mbar_wait_bounded_sleep(bar, parity)) return true;
  *failed = 1;
  set_error(err, KVQ_ERR_TIMEOUT);
  return false;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// 1 when v >= thr, else 0, on the FMA pipe: sat(v 2^90 + (1 - thr 2^90)). v 2^90 rounds to
// ~2^-24 of itself, so values within a few ulps of thr may land either way; the error band
// around the best is far wider than that.
__device__ __forceinline__ float at_least(float v, float cth) {
  float d;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(v), "f"(1.2379400392853803e27f), "f"(cth));
  return d;
}

template <int TC, int C, bool kRoll>
__global__ void __launch_bounds__(kEncThreads, 1) encode_tc_kernel(const VqEncodeArgs a, const int U,
                                                                  const int tiles_per_plane) {
  using Lay = TcLayout<TC, C, kRoll>;
  constexpr int KC = Lay::KC, DC = Lay::DC;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* sa0 = smem + Lay::kOffA;
  unsigned char* sb = smem + Lay::kOffB;
  uint64_t* afull = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);  // rows landed (32 loader lanes)
  uint64_t* aempty = afull + kAStages;                                  // rows released (4 epilogue warps)
  uint64_t* accfull = aempty + kAStages;                                // MMAs done (commit)
  uint64_t* accempty = accfull + 2;                                     // accumulator read (4 warps)
  uint64_t* bdone = accempty + 2;                                       // tile done with the codebook (4 warps)
  uint64_t* bfull = bdone + 2;                                          // roll: codebook buffer landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bfull + 2);
  volatile int* failed = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* done = reinterpret_cast<int*>(tmem_slot + 2);  // roll, per epilogue warpgroup: tiles finished x 4 warps

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Block k encodes group gi = k mod g_count over slots [m S / sets, (m + 1) S / sets) of the
  // (sequence, head, block beta, tile) slots, m = k / g_count: the g_count blocks of a set walk
  // the same token rows at the same time, so each row's 16-byte group slices come from DRAM
  // once and from L2 for the other groups.
  const int gsel = blockIdx.x % a.g_count, set = blockIdx.x / a.g_count, n_sets = gridDim.x / a.g_count;
  const int lo = (int)((long long)U * set / n_sets), hi = (int)((long long)U * (set + 1) / n_sets);
  if (lo >= hi) return;  // uniform
  if constexpr (kRoll) {  // between rolls no request is due: leave before anything is set up
    int any = 0;
    for (int b = tid; b < a.n_req; b += kEncThreads) {
      int bb, jj, np;
      any |= roll_row(a, kPage * b, bb, jj, np) ? 1 : 0;
    }
    if (!__syncthreads_or(any)) return;
  }
  const int n = hi - lo;  // tiles of this block
  // tile i of the block: slot lo + i -> plane ((sequence, head, beta) of the slot, group gsel), tile
  auto plane_at = [&](int i) { return ((lo + i) / tiles_per_plane) * a.g_count + gsel; };
  auto tile_at = [&](int i) { return (lo + i) % tiles_per_plane; };
  // roll: the block's planes in order (ordinal of tile i's plane, first tile of ordinal q);
  // plane ordinal q uses codebook buffer q & 1, copied once the plane two before it is done
  auto pk_of = [&](int i) { return (lo + i) / tiles_per_plane - lo / tiles_per_plane; };
  auto first_of = [&](int q) { return q == 0 ? 0 : (lo / tiles_per_plane + q) * tiles_per_plane - lo; };

  // ---- TMEM (warp 0), barriers, constant A chunks, the first plane's codebook (all threads) ----
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&afull[s], 32);
      mbar_init(&aempty[s], 4);
    }
    for (int e = 0; e < 2; ++e) {
      mbar_init(&accfull[e], 1);
      mbar_init(&accempty[e], 4);
      mbar_init(&bdone[e], 4);
      mbar_init(&bfull[e], 1);
      done[e] = 0;
    }
    *failed = 0;
    fence_mbar_init();
    // the codebooks of the block's later planes: HBM -> L2 while the pipeline starts
    for (int pl = plane_at(0) + a.g_count; !kRoll && pl <= plane_at(n - 1); pl += a.g_count) {
      const Plane P = plane_of(a, pl);
      bulk_prefetch_l2(a.cb + (((size_t)P.beta * a.H + P.h) * Lay::NG + a.g_begin + P.gi) * (size_t)kCB * Lay::G,
                       kCB * Lay::G * 4);
    }
  }
  for (int i = tid; i < kAStages * kTcM * (KC - DC); i += kEncThreads) {  // the ones column, zero padding
    const int st = i / (kTcM * (KC - DC)), rem = i % (kTcM * (KC - DC));
    const int r = rem / (KC - DC), c = DC + rem % (KC - DC);
    *reinterpret_cast<uint4*>(sa0 + st * Lay::kABytes + op_off(r, c, KC)) = make_uint4(c == DC ? 0x3F80u : 0u, 0u, 0u, 0u);
  }
  if constexpr (!kRoll) stage_codebook<TC, C>(a, plane_at(0), sb, tid, kEncThreads);
  fence_proxy_async_smem();  // generic writes -> the tensor cores' view
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kLoadWarp) {
    // ================= loader: vector rows of tile i -> ring stage i % kAStages ================
    auto land = [&](int i) {  // tile i's copies by this lane are complete: publish them
      fence_proxy_async_smem();
      mbar_arrive(&afull[i % kAStages]);
    };
    // roll: the codebook parts of the block's planes, one bulk copy each into buffer q & 1
    // (completion q >> 1 of bfull[q & 1]) once plane q - 2 is done with that buffer
    const int n_planes = kRoll ? pk_of(n - 1) + 1 : 1;
    int copied = -1;  // planes 0 .. copied have been issued
    volatile int* vdone = done;
    auto done_below = [&](int X) {  // every tile < X is finished by its epilogue warpgroup
      return vdone[0] >= 4 * ((X + 1) / 2) && vdone[1] >= 4 * (X / 2);
    };
    auto copy_parts = [&](int q) {  // lane 0
      const Plane P = plane_of(a, plane_at(first_of(q)));
      const uint8_t* src = ((P.b & 1) ? a.cbp2 : a.cbp) + (size_t)(P.b >> 1) * a.cbp_layer +
                           (((size_t)P.beta * a.H + P.h) * Lay::NG + P.gi) * (size_t)Lay::kBufBytes;
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&bfull[q & 1], Lay::kBufBytes);
      bulk_g2s(sb + (q & 1) * Lay::kBufBytes, src, Lay::kBufBytes, &bfull[q & 1]);
    };
    if constexpr (kRoll) {
      if (lane == 0)
        for (int q = 0; q < min(2, n_planes); ++q) copy_parts(q);
      copied = min(2, n_planes) - 1;
    }
    int i = 0;
    for (; i < n; ++i) {
      const int st = i % kAStages;
      if constexpr (kRoll) {
        // the next plane's parts, once the plane two before it is done (needed before this
        // tile's MMAs when it starts that plane: then wait for the buffer)
        const int q = copied + 1;
        if (q < n_planes) {
          const bool need = q <= pk_of(i);
          bool free_buf = __all_sync(0xFFFFFFFFu, done_below(first_of(q - 1)));
          if (need && !free_buf) {
            const uint64_t t0 = global_ns();
            while (!free_buf) {
              if (*failed) break;
              if (global_ns() - t0 > 1000000000ull) {
                *failed = 1;
                set_error(a.err, KVQ_ERR_TIMEOUT);
                break;
              }
              __nanosleep(64);
              free_buf = __all_sync(0xFFFFFFFFu, done_below(first_of(q - 1)));
            }
            if (!free_buf) break;  // warp-uniform
          }
          if (free_buf) {
            if (lane == 0) copy_parts(q);
            copied = q;
          }
        }
      }
      if (i >= kAStages && !__all_sync(0xFFFFFFFFu, enc_wait(&aempty[st], ((i / kAStages) - 1) & 1, failed, a.err)))
        break;  // warp-uniform
      const int plane = plane_at(i), t = tile_at(i);
      const Plane P = plane_of(a, plane);
      const uint16_t* xb = a.x + (size_t)P.b * a.sb + (size_t)P.h * a.sh + (size_t)(a.g_begin + P.gi) * C;
      if constexpr (kRoll) xb = ((P.b & 1) ? a.x2 : a.x) + (size_t)(P.b >> 1) * a.x_layer + (size_t)P.h * a.sh + (size_t)P.gi * C;
      unsigned char* sa = sa0 + st * Lay::kABytes;
      for (int q = lane; q < kTcM * DC; q += 32) {  // chunk d of row r: coordinates 8d .. 8d + 7
        const int r = q / DC, d = q % DC, j = t * kTcM + r;
        bool in = j < a.n_tok;
        const uint16_t* xr = xb + (size_t)(in ? j : 0) * kD;
        if constexpr (kRoll) {  // the request's window slot of the token
          int b, jj, np;
          in = roll_row(a, j, b, jj, np);
          const int pos = a.sink + kPage * np + jj;
          const int slot = a.sink + (pos - a.sink) % (a.recent + kPage);
          xr = xb + (in ? (size_t)b * a.sb + (size_t)slot * kD : 0);
        }
        unsigned char* dst = sa + op_off(r, d, KC);
        if constexpr (C >= 8) {
          cp_async16(dst, xr + (size_t)(P.beta * TC + (8 * d) / C) * a.st + (8 * d) % C, in);
        } else {  // two loop steps of 4 channels
          cp_async8(dst, xr + (size_t)(P.beta * TC + 2 * d) * a.st, in);
          cp_async8(dst + 8, xr + (size_t)(P.beta * TC + 2 * d + 1) * a.st, in);
        }
      }
      cp_async_commit();
      if (i >= kLoadDepth - 1) {
        cp_async_wait<kLoadDepth - 1>();
        land(i - (kLoadDepth - 1));
      }
    }
    cp_async_wait<0>();  // nothing of this block's may land after it exits
    for (int k = max(0, i - (kLoadDepth - 1)); k < i; ++k) land(k);
    if constexpr (kRoll) {  // the last codebook copies issued: let them land (bounded)
      if (lane == 0)
        for (int q = max(0, copied - 1); q <= copied; ++q) mbar_wait_bounded(&bfull[q & 1], (uint32_t)((q >> 1) & 1));
    }
  } else if (warp == kMmaWarp) {
    // ================= MMA issue; codebook restaging at plane changes ==========================
    const uint64_t a_desc0 = umma_desc(smem_u32(sa0), 128, KC * 128);
    const uint64_t b_desc0 = umma_desc(smem_u32(sb), 128, KC * 128);
    int cur_plane = plane_at(0);
    int last = -1;  // last tile whose MMAs were committed
    for (int i = 0; i < n; ++i) {
      const int st = i % kAStages, e = i & 1;
      const int plane = plane_at(i);
      const int bufo = kRoll ? (pk_of(i) & 1) * Lay::kBufBytes : 0;  // this plane's codebook buffer
      if (!kRoll && plane != cur_plane) {
        // every earlier tile is done with the codebook: its MMAs and its epilogue (near-ties
        // read the parts)
        bool ok = true;
        if (lane == 0) {
          ok = enc_wait(&bdone[(i - 1) & 1], ((i - 1) >> 1) & 1, failed, a.err);
          if (ok && i >= 2) ok = enc_wait(&bdone[i & 1], ((i - 2) >> 1) & 1, failed, a.err);
        }
        if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) break;
        stage_codebook<TC, C>(a, plane, sb, lane, 32);
        fence_proxy_async_smem();
        __syncwarp();
        cur_plane = plane;
      }
      int ok = 1;
      if (lane == 0) {
        if (kRoll && (i == 0 || pk_of(i - 1) != pk_of(i))) {  // the plane's parts have landed
          const int pk = pk_of(i);
          ok = enc_wait(&bfull[pk & 1], (pk >> 1) & 1, failed, a.err);
        }
        if (ok) ok = enc_wait(&afull[st], (i / kAStages) & 1, failed, a.err);
        if (ok && i >= 2) ok = enc_wait(&accempty[e], ((i >> 1) - 1) & 1, failed, a.err);
        if (ok) {
          tc_fence_after();
          // start addresses advance in 16-byte units in the low descriptor bits (no carry: every
          // operand lies below 256 KB of shared memory)
#pragma unroll
          for (int p = 0; p < kParts; ++p)
#pragma unroll
            for (int s = 0; s < KC / 2; ++s)
              umma_bf16(tmem + kTcN * e, a_desc0 + (uint64_t)((st * Lay::kABytes + s * 256) >> 4),
                        b_desc0 + (uint64_t)((bufo + p * Lay::kBPartBytes + s * 256) >> 4), (p | s) != 0);
          umma_commit(&accfull[e]);
          last = i;
        }
      }
      if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;
    }
    // the block may only free TMEM once its last MMAs have landed
    if (lane == 0 && last >= 0) mbar_wait_bounded(&accfull[last & 1], (last >> 1) & 1);
  } else {
    // ================= epilogue: warpgroup e takes tiles e, e + 2, ...; a thread owns a row =====
    // Pass 1: the best acc of the row (3-input max). Pass 2: with thr = best - band, the number
    // of columns at or above thr and, when that is one, its column, as sum [v >= thr] (1 + col/512)
    // on the FMA pipe. More than one column in the band: the row is decided on exact distances.
    const int e = warp >> 2, row = 32 * (warp & 3) + lane;
    uint32_t* near_list = reinterpret_cast<uint32_t*>(smem + Lay::kOffNear) + warp * kNearCap;
    float* near_d = reinterpret_cast<float*>(smem + Lay::kOffNear) + kEpiWarps * kNearCap + warp * kNearCap;
    const uint32_t row_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(kTcN * e);
    int ties = 0;
    for (int i = e; i < n; i += 2) {
      const int st = i % kAStages;
      // warp-uniform: the accumulator reads below are warp-collective
      if (!__all_sync(0xFFFFFFFFu, enc_wait(&accfull[e], (i >> 1) & 1, failed, a.err))) break;
      tc_fence_after();
      float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll 1
      for (int k = 0; k < kTcN / 128; ++k) {
        float v[128];
        tmem_ld<128>(row_addr + 128 * k, v);
#pragma unroll
        for (int c = 0; c < 128; c += 8) {
          m0 = max3f(m0, v[c], v[c + 1]);
          m1 = max3f(m1, v[c + 2], v[c + 3]);
          m2 = max3f(m2, v[c + 4], v[c + 5]);
          m3 = max3f(m3, v[c + 6], v[c + 7]);
        }
      }
      const float best = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
      const int plane = plane_at(i), t = tile_at(i);
      const unsigned char* sa = sa0 + st * Lay::kABytes;
      const unsigned char* sbt = sb + (kRoll ? (pk_of(i) & 1) * Lay::kBufBytes : 0);  // this tile's codebook
      float z2 = 0.f;
#pragma unroll
      for (int c = 0; c < DC; ++c) {
        const uint4 w = *reinterpret_cast<const uint4*>(sa + op_off(row, c, KC));
        const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float l = bf16_lo(w4[q]), hh = bf16_hi(w4[q]);
          z2 = fmaf(l, l, fmaf(hh, hh, z2));
        }
      }
      const float band = acc_band<KC>(z2, best);
      const float thr = best - band;
      const float cth = fmaf(-thr, 1.2379400392853803e27f, 1.0f);
      // per 64-column chunk k: sum [v >= thr] (1 + c/512), c the column within the chunk; the
      // whole row's tally is below 1.5 exactly when one column is in the band, and then the
      // chunk holding it has a sum of 1 + c/512
      float tally = 0.f, ksum = 0.f;
      int ksel = 0;
      uint32_t kmask = 0;  // chunks holding a column in the band
#pragma unroll 1
      for (int k2 = 0; k2 < kTcN / 128; ++k2) {
        float v[128];
        tmem_ld<128>(row_addr + 128 * k2, v);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int k = 2 * k2 + hh;
          const float* vk = v + 64 * hh;
          float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            const float2 f01 = make_float2(at_least(vk[c], cth), at_least(vk[c + 1], cth));
            const float2 f23 = make_float2(at_least(vk[c + 2], cth), at_least(vk[c + 3], cth));
            s01 = __ffma2_rn(f01, make_float2(1.f + c / 512.f, 1.f + (c + 1) / 512.f), s01);
            s23 = __ffma2_rn(f23, make_float2(1.f + (c + 2) / 512.f, 1.f + (c + 3) / 512.f), s23);
          }
          const float sk = (s01.x + s01.y) + (s23.x + s23.y);
          if (sk > 0.5f) {
            ksel = k;
            ksum = sk;
            kmask |= 1u << k;
          }
          tally += sk;
        }
      }
      const int j = t * kTcM + row;
      int rb = 0, rj = 0, rnp = 0;
      bool valid = j < a.n_tok;
      if constexpr (kRoll) valid = roll_row(a, j, rb, rj, rnp);
      const bool need = valid && !*failed && !(tally < 1.5f);
      int result = 64 * ksel + __float2int_rn((ksum - 1.f) * 512.f);
      uint32_t cand[kTcN / 32];  // candidate masks of this row (need only)
#pragma unroll
      for (int q = 0; q < kTcN / 32; ++q) cand[q] = 0;
      const bool any_need = __any_sync(0xFFFFFFFFu, need);
      if (any_need) {  // candidate masks, reading only the chunks some row of the warp needs
#pragma unroll
        for (int k = 0; k < kTcN / 64; ++k) {
          const bool mine = need && ((kmask >> k) & 1u);
          if (!__any_sync(0xFFFFFFFFu, mine)) continue;  // warp-uniform
          float v[64];
          tmem_ld<64>(row_addr + 64 * k, v);  // warp-wide load: every lane takes part
          if (mine) {
#pragma unroll
            for (int b = 0; b < 32; ++b) {
              cand[2 * k] |= (v[b] >= thr) ? (1u << b) : 0u;
              cand[2 * k + 1] |= (v[32 + b] >= thr) ? (1u << b) : 0u;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&accempty[e]);  // the accumulator is read: the next MMAs may go
      if (any_need) {
        // every candidate in the band, decided on compensated fp32 distances (lowest index wins
        // exact ties); a runner-up within 1e-6 of the best is reported as a tie. The warp's
        // (row, candidate) pairs go to a list that all 32 lanes work through together (a row
        // rarely has more than a few candidates, and only some rows of a warp have any); a
        // longer list than kNearCap is done row by row.
        float bd = INFINITY, sd = INFINITY;
        int bdi = result;
        auto consider = [&](int r, float dd) {  // in increasing column order: the lowest wins exact ties
          if (dd < bd) {
            sd = bd;
            bd = dd;
            bdi = r;
          } else if (dd < sd) {
            sd = dd;
          }
        };
        // e = hi + mid + lo exactly (each residual is a multiple of e's ulp that fits the next
        // part), so the staged parts give the fp32 entries back
        auto exact_d = [&](int rr, int r) {
          float dh = 0.f, dl = 0.f;
#pragma unroll 1
          for (int c = 0; c < DC; ++c) {
            const uint4 w = *reinterpret_cast<const uint4*>(sa + op_off(rr, c, KC));
            const uint4 e0 = *reinterpret_cast<const uint4*>(sbt + op_off(r, c, KC));
            const uint4 e1 = *reinterpret_cast<const uint4*>(sbt + Lay::kBPartBytes + op_off(r, c, KC));
            const uint4 e2 = *reinterpret_cast<const uint4*>(sbt + 2 * Lay::kBPartBytes + op_off(r, c, KC));
            const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
            const uint32_t h4[4] = {e0.x, e0.y, e0.z, e0.w}, m4[4] = {e1.x, e1.y, e1.z, e1.w},
                           l4[4] = {e2.x, e2.y, e2.z, e2.w};
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
              add_sq_diff(bf16_lo(w4[q2]), __fadd_rn(__fadd_rn(bf16_lo(h4[q2]), bf16_lo(m4[q2])), bf16_lo(l4[q2])), dh, dl);
              add_sq_diff(bf16_hi(w4[q2]), __fadd_rn(__fadd_rn(bf16_hi(h4[q2]), bf16_hi(m4[q2])), bf16_hi(l4[q2])), dh, dl);
            }
          }
          return __fadd_rn(dh, dl);
        };
        int cnt = 0;
#pragma unroll
        for (int q = 0; q < kTcN / 32; ++q) cnt += __popc(need ? cand[q] : 0u);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += y;
        }
        const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
        if (total <= kNearCap) {  // warp-uniform
          int en = incl - cnt;
#pragma unroll
          for (int q = 0; q < kTcN / 32; ++q) {
            uint32_t cm = need ? cand[q] : 0u;
            while (cm) {
              near_list[en++] = ((uint32_t)row << 8) | (uint32_t)(32 * q + __ffs(cm) - 1);
              cm &= cm - 1;
            }
          }
          __syncwarp();
          for (int e2 = lane; e2 < total; e2 += 32) {
            const uint32_t v = near_list[e2];
            near_d[e2] = exact_d((int)(v >> 8), (int)(v & 255u));
          }
          __syncwarp();
          for (int e2 = incl - cnt; e2 < incl; ++e2) consider((int)(near_list[e2] & 255u), near_d[e2]);
          __syncwarp();  // the list is free for the next tile
        } else {
#pragma unroll
          for (int q = 0; q < kTcN / 32; ++q) {
            uint32_t cm = need ? cand[q] : 0u;
            while (cm) {
              const int r = 32 * q + __ffs(cm) - 1;
              cm &= cm - 1;
              consider(r, exact_d(row, r));
            }
          }
        }
        if (need) {
          result = bdi;
          ties += (sd <= bd * (1.f + 1e-6f)) ? 1 : 0;
        }
      }
      if (valid && !*failed) {
        const Plane P = plane_of(a, plane);
        if constexpr (kRoll) {
          uint8_t* out = ((P.b & 1) ? a.idx2 : a.idx) + (size_t)(P.b >> 1) * a.idx_layer +
                         (((size_t)P.beta * a.max_batch + rb) * a.H + P.h) * (size_t)a.max_pages * Lay::kPageBytes;
          out[(size_t)rnp * Lay::kPageBytes + page_byte(P.gi, rj, Lay::NG)] = (uint8_t)result;
        } else {
          uint8_t* out = a.idx + (((size_t)P.beta * a.max_batch + (a.seq_begin + P.b)) * a.H + P.h) *
                                     (size_t)a.max_pages * Lay::kPageBytes;
          out[(size_t)(a.page_begin + j / kPage) * Lay::kPageBytes + page_byte(a.g_begin + P.gi, j % kPage, Lay::NG)] =
              (uint8_t)result;
        }
      }
      __syncwarp();
      if (lane == 0) {  // this warp is done with the vector rows and the codebook
        mbar_arrive(&aempty[st]);
        if constexpr (kRoll) atomicAdd(&done[e], 1);  // after __syncwarp: the warp's reads are done
        else mbar_arrive(&bdone[e]);
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ties += __shfl_xor_sync(0xFFFFFFFFu, ties, off);
    if (lane == 0 && ties && a.n_ties) atomicAdd(a.n_ties, ties);
  }

  // ---- free TMEM once every warp is out of its loop (the MMA warp saw its last MMAs land) ----
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int TC, int C, bool kRoll>
cudaError_t launch_tc(const VqEncodeArgs& a, cudaStream_t s) {
  using Lay = TcLayout<TC, C, kRoll>;
  cudaError_t e =
      cudaFuncSetAttribute(encode_tc_kernel<TC, C, kRoll>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmemLaunch);
  if (e != cudaSuccess) return e;
  const int tiles = (a.n_tok + kTcM - 1) / kTcM;
  const long long U = (long long)a.n_seq * a.H * a.NB * tiles;  // (sequence, head, beta, tile) slots
  if (U * a.g_count >= (1ll << 31)) return cudaErrorInvalidValue;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // sets of g_count blocks (one per group), as many as fit one block per SM and have slots
  const long long sets = std::max(1ll, std::min<long long>(U, sms / std::max(1, a.g_count)));
  const long long blocks = sets * a.g_count;
  encode_tc_kernel<TC, C, kRoll><<<(unsigned)blocks, kEncThreads, Lay::kSmemLaunch, s>>>(a, (int)U, tiles);
  return cudaGetLastError();
}


template <bool kRoll>
cudaError_t launch_encode_any(const VqEncodeArgs& a, cudaStream_t s) {
  if (a.n_tok <= 0 || a.n_seq <= 0 || a.g_count <= 0) return cudaSuccess;
  const int C = a.G / a.Tc;
  if (a.Tc == 1 && C == 8) return launch_tc<1, 8, kRoll>(a, s);
  if (a.Tc == 2 && C == 8) return launch_tc<2, 8, kRoll>(a, s);
  if (a.Tc == 4 && C == 8) return launch_tc<4, 8, kRoll>(a, s);
  if (a.Tc == 1 && C == 16) return launch_tc<1, 16, kRoll>(a, s);
  if (a.Tc == 4 && C == 4) return launch_tc<4, 4, kRoll>(a, s);
  return cudaErrorInvalidValue;
}

template <int TC, int C>
cudaError_t launch_split(const float* cb, uint8_t* cbp, long long n, cudaStream_t s) {
  split_codebooks_kernel<TC, C><<<(unsigned)n, 256, 0, s>>>(cb, cbp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_vq_encode(const VqEncodeArgs& a, cudaStream_t s) { return launch_encode_any<false>(a, s); }
cudaError_t launch_vq_roll_tc(const VqEncodeArgs& a, cudaStream_t s) { return launch_encode_any<true>(a, s); }

size_t split_codebook_bytes(int G) { return (size_t)kParts * kTcN * tc_chunks(G / 8) * 16; }

cudaError_t launch_split_codebooks(const float* cb, uint8_t* cbp, long long n, int Tc, int G, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (n >= (1ll << 31)) return cudaErrorInvalidValue;
  const int C = G / Tc;
  if (Tc == 1 && C == 8) return launch_split<1, 8>(cb, cbp, n, s);
  if (Tc == 2 && C == 8) return launch_split<2, 8>(cb, cbp, n, s);
  if (Tc == 4 && C == 8) return launch_split<4, 8>(cb, cbp, n, s);
  if (Tc == 1 && C == 16) return launch_split<1, 16>(cb, cbp, n, s);
  if (Tc == 4 && C == 4) return launch_split<4, 4>(cb, cbp, n, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
