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
// GB300 mapping. Persistent 512-thread blocks, two per SM (each holds a 128 x 256 fp32
// accumulator in 256 TMEM columns), over equal contiguous shares of the (plane, 128-vector
// tile) units, a plane being one (sequence, head, block beta, group) with its codebook. A
// block stages the three codebook parts in shared memory (K-major, no swizzle: 8-row x
// 16-byte core matrices) when its share enters a plane. Per tile: the block loads the vector
// rows into one of two A buffers, one thread issues the tcgen05.mma chain (3 parts x K steps
// of 16) and commits to an mbarrier; the four warpgroups each read 64 accumulator columns of
// every row (tcgen05.ld) and keep the best two; warpgroup 0 merges the four and writes the
// index while the others load the next tile. Every wait is bounded.
#include <cuda_fp16.h>

#include <algorithm>

#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "../../include/kvq.h"

namespace kvq {
namespace {

constexpr int kTcThreads = 512;      // 4 warpgroups; a thread reads one TMEM lane
constexpr int kTcM = 128;            // vectors per tile (MMA M)
constexpr int kTcN = 256;            // codewords (MMA N)
constexpr int kQCols = kTcN / 4;     // accumulator columns each warpgroup reads
constexpr uint32_t kTmemCols = 256;  // fp32 accumulator columns
constexpr int kParts = 3;            // hi, mid, lo bf16 parts of the fp32 codebook
constexpr int kTcBlocksPerSm = 2;    // 2 x 256 TMEM columns

// 16-byte K chunks per row: G/8 chunks of data (row coordinate k' = m c + i holds channel
// g c + i of loop step m, i.e. coupled coordinate i Tc + m), one augmented chunk (A: 1, 0..;
// B: -||e||^2 / 2, 0..), padded to whole MMA K steps of 32 bytes
__host__ __device__ constexpr int tc_chunks(int DC) { return 2 * ((DC + 2) / 2); }

template <int TC, int C>
struct TcLayout {
  static constexpr int G = TC * C;
  static constexpr int DC = G / 8;                          // data chunks per row
  static constexpr int NG = kD / C;                         // groups per token
  static constexpr int kPageBytes = kPage * NG;
  static constexpr int KC = tc_chunks(DC);
  static constexpr int kRowBytes = KC * 16;
  static constexpr int kABytes = kTcM * kRowBytes;          // one tile of vectors
  static constexpr int kBPartBytes = kTcN * kRowBytes;      // one codebook part
  static constexpr int kOffA = 0;                           // two tile buffers
  static constexpr int kOffB = kOffA + 2 * kABytes;
  static constexpr int kOffPart = kOffB + kParts * kBPartBytes;  // [row][warpgroup] best two
  static constexpr int kOffBar = kOffPart + kTcM * 4 * 16;       // mbarrier + TMEM address
  static constexpr int kSmem = kOffBar + 32;
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

// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint16_t bf16_rn_bits(float f) { return f32_to_bf16(f); }

// one warpgroup's share of a row: its maximum, the band it used, how many of its columns lie
// within that band of its maximum, and the first of them
struct Quarter {
  float best, band;
  int count, first;
};

// Error band in acc units for a row with |z|^2 = z2 whose best acc is `best`. A codeword that
// can compete with the best lies within |z| + sqrt(d_best) of the origin, and its
// acc = z.e - |e|^2/2 is accumulated over 3 x KC/2 MMAs of exact bf16 products: its error is
// below about 3 (KC/2) 17 2^-24 (|z||e| + |e|^2/2) plus the 2^-24 |z||e| of the split. The
// band takes 8 times that for two candidates, plus the 1e-6 tie threshold of the best
// distance. A larger `best` (a better candidate) never widens it.
template <int KC>
__device__ __forceinline__ float acc_band(float z2, float best) {
  const float znorm = sqrtf(z2);
  const float dbest = fmaxf(0.f, z2 - 2.f * best);
  const float enear = znorm + 1.01f * sqrtf(dbest) + 1e-3f * znorm + 1e-6f;
  return 8.f * 3.f * (KC / 2) * 18.f * 5.97e-8f * (znorm * enear + 0.5f * enear * enear) + 1e-6f * dbest + 1e-30f;
}

template <int TC, int C>
__global__ void __launch_bounds__(kTcThreads, kTcBlocksPerSm) encode_tc_kernel(const VqEncodeArgs a, const int U,
                                                                                const int tiles_per_plane) {
  using Lay = TcLayout<TC, C>;
  constexpr int G = Lay::G, KC = Lay::KC, DC = Lay::DC;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* sb = smem + Lay::kOffB;
  Quarter* part = reinterpret_cast<Quarter*>(smem + Lay::kOffPart);
  uint64_t* mma_bar = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffBar + 8);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + Lay::kOffBar + 12);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wg = warp >> 2;                    // warpgroup: accumulator columns 64 wg ..
  const int row = 32 * (warp & 3) + lane;      // TMEM lane = vector row of the tile
  const int lo = (int)((long long)U * blockIdx.x / gridDim.x), hi = (int)((long long)U * (blockIdx.x + 1) / gridDim.x);
  if (lo >= hi) return;

  // ---- TMEM accumulator (warp 0), barrier ----------------------------------------------
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    mbar_init(mma_bar, 1);
    *failed = 0;
    fence_mbar_init();
  }
  // constant chunks of both A buffers: the ones column, zero padding
  for (int i = tid; i < 2 * kTcM * (KC - DC); i += kTcThreads) {
    const int buf = i / (kTcM * (KC - DC)), rem = i % (kTcM * (KC - DC));
    const int r = rem / (KC - DC), c = DC + rem % (KC - DC);
    *reinterpret_cast<uint4*>(smem + Lay::kOffA + buf * Lay::kABytes + op_off(r, c, KC)) =
        make_uint4(c == DC ? 0x3F80u : 0u, 0u, 0u, 0u);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kQCols * wg;

  int ties = 0;
  uint32_t phase = 0;
  int pending = -1;  // thread 0: phase of an MMA chain whose completion it gave up waiting for
  int cur_plane = -1, buf = 0;
  const float* cb = nullptr;
  uint8_t* out = nullptr;
  int g = 0;
  // chunk i (< kTcM * DC) of unit u: 16 bytes of one vector row (zeros past the tokens):
  // row coordinates 8d .. 8d + 7 of chunk d are channels of one loop step (c >= 8) or of
  // two (c = 4)
  auto load_chunk = [&](int u) {
    uint4 v = make_uint4(0, 0, 0, 0);
    const int i = tid;
    if (u < hi && i < kTcM * DC) {
      const int pl = u / tiles_per_plane, tt = u - pl * tiles_per_plane;
      const int gi2 = pl % a.g_count, be = (pl / a.g_count) % a.NB, hh = (pl / (a.g_count * a.NB)) % a.H;
      const int bb = pl / (a.g_count * a.NB * a.H);
      const int r = i / DC, d = i % DC;
      const int j = tt * kTcM + r;
      if (j < a.n_tok) {
        const uint16_t* xr = a.x + (size_t)bb * a.sb + (size_t)hh * a.sh + (size_t)j * kD + (a.g_begin + gi2) * C;
        if constexpr (C >= 8) {
          v = __ldg(reinterpret_cast<const uint4*>(xr + (size_t)(be * TC + (8 * d) / C) * a.st + (8 * d) % C));
        } else {
          const uint2 w0 = __ldg(reinterpret_cast<const uint2*>(xr + (size_t)(be * TC + 2 * d) * a.st));
          const uint2 w1 = __ldg(reinterpret_cast<const uint2*>(xr + (size_t)(be * TC + 2 * d + 1) * a.st));
          v = make_uint4(w0.x, w0.y, w1.x, w1.y);
        }
      }
    }
    return v;
  };
  uint4 pre = load_chunk(lo);
  // descriptors of the operands: A buffer 0, codebook part 0 (the others are fixed offsets)
  const uint64_t a_desc0 = umma_desc(smem_u32(smem + Lay::kOffA), 128, KC * 128);
  const uint64_t b_desc0 = umma_desc(smem_u32(sb), 128, KC * 128);
  for (int u = lo; u < hi; ++u, buf ^= 1) {
    const int plane = u / tiles_per_plane, t = u - plane * tiles_per_plane;
    const int gi = plane % a.g_count;
    const int beta = (plane / a.g_count) % a.NB;
    const int h = (plane / (a.g_count * a.NB)) % a.H;
    const int b = plane / (a.g_count * a.NB * a.H);
    if (plane != cur_plane) {  // uniform
      // ---- codebook of this plane: three bf16 parts with the -||e||^2/2 column ------------
      // row coordinate k' = 8 c + i (chunk c < DC, i < 8) = m C + i2 is coupled coordinate i2 TC + m
      g = a.g_begin + gi;
      cb = a.cb + (((size_t)beta * a.H + h) * Lay::NG + g) * (size_t)kCB * G;
      out = a.idx + (((size_t)beta * a.max_batch + (a.seq_begin + b)) * a.H + h) * (size_t)a.max_pages * Lay::kPageBytes;
      __syncthreads();  // the previous plane's MMAs have all been waited for
      for (int r = tid; r < kTcN; r += kTcThreads) {
        float nh_hi = 0.f, nh_lo = 0.f;  // |e|^2, compensated
#pragma unroll 4
        for (int k = 0; k < G; ++k) add_sq_diff(__ldg(cb + (size_t)r * G + k), 0.f, nh_hi, nh_lo);
        const float nh = -0.5f * __fadd_rn(nh_hi, nh_lo);
        // one 16-byte chunk at a time; parts: hi = bf16(v), mid = bf16(v - hi), lo = bf16(v - hi - mid)
#pragma unroll 1
        for (int c = 0; c < KC; ++c) {
          uint32_t w[kParts][4];
#pragma unroll
          for (int i2 = 0; i2 < 4; ++i2) {
            uint16_t pb[kParts][2];
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const int i = 2 * i2 + e2;
              float v = 0.f;
              if (c < DC) {
                const int kk = 8 * c + i;
                v = __ldg(cb + (size_t)r * G + (kk % C) * TC + kk / C);
              } else if (c == DC && i == 0) {
                v = nh;
              }
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
      cur_plane = plane;
    }

    // ---- vector rows of tile t -> A buffer (DC 16-byte chunks per row); the next tile's
    //      rows are loaded now and land during this tile's work --------------------------------
    unsigned char* sa = smem + Lay::kOffA + buf * Lay::kABytes;
    static_assert(kTcM * DC <= kTcThreads, "one chunk per thread");
    if (tid < kTcM * DC) *reinterpret_cast<uint4*>(sa + op_off(tid / DC, tid % DC, KC)) = pre;
    pre = load_chunk(u + 1);
    fence_proxy_async_smem();  // A (and a new codebook) are read by the tensor cores
    tc_fence_before();
    __syncthreads();  // operands written; the previous tile's accumulator reads are done

    // ---- one thread: 3 parts x K steps into the accumulator, commit, wait ------------------
    if (tid == 0 && !*failed) {
      tc_fence_after();
      // start addresses advance in 16-byte units in the low descriptor bits (no carry: every
      // operand lies below 256 KB of shared memory)
#pragma unroll
      for (int p = 0; p < kParts; ++p)
#pragma unroll
        for (int s = 0; s < KC / 2; ++s)
          umma_bf16(tmem, a_desc0 + (uint64_t)((buf * Lay::kABytes + s * 256) >> 4),
                    b_desc0 + (uint64_t)((p * Lay::kBPartBytes + s * 256) >> 4), (p | s) != 0);
      umma_commit(mma_bar);
      if (!mbar_wait_bounded(mma_bar, phase)) {
        *failed = 1;
        pending = (int)phase;
        set_error(a.err, KVQ_ERR_TIMEOUT);
      }
    }
    phase ^= 1u;
    __syncthreads();  // thread 0 saw the accumulator complete (or gave up)
    tc_fence_after();

    // ---- each warpgroup, its 64 columns of the row: maximum of acc = z.e - |e|^2/2, then the
    //      columns within the error band of it (a bit mask per 32 columns) --------------------
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
    {
      float run = -INFINITY, cmax[kQCols / 32];
      uint32_t mask[kQCols / 32];
#pragma unroll
      for (int k = 0; k < kQCols / 32; ++k) {
        float v[32];
        tmem_ld32(lane_addr + 32 * k, v);
        float cm = v[0];
#pragma unroll
        for (int i = 1; i < 32; ++i) cm = fmaxf(cm, v[i]);
        run = fmaxf(run, cm);
        const float thr = run - acc_band<KC>(z2, run);
        uint32_t mk = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) mk |= (v[i] >= thr) ? (1u << i) : 0u;
        cmax[k] = cm;
        mask[k] = mk;
      }
      Quarter qr;
      qr.best = run;
      qr.band = acc_band<KC>(z2, run);
      qr.count = 0;
      qr.first = kTcN;
#pragma unroll
      for (int k = kQCols / 32 - 1; k >= 0; --k) {  // a chunk far below the maximum has no candidate
        if (cmax[k] < run - qr.band) continue;
        qr.count += __popc(mask[k]);
        if (mask[k]) qr.first = kQCols * wg + 32 * k + __ffs(mask[k]) - 1;
      }
      part[row * 4 + wg] = qr;
    }
    tc_fence_before();
    __syncthreads();  // the four quarters of every row are in shared memory

    // ---- warpgroup 0: merge the quarters; one candidate is the answer, several are decided
    //      on compensated distances --------------------------------------------------------------
    if (wg == 0) {
      float best = -INFINITY;
#pragma unroll
      for (int q = 0; q < 4; ++q) best = fmaxf(best, part[row * 4 + q].best);
      const float band = acc_band<KC>(z2, best);
      int count = 0, first = kTcN;
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // each quarter's band is at least this one: its mask covers
        const Quarter o = part[row * 4 + q];
        if (o.best < best - band) continue;
        count += o.count;
        first = min(first, o.first);
      }
      const int j = t * kTcM + row;
      const bool valid = j < a.n_tok;
      const bool need = valid && !*failed && count > 1;
      struct { float best; int col; } m = {best, first};
      int result = m.col;
      if (__any_sync(0xFFFFFFFFu, need)) {
        // every candidate in the band, decided on compensated fp32 distances (lowest index wins
        // exact ties); a runner-up within 1e-6 of the best is reported as a tie
        float bd = INFINITY, sd = INFINITY;
        int bdi = m.col;
        const uint32_t row_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
#pragma unroll 1
        for (int c0 = 0; c0 < kTcN; c0 += 32) {
          uint32_t cand = 0;  // columns of this chunk inside the band
          {
            float v[32];
            tmem_ld32(row_addr + c0, v);  // warp-wide load: every lane takes part
#pragma unroll
            for (int i = 0; i < 32; ++i) cand |= (v[i] >= m.best - band) ? (1u << i) : 0u;
          }
          if (!need) cand = 0;
          while (cand) {
            const int r = c0 + __ffs(cand) - 1;
            cand &= cand - 1;
            // e = hi + mid + lo exactly (each residual is a multiple of e's ulp that fits the
            // next part), so the staged parts give the fp32 entries back
            float dh = 0.f, dl = 0.f;
#pragma unroll 1
            for (int c = 0; c < DC; ++c) {
              const uint4 w = *reinterpret_cast<const uint4*>(sa + op_off(row, c, KC));
              const uint4 e0 = *reinterpret_cast<const uint4*>(sb + op_off(r, c, KC));
              const uint4 e1 = *reinterpret_cast<const uint4*>(sb + Lay::kBPartBytes + op_off(r, c, KC));
              const uint4 e2 = *reinterpret_cast<const uint4*>(sb + 2 * Lay::kBPartBytes + op_off(r, c, KC));
              const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
              const uint32_t h4[4] = {e0.x, e0.y, e0.z, e0.w}, m4[4] = {e1.x, e1.y, e1.z, e1.w},
                             l4[4] = {e2.x, e2.y, e2.z, e2.w};
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                add_sq_diff(bf16_lo(w4[q]), __fadd_rn(__fadd_rn(bf16_lo(h4[q]), bf16_lo(m4[q])), bf16_lo(l4[q])), dh, dl);
                add_sq_diff(bf16_hi(w4[q]), __fadd_rn(__fadd_rn(bf16_hi(h4[q]), bf16_hi(m4[q])), bf16_hi(l4[q])), dh, dl);
              }
            }
            const float dd = __fadd_rn(dh, dl);
            if (dd < bd) {  // columns are visited in increasing order: the lowest wins exact ties
              sd = bd;
              bd = dd;
              bdi = r;
            } else if (dd < sd) {
              sd = dd;
            }
          }
        }
        if (need) {
          result = bdi;
          ties += (sd <= bd * (1.f + 1e-6f)) ? 1 : 0;
        }
      }
      if (valid && !*failed)
        out[(size_t)(a.page_begin + j / kPage) * Lay::kPageBytes + page_byte(g, j % kPage, Lay::NG)] = (uint8_t)result;
    }
  }

  // ---- tie count, then free TMEM (after the last MMA has landed) --------------------------
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) ties += __shfl_xor_sync(0xFFFFFFFFu, ties, off);
  if (lane == 0 && ties && a.n_ties) atomicAdd(a.n_ties, ties);
  if (tid == 0 && pending >= 0) mbar_wait_bounded(mma_bar, (uint32_t)pending);  // an MMA still in flight
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int TC, int C>
cudaError_t launch_tc(const VqEncodeArgs& a, cudaStream_t s) {
  using Lay = TcLayout<TC, C>;
  cudaError_t e = cudaFuncSetAttribute(encode_tc_kernel<TC, C>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmem);
  if (e != cudaSuccess) return e;
  const long long planes = (long long)a.n_seq * a.H * a.NB * a.g_count;
  const int tiles = (a.n_tok + kTcM - 1) / kTcM;
  const long long U = planes * tiles;
  if (U >= (1ll << 31)) return cudaErrorInvalidValue;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long blocks = std::min<long long>(U, (long long)kTcBlocksPerSm * sms);
  encode_tc_kernel<TC, C><<<(unsigned)blocks, kTcThreads, Lay::kSmem, s>>>(a, (int)U, tiles);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_vq_encode(const VqEncodeArgs& a, cudaStream_t s) {
  if (a.n_tok <= 0 || a.n_seq <= 0 || a.g_count <= 0) return cudaSuccess;
  const int C = a.G / a.Tc;
  if (a.Tc == 1 && C == 8) return launch_tc<1, 8>(a, s);
  if (a.Tc == 2 && C == 8) return launch_tc<2, 8>(a, s);
  if (a.Tc == 4 && C == 8) return launch_tc<4, 8>(a, s);
  if (a.Tc == 1 && C == 16) return launch_tc<1, 16>(a, s);
  if (a.Tc == 4 && C == 4) return launch_tc<4, 4>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
