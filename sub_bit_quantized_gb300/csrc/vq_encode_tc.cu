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
// decided again in fp64 over the candidates in the band: the result is the exact argmin
// with the lowest index on exact ties, and a tie is reported when the runner-up's fp64
// distance is within 1e-6 (relative) of the best.
//
// GB300 mapping. One 128-thread block per (sequence, head, block beta, group) x 32 tiles of 128
// vectors. The block stages the three codebook parts in shared memory once (K-major, no
// swizzle: 8-row x 16-byte core matrices), holds a 128 x 256 fp32 accumulator in TMEM
// (256 columns), and per tile: threads load their vector rows, one thread issues the
// tcgen05.mma chain (3 parts x K steps of 16) and commits to an mbarrier, then each thread
// reads its accumulator row with tcgen05.ld and keeps the best two. Every wait is bounded.
#include <cuda_fp16.h>

#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "../../include/kvq.h"

namespace kvq {
namespace {

constexpr int kTcThreads = 128;      // one vector row per thread = one TMEM lane
constexpr int kTcM = 128;            // vectors per tile (MMA M)
constexpr int kTcN = 256;            // codewords (MMA N)
constexpr int kTilesPerBlock = 32;
constexpr uint32_t kTmemCols = 256;  // fp32 accumulator columns
constexpr int kParts = 3;            // hi, mid, lo bf16 parts of the fp32 codebook
constexpr int kTcMinSmem = 80 * 1024;  // keeps at most two blocks (2 x 256 TMEM columns) per SM

// 16-byte K chunks per row: TC chunks of data (8 coordinates of one loop step each), one
// augmented chunk (A: 1, 0..; B: -||e||^2 / 2, 0..), padded to whole MMA K steps of 32 bytes
__host__ __device__ constexpr int tc_chunks(int TC) { return 2 * ((TC + 2) / 2); }

template <int TC>
struct TcLayout {
  static constexpr int G = TC * kC;
  static constexpr int KC = tc_chunks(TC);
  static constexpr int kRowBytes = KC * 16;
  static constexpr int kABytes = kTcM * kRowBytes;          // one tile of vectors
  static constexpr int kBPartBytes = kTcN * kRowBytes;      // one codebook part
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kABytes;
  static constexpr int kOffCb = kOffB + kParts * kBPartBytes;  // fp32 codebook [256][G], chunk order
  static constexpr int kOffRed = kOffCb + kTcN * G * 4;         // float [4] block reduction
  static constexpr int kOffBar = kOffRed + 32;                  // mbarrier + TMEM address
  static constexpr int kBytes = kOffBar + 32;
  static constexpr int kSmem = kBytes > kTcMinSmem ? kBytes : kTcMinSmem;
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

__device__ __forceinline__ size_t page_byte_tc(int g, int j) {  // in-page byte of (group, token)
  return (size_t)(((g & 7) * kPage + (j & 7)) * 2 + (g >> 3));
}

template <int TC>
__global__ void __launch_bounds__(kTcThreads) encode_tc_kernel(const VqEncodeArgs a) {
  using Lay = TcLayout<TC>;
  constexpr int G = Lay::G, KC = Lay::KC;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char* sa = smem + Lay::kOffA;
  unsigned char* sb = smem + Lay::kOffB;
  float* cbp = reinterpret_cast<float*>(smem + Lay::kOffCb);
  uint64_t* mma_bar = reinterpret_cast<uint64_t*>(smem + Lay::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lay::kOffBar + 8);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + Lay::kOffBar + 12);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gq = blockIdx.y;  // (b, h, beta, gi) flattened
  const int gi = gq % a.g_count;
  const int beta = (gq / a.g_count) % a.NB;
  const int h = (gq / (a.g_count * a.NB)) % a.H;
  const int b = gq / (a.g_count * a.NB * a.H);
  const int g = a.g_begin + gi;

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

  // ---- codebook: three bf16 parts (with the -||e||^2/2 column) and an fp32 copy ----------
  // coordinate k' = c*8 + i of a row (chunk c < TC, i < 8) is coupled coordinate i*TC + c
  const float* cb = a.cb + (((size_t)beta * a.H + h) * kNG + g) * (size_t)kCB * G;
  for (int r = tid; r < kTcN; r += kTcThreads) {
    float e[G];
    double n2 = 0.0;
#pragma unroll
    for (int c = 0; c < TC; ++c)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        e[c * 8 + i] = __ldg(cb + (size_t)r * G + i * TC + c);
        n2 = fma((double)e[c * 8 + i], (double)e[c * 8 + i], n2);
      }
#pragma unroll
    for (int k = 0; k < G; ++k) cbp[r * G + k] = e[k];
    const float nh = (float)(-0.5 * n2);
    // parts: hi = bf16(v), mid = bf16(v - hi), lo = bf16(v - hi - mid)
    for (int c = 0; c < KC; ++c) {
      uint32_t w[kParts][4];
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) {
        uint16_t pb[kParts][2];
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int i = 2 * i2 + e2;
          float v = 0.f;
          if (c < TC) v = e[c * 8 + i];
          else if (c == TC && i == 0) v = nh;
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
  fence_proxy_async_smem();  // codebook parts are read by the tensor cores
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t my_lane_addr = tmem + ((uint32_t)(32 * warp) << 16);

  uint8_t* out = a.idx + (((size_t)beta * a.max_batch + (a.seq_begin + b)) * a.H + h) * (size_t)a.max_pages * kPageBytes;
  const int n_tiles = (a.n_tok + kTcM - 1) / kTcM;
  const int t_begin = blockIdx.x * kTilesPerBlock;
  const int t_end = min(n_tiles, t_begin + kTilesPerBlock);
  int ties = 0;
  uint32_t phase = 0;
  int pending = -1;  // thread 0: phase of an MMA chain whose completion it gave up waiting for
  // this thread's vector row of tile t (zeros past the end)
  auto load_row = [&](int t, uint4 (&zr)[TC]) {
    const int j = t * kTcM + tid;
#pragma unroll
    for (int m = 0; m < TC; ++m) {
      zr[m] = make_uint4(0, 0, 0, 0);
      if (t < t_end && j < a.n_tok) {
        const uint16_t* xp = a.x + (size_t)(beta * TC + m) * a.st + (size_t)b * a.sb + (size_t)h * a.sh +
                             (size_t)j * kD + g * kC;
        zr[m] = __ldg(reinterpret_cast<const uint4*>(xp));
      }
    }
  };
  uint4 znext[TC];
  load_row(t_begin, znext);
  for (int t = t_begin; t < t_end; ++t) {
    // ---- this thread's vector row -> A tile (chunks: TC data, ones column, zero pad) ----
    const int j = t * kTcM + tid;
    const bool valid = j < a.n_tok;
    uint4 zr[TC];
    float z2 = 0.f;
#pragma unroll
    for (int m = 0; m < TC; ++m) {
      zr[m] = znext[m];
      const uint32_t w4[4] = {zr[m].x, zr[m].y, zr[m].z, zr[m].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float lo = bf16_lo(w4[q]), hi = bf16_hi(w4[q]);
        z2 = fmaf(lo, lo, fmaf(hi, hi, z2));
      }
      *reinterpret_cast<uint4*>(sa + op_off(tid, m, KC)) = zr[m];
    }
#pragma unroll
    for (int c = TC; c < KC; ++c)
      *reinterpret_cast<uint4*>(sa + op_off(tid, c, KC)) = make_uint4(c == TC ? 0x3F80u : 0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();  // A tile written; the previous tile's accumulator reads are done

    // ---- one thread: 3 parts x K steps into the accumulator, commit -----------------------
    if (tid == 0 && !*failed) {
      tc_fence_after();
#pragma unroll
      for (int p = 0; p < kParts; ++p)
#pragma unroll
        for (int s = 0; s < KC / 2; ++s) {
          const uint64_t ad = umma_desc(smem_u32(sa) + s * 256, 128, KC * 128);
          const uint64_t bd = umma_desc(smem_u32(sb + p * Lay::kBPartBytes) + s * 256, 128, KC * 128);
          umma_bf16(tmem, ad, bd, (p | s) != 0);
        }
      umma_commit(mma_bar);
      if (!mbar_wait_bounded(mma_bar, phase)) {
        *failed = 1;
        pending = (int)phase;
        set_error(a.err, KVQ_ERR_TIMEOUT);
      }
    }
    phase ^= 1u;
    load_row(t + 1, znext);  // in flight during this tile's epilogue
    __syncthreads();  // thread 0 saw the accumulator complete (or gave up)
    tc_fence_after();

    // ---- epilogue: best and runner-up of acc_r = z.e_r - ||e_r||^2/2 over 256 columns ----
    float best = -INFINITY, second = -INFINITY;
    int bi = 0;
#pragma unroll 1
    for (int c0 = 0; c0 < kTcN; c0 += 32) {
      float v[32];
      tmem_ld32(my_lane_addr + c0, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const bool gt = v[i] > best;
        second = fmaxf(second, fminf(v[i], best));
        bi = gt ? c0 + i : bi;
        best = fmaxf(best, v[i]);
      }
    }
    // Error band in acc units. A codeword that can compete with the best lies within
    // |z| + sqrt(d_best) of the origin, and its acc = z.e - |e|^2/2 is accumulated over 3 x K/16
    // MMAs of exact bf16 products: its error is below about 3 (K/16) 17 2^-24 (|z||e| + |e|^2/2)
    // plus the 2^-24 |z||e| of the split. The band takes 8 times that for two candidates, plus
    // the 1e-6 tie threshold of the best distance.
    const float znorm = sqrtf(z2);
    const float dbest = fmaxf(0.f, z2 - 2.f * best);
    const float enear = znorm + 1.01f * sqrtf(dbest) + 1e-3f * znorm + 1e-6f;
    const float band = 8.f * 3.f * (KC / 2) * 18.f * 5.97e-8f * (znorm * enear + 0.5f * enear * enear) +
                       1e-6f * dbest + 1e-30f;
    const bool need = valid && !*failed && (second >= best - band);
    int result = bi;
    if (__any_sync(0xFFFFFFFFu, need)) {
      // exact decision over every candidate in the band, in fp64 (lowest index wins ties)
      float zf[G];
#pragma unroll
      for (int m = 0; m < TC; ++m) {
        const uint32_t w4[4] = {zr[m].x, zr[m].y, zr[m].z, zr[m].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          zf[m * 8 + 2 * q] = bf16_lo(w4[q]);
          zf[m * 8 + 2 * q + 1] = bf16_hi(w4[q]);
        }
      }
      double b64 = INFINITY, s64 = INFINITY;
      int b64i = bi;
#pragma unroll 1
      for (int c0 = 0; c0 < kTcN; c0 += 32) {
        float v[32];
        tmem_ld32(my_lane_addr + c0, v);  // every lane of the warp reads (the load is warp-wide)
        if (need) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (v[i] < best - band) continue;
            const int r = c0 + i;
            const float* er = cbp + r * G;
            double dd = 0.0;
#pragma unroll
            for (int k = 0; k < G; ++k) {
              const double df = (double)zf[k] - (double)er[k];
              dd = fma(df, df, dd);
            }
            if (dd < b64) {
              s64 = b64;
              b64 = dd;
              b64i = r;
            } else if (dd < s64) {
              s64 = dd;
            }
          }
        }
      }
      if (need) {
        result = b64i;
        ties += (s64 <= b64 * (1.0 + 1e-6)) ? 1 : 0;
      }
    }
    if (valid && !*failed) out[(size_t)(a.page_begin + j / kPage) * kPageBytes + page_byte_tc(g, j)] = (uint8_t)result;
    tc_fence_before();
  }

  // ---- tie count, then free TMEM (after the last MMA has landed) --------------------------
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) ties += __shfl_xor_sync(0xFFFFFFFFu, ties, off);
  if (lane == 0 && ties && a.n_ties) atomicAdd(a.n_ties, ties);
  if (tid == 0 && pending >= 0) mbar_wait_bounded(mma_bar, (uint32_t)pending);  // an MMA still in flight
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int TC>
cudaError_t launch_tc(const VqEncodeArgs& a, cudaStream_t s) {
  using Lay = TcLayout<TC>;
  cudaError_t e = cudaFuncSetAttribute(encode_tc_kernel<TC>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kSmem);
  if (e != cudaSuccess) return e;
  const long long planes = (long long)a.n_seq * a.H * a.NB * a.g_count;
  const int tiles = (a.n_tok + kTcM - 1) / kTcM;
  dim3 grid((tiles + kTilesPerBlock - 1) / kTilesPerBlock, (unsigned)planes);
  encode_tc_kernel<TC><<<grid, kTcThreads, Lay::kSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_vq_encode(const VqEncodeArgs& a, cudaStream_t s) {
  if (a.n_tok <= 0 || a.n_seq <= 0 || a.g_count <= 0) return cudaSuccess;
  switch (a.Tc) {
    case 1: return launch_tc<1>(a, s);
    case 2: return launch_tc<2>(a, s);
    case 4: return launch_tc<4>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
