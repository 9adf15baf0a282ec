// KIVI KV cache: group quantization with 2- or 4-bit codes, the streaming cache of
// Algorithm 1 (prefill and decode append) and decode attention with grouped-query heads.
//
// "KIVI 完全拆解：非对称 2-bit KV Cache 量化":
//  * quantization-direction section: q = clamp(round(X/s + z), 0, 2^b - 1), X_hat = s(q - z),
//    [min, max] split evenly by s; keys per channel, values per token (core design);
//  * core design, eq. (3) and Algorithm 1: grouped (quantized) + fp16 residual segments,
//    logits of both concatenated before one softmax; during decoding a full key residual is
//    quantized whole and the value window drops its oldest token into the quantized part;
//  * implementation section: the Q_MatMul kernel fuses dequantization into the product;
//    key and value bit widths are configured independently (2 or 4); GQA.
//
// Quantize: one fp32 sequence (IEEE division, separate rounding of every step, round half
// to even) so codes, scales and zero-points match a reference that follows the same steps
// bit for bit. Attention: keys dequantize into the query instead of the cache -
// sum_ch q_ch s_ch (code - z_ch) = sum_ch (q_ch s_ch) code + bias - so each 32-token group
// folds its per-channel scale into the query once; values accumulate
// sum_j p_j s_jg code_j,ch and subtract sum_j p_j s_jg z_jg per channel group at the end.
// Under GQA one block serves up to four query heads of a KV head: the codes are read from
// HBM and unpacked once for all of them. With one query head per block the value codes feed
// the mixed-precision FMA directly (fp16 operands, fp32 sums) with the token weight p_j s_jg
// rounded to fp16 once (relative error 2^-12 per token, in the code and zero-point terms
// alike).
#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "../../include/kvq.h"

#include <cuda_fp16.h>

namespace kvq {
namespace {

constexpr int kGroup = 32;  // tokens per key group, channels per value group (checked by the host)

struct GroupQ {
  float s16f, z16f, rs;  // rs = 1 / s16f, correctly rounded
  uint16_t s_bits, z_bits;
};

template <int BITS>
__device__ __forceinline__ GroupQ group_params(float mn, float mx) {
  const float s = __fdiv_rn(__fsub_rn(mx, mn), (float)((1 << BITS) - 1));
  __half s16 = __float2half_rn(s);
  if (__half2float(s16) == 0.0f) s16 = __float2half_rn(1.0f);
  const float s16f = __half2float(s16);
  const __half z16 = __float2half_rn(__fdiv_rn(-mn, s16f));
  GroupQ g;
  g.s16f = s16f;
  g.rs = __frcp_rn(s16f);
  g.z16f = __half2float(z16);
  g.s_bits = __half_as_ushort(s16);
  g.z_bits = __half_as_ushort(z16);
  return g;
}

// The codes of four values x_i (group parameters g_i): clamp(rint(t_i), 0, 2^b - 1) with
// t = (x / s) + z, an IEEE division and a separate rounded add. t' = fma(x, 1/s, z) differs
// from t by at most about 2^-23 (|x / s| + |t'|) (one rounding each in 1/s, the fma, x / s
// and the add), so when every t'_i lies farther than four times that from the rounding
// boundary k + 1/2 nearest to it, rint(t) = rint(t') and the codes are the same; otherwise
// (about 1e-6 of the values, |t'| >= 2^23 and any NaN) the exact sequence decides all four.
template <int BITS>
__device__ __forceinline__ void quant_codes4(const float (&x)[4], const GroupQ* const (&g)[4], uint32_t (&c)[4]) {
  float k[4];
  bool fast = true;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float tf = __fmaf_rn(x[i], g[i]->rs, g[i]->z16f);
    k[i] = rintf(tf);
    const float bound = __fmul_rn(__fmaf_rn(fabsf(x[i]), g[i]->rs, fabsf(tf)), 4.8e-7f);  // 4 x 2^-23 (...)
    fast = fast && (fabsf(tf - k[i]) < 0.5f - bound);
  }
  if (!fast) {
#pragma unroll
    for (int i = 0; i < 4; ++i) k[i] = rintf(__fadd_rn(__fdiv_rn(x[i], g[i]->s16f), g[i]->z16f));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = (uint32_t)fminf(fmaxf(k[i], 0.0f), (float)((1 << BITS) - 1));
}

__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }

__device__ __forceinline__ void unpack4(const uint2 r, float v[4]) {
  v[0] = h2f(r.x & 0xFFFFu);
  v[1] = h2f(r.x >> 16);
  v[2] = h2f(r.y & 0xFFFFu);
  v[3] = h2f(r.y >> 16);
}

// The codes of a lane's four channels 4 lane .. 4 lane + 3 as stored: channel (8/b)k + i of a
// token sits in bits [b i, b i + b) of byte k, so 2-bit codes fill byte `lane` and 4-bit
// codes bytes 2 lane and 2 lane + 1.
template <int BITS>
__device__ __forceinline__ void store_codes4(uint8_t* row, int lane, const uint32_t c[4]) {
  if constexpr (BITS == 2) row[lane] = (uint8_t)(c[0] | (c[1] << 2) | (c[2] << 4) | (c[3] << 6));
  else *reinterpret_cast<uint16_t*>(row + 2 * lane) = (uint16_t)(c[0] | (c[1] << 4) | (c[2] << 8) | (c[3] << 12));
}

// 8 bytes of a row (4 fp16 values), through the read-only cache when the data is not written
// by the same kernel
template <bool kReadOnly>
__device__ __forceinline__ uint2 load_row(const uint16_t* p) {
  return kReadOnly ? __ldg(reinterpret_cast<const uint2*>(p)) : *reinterpret_cast<const uint2*>(p);
}

// One warp quantizes one 32-token key group over all 128 channels; lane l owns channels
// 4l .. 4l + 3, so each token row is one coalesced 256-byte read, all 32 rows in flight. The
// first pass finds each channel's minimum and maximum, the second reads the rows again (from
// L1: the warp read them just before) and writes the codes, so the rows need no registers.
// src: row j at src + j * src_row elements; codes: row j at codes + j * (D b / 8) bytes;
// scale / zero: the group's [D] row.
template <int BITS, bool kReadOnly>
__device__ __forceinline__ void quant_key_group(const uint16_t* src, size_t src_row, uint8_t* codes,
                                                uint16_t* scale, uint16_t* zero, int lane) {
  constexpr int kRow = kD * BITS / 8;
  const uint16_t* base = src + 4 * lane;
  float mn[4], mx[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    mn[i] = INFINITY;
    mx[i] = -INFINITY;
  }
#pragma unroll 8
  for (int j = 0; j < kGroup; ++j) {
    float v[4];
    unpack4(load_row<kReadOnly>(base + (size_t)j * src_row), v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      mn[i] = fminf(mn[i], v[i]);
      mx[i] = fmaxf(mx[i], v[i]);
    }
  }
  GroupQ g[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) g[i] = group_params<BITS>(mn[i], mx[i]);
  *reinterpret_cast<uint2*>(scale + 4 * lane) =
      make_uint2(g[0].s_bits | ((uint32_t)g[1].s_bits << 16), g[2].s_bits | ((uint32_t)g[3].s_bits << 16));
  *reinterpret_cast<uint2*>(zero + 4 * lane) =
      make_uint2(g[0].z_bits | ((uint32_t)g[1].z_bits << 16), g[2].z_bits | ((uint32_t)g[3].z_bits << 16));
#pragma unroll 8
  for (int j = 0; j < kGroup; ++j) {
    float v[4];
    unpack4(load_row<kReadOnly>(base + (size_t)j * src_row), v);
    uint32_t c[4];
    const GroupQ* const gp[4] = {&g[0], &g[1], &g[2], &g[3]};
    quant_codes4<BITS>(v, gp, c);
    store_codes4<BITS>(codes + (size_t)j * kRow, lane, c);
  }
}

// One warp quantizes one token's 128 values (four 32-channel groups): lane l owns channels
// 4l .. 4l + 3 (raw), the 8 lanes of a group reduce min and max by shuffles. All 32 lanes
// must call it. scale / zero: the token's [D/32] row.
template <int BITS>
__device__ __forceinline__ void quant_value_row(const uint2 raw, uint8_t* codes, uint16_t* scale, uint16_t* zero,
                                                int lane) {
  float v[4];
  unpack4(raw, v);
  float mn = fminf(fminf(v[0], v[1]), fminf(v[2], v[3]));
  float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
#pragma unroll
  for (int off = 4; off >= 1; off >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
  }
  const GroupQ g = group_params<BITS>(mn, mx);
  if ((lane & 7) == 0) {
    scale[lane >> 3] = g.s_bits;
    zero[lane >> 3] = g.z_bits;
  }
  uint32_t c[4];
  const GroupQ* const gp[4] = {&g, &g, &g, &g};
  quant_codes4<BITS>(v, gp, c);
  store_codes4<BITS>(codes, lane, c);
}

// ---------------------------------------------------------------- kvq_quantize_kivi
// Persistent warps, each with a one-tile stage of shared memory (8 KB: 32 tokens x 128
// channels of one (b, h)) filled by one bulk copy. A warp moves the tile into registers as
// packed halves (lane l: channels 4l .. 4l + 3 of every row, 64 registers) and at once
// issues the copy of its next tile into the stage, so the copy runs while it quantizes.
// A warp takes a contiguous range of the tiles.
constexpr int kQWarps = 16;
constexpr int kQThreads = kQWarps * 32;
constexpr int kQTileB = kGroup * kD * 2;
constexpr int kQParB = 8 * 4 * 16;  // per warp: (rs, z16, threshold, s16) of 8 rows x 4 groups
constexpr int kQOffPar = kQWarps * kQTileB;
constexpr int kQOffBar = kQOffPar + kQWarps * kQParB;
constexpr int kQSmem = kQOffBar + kQWarps * 8;
static_assert(kQSmem <= 232448, "shared memory");

// A group's quantization constants for the fast path. The per-value bound of quant_codes4,
// 4 x 2^-23 (|x / s| + |t'|), is at most 4.8e-7 (2 M / s + |z|) for every x of a group whose
// largest magnitude is M (|t'| <= |x| / s + |z|), so one threshold serves the whole group:
// rint(t') is the reading's code when |t' - rint(t')| < 0.5 - that bound. A group with
// infinite members gets a NaN or negative threshold and always takes the exact path; a NaN
// member fails its own comparison.
struct GroupF {
  float rs, z, th, s;
};
__device__ __forceinline__ GroupF group_fast(const GroupQ& g, float mn, float mx) {
  GroupF f;
  f.rs = g.rs;
  f.z = g.z16f;
  f.s = g.s16f;
  f.th = 0.5f - 4.8e-7f * (2.0f * fmaxf(fabsf(mn), fabsf(mx)) * g.rs + fabsf(g.z16f));
  return f;
}

__device__ __forceinline__ __half2 u2h2(uint32_t w) { return *reinterpret_cast<const __half2*>(&w); }
__device__ __forceinline__ uint32_t h22u(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }

// The codes of four values of (up to) four groups, packed as stored: code i in bits
// [b i, b i + b). The packing runs in float arithmetic on small integers (exact) above 2^23,
// whose low mantissa bits are then the packed codes.
template <int BITS, bool kClamp>
__device__ __forceinline__ uint32_t pack_codes4(const float (&k)[4]) {
  constexpr float kMax = (float)((1 << BITS) - 1);
  float c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = kClamp ? fminf(fmaxf(k[i], 0.0f), kMax) : k[i];
  float acc = c[0] + 8388608.0f;
#pragma unroll
  for (int i = 1; i < 4; ++i) acc = __fmaf_rn(c[i], (float)(1 << (BITS * i)), acc);
  return __float_as_uint(acc);
}

// Packed constants of a lane's four values: (rs, z, th) of channels (0, 1) and (2, 3).
struct Quad {
  float2 rs01, rs23, z01, z23, th01, th23;
};

// Fast codes of one row (four fp16 values): t' = fma(x, 1/s, z) and its rounding to nearest
// even by adding and removing 1.5 * 2^23 (exact for |t'| < 2^22), two values per packed
// operation; `bad` is set when a value lies too close to a rounding boundary (or is NaN, or
// |t'| is too large for the rounding: the threshold is negative then). kClamp: the group's
// extremes may round outside [0, 2^b - 1].
template <int BITS, bool kClamp>
__device__ __forceinline__ uint32_t row_codes_fast(const uint2 w, const Quad& q, bool& bad) {
  const float2 x01 = __half22float2(u2h2(w.x)), x23 = __half22float2(u2h2(w.y));
  const float2 M2 = make_float2(12582912.0f, 12582912.0f), nM2 = make_float2(-12582912.0f, -12582912.0f);
  const float2 m1 = make_float2(-1.0f, -1.0f);
  const float2 t01 = __ffma2_rn(x01, q.rs01, q.z01), t23 = __ffma2_rn(x23, q.rs23, q.z23);
  const float2 k01 = __fadd2_rn(__fadd2_rn(t01, M2), nM2), k23 = __fadd2_rn(__fadd2_rn(t23, M2), nM2);
  const float2 d01 = __ffma2_rn(k01, m1, t01), d23 = __ffma2_rn(k23, m1, t23);
  bad = !(fabsf(d01.x) < q.th01.x) || !(fabsf(d01.y) < q.th01.y) || !(fabsf(d23.x) < q.th23.x) ||
        !(fabsf(d23.y) < q.th23.y);
  const float k[4] = {k01.x, k01.y, k23.x, k23.y};
  return pack_codes4<BITS, kClamp>(k);
}

// The reading's sequence for one row: rint(x / s + z), clamped
template <int BITS>
__device__ __forceinline__ uint32_t row_codes_exact(const uint2 w, const GroupF (&g)[4]) {
  float x[4], k[4];
  unpack4(w, x);
#pragma unroll
  for (int i = 0; i < 4; ++i) k[i] = rintf(__fadd_rn(__fdiv_rn(x[i], g[i].s), g[i].z));
  return pack_codes4<BITS, true>(k);
}

// true when every x of the group [mn, mx] has a fast-path code inside [0, 2^b - 1]: t' and
// its rounding are monotone in x, so the extremes decide
template <int BITS>
__device__ __forceinline__ bool group_in_range(const GroupF& f, float mn, float mx) {
  const float lo = rintf(__fmaf_rn(mn, f.rs, f.z)), hi = rintf(__fmaf_rn(mx, f.rs, f.z));
  return lo >= 0.0f && hi <= (float)((1 << BITS) - 1);
}

template <int BITS>
__device__ __forceinline__ void store_packed4(uint8_t* row, int lane, uint32_t packed) {
  if constexpr (BITS == 2) row[lane] = (uint8_t)packed;
  else *reinterpret_cast<uint16_t*>(row + 2 * lane) = (uint16_t)packed;
}


// keys of one tile (held as t[row] = the lane's 4 fp16 channels): one 32-token group per
// channel. Minimum and maximum on packed halves (exact: the order of fp16 values is that of
// their fp32 conversions), then the codes.
template <int BITS>
__device__ __forceinline__ void quant_key_tile(const uint2 (&t)[kGroup], const uint16_t* gsrc, uint8_t* codes,
                                               uint16_t* scale, uint16_t* zero, int lane) {
  constexpr int kRow = kD * BITS / 8;
  __half2 mn0 = u2h2(t[0].x), mn1 = u2h2(t[0].y), mx0 = mn0, mx1 = mn1;
#pragma unroll
  for (int j = 1; j < kGroup; ++j) {
    mn0 = __hmin2(mn0, u2h2(t[j].x));
    mn1 = __hmin2(mn1, u2h2(t[j].y));
    mx0 = __hmax2(mx0, u2h2(t[j].x));
    mx1 = __hmax2(mx1, u2h2(t[j].y));
  }
  const float2 a0 = __half22float2(mn0), a1 = __half22float2(mn1), b0 = __half22float2(mx0), b1 = __half22float2(mx1);
  const float mn[4] = {a0.x, a0.y, a1.x, a1.y}, mx[4] = {b0.x, b0.y, b1.x, b1.y};
  GroupF f[4];
  uint32_t sb[4], zb[4];
  bool in_range = true;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const GroupQ g = group_params<BITS>(mn[i], mx[i]);
    f[i] = group_fast(g, mn[i], mx[i]);
    in_range = in_range && group_in_range<BITS>(f[i], mn[i], mx[i]);
    sb[i] = g.s_bits;
    zb[i] = g.z_bits;
  }
  *reinterpret_cast<uint2*>(scale + 4 * lane) = make_uint2(sb[0] | (sb[1] << 16), sb[2] | (sb[3] << 16));
  *reinterpret_cast<uint2*>(zero + 4 * lane) = make_uint2(zb[0] | (zb[1] << 16), zb[2] | (zb[3] << 16));
  const Quad q = {make_float2(f[0].rs, f[1].rs), make_float2(f[2].rs, f[3].rs), make_float2(f[0].z, f[1].z),
                  make_float2(f[2].z, f[3].z),   make_float2(f[0].th, f[1].th), make_float2(f[2].th, f[3].th)};
  uint32_t badrows = 0;
  if (__all_sync(0xFFFFFFFFu, in_range)) {
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      bool bad;
      store_packed4<BITS>(codes + (size_t)j * kRow, lane, row_codes_fast<BITS, false>(t[j], q, bad));
      badrows |= (uint32_t)bad << j;
    }
  } else {
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      bool bad;
      store_packed4<BITS>(codes + (size_t)j * kRow, lane, row_codes_fast<BITS, true>(t[j], q, bad));
      badrows |= (uint32_t)bad << j;
    }
  }
  while (badrows) {  // rare: rows with a value near a rounding boundary, re-read from HBM
    const int j = __ffs(badrows) - 1;
    badrows &= badrows - 1;
    store_packed4<BITS>(codes + (size_t)j * kRow, lane,
                        row_codes_exact<BITS>(__ldg(reinterpret_cast<const uint2*>(gsrc + (size_t)j * kD + 4 * lane)), f));
  }
}

// fast codes of rows r0 .. r0 + 7 of a value tile (constants of row k, group grp at
// par[4 k + grp]); returns the rows (bit k) with a value near a rounding boundary
template <int BITS, bool kClamp>
__device__ __forceinline__ uint32_t value_rows8(const uint2 (&t)[kGroup], const int r0, const int rows,
                                                uint8_t* codes, const float4* par, const int grp, const int lane) {
  constexpr int kRow = kD * BITS / 8;
  uint32_t badrows = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float4 p = par[k * 4 + grp];
    const Quad q = {make_float2(p.x, p.x), make_float2(p.x, p.x), make_float2(p.y, p.y),
                    make_float2(p.y, p.y), make_float2(p.z, p.z), make_float2(p.z, p.z)};
    bool bad;
    const uint32_t c = row_codes_fast<BITS, kClamp>(t[r0 + k], q, bad);
    if (r0 + k < rows) {
      store_packed4<BITS>(codes + (size_t)(r0 + k) * kRow, lane, c);
      badrows |= (uint32_t)bad << k;
    }
  }
  return badrows;
}

// values of one tile (rows < 32 valid), 8 rows at a time: lane l holds channels 4l .. 4l + 3
// of each row, i.e. group l / 8. Each row's (min, -max) over the lane's 4 channels is one
// packed half pair; a transposing reduction over the 8 lanes of a group leaves lane 8g + k
// with row k's extremes of group g. That lane computes the group's constants once, writes
// its scale and zero-point, and posts the constants for the other lanes in shared memory.
template <int BITS>
__device__ __forceinline__ void quant_value_tile(const uint2 (&t)[kGroup], const uint16_t* gsrc, int rows,
                                                 uint8_t* codes, uint16_t* scale, uint16_t* zero, float4* par,
                                                 int lane) {
  constexpr int kRow = kD * BITS / 8;
  const int kk = lane & 7, grp = lane >> 3;
#pragma unroll
  for (int r0 = 0; r0 < kGroup; r0 += 8) {
    if (r0 >= rows) break;  // uniform across the warp
    uint32_t e[8];  // (min, -max) of row r0 + k over the lane's channels
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const __half2 m = __hmin2(u2h2(t[r0 + k].x), u2h2(t[r0 + k].y));
      const uint32_t nM = h22u(__hmax2(u2h2(t[r0 + k].x), u2h2(t[r0 + k].y))) ^ 0x80008000u;
      const uint32_t um = h22u(m);
      e[k] = h22u(__hmin2(u2h2(__byte_perm(um, nM, 0x5410)), u2h2(__byte_perm(um, nM, 0x7632))));
    }
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1) {
      const bool up = (lane & w) != 0;
#pragma unroll
      for (int k = 0; k < w; ++k) {
        const uint32_t send = up ? e[k] : e[k + w], keep = up ? e[k + w] : e[k];
        e[k] = h22u(__hmin2(u2h2(keep), u2h2(__shfl_xor_sync(0xFFFFFFFFu, send, w))));
      }
    }
    const float2 ex = __half22float2(u2h2(e[0]));
    const float mn = ex.x, mx = -ex.y;
    const GroupQ g = group_params<BITS>(mn, mx);
    const GroupF f = group_fast(g, mn, mx);
    const bool in_range = group_in_range<BITS>(f, mn, mx) || r0 + kk >= rows;
    if (r0 + kk < rows) {  // lane 8 grp + kk: row r0 + kk, group grp
      scale[(size_t)(r0 + kk) * (kD / kGroup) + grp] = g.s_bits;
      zero[(size_t)(r0 + kk) * (kD / kGroup) + grp] = g.z_bits;
    }
    par[kk * 4 + grp] = make_float4(f.rs, f.z, f.th, f.s);
    __syncwarp();
    uint32_t badrows;
    if (__all_sync(0xFFFFFFFFu, in_range))
      badrows = value_rows8<BITS, false>(t, r0, rows, codes, par, grp, lane);
    else
      badrows = value_rows8<BITS, true>(t, r0, rows, codes, par, grp, lane);
    while (badrows) {  // rare: rows with a value near a rounding boundary, re-read from HBM
      const int k = __ffs(badrows) - 1;
      badrows &= badrows - 1;
      const float4 p = par[k * 4 + grp];
      const GroupF gk = {p.x, p.y, p.z, p.w};
      const GroupF gg[4] = {gk, gk, gk, gk};
      store_packed4<BITS>(codes + (size_t)(r0 + k) * kRow, lane,
                          row_codes_exact<BITS>(__ldg(reinterpret_cast<const uint2*>(gsrc + (size_t)(r0 + k) * kD + 4 * lane)), gg));
    }
    __syncwarp();  // before the constants are overwritten
  }
}

template <int BITS, bool kKeys>
__global__ void __launch_bounds__(kQThreads, 1) kivi_quant_kernel(const KiviQuantArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int kRow = kD * BITS / 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned char* stage = smem + warp * kQTileB;
  float4* par = reinterpret_cast<float4*>(smem + kQOffPar + warp * kQParB);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kQOffBar) + warp;
  const int n_gi = (a.n_tok + kGroup - 1) / kGroup;
  const long long T = (long long)a.B * a.H * n_gi;
  const long long W = (long long)gridDim.x * kQWarps, gw = (long long)blockIdx.x * kQWarps + warp;
  const long long t0 = T * gw / W, t1 = T * (gw + 1) / W;
  if (lane == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  auto tile_rows = [&](long long t) { return min(kGroup, a.n_tok - (int)(t % n_gi) * kGroup); };
  auto issue = [&](long long t) {  // lane 0: tile t into the stage
    const long long bh = t / n_gi;
    const int gi = (int)(t - bh * n_gi), b = (int)(bh / a.H), h = (int)(bh - (long long)b * a.H);
    const uint16_t* src = a.x + (size_t)b * a.sb + (size_t)h * a.sh + (size_t)gi * kGroup * kD;
    const uint32_t bytes = (uint32_t)tile_rows(t) * kD * 2;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(stage, src, bytes, bar);
  };
  if (lane == 0 && t0 < t1) issue(t0);
  for (long long t = t0; t < t1; ++t) {
    if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(bar, (uint32_t)((t - t0) & 1)))) {
      // the copy did not land in time: record it, let it land (bounded) and leave
      if (lane == 0) {
        set_error(a.err, KVQ_ERR_TIMEOUT);
        mbar_wait_bounded(bar, (uint32_t)((t - t0) & 1));
      }
      __syncwarp();
      return;
    }
    uint2 tl[kGroup];
    const uint16_t* tp = reinterpret_cast<const uint16_t*>(stage) + 4 * lane;
#pragma unroll
    for (int j = 0; j < kGroup; ++j) tl[j] = *reinterpret_cast<const uint2*>(tp + j * kD);
    const int rows = tile_rows(t);
    __syncwarp();  // every lane has its rows: the stage takes the next tile
    if (lane == 0 && t + 1 < t1) issue(t + 1);
    const long long bh = t / n_gi;
    const int gi = (int)(t - bh * n_gi), b = (int)(bh / a.H), h = (int)(bh - (long long)b * a.H);
    const uint16_t* gsrc = a.x + (size_t)b * a.sb + (size_t)h * a.sh + (size_t)gi * kGroup * kD;
    const size_t tok = (size_t)bh * a.max_tokens + a.tok_begin + (size_t)gi * kGroup;
    if constexpr (kKeys) {
      const size_t sz = ((size_t)bh * (a.max_tokens / kGroup) + a.tok_begin / kGroup + gi) * kD;
      quant_key_tile<BITS>(tl, gsrc, a.codes + tok * kRow, a.scale + sz, a.zero + sz, lane);
    } else {
      quant_value_tile<BITS>(tl, gsrc, rows, a.codes + tok * kRow, a.scale + tok * (kD / kGroup),
                             a.zero + tok * (kD / kGroup), par, lane);
    }
  }
}

// ---------------------------------------------------------------- streaming cache
// Prefill tail: block (b, h) copies tokens [nq, n) to the residuals (keys from row 0, values
// at row t % R) and block (b, 0) sets the request's lengths.
__global__ void __launch_bounds__(128) kivi_prefill_tail_kernel(const KiviTailArgs a) {
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int n_tail = a.n_tok_new - a.nq;
  const size_t row0 = ((size_t)(a.b0 + b) * a.H + h) * a.residual;
  const uint16_t* ks = a.k + (size_t)b * a.sb + (size_t)h * a.sh + (size_t)a.nq * kD;
  const uint16_t* vs = a.v + (size_t)b * a.sb + (size_t)h * a.sh + (size_t)a.nq * kD;
  for (int i = tid; i < n_tail * (kD / 8); i += blockDim.x) {  // one 16-byte piece per thread
    const int r = i / (kD / 8), c8 = (i % (kD / 8)) * 8;
    const int slot = (a.nq + r) % a.residual;
    *reinterpret_cast<uint4*>(a.k_resid + (row0 + r) * kD + c8) = __ldg(reinterpret_cast<const uint4*>(ks + (size_t)r * kD + c8));
    *reinterpret_cast<uint4*>(a.v_resid + (row0 + slot) * kD + c8) = __ldg(reinterpret_cast<const uint4*>(vs + (size_t)r * kD + c8));
  }
  if (h == 0 && tid == 0) {
    a.n_tok[a.b0 + b] = a.n_tok_new;
    a.n_quant_k[a.b0 + b] = a.nq;
    a.n_quant_v[a.b0 + b] = a.nq;
  }
}

// Decode append: one 128-thread block per (request, KV head). Every block of a request reads
// the request's lengths and takes the same decisions; the last block of the request to finish
// (an arrival counter in the cache's sync array) advances the lengths, so no block reads them
// after they changed. Quantization (a key flush: warp w takes 32-token groups w, w + 4, ...;
// a value eviction: warp 0) reads the residual rows before the barrier; the new token is
// written after it, because the evicted value and the new value share a ring row and the
// flushed key residual restarts at row 0.
template <int KB, int VB>
__global__ void __launch_bounds__(128) kivi_append_kernel(const KiviAppendArgs a) {
  constexpr int kKRow = kD * KB / 8, kVRow = kD * VB / 8;
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_warps = blockDim.x >> 5;
  const int R = a.residual, H = a.H;
  const int n = a.n_tok[b], nqk = a.n_quant_k[b], nqv = a.n_quant_v[b];
  const bool valid = nqk >= 0 && nqk % kGroup == 0 && nqv >= 0 && nqv <= nqk && nqk <= n && n - nqv <= R &&
                     nqk <= a.max_tokens;
  const bool flush = valid && (n - nqk == R);
  if (!valid || (flush && nqk + R > a.max_tokens)) {  // every block of the request leaves it as it is
    if (h == 0 && tid == 0) set_error(a.err, KVQ_ERR_CAPACITY);
    return;
  }
  const bool evict = (n + 1 - nqv > R);
  const size_t bh = (size_t)b * H + h;
  if (flush) {
    for (int gi = warp; gi < R / kGroup; gi += n_warps) {
      const size_t sz = (bh * (a.max_tokens / kGroup) + nqk / kGroup + gi) * kD;
      quant_key_group<KB, false>(a.k_resid + (bh * R + (size_t)gi * kGroup) * kD, kD,
                                 a.k_codes + (bh * a.max_tokens + nqk + (size_t)gi * kGroup) * kKRow, a.k_scale + sz,
                                 a.k_zero + sz, lane);
    }
  }
  if (evict && warp == 0) {
    const uint2 raw = *reinterpret_cast<const uint2*>(a.v_resid + (bh * R + nqv % R) * kD + 4 * lane);
    const size_t tok = bh * a.max_tokens + nqv;
    quant_value_row<VB>(raw, a.v_codes + tok * kVRow, a.v_scale + tok * (kD / kGroup), a.v_zero + tok * (kD / kGroup),
                        lane);
  }
  __syncthreads();
  const int kslot = flush ? 0 : n - nqk, vslot = n % R;
  if (tid < 2 * (kD / 8)) {  // 16 threads per fp16 row: the key, then the value
    const int c8 = (tid % (kD / 8)) * 8;
    const bool is_v = tid >= kD / 8;
    const uint4 x = __ldg(reinterpret_cast<const uint4*>((is_v ? a.v_new : a.k_new) + bh * kD + c8));
    uint16_t* dst = is_v ? a.v_resid + (bh * R + vslot) * kD : a.k_resid + (bh * R + kslot) * kD;
    *reinterpret_cast<uint4*>(dst + c8) = x;
  }
  __syncthreads();
  if (tid == 0 && atomicAdd(&a.sync[b], 1) == H - 1) {  // every block of the request has read the lengths
    a.n_tok[b] = n + 1;
    if (flush) a.n_quant_k[b] = nqk + R;
    if (evict) a.n_quant_v[b] = nqv + 1;
    a.sync[b] = 0;
  }
}

// ---------------------------------------------------------------- attention
// Blocks (split, head subgroup) x request x KV head; splits 0 .. n_split-1 take equal token
// ranges of the quantized keys, the last split the fp16 key residual. A subgroup is RH query
// heads of the KV head (RH = 4 when the GQA ratio allows), and the blocks of one split's
// subgroups are adjacent in launch order so their code reads meet in L2. A quantized split
// streams its tokens through a 3- or 4-stage shared-memory ring of 128-token chunks (TMA bulk
// copies of the chunk's key codes, key scales and zeros, value codes, value scales and
// zeros); each warp takes its tokens of a chunk (one head: a whole 32-token key group of
// every other chunk; RH > 1 heads: 16 tokens of every chunk), computes their scores (RH > 1:
// a tensor-core product per key group, fp16 code fragments against q' = q s split into fp16
// high and low parts; one head: on the CUDA cores), keeps its own online softmax per query
// head, and sums the values on the CUDA cores; the block merges the warps at the end. Tokens whose key is quantized but whose
// value is still in the fp16 window (the streaming cache's tail) take the value from the
// window. Partials of all splits merge exactly in the last block of a (request, subgroup) to
// finish (arrival counter, no spin-wait).
constexpr int kAThreads = 256;
constexpr int kAWarps = kAThreads / 32;
constexpr int kAChunk = 128;  // tokens per ring stage (4 key groups of 32)

template <int KB, int VB, int RH>
struct AttnLayout {
  // ring depth: 4 stages of 12 KB at 2 bits; 3 of up to 20 KB at 4 bits, so that three blocks
  // of the multi-head-group variants fit an SM
  static constexpr int kAStages = (KB + VB >= 6) ? 3 : 4;
  // resident blocks per SM the register budget targets: four with one query head and 2-bit
  // codes (64 registers), three otherwise, two for 2-bit values with four heads (64
  // accumulators a thread)
  static constexpr int kMinBlocks = (RH == 1) ? ((KB + VB == 4) ? 4 : 3) : (VB == 2 && RH == 4) ? 2 : 3;
  // log2 headroom of each warp's running maximum: weights p = exp2(s - M) stay below
  // 2^kSlack. One head rounds its value weights p s_v to fp16, so p <= 4 keeps |p s_v| <=
  // 4 (131008 / 15) < 65504 for any fp16 values; grouped heads keep their weights in fp32
  static constexpr float kSlack = (RH == 1) ? 2.f : 8.f;
  // tokens a warp takes of a chunk it works on: with one head a whole 32-token key group
  // (warps 0-3 on even chunks, 4-7 on odd ones), so a warp builds its group's q' alone and
  // no pair of warps meets; with grouped heads 16, the m16n8k16 tile's rows
  static constexpr int kTPW = (RH == 1) ? 32 : 16;
  static constexpr int kWPC = kAChunk / kTPW;             // warps per chunk
  static constexpr int kNPar = kAThreads / 32 / kWPC;     // chunk parities
  static constexpr int kKRow = kD * KB / 8;               // key code bytes per token
  static constexpr int kVRow = kD * VB / 8;               // value code bytes per token
  static constexpr int kCKc = 0;                          // stage layout (bytes)
  static constexpr int kCKs = kCKc + kAChunk * kKRow;     // key scales [4 groups][128] fp16
  static constexpr int kCKz = kCKs + 4 * kD * 2;
  static constexpr int kCVc = kCKz + 4 * kD * 2;
  static constexpr int kCVs = kCVc + kAChunk * kVRow;     // value scales [128 tokens][4 groups] fp16
  static constexpr int kCVz = kCVs + kAChunk * 4 * 2;
  static constexpr int kStage = kCVz + kAChunk * 4 * 2;
  static constexpr int kOffQ = kAStages * kStage;         // float q [RH][128]
  // q': with grouped heads the B fragments of the 4 key groups (4 x kQfWords words); with one
  // head a float [128] per warp (each warp takes a whole key group, below)
  static constexpr int kOffQf = kOffQ + RH * kD * 4;
  static constexpr int kOffBias = kOffQf + ((RH == 1) ? kAThreads / 32 : RH * 4) * kD * 4;  // float [RH][4 groups][2 halves]
  // float l [8 warps][RH], float M [8 warps][RH], int flag, int released [stages], int issued
  static constexpr int kOffRed = kOffBias + RH * 8 * 4;
  static constexpr int kOffBar = kOffRed + ((2 * kAWarps * RH + 2 + kAStages) * 4 + 15) / 16 * 16;  // mbarriers + failed
  // With grouped heads the scores are a tensor-core product (with one head the CUDA-core
  // path, below, measured faster): the q' area holds each key group's B fragments
  // ([k-step pair][kNC columns][4 threads][k-step parity][2 registers] words, so a thread
  // loads two k-steps with one 16-byte read; head r's high q' parts in column 2 r, its low
  // parts in 2 r + 1), and each warp's [16 tokens][RH heads] scores pass through
  // kOffS to the lanes that own the tokens
  static constexpr int kNC = 2 * RH;                      // B columns in use (of 8)
  static constexpr int kQfWords = 8 * kNC * 4 * 2;        // per key group (= RH 128 floats)
  static_assert(KB == 2 || KB == 4, "2- or 4-bit keys");
  static constexpr int kWPS = 16 * KB / 32;               // code words per 16-channel k-step
  static constexpr bool kMma = RH > 1;
  static constexpr int kOffS = kOffBar + 64;
  static constexpr int kSmem = kOffS + (kMma ? kAWarps * 16 * RH * 4 : 0);
  // value phase: a lane takes kLW code words of one token, all in one value group (with one
  // query head the whole group, so its scale and zero-point are read once); a warp-step
  // covers kTS tokens
  static constexpr int kVW = kVRow / 4;                   // code words per token
  static constexpr int kCPWv = 32 / VB;                   // value channels per word
  static constexpr int kPV = kCPWv / 2;                   // channel pairs per word
  static constexpr int kWPG = kGroup / kCPWv;             // words per value group
  static constexpr int kLW = (RH == 1 && VB == 4) ? kWPG : 1;  // words per lane
  static constexpr int kLPT = kVW / kLW;                  // lanes per token
  static constexpr int kTS = 32 / kLPT;                   // tokens per warp-step
  static constexpr int kOV = kLW * kCPWv;                 // value accumulators per lane and head
  // one-head score phase: a lane covers 64 channels of one token
  static constexpr int kKW = kKRow / 8;                   // key code words per half token
  static constexpr int kPK = 16 / KB;                     // channel pairs per key word
  static_assert(kStage % 128 == 0 && kOffBar % 8 == 0, "alignment");
  static_assert(kAWarps * RH * kD * 4 <= kAStages * kStage, "block reduction fits in the ring");
};

// Codes j and j + 16/b (j < 16/b) of a 32-bit word of b-bit codes, each as (code * 2^(b j))
// in fp32: the code is masked in place inside the mantissa of 2^23 and 2^23 is subtracted,
// all exact. A byte permute puts each 16-bit half of the word under the exponent of 2^23
// once per word (magic_lo / magic_hi); then every code costs one AND with an immediate and
// every pair one packed add, instead of shift + int-to-float conversion. The 2^(-b j) scale
// is folded into the other operand.
constexpr uint32_t kMagic = 0x4B000000u;  // 2^23
__device__ __forceinline__ uint32_t magic_lo(uint32_t w) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, 0x7410;" : "=r"(r) : "r"(w), "r"(kMagic));
  return r;
}
__device__ __forceinline__ uint32_t magic_hi(uint32_t w) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, 0x7432;" : "=r"(r) : "r"(w), "r"(kMagic));
  return r;
}
template <int BITS>
__device__ __forceinline__ float2 code_pair(uint32_t ml, uint32_t mh, int j) {
  const uint32_t m = (((1u << BITS) - 1u) << (BITS * j)) | kMagic;
  const float2 f = make_float2(__uint_as_float(ml & m), __uint_as_float(mh & m));
  return __fadd2_rn(f, make_float2(-8388608.f, -8388608.f));
}
// One query head per block (no grouped heads): the value codes go straight into the
// mixed-precision FMA (fp16 operands, fp32 sums), one FMA per code and no conversion. A masked
// code word is read as two fp16 bit patterns; an integer pattern n below 2^11 is exactly the
// fp16 n * 2^-24 (subnormal below 2^10, the first binade above), so code c at bit position k
// of a half reads as c * 2^(k - 24). Codes j < kSplit of each half are masked in place; the
// rest come from the word shifted right by b * kSplit. Accumulator pair (2j, 2j + 1) therefore
// holds 2^(b jj - 24) * sum(w c) with jj = j or j - kSplit (value_scale_exp gives b jj - 24),
// w being the token's weight p * s_v rounded to fp16 once.
template <int BITS>
struct HalfCodes {
  static constexpr int kSplit = (BITS == 2) ? 5 : 2;  // codes per half below bit 11
  static __device__ __forceinline__ int value_scale_exp(int j) { return BITS * (j < kSplit ? j : j - kSplit) - 24; }
};
// a0 += lo16(m) * wh, a1 += hi16(m) * wh, lo16 / hi16 and wh (low 16 bits) as fp16
__device__ __forceinline__ void fma_f16x2(float& a0, float& a1, uint32_t m, uint32_t wh) {
  asm("{\n\t.reg .b16 l, h, p;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.u16.u32 p, %3;\n\t"
      "fma.rn.f32.f16 %0, l, p, %0;\n\t"
      "fma.rn.f32.f16 %1, h, p, %1;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "r"(m), "r"(wh));
}
// a (low 16 bits, fp16) x b (low 16 bits, fp16) + c, product and sum in fp32
__device__ __forceinline__ float fma_f16_f32(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 x, y;\n\t"
      "cvt.u16.u32 x, %1;\n\t"
      "cvt.u16.u32 y, %2;\n\t"
      "fma.rn.f32.f16 %0, x, y, %3;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}
template <bool B>
struct BoolTag {
  static constexpr bool value = B;
};
// barrier of the two warps 2g and 2g + 1 (named barrier 1 + g, 64 threads)
__device__ __forceinline__ void pair_sync(int g) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + g) : "memory");
}
// K consecutive 32-bit words from shared memory (p aligned to 4 K bytes)
template <int K>
__device__ __forceinline__ void load_words(const unsigned char* p, uint32_t (&w)[K]) {
  if constexpr (K == 4) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else if constexpr (K == 2) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x; w[1] = v.y;
  } else {
    static_assert(K == 1, "1, 2 or 4 words");
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  }
}
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }
__device__ __forceinline__ float pow2_pos(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// position of channel c (< 64) of a key half in the query pair layout: word k = c / (32/b),
// within it pair j and member (low or high half word)
template <int BITS>
__device__ __forceinline__ int qpair_index(int c, int& j) {
  constexpr int kCPW = 32 / BITS, kP = kCPW / 2;
  const int k = c / kCPW, p = c % kCPW;
  j = p % kP;
  return 2 * (k * kP + j) + p / kP;
}

// D += A B for one m16n8k16 tile: fp16 A (16 x 16, row-major) and B (16 x 8, column-major)
// fragments, fp32 accumulators (the warp-wide tensor-core product of this architecture's
// instruction set; a 16-token x 8-head tile is below the smallest tcgen05 shape)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// The A fragments of one 16-channel k-step from the code words of two token rows (wa: row
// g8, wb: row g8 + 8; kWPS words each), thread t4 taking byte t4 of each word. A code c at
// bit k of a 16-bit half reads as the fp16 subnormal c 2^(k-24), exact, so every register is
// one byte permute (sel puts byte t4 under both halves) and one AND; the 2^k is folded into
// that channel's q'.
//   4-bit: byte t4 of word 0 (1) holds channels 2 t4, 2 t4 + 1 (+ 8) as (c, 16 c): k-step
//          columns 2 t4, 2 t4 + 1 (+ 8) are the channels in order.
//   2-bit: byte t4 of the word holds channels 4 t4 .. 4 t4 + 3 as (c, 4 c) and (16 c, 64 c):
//          columns 2 t4, 2 t4 + 1 are channels 4 t4, 4 t4 + 1, columns 2 t4 + 8, 2 t4 + 9
//          channels 4 t4 + 2, 4 t4 + 3.
template <int KB>
__device__ __forceinline__ void code_frag(const uint32_t* wa, const uint32_t* wb, uint32_t sel, uint32_t (&af)[4]) {
  if constexpr (KB == 4) {
    af[0] = __byte_perm(wa[0], 0u, sel) & 0x00F0000Fu;
    af[1] = __byte_perm(wb[0], 0u, sel) & 0x00F0000Fu;
    af[2] = __byte_perm(wa[1], 0u, sel) & 0x00F0000Fu;
    af[3] = __byte_perm(wb[1], 0u, sel) & 0x00F0000Fu;
  } else {
    const uint32_t pa = __byte_perm(wa[0], 0u, sel), pb = __byte_perm(wb[0], 0u, sel);
    af[0] = pa & 0x000C0003u;
    af[1] = pb & 0x000C0003u;
    af[2] = pa & 0x00C00030u;
    af[3] = pb & 0x00C00030u;
  }
}

__device__ __forceinline__ bool kivi_wait(uint64_t* bar, uint32_t parity, volatile int* failed, int* err) {
  if (*failed) return false;
  if (mbar_wait_bounded(bar, parity)) return true;
  *failed = 1;
  set_error(err, KVQ_ERR_TIMEOUT);
  return false;
}

template <int KB, int VB, int RH>
__global__ void __launch_bounds__(kAThreads, AttnLayout<KB, VB, RH>::kMinBlocks)
    kivi_attn_kernel(const KiviAttnArgs a, const float scale_log2) {
  using L = AttnLayout<KB, VB, RH>;
  extern __shared__ __align__(128) unsigned char sma[];
  float* qs = reinterpret_cast<float*>(sma + L::kOffQ);
  float* qf = reinterpret_cast<float*>(sma + L::kOffQf);
  float* bias = reinterpret_cast<float*>(sma + L::kOffBias);
  float* red = reinterpret_cast<float*>(sma + L::kOffRed);  // l per warp and head
  float* redm = red + kAWarps * RH;                          // running max per warp and head
  int* flag = reinterpret_cast<int*>(redm + kAWarps * RH);
  int* released = flag + 1;                                  // warps done with a stage's chunk
  int* issued = released + L::kAStages;                      // chunks whose copies were issued
  uint64_t* full = reinterpret_cast<uint64_t*>(sma + L::kOffBar);
  volatile int* failed = reinterpret_cast<volatile int*>(sma + L::kOffBar + L::kAStages * 8);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rep = a.Hq / a.H, n_sub = rep / RH;
  const int split = blockIdx.x / n_sub, sub = blockIdx.x % n_sub, b = blockIdx.y, hk = blockIdx.z;
  const int n_total = gridDim.x / n_sub;  // token splits; the last one also takes the fp16 residual
  const int R = a.residual;
  const bool has_resid = (R > 0) && (split == n_total - 1);
  const size_t bh = (size_t)b * a.H + hk;                       // KV row of (b, hk)
  const size_t bq0 = (size_t)b * a.Hq + (size_t)hk * rep + sub * RH;  // first query row
  const int NQK = min(max(a.n_quant_k[b], 0), a.max_tokens) / kGroup * kGroup;
  const int NQV = (R > 0) ? min(max(a.n_quant_v[b], 0), NQK) : NQK;
  for (int i = tid; i < RH * kD; i += kAThreads) qs[i] = bf16_to_f32(a.q[bq0 * kD + i]);
  if (tid == 0) {
    for (int s = 0; s < L::kAStages; ++s) {
      mbar_init(&full[s], 1);
      released[s] = 0;
    }
    *issued = 0;
    *failed = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // running softmax state per query head, per warp; a lane holds the kOV channels of code
  // words kLW (lane % kLPT) .. + kLW - 1 of its token slot (kTS token slots per warp step)
  float M[RH], l[RH], oz[RH];
  float o[RH][L::kOV];
  const int lt = lane % L::kLPT, ts = lane / L::kLPT;
  const int w0 = lt * L::kLW, gv = w0 / L::kWPG;  // the lane's first code word, its value group
#pragma unroll
  for (int r = 0; r < RH; ++r) {
    M[r] = -INFINITY;
    l[r] = 0.f;
    oz[r] = 0.f;
#pragma unroll
    for (int i = 0; i < L::kOV; ++i) o[r][i] = 0.f;
  }
  // raise head r's running max to Mn
  auto rescale_to = [&](int r, float Mn) {
    const float f = (M[r] == -INFINITY) ? 0.f : exp2f(M[r] - Mn);
#pragma unroll
    for (int i = 0; i < L::kOV; ++i) o[r][i] *= f;
    oz[r] *= f;
    l[r] *= f;
    M[r] = Mn;
  };
  // the lane's value channels of fp16 value-ring row t % R, weighted by p[r]
  auto value_fp16 = [&](int t, const float (&p)[RH]) {
#pragma unroll
    for (int w = 0; w < L::kLW; ++w) {
      const uint4* vr = reinterpret_cast<const uint4*>(a.v_resid + (bh * R + t % R) * kD + (w0 + w) * L::kCPWv);
      uint32_t hv[L::kCPWv / 2];
#pragma unroll
      for (int k4 = 0; k4 < L::kCPWv / 8; ++k4) {
        const uint4 u = __ldg(vr + k4);
        hv[4 * k4] = u.x;
        hv[4 * k4 + 1] = u.y;
        hv[4 * k4 + 2] = u.z;
        hv[4 * k4 + 3] = u.w;
      }
#pragma unroll
      for (int j = 0; j < L::kPV; ++j) {
        const int e0 = j, e1 = L::kPV + j, i = w * L::kCPWv + 2 * j;
        const float v0 = h2f((e0 & 1) ? (hv[e0 >> 1] >> 16) : (hv[e0 >> 1] & 0xFFFFu));
        const float v1 = h2f((e1 & 1) ? (hv[e1 >> 1] >> 16) : (hv[e1 >> 1] & 0xFFFFu));
        // the scale of accumulator pair j: 2^(b j) for grouped heads, 2^(b jj - 24) for one head
        const float sj = (RH == 1) ? pow2_pos(HalfCodes<VB>::value_scale_exp(j)) : pow2_pos(VB * j);
#pragma unroll
        for (int r = 0; r < RH; ++r) {
          o[r][i] = fmaf(p[r] * sj, v0, o[r][i]);
          o[r][i + 1] = fmaf(p[r] * sj, v1, o[r][i + 1]);
        }
      }
    }
  };

  {
    // ================================ quantized keys ========================================
    const int t0 = split * a.tok_per_split;
    const int t1 = min(NQK, t0 + a.tok_per_split);
    const int n_tok = max(0, t1 - t0);
    const int n_chunks = (n_tok + kAChunk - 1) / kAChunk;
    const size_t tok0 = bh * a.max_tokens;              // token row base of (b, hk)
    const size_t grp0 = bh * (a.max_tokens / kGroup);   // key group row base of (b, hk)
    auto produce = [&](int c) {                         // thread 0
      const int st = c % L::kAStages;
      unsigned char* dst = sma + st * L::kStage;
      const int t = t0 + c * kAChunk;
      const int n = min(kAChunk, t1 - t), ng = n / kGroup;
      mbar_arrive_expect_tx(&full[st], (uint32_t)(n * (L::kKRow + L::kVRow) + ng * kD * 2 * 2 + n * 8 * 2));
      bulk_g2s(dst + L::kCKc, a.k_codes + (tok0 + t) * L::kKRow, n * L::kKRow, &full[st]);
      bulk_g2s(dst + L::kCVc, a.v_codes + (tok0 + t) * L::kVRow, n * L::kVRow, &full[st]);
      bulk_g2s(dst + L::kCKs, a.k_scale + (grp0 + t / kGroup) * kD, ng * kD * 2, &full[st]);
      bulk_g2s(dst + L::kCKz, a.k_zero + (grp0 + t / kGroup) * kD, ng * kD * 2, &full[st]);
      bulk_g2s(dst + L::kCVs, a.v_scale + (tok0 + t) * 4, n * 8, &full[st]);
      bulk_g2s(dst + L::kCVz, a.v_zero + (tok0 + t) * 4, n * 8, &full[st]);
    };
    if (tid == 0) {
      for (int c = 0; c < min(L::kAStages, n_chunks); ++c) produce(c);
      *issued = min(L::kAStages, n_chunks);
    }

    // Every warp works on its kTPW tokens of each chunk it takes with a warp-local online
    // softmax, warps meet only at the end, and the last warp done with a stage refills it.
    // Grouped heads: 16 tokens of every chunk (half of one key group); the two warps of a
    // group share its q' fragments and bias (each builds one channel half; a 64-thread named
    // barrier per pair before and after). One head: a whole key group of every other chunk,
    // q' in the warp's own area and the bias in a register.
    const int wc = warp % L::kWPC;                     // the warp's slot in its chunks
    const int tb = L::kTPW * wc, g = (RH == 1) ? wc : warp >> 1, hf = warp & 1;
    for (int c = warp / L::kWPC; c < n_chunks; c += L::kNPar) {
      const int st = c % L::kAStages;
      kivi_wait(&full[st], (c / L::kAStages) & 1, failed, a.err);  // a timeout leaves stale data: harmless, reported
      const unsigned char* stage = sma + st * L::kStage;
      const int tc0 = t0 + c * kAChunk;  // token of chunk row 0
      const int n = min(kAChunk, t1 - tc0);  // a multiple of 32: a key group's warps have all its tokens or none
      float bias_w = 0.f;                    // one head: -sum q' z of the warp's key group
      if (tb < n && RH == 1) {
        // ---- one head: q' = q s of key group g (the scale folds into the query) in the code-
        //      pair order of each 64-channel half, divided by 2^(b j); lane l builds channels
        //      2 l, 2 l + 1 of both halves ----
        float* qr = qf + warp * kD;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int ch = 64 * hh + 2 * lane;
          const uint32_t s2 = *reinterpret_cast<const uint32_t*>(stage + L::kCKs + (g * kD + ch) * 2);
          const uint32_t z2 = *reinterpret_cast<const uint32_t*>(stage + L::kCKz + (g * kD + ch) * 2);
          const float qa = qs[ch] * h2f(s2 & 0xFFFFu), qb = qs[ch + 1] * h2f(s2 >> 16);
          int ja, jb;
          const int ia = qpair_index<KB>(2 * lane, ja), ib = qpair_index<KB>(2 * lane + 1, jb);
          qr[64 * hh + ia] = qa * pow2_neg(KB * ja);
          qr[64 * hh + ib] = qb * pow2_neg(KB * jb);
          bias_w -= qa * h2f(z2 & 0xFFFFu) + qb * h2f(z2 >> 16);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) bias_w += __shfl_xor_sync(0xFFFFFFFFu, bias_w, off);
        __syncwarp();  // q' written before the lanes read it
      }
      if (tb < n) {
        if constexpr (RH > 1) {
        // ---- grouped heads: q' = q s per key group and bias = -sum q' z; warp hf builds
        //      channels 64 hf .. 64 hf + 63 ----
        pair_sync(g);  // the partner is done reading the previous chunk's q'
        {
          const int ch = 64 * hf + 2 * lane;
          const uint32_t s2 = *reinterpret_cast<const uint32_t*>(stage + L::kCKs + (g * kD + ch) * 2);
          const uint32_t z2 = *reinterpret_cast<const uint32_t*>(stage + L::kCKz + (g * kD + ch) * 2);
          const float sa = h2f(s2 & 0xFFFFu), sb = h2f(s2 >> 16), za = h2f(z2 & 0xFFFFu), zb = h2f(z2 >> 16);
          // channels (ch, ch + 1) are one fp16 pair of the B fragments of k-step ch / 16 (thread
          // t4, register reg), each channel's q' divided by the power of two its code carries in
          // the A fragment (code_frag)
          int t4, reg;
          float fa = 1.f, fb;
          if constexpr (KB == 4) {
            t4 = (ch & 7) >> 1, reg = (ch >> 3) & 1, fb = 0.0625f;
          } else {
            t4 = (ch & 15) >> 2, reg = (ch >> 1) & 1, fa = reg ? 0.0625f : 1.f, fb = reg ? 0.015625f : 0.25f;
          }
          const int kk = ch >> 4;
          uint32_t* qbf = reinterpret_cast<uint32_t*>(qf) + g * L::kQfWords + ((kk >> 1) * L::kNC * 4 + t4) * 4 + (kk & 1) * 2 + reg;
#pragma unroll
          for (int r = 0; r < RH; ++r) {
            const float qa = qs[r * kD + ch] * sa, qb = qs[r * kD + ch + 1] * sb;
            {  // q' = hi + lo in fp16: column 2 r holds the high parts, 2 r + 1 the low
              const float qe = qa * fa, qo = qb * fb;
              const __half he = __float2half_rn(qe), ho = __float2half_rn(qo);
              const __half le = __float2half_rn(qe - __half2float(he)), lo = __float2half_rn(qo - __half2float(ho));
              qbf[(2 * r) * 4 * 4] = (uint32_t)__half_as_ushort(he) | ((uint32_t)__half_as_ushort(ho) << 16);
              qbf[(2 * r + 1) * 4 * 4] = (uint32_t)__half_as_ushort(le) | ((uint32_t)__half_as_ushort(lo) << 16);
            }
            float pb = -(qa * za + qb * zb);
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) pb += __shfl_xor_sync(0xFFFFFFFFu, pb, off);
            if (lane == 0) bias[(r * 4 + g) * 2 + hf] = pb;
          }
        }
        pair_sync(g);  // both halves written
        }
        // ---- scores of the warp's kTPW tokens ----
        float pk[RH];
        float raw[RH];  // dot products q' . codes: lane l's token (grouped heads: l and l + 16 share token l)
        if constexpr (L::kMma) {
          // scores[16 tokens][RH heads] = codes[16 x 128] . q'[128 x RH] on the tensor cores, one
          // m16n8k16 product per 16 channels: the A fragments come straight from the code bytes
          // (tokens tb + g8 and tb + g8 + 8, byte t4 of the k-step's words), the B fragments from
          // the q' area; column 2 r holds head r's high q' parts and 2 r + 1 its low parts, so
          // thread (g8, t4 < RH) ends with head t4's two partial sums of both tokens. Scores reach
          // the lanes of their tokens through the warp's kOffS area.
          const int g8 = lane >> 2, t4 = lane & 3;
          const uint32_t sel = (uint32_t)t4 * 0x101u + 0x4040u;
          const unsigned char* rowa = stage + L::kCKc + (tb + g8) * L::kKRow;
          const unsigned char* rowb = rowa + 8 * L::kKRow;
          const uint32_t* qbf = reinterpret_cast<const uint32_t*>(qf) + g * L::kQfWords + (g8 * 4 + t4) * 4;
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int w4 = 0; w4 < L::kKRow / 16; ++w4) {  // 4 code words of both rows
            const uint4 ua = *reinterpret_cast<const uint4*>(rowa + 16 * w4);
            const uint4 ub = *reinterpret_cast<const uint4*>(rowb + 16 * w4);
            const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
#pragma unroll
            for (int h2 = 0; h2 < 2 / L::kWPS; ++h2) {  // k-steps kk, kk + 1: one B load
              const int kk = (4 / L::kWPS) * w4 + 2 * h2;
              uint4 bq = make_uint4(0u, 0u, 0u, 0u);
              if (g8 < L::kNC) bq = *reinterpret_cast<const uint4*>(qbf + (kk >> 1) * L::kNC * 4 * 4);
              uint32_t af[4];
              code_frag<KB>(wa + L::kWPS * 2 * h2, wb + L::kWPS * 2 * h2, sel, af);
              mma_16816(acc, af, bq.x, bq.y);
              code_frag<KB>(wa + L::kWPS * (2 * h2 + 1), wb + L::kWPS * (2 * h2 + 1), sel, af);
              mma_16816(acc, af, bq.z, bq.w);
            }
          }
          float* ss = reinterpret_cast<float*>(sma + L::kOffS) + warp * 16 * RH;
          if (t4 < RH) {  // head t4 of tokens g8, g8 + 8 (x 2^24: the codes' fp16 scale)
            ss[g8 * RH + t4] = (acc[0] + acc[1]) * 16777216.f;
            ss[(g8 + 8) * RH + t4] = (acc[2] + acc[3]) * 16777216.f;
          }
          __syncwarp();
#pragma unroll
          for (int r = 0; r < RH; ++r) raw[r] = ss[(lane & 15) * RH + r];
          __syncwarp();  // read before the next chunk overwrites it
        } else {
          // one head: lane l takes all 128 channels of token tb + l, one 64-channel half at a
          // time; a byte permute per code word puts the codes under the exponent of 2^23, then
          // one AND per code, one packed add and one packed FMA per code pair
          const float* qw = qf + warp * kD;
          float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t wds[L::kKW];
#pragma unroll
            for (int k4 = 0; k4 < L::kKW / 4; ++k4) {
              const uint4 cw = *reinterpret_cast<const uint4*>(stage + L::kCKc + (tb + lane) * L::kKRow + hh * (L::kKRow / 2) + 16 * k4);
              wds[4 * k4] = cw.x;
              wds[4 * k4 + 1] = cw.y;
              wds[4 * k4 + 2] = cw.z;
              wds[4 * k4 + 3] = cw.w;
            }
#pragma unroll
            for (int k = 0; k < L::kKW; ++k) {
              const uint32_t ml = magic_lo(wds[k]), mh = magic_hi(wds[k]);
#pragma unroll
              for (int j = 0; j < L::kPK; j += 2) {  // two code pairs per 16-byte q' load
                const float4 q4 = *reinterpret_cast<const float4*>(qw + 64 * hh + 2 * (k * L::kPK + j));
                acc2 = __ffma2_rn(make_float2(q4.x, q4.y), code_pair<KB>(ml, mh, j), acc2);
                acc2 = __ffma2_rn(make_float2(q4.z, q4.w), code_pair<KB>(ml, mh, j + 1), acc2);
              }
            }
          }
          raw[0] = acc2.x + acc2.y;
        }
        // ---- warp-local online softmax over the warp's kTPW tokens ----
        constexpr int kRed = L::kTPW / 2;  // first xor distance of the reductions over the tokens
#pragma unroll
        for (int r = 0; r < RH; ++r) {
          const float bsum = (RH == 1) ? bias_w : bias[(r * 4 + g) * 2] + bias[(r * 4 + g) * 2 + 1];
          const float sc_r = (raw[r] + bsum) * scale_log2;
          float mx = sc_r;
#pragma unroll
          for (int off = kRed; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
          // the running maximum is raised only when a score passes it by more than kSlack (or
          // on the first chunk): the sums stay exact relative to M, and most chunks skip the
          // rescale (warp-uniform)
          if (mx > M[r] + L::kSlack) rescale_to(r, mx);
          pk[r] = exp2f(sc_r - M[r]);
          float ls = pk[r];
#pragma unroll
          for (int off = kRed; off >= 1; off >>= 1) ls += __shfl_xor_sync(0xFFFFFFFFu, ls, off);
          l[r] += ls;
        }
        // ---- values: kTS tokens of the warp per step ----
        // kFull: every token of the warp has a quantized value, so the steps need no per-token
        // test (warp-uniform; only the streaming cache's tail takes the checked path)
        auto value_steps = [&](auto full_tag) {
          constexpr bool kFull = decltype(full_tag)::value;
#pragma unroll
          for (int step = 0; step < L::kTPW / L::kTS; ++step) {
            float p[RH];
#pragma unroll
            for (int r = 0; r < RH; ++r) p[r] = __shfl_sync(0xFFFFFFFFu, pk[r], L::kTS * step + ts);
            const int tv = tb + L::kTS * step + ts;
            if (kFull || tc0 + tv < NQV) {
              uint32_t wv[L::kLW];
              load_words<L::kLW>(stage + L::kCVc + tv * L::kVRow + 4 * w0, wv);
              const uint32_t svh = *reinterpret_cast<const uint16_t*>(stage + L::kCVs + (tv * 4 + gv) * 2);
              const uint32_t zvh = *reinterpret_cast<const uint16_t*>(stage + L::kCVz + (tv * 4 + gv) * 2);
              if constexpr (RH == 1) {
                // the weight fp16(p) x s_v in one half multiply (p <= 2^kSlack); the zero-point
                // term takes the same rounded weight, through the mixed-precision FMA
                const __half wgt = __hmul(__float2half_rn(p[0]), __ushort_as_half((unsigned short)svh));
                const uint32_t wh = __half_as_ushort(wgt);
                oz[0] = fma_f16_f32(wh, zvh, oz[0]);
                constexpr int kSp = HalfCodes<VB>::kSplit;
#pragma unroll
                for (int w = 0; w < L::kLW; ++w) {
                  const uint32_t hi_codes = wv[w] >> (VB * kSp);
#pragma unroll
                  for (int j = 0; j < L::kPV; ++j) {  // (channel j, channel kPV + j) of the word
                    const int jj = (j < kSp) ? j : j - kSp;
                    const uint32_t m = ((j < kSp) ? wv[w] : hi_codes) & ((((1u << VB) - 1u) << (VB * jj)) * 0x10001u);
                    const int i = w * L::kCPWv + 2 * j;
                    fma_f16x2(o[0][i], o[0][i + 1], m, wh);
                  }
                }
              } else {
                const float sv = h2f(svh), zv = h2f(zvh);
                float2 w2[RH];
#pragma unroll
                for (int r = 0; r < RH; ++r) {
                  const float wgt = p[r] * sv;
                  oz[r] = fmaf(wgt, zv, oz[r]);
                  w2[r] = make_float2(wgt, wgt);
                }
#pragma unroll
                for (int w = 0; w < L::kLW; ++w) {
                  const uint32_t ml = magic_lo(wv[w]), mh = magic_hi(wv[w]);
#pragma unroll
                  for (int j = 0; j < L::kPV; ++j) {  // (channel j, channel kPV + j) of the word, x 2^(b j)
                    const float2 cp = code_pair<VB>(ml, mh, j);
                    const int i = w * L::kCPWv + 2 * j;
#pragma unroll
                    for (int r = 0; r < RH; ++r) {
                      const float2 acc = __ffma2_rn(w2[r], cp, make_float2(o[r][i], o[r][i + 1]));
                      o[r][i] = acc.x;
                      o[r][i + 1] = acc.y;
                    }
                  }
                }
              }
            } else {  // key quantized, value still in the fp16 window
              value_fp16(tc0 + tv, p);
            }
          }
        };
        if (tc0 + tb + L::kTPW <= NQV) value_steps(BoolTag<true>{});
        else value_steps(BoolTag<false>{});
      }
      // ---- this warp is done with the stage; the last one refills it ----
      __syncwarp();
      if (lane == 0 && atom_add_acq_rel_shared(&released[st], 1) == L::kWPC - 1) {
        released[st] = 0;
        if (c + L::kAStages < n_chunks && !*failed) {
          fence_proxy_async_smem();
          produce(c + L::kAStages);
          atomicAdd(issued, 1);
        }
      }
    }
    __syncthreads();  // every warp is out of the loop
    // after a timed-out wait, let this block's copies still in flight land first
    if (tid == 0 && *failed)
      for (int c = max(0, *issued - L::kAStages); c < *issued; ++c)
        mbar_wait_bounded(&full[c % L::kAStages], (c / L::kAStages) & 1);
  }
  if (has_resid) {
    // ============ fp16 residual (keys and values), after the last split's quantized keys ============
    // warp w takes residual tokens 16 w .. 16 w + 15 of every 128: scores with lanes 0-15 on
    // channels 0-63 and lanes 16-31 on 64-127, the same warp-local softmax, then the values
    // from the fp16 ring
    const int NR = max(0, min(a.n_tok[b] - NQK, R));
    for (int rb = 0; rb < NR; rb += 16 * kAWarps) {
      const int tw = rb + 16 * warp;
      if (tw >= NR) continue;  // warp-uniform
      const int rr = tw + (lane & 15), chh = lane >> 4;
      const bool valid = rr < NR;
      float acc[RH];
#pragma unroll
      for (int r = 0; r < RH; ++r) acc[r] = 0.f;
      const uint4* kr = reinterpret_cast<const uint4*>(a.k_resid + (bh * R + min(rr, NR - 1)) * kD + 64 * chh);
#pragma unroll 1
      for (int k8 = 0; k8 < 8; ++k8) {
        const uint4 v = __ldg(kr + k8);
        const uint32_t hw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hw[i]));
#pragma unroll
          for (int r = 0; r < RH; ++r) {
            const float2 q2 = *reinterpret_cast<const float2*>(qs + r * kD + 64 * chh + 8 * k8 + 2 * i);
            acc[r] = fmaf(q2.x, f.x, fmaf(q2.y, f.y, acc[r]));
          }
        }
      }
      float pk[RH];
#pragma unroll
      for (int r = 0; r < RH; ++r) {
        float sc_r = acc[r] + __shfl_xor_sync(0xFFFFFFFFu, acc[r], 16);
        sc_r = valid ? sc_r * scale_log2 : -INFINITY;
        float mx = sc_r;
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
        if (mx > M[r] + L::kSlack) rescale_to(r, mx);  // warp-uniform; token tw is valid
        pk[r] = valid ? exp2f(sc_r - M[r]) : 0.f;
        float ls = pk[r];
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) ls += __shfl_xor_sync(0xFFFFFFFFu, ls, off);
        l[r] += ls;
      }
#pragma unroll
      for (int step = 0; step < 16 / L::kTS; ++step) {
        float p[RH];
#pragma unroll
        for (int r = 0; r < RH; ++r) p[r] = __shfl_sync(0xFFFFFFFFu, pk[r], L::kTS * step + ts);
        const int tv = tw + L::kTS * step + ts;
        if (tv < NR) value_fp16(NQK + tv, p);
      }
    }
  }

  // ---- warps -> block: sum o - oz and l over the warps (one max per head for the block) ----
  __syncthreads();  // the ring is idle
  float* ored = reinterpret_cast<float*>(sma);  // [warp][RH][128]
  {  // the token slots of a lane position meet, then kLPT lanes hold 128 channels
#pragma unroll
    for (int r = 0; r < RH; ++r) {
#pragma unroll
      for (int off = L::kLPT; off < 32; off <<= 1) {
#pragma unroll
        for (int i = 0; i < L::kOV; ++i) o[r][i] += __shfl_xor_sync(0xFFFFFFFFu, o[r][i], off);
        oz[r] += __shfl_xor_sync(0xFFFFFFFFu, oz[r], off);
      }
    }
    if (lane < L::kLPT) {  // o[r][w kCPWv + 2j] is channel j of word w, + 1 channel kPV + j, x 2^(b j)
#pragma unroll
      for (int r = 0; r < RH; ++r) {
#pragma unroll
        for (int w = 0; w < L::kLW; ++w) {
          float* dst = ored + (warp * RH + r) * kD + (lane * L::kLW + w) * L::kCPWv;
#pragma unroll
          for (int j = 0; j < L::kPV; ++j) {
            const float sc = (RH == 1) ? pow2_pos(-HalfCodes<VB>::value_scale_exp(j)) : pow2_neg(VB * j);
            dst[j] = o[r][w * L::kCPWv + 2 * j] * sc - oz[r];
            dst[L::kPV + j] = o[r][w * L::kCPWv + 2 * j + 1] * sc - oz[r];
          }
        }
      }
    }
  }
  if (lane == 0)
#pragma unroll
    for (int r = 0; r < RH; ++r) {
      red[warp * RH + r] = l[r];
      redm[warp * RH + r] = M[r];
    }
  __syncthreads();
  if (*failed) return;  // uniform after the barrier

  constexpr int kIt = (RH * kD + kAThreads - 1) / kAThreads;  // outputs per thread
  float ov[kIt], Ls[kIt], Mv[kIt];
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    const int i = it * kAThreads + tid, r = i / kD, ch = i % kD;
    ov[it] = 0.f;
    Ls[it] = 0.f;
    Mv[it] = -INFINITY;
    if (i < RH * kD) {  // each warp's running max differs: rescale to the block's
      for (int w = 0; w < kAWarps; ++w) Mv[it] = fmaxf(Mv[it], redm[w * RH + r]);
      if (Mv[it] != -INFINITY)
        for (int w = 0; w < kAWarps; ++w) {
          const float mw = redm[w * RH + r];
          if (mw == -INFINITY) continue;
          const float f = exp2f(mw - Mv[it]);
          ov[it] = fmaf(f, ored[(w * RH + r) * kD + ch], ov[it]);
          Ls[it] = fmaf(f, red[w * RH + r], Ls[it]);
        }
    }
  }
  auto write_out = [&](int i, float val) {
    if (a.out_fp32) reinterpret_cast<float*>(a.out)[bq0 * kD + i] = val;
    else reinterpret_cast<uint16_t*>(a.out)[bq0 * kD + i] = f32_to_bf16(val);
  };

  if (n_total == 1) {
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int i = it * kAThreads + tid;
      if (i < RH * kD) write_out(i, (Ls[it] > 0.f) ? ov[it] / Ls[it] : 0.f);
    }
    return;
  }
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    const int i = it * kAThreads + tid, r = i / kD, ch = i % kD;
    if (i < RH * kD) {
      float* pp = a.part + ((bq0 + r) * n_total + split) * (kD + 2);
      pp[2 + ch] = ov[it];
      if (ch == 0) {
        pp[0] = Mv[it];
        pp[1] = Ls[it];
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) *flag = (atomicAdd(&a.counters[bq0], 1) == n_total - 1);
  __syncthreads();
  if (!*flag) return;
  __threadfence();
#pragma unroll
  for (int it = 0; it < kIt; ++it) {
    const int i = it * kAThreads + tid, r = i / kD, ch = i % kD;
    if (i >= RH * kD) continue;
    const float* base = a.part + (bq0 + r) * n_total * (kD + 2);
    float Mx = -INFINITY;
    for (int s = 0; s < n_total; ++s) Mx = fmaxf(Mx, __ldcg(base + s * (kD + 2)));
    float Lt = 0.f, acc = 0.f;
    if (Mx != -INFINITY) {
      for (int s = 0; s < n_total; ++s) {
        const float ms = __ldcg(base + s * (kD + 2));
        if (ms == -INFINITY) continue;
        const float w = exp2f(ms - Mx);
        Lt = fmaf(w, __ldcg(base + s * (kD + 2) + 1), Lt);
        acc = fmaf(w, __ldcg(base + s * (kD + 2) + 2 + ch), acc);
      }
    }
    write_out(i, (Lt > 0.f) ? acc / Lt : 0.f);
  }
  if (tid == 0) a.counters[bq0] = 0;
}

template <int KB, int VB, int RH>
size_t attn_smem(int) {
  return (size_t)AttnLayout<KB, VB, RH>::kSmem;
}

template <int KB, int VB, int RH>
cudaError_t launch_attn(const KiviAttnArgs& a, cudaStream_t st) {
  const size_t smem = attn_smem<KB, VB, RH>(a.residual);
  cudaError_t e = cudaFuncSetAttribute(kivi_attn_kernel<KB, VB, RH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)kD);
  const int n_sub = (a.Hq / a.H) / RH;
  // token splits per head subgroup; the last split also attends the fp16 residual
  dim3 grid(a.n_split * n_sub, a.B, a.H);
  kivi_attn_kernel<KB, VB, RH><<<grid, kAThreads, smem, st>>>(a, scale_log2);
  return cudaGetLastError();
}

template <int KB, int VB>
cudaError_t launch_attn_rh(const KiviAttnArgs& a, int rh, cudaStream_t st) {
  if (rh == 4) return launch_attn<KB, VB, 4>(a, st);
  if (rh == 2) return launch_attn<KB, VB, 2>(a, st);
  return launch_attn<KB, VB, 1>(a, st);
}

template <int KB, int VB>
size_t smem_rh(int rh, int residual) {
  if (rh == 4) return attn_smem<KB, VB, 4>(residual);
  if (rh == 2) return attn_smem<KB, VB, 2>(residual);
  return attn_smem<KB, VB, 1>(residual);
}

int sm_count_cached() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

}  // namespace

int kivi_heads_per_block(int rep) { return (rep % 4 == 0) ? 4 : (rep % 2 == 0) ? 2 : 1; }

int kivi_attn_max_tok_per_split(int) { return 1 << 30; }  // tokens stream through the ring

size_t kivi_attn_smem_bytes(int k_bits, int v_bits, int rh, int residual) {
  if (k_bits == 2 && v_bits == 2) return smem_rh<2, 2>(rh, residual);
  if (k_bits == 2 && v_bits == 4) return smem_rh<2, 4>(rh, residual);
  if (k_bits == 4 && v_bits == 2) return smem_rh<4, 2>(rh, residual);
  return smem_rh<4, 4>(rh, residual);
}

template <int KB, int VB, int RH>
int blocks_per_sm_of() {
  int n = 0;
  const size_t smem = attn_smem<KB, VB, RH>(0);
  if (cudaFuncSetAttribute(kivi_attn_kernel<KB, VB, RH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kivi_attn_kernel<KB, VB, RH>, kAThreads, smem) != cudaSuccess)
    return 4;
  return n > 0 ? n : 1;
}
template <int KB, int VB>
int blocks_per_sm_rh(int rh) {
  if (rh == 4) return blocks_per_sm_of<KB, VB, 4>();
  if (rh == 2) return blocks_per_sm_of<KB, VB, 2>();
  return blocks_per_sm_of<KB, VB, 1>();
}

int kivi_attn_blocks_per_sm(int k_bits, int v_bits, int rh) {
  // one query per kernel instance and process (a property of the build and the GPU model)
  static int cached[2][2][3] = {};
  int& c = cached[k_bits == 4][v_bits == 4][rh == 4 ? 2 : rh == 2 ? 1 : 0];
  if (c == 0) {
    if (k_bits == 2 && v_bits == 2) c = blocks_per_sm_rh<2, 2>(rh);
    else if (k_bits == 2 && v_bits == 4) c = blocks_per_sm_rh<2, 4>(rh);
    else if (k_bits == 4 && v_bits == 2) c = blocks_per_sm_rh<4, 2>(rh);
    else c = blocks_per_sm_rh<4, 4>(rh);
  }
  return c;
}

template <int BITS, bool kKeys>
cudaError_t launch_quant(const KiviQuantArgs& a, int blocks, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kivi_quant_kernel<BITS, kKeys>, cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmem);
  if (e != cudaSuccess) return e;
  kivi_quant_kernel<BITS, kKeys><<<blocks, kQThreads, kQSmem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_kivi_quantize(const KiviQuantArgs& a, cudaStream_t s) {
  // one block of kQWarps persistent warps per SM, fewer when there are few tiles
  const long long tiles = (long long)a.B * a.H * ((a.n_tok + kGroup - 1) / kGroup);
  if (tiles <= 0) return cudaSuccess;
  const int blocks = (int)std::min<long long>(sm_count_cached(), (tiles + kQWarps - 1) / kQWarps);
  const bool keys = (a.axis == KVQ_PER_CHANNEL);
  if (a.bits == 4) return keys ? launch_quant<4, true>(a, blocks, s) : launch_quant<4, false>(a, blocks, s);
  return keys ? launch_quant<2, true>(a, blocks, s) : launch_quant<2, false>(a, blocks, s);
}

cudaError_t launch_kivi_prefill_tail(const KiviTailArgs& a, cudaStream_t s) {
  if (a.B <= 0) return cudaSuccess;
  kivi_prefill_tail_kernel<<<dim3(a.B, a.H), 128, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_kivi_append(const KiviAppendArgs& a, cudaStream_t s) {
  if (a.n_seq <= 0) return cudaSuccess;
  const dim3 grid(a.n_seq, a.H);
  if (a.k_bits == 2 && a.v_bits == 2) kivi_append_kernel<2, 2><<<grid, 128, 0, s>>>(a);
  else if (a.k_bits == 2) kivi_append_kernel<2, 4><<<grid, 128, 0, s>>>(a);
  else if (a.v_bits == 2) kivi_append_kernel<4, 2><<<grid, 128, 0, s>>>(a);
  else kivi_append_kernel<4, 4><<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_kivi_attn(const KiviAttnArgs& a, cudaStream_t st) {
  const int rh = kivi_heads_per_block(a.Hq / a.H);
  if (a.k_bits == 2 && a.v_bits == 2) return launch_attn_rh<2, 2>(a, rh, st);
  if (a.k_bits == 2 && a.v_bits == 4) return launch_attn_rh<2, 4>(a, rh, st);
  if (a.k_bits == 4 && a.v_bits == 2) return launch_attn_rh<4, 2>(a, rh, st);
  return launch_attn_rh<4, 4>(a, rh, st);
}

}  // namespace kvq
