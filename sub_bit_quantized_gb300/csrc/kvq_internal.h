// Internal launch interface between the C ABI layer (kvq_api.cu) and the kernel files.
// Not exported; no validation here (kvq_api.cu checks every argument first).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

// stores the detail message kvq_last_error() returns on this host thread
void set_last_error(const char* msg);

// every host-side check of kvq_decode_attn except the workspace (fn names the caller in the
// message kvq_last_error() returns)
kvq_status check_decode_args(int format, const void* cfg, const void* cache, int layer, int loop_step,
                             const uint16_t* q, int B, const void* out, int out_dtype, int n_splits, const char* fn);

constexpr int kD = 128;        // head dimension
constexpr int kPage = 8;       // tokens per index page
constexpr int kCB = 256;       // codebook entries

// In-page byte of (group g, token j) for NG index groups per token (pages of 8 NG bytes):
// byte (p * 8 + j) * 2 + h holds group p + h NG/2, so the two groups whose channels are RoPE
// partners (channel ch and ch + 64) sit side by side and a lane reads its 8 tokens' pairs as
// one 16-byte row.
__host__ __device__ inline size_t page_byte(int g, int j, int NG) {
  const int half = NG / 2;
  return (size_t)(((g % half) * kPage + j) * 2 + g / half);
}

// ---------------------------------------------------------------- LoopVQ decode attention
// One persistent launch per call. The quantized pages of every (head, request) segment,
// head-major, form one list of page positions; block k of G takes positions
// [k P / G, (k + 1) P / G). Inside a block, 16 compute warps score the keys of up to
// kVqSubPages pages (pass 1), then add the fixed-point softmax weights of the same pages into
// a per-(group, codeword) histogram (pass 2); aux warps turn each histogram into value sums
// and merge; window warps attend the bf16 window of every segment whose first page the block
// holds, and the aux warps merge that in too. A
// segment split over several blocks is merged by the last block to finish its part: each
// writes a partial (M, l, o[128]) to a per-block slot and counts itself in cnt[segment]; the
// last one merges the slots, writes the output and resets the counter to 0.
constexpr int kVqComputeWarps = 16;              // compute warps per block
constexpr int kVqSubPages = 384;                 // index pages per sub-piece (fixed-point capacity)
constexpr int kVqSlotFloats = 132;               // one partial: M, l, 2 pad, o[128]
constexpr int kVqMaxBatch = 8191;                // requests per call (prefix scan in shared memory)

struct VqAttnArgs {
  const uint8_t* idx_k;      // [max_batch][H][max_pages][8 NG] of (layer, block)
  const uint8_t* idx_v;
  const uint16_t* win_k;     // [max_batch][H][win_slots][D] of (layer, step)
  const uint16_t* win_v;
  const float* bt_k;         // [H][2][256][D/2] of (layer, step)
  const uint16_t* bt_v;      // fp16 [H][256][D] of (layer, step)
  const float* rope_cos;     // [max_ctx][D/2]
  const float* rope_sin;
  const int32_t* seq_len;    // [max_batch]
  const int32_t* n_pages;
  const uint16_t* q;         // [B][H][D] bf16
  void* out;                 // [B][H][D]
  int out_fp32;
  int32_t* cnt;              // [B * H] merge counters (zero between calls)
  float* slots;              // [G][2][kVqSlotFloats] partials of segments shared between blocks
  int* err;
  int B, H, max_pages, max_ctx, sink, recent, win_slots;
  int G;                     // blocks
  int NG;                    // index groups per token (8, 16 or 32): pages of 8 NG bytes
};
size_t vq_attn_ws_bytes(int B, int H, int G);
cudaError_t launch_vq_attn(const VqAttnArgs& a, void* ws, cudaStream_t s);

// ---------------------------------------------------------------- LoopVQ encode and friends
struct VqEncodeArgs {
  const uint16_t* x;               // bf16, element (t, b, h, j, ch)
  int64_t st, sb, sh;              // element strides of t, b, h (token stride D)
  const float* cb;                 // [NB][H][NG][256][G] of one layer
  uint8_t* idx;                    // [NB][max_batch][H][max_pages][128] of one layer
  int32_t* n_ties;
  int* err;
  int T, Tc, G, NB, H, max_batch, max_pages;
  int seq_begin, n_seq, n_tok, page_begin, g_begin, g_count;
  // Page roll (launch_vq_roll_tc): the planes' sequence index is (layer, K/V) = 2 layer + kv,
  // the rows of a plane are (request b, token j of b's oldest recent page) = 8 b + j, read
  // from the bf16 windows (x: win_k of layer 0, x2: win_v; st, sb, sh: loop-step, request and
  // head strides, rows at slot * D) and written to page n_pages[b] of the requests that are
  // due (idx: idx_k of layer 0, idx2: idx_v); codebook parts from cbp (K) and cbp2 (V);
  // n_tok = 8 n_req.
  const uint16_t* x2; uint8_t* idx2;
  const uint8_t* cbp; const uint8_t* cbp2;
  int64_t x_layer, cbp_layer, idx_layer;  // per-layer strides: elements, bytes, bytes
  const int32_t* seq_len; const int32_t* n_pages;
  int sink, recent, n_req;
};
cudaError_t launch_vq_encode(const VqEncodeArgs& a, cudaStream_t s);

cudaError_t launch_rope_table(float* cos_t, float* sin_t, int max_ctx, int D, float base, cudaStream_t s);
cudaError_t launch_slice_codebooks(const float* cb, float* bt, int L, int T, int Tc, int G, int H,
                                   cudaStream_t s);
cudaError_t launch_slice_codebooks_fp16(const float* cb, uint16_t* bt16, int L, int T, int Tc, int G, int H,
                                        cudaStream_t s);

struct VqWindowArgs {              // copy prefill tokens into the bf16 windows
  const uint16_t* xk; const uint16_t* xv;
  int64_t st, sb, sh;
  uint16_t* win_k; uint16_t* win_v;  // [T][max_batch][H][win_slots][D] of one layer
  int32_t* seq_len; int32_t* n_pages;  // set for the requests (may be null)
  int T, H, max_batch, win_slots, sink, recent;
  int seq_begin, n_seq, L, n_pages_val;
};
cudaError_t launch_vq_prefill_window(const VqWindowArgs& a, cudaStream_t s);

struct VqAppendArgs {
  const uint16_t* k_new; const uint16_t* v_new;   // [n_seq][H][D]
  uint16_t* win_k; uint16_t* win_v;               // of (layer, step): [max_batch][H][win_slots][D]
  int32_t* seq_len; int32_t* n_pages;
  int* err;
  int H, n_seq, win_slots, sink, recent, max_pages, max_ctx;
  int advance;                                    // first (layer, step) of the token
};
cudaError_t launch_vq_append(const VqAppendArgs& a, cudaStream_t s);

struct VqRollArgs {                // encode the oldest recent page where the ring is full
  const uint16_t* win_k; const uint16_t* win_v;   // full [L][T][max_batch][H][win_slots][D]
  const float* cb_k; const float* cb_v;           // [L][NB][H][NG][256][G]
  uint8_t* idx_k; uint8_t* idx_v;                 // [L][NB][max_batch][H][max_pages][128]
  int32_t* seq_len; int32_t* n_pages;
  const uint8_t* cbp_k; const uint8_t* cbp_v;     // split codebook parts (null: CUDA-core roll)
  int* err;
  int L, T, Tc, G, NB, H, n_seq, max_batch, max_pages, win_slots, sink, recent;
};
cudaError_t launch_vq_roll(const VqRollArgs& a, cudaStream_t s);
// the roll's encode on the tensor cores (needs the split codebook parts)
cudaError_t launch_vq_roll_tc(const VqEncodeArgs& a, cudaStream_t s);
// three bf16 parts of every [256][G] codebook of cb (n codebooks) in the tensor-core operand
// layout; bytes per codebook from split_codebook_bytes
cudaError_t launch_split_codebooks(const float* cb, uint8_t* cbp, long long n, int Tc, int G, cudaStream_t s);
size_t split_codebook_bytes(int G);

// ---------------------------------------------------------------- KIVI
struct KiviQuantArgs {
  const uint16_t* x;               // fp16 (b, h, j, ch)
  int64_t sb, sh;
  uint8_t* codes; uint16_t* scale; uint16_t* zero;
  int axis, bits, B, H, n_tok, tok_begin, max_tokens, group;
  int* err;  // device error word (a bounded wait that timed out)
};
cudaError_t launch_kivi_quantize(const KiviQuantArgs& a, cudaStream_t s);

// prefill tail: copy tokens [nq, n_tok) to the residuals and set the lengths
struct KiviTailArgs {
  const uint16_t* k; const uint16_t* v;  // fp16 (b, h, j, ch), b relative to b0
  int64_t sb, sh;
  uint16_t* k_resid; uint16_t* v_resid;
  int32_t* n_tok; int32_t* n_quant_k; int32_t* n_quant_v;
  int b0, B, H, n_tok_new, nq, residual;
};
cudaError_t launch_kivi_prefill_tail(const KiviTailArgs& a, cudaStream_t s);

struct KiviAppendArgs {
  const uint16_t* k_new; const uint16_t* v_new;  // fp16 [n_seq][H][D]
  uint8_t* k_codes; uint16_t* k_scale; uint16_t* k_zero;
  uint8_t* v_codes; uint16_t* v_scale; uint16_t* v_zero;
  uint16_t* k_resid; uint16_t* v_resid;
  int32_t* n_tok; int32_t* n_quant_k; int32_t* n_quant_v; int32_t* sync;
  int* err;
  int n_seq, H, k_bits, v_bits, residual, max_tokens;
};
cudaError_t launch_kivi_append(const KiviAppendArgs& a, cudaStream_t s);

struct KiviAttnArgs {
  const uint8_t* k_codes; const uint16_t* k_scale; const uint16_t* k_zero;
  const uint8_t* v_codes; const uint16_t* v_scale; const uint16_t* v_zero;
  const uint16_t* k_resid; const uint16_t* v_resid;
  const int32_t* n_tok; const int32_t* n_quant_k; const int32_t* n_quant_v;
  const uint16_t* q;               // bf16 [B][Hq][D]
  void* out; int out_fp32;
  float* part; int* counters; int* err;
  int B, H, Hq, k_bits, v_bits, max_tokens, residual, group;
  int n_split, tok_per_split;
};
// query heads one attention block serves (a divisor of Hq / H, at most 4)
int kivi_heads_per_block(int rep);
size_t kivi_attn_smem_bytes(int k_bits, int v_bits, int heads_per_block, int residual);
int kivi_attn_blocks_per_sm(int k_bits, int v_bits, int heads_per_block);  // resident attention blocks per SM
int kivi_attn_max_tok_per_split(int residual);
cudaError_t launch_kivi_attn(const KiviAttnArgs& a, cudaStream_t s);

}  // namespace kvq
