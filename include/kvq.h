/*
 * kvq.h - C ABI of libkvq: decode attention over quantized KV caches on one NVIDIA GB300
 * (sm_103a). Two cache formats:
 *
 *   LoopVQ  "LoopVQ: Sub 1-bit KV Cache Quantization for Looped Transformers" (paper
 *           digest): one 8-bit codeword covers c = G/Tc channels over Tc consecutive loop
 *           steps (method step 1, Figure 3); 256-entry codebooks per (loop block, layer,
 *           head, channel group); keys quantized before RoPE; 8 sink and W recent tokens
 *           kept in bf16 at every loop step, the rest in 8-token index pages (method
 *           step 4, Figure 5); decode attention looks codewords up through the per-step
 *           slice B_t, applies RoPE and merges the bf16 and quantized partials exactly
 *           (method step 5, Algorithm 1).
 *   KIVI    "KIVI 完全拆解：非对称 2-bit KV Cache 量化": asymmetric 2- or 4-bit quantization
 *           q = clamp(round(X/s + z), 0, 2^b - 1) with fp16 scale and zero-point per group
 *           (section on per-token / per-channel quantization); keys per channel over 32
 *           tokens, values per token over 32 channels, fp16 residual windows filled and
 *           drained as Algorithm 1 streams tokens in, and one softmax over both segments
 *           (core design, eq. (3)); grouped-query heads (implementation section).
 *
 * Conventions for every call:
 *   - Pointers are CUDA device pointers unless stated otherwise, owned by the caller; the
 *     library never allocates, frees or keeps them. Device pointers must be 16-byte
 *     aligned (checked: KVQ_ERR_INVALID_ARG).
 *   - bf16 and fp16 values are passed as uint16_t bit patterns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and return a status at once. KVQ_ERR_CUDA means a launch failed; kvq_last_error()
 *     gives the detail. Argument errors are detected on the host before anything is
 *     launched, so an error return leaves all buffers untouched.
 *   - Device-side waits (the TMA completion barrier) are bounded; a timed-out wait sets a
 *     device error word that kvq_device_error() reads after the stream has drained.
 *   - Loop steps are 1-based (t = 1..T) as on the LoopVQ page; layers and heads 0-based.
 *   - Head dimension D = 128 and page size 8. LoopVQ shapes built: c = G/Tc = 8 with
 *     Tc = 1, 2, 4 (G = 8, 16, 32: 1, 0.5, 0.25 bit), and at G = 16 (0.5 bit) also Tc = 1
 *     (c = 16, codewords of one loop step) and Tc = 4 (c = 4, one index for four steps);
 *     other shapes return KVQ_ERR_UNSUPPORTED.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int kvq_status;
enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, inconsistent shape            */
  KVQ_ERR_CAPACITY = 2,     /* more tokens, pages or requests than the buffers hold      */
  KVQ_ERR_UNSUPPORTED = 3,  /* a valid shape this build has no kernel for               */
  KVQ_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed                     */
  KVQ_ERR_WORKSPACE = 5,    /* workspace smaller than kvq_decode_workspace_size()       */
  KVQ_ERR_TIMEOUT = 6       /* a device-side wait ran out of time (device error word)   */
};

enum { KVQ_FMT_LOOPVQ = 0, KVQ_FMT_KIVI = 1 };
enum { KVQ_OUT_BF16 = 0, KVQ_OUT_FP32 = 1 };
enum { KVQ_PER_CHANNEL = 0, KVQ_PER_TOKEN = 1 };

typedef void* kvq_stream; /* cudaStream_t */

/* ---------------------------------------------------------------------------------- */
/* LoopVQ                                                                              */
/* ---------------------------------------------------------------------------------- */

/* Shape of a LoopVQ cache. NB = T/Tc loop blocks, c = G/Tc, NG = D/c index groups, a page
 * holds 8 tokens and is 8*NG bytes. `recent` is W, the bf16 recent window (64, or 256
 * for long contexts). */
typedef struct {
  int D;            /* head dimension (128)                                  */
  int T;            /* loop steps                                            */
  int Tc;           /* loop steps per block; divides T and G                 */
  int G;            /* coupled dimensions per codeword                      */
  int K;            /* codebook entries (256: 8-bit indices)                 */
  int n_layers;
  int n_heads;      /* KV heads (= query heads: dense multi-head attention) */
  int sink;         /* bf16 sink tokens (8)                                  */
  int recent;       /* W                                                     */
  int max_pages;    /* index pages per (layer, block, request, head)         */
  int max_batch;    /* requests the buffers hold                             */
  int max_ctx;      /* rows of the RoPE table (largest position + 1)         */
  float rope_base;  /* RoPE base (1e4)                                       */
} kvq_vq_cfg;

/* Device buffers of a LoopVQ cache (all caller-owned, sizes from kvq_vq_cache_sizes).
 *
 * idx_k, idx_v  uint8  [n_layers][NB][max_batch][n_heads][max_pages][8*NG]
 *     Index page p of (layer, block, request, head) holds the 8 tokens at positions
 *     sink + 8p .. sink + 8p + 7. In-page byte order pairs the RoPE partner groups
 *     s and s + NG/2 (channels s*c.. and D/2 + s*c..): byte (s*8 + j)*2 + 0 is the index
 *     of group s for token j, byte (s*8 + j)*2 + 1 that of group s + NG/2.
 * win_k, win_v  bf16   [n_layers][T][max_batch][n_heads][sink + recent + 8][D]
 *     Pre-RoPE keys / values of the bf16 tokens at each loop step. Position p < sink sits
 *     in slot p; a recent position p in slot sink + (p - sink) mod (recent + 8).
 * bt_k          fp32   [n_layers][T][n_heads][2][K][D/2]
 *     Per-loop-step key codebook slices B_t, cut once by kvq_slice_codebooks. Channel
 *     ch = g*c + i of codeword r sits in half ch / (D/2) at column ch % (D/2):
 *     bt[l][t][h][ch/(D/2)][r][ch%(D/2)] = cb[l][beta][h][g][r][i*Tc + m],
 *     beta = (t-1)/Tc, m = (t-1)%Tc. (The halves hold the RoPE partner channels.)
 * bt_v          fp16   [n_layers][T][n_heads][K][D]
 *     Per-loop-step value codebook slices, cut once by kvq_slice_codebooks_fp16 and
 *     rounded to fp16 (nearest even): bt_v[l][t][h][r][ch] = fp16(cb[l][beta][h][g][r][i*Tc + m]).
 * cb_k, cb_v    fp32   [n_layers][NB][n_heads][NG][K][G]   full codebooks (encode, roll)
 * cbp_k, cbp_v  bytes  [n_layers][NB][n_heads][NG][3 parts][K rows x KC 16-byte chunks]
 *     Optional (may be NULL): each codebook split into three bf16 parts hi + mid + lo (hi =
 *     bf16(e), mid = bf16(e - hi), lo = bf16(e - hi - mid), round to nearest even) with the
 *     -|e|^2/2 column appended, in the tensor cores' operand layout (kvq_split_codebooks).
 *     With both set, the page roll of kvq_append_page runs on the tensor cores; with either
 *     NULL it runs on CUDA cores (same decisions).
 * rope_cos, rope_sin fp32 [max_ctx][D/2]: cos / sin(p * base^(-2i/D)) (kvq_rope_table)
 * seq_len       int32  [max_batch]: tokens cached per request, including the newest one
 *                      (the query position is seq_len - 1)
 * n_pages       int32  [max_batch]: index pages in use per request
 */
typedef struct {
  uint8_t* idx_k;
  uint8_t* idx_v;
  uint16_t* win_k;
  uint16_t* win_v;
  float* bt_k;
  uint16_t* bt_v;
  const float* cb_k;
  const float* cb_v;
  const float* rope_cos;
  const float* rope_sin;
  int32_t* seq_len;
  int32_t* n_pages;
  uint8_t* cbp_k;
  uint8_t* cbp_v;
} kvq_vq_cache;

/* Byte sizes of each buffer of kvq_vq_cache for `cfg` (host-only, no device work).
 * Order: idx (each of k, v), win (each), bt (bt_k), bt_v, cb (each), rope (each of cos,
 * sin), per-request int32 arrays (each), cbp (each of cbp_k, cbp_v). Returns
 * KVQ_ERR_INVALID_ARG for an invalid cfg. */
typedef struct {
  size_t idx, win, bt, bt_v, cb, rope, per_request, cbp;
} kvq_vq_sizes;
kvq_status kvq_vq_cache_sizes(const kvq_vq_cfg* cfg, kvq_vq_sizes* out /* host */);

/* RoPE table: cos/sin(p * theta_i), theta_i = base^(-2i/D), p < max_ctx, i < D/2, computed
 * in fp64 and rounded to fp32 (LoopVQ page, background "RoPE" and method step 5:
 * reconstructed keys are rotated with a precomputed cos/sin table). The pairing is
 * rotate-half: channel i with channel i + D/2 (a reading; the page names no convention). */
kvq_status kvq_rope_table(const kvq_vq_cfg* cfg, float* rope_cos, float* rope_sin, kvq_stream stream);

/* Cut the per-loop-step slices B_t out of the full codebooks, once at load time
 * (LoopVQ method step 5 and Figure 3: step t reads the shared indices through its own
 * slice). cb: [n_layers][NB][n_heads][NG][K][G]; bt: [n_layers][T][n_heads][2][K][D/2]
 * (layout in kvq_vq_cache). */
kvq_status kvq_slice_codebooks(const kvq_vq_cfg* cfg, const float* cb, float* bt, kvq_stream stream);

/* The same cut for the value codebooks, rounded to fp16 (round to nearest even) in codeword
 * rows of natural channel order: bt16 is [n_layers][T][n_heads][K][D] (layout of bt_v in
 * kvq_vq_cache). Decode attention accumulates values from these fp16 rows; the rounding
 * (relative 2^-11 per entry) is far inside the attention output tolerance. */
kvq_status kvq_slice_codebooks_fp16(const kvq_vq_cfg* cfg, const float* cb, uint16_t* bt16,
                                    kvq_stream stream);

/* Split every codebook of cb ([n_layers][NB][n_heads][NG][K][G] fp32) into the three bf16
 * parts the tensor-core encode multiplies (layout of cbp_k in kvq_vq_cache), once at load
 * time, for the page roll (LoopVQ method step 4: the oldest recent page is encoded during
 * decode; each roll reads every codebook, so the split is not redone per roll). The parts sum
 * back to the fp32 entries exactly. Errors: KVQ_ERR_INVALID_ARG (cfg, pointers). */
kvq_status kvq_split_codebooks(const kvq_vq_cfg* cfg, const float* cb, uint8_t* cbp, kvq_stream stream);

/* Nearest-codeword encode of coupled vectors (LoopVQ background: a(z) = argmin_r
 * ||z - e_r||^2; method step 1 for the coupling, method step 4 for prefill encoding).
 *
 * x: bf16 pre-RoPE keys (or values) of ONE layer, element (t, b, h, j, ch) at
 *    x[t*x_stride_t + b*x_stride_b + h*x_stride_h + j*D + ch], t the 0-based loop step,
 *    b < n_seq, j < n_tok (n_tok a multiple of 8: whole pages).
 * cb: fp32 [NB][n_heads][NG][K][G] codebooks of this layer.
 * idx: this layer's index pages, [NB][max_batch][n_heads][max_pages][8*NG] (in-page order
 *    as in kvq_vq_cache); token j of request b goes to page page_begin + j/8 of request
 *    seq_begin + b. Only groups [g_begin, g_begin + g_count) are written.
 * n_ties: optional device int32 counter (may be NULL); incremented once per (vector) whose
 *    two best distances lie within 1e-6 relative of each other, where either index is a
 *    correct encoding. The arithmetic is exact enough that any other decision equals the
 *    exact-arithmetic argmin with the lowest index on ties.
 * Errors: KVQ_ERR_CAPACITY if pages or requests exceed max_pages / max_batch. */
kvq_status kvq_encode_vq(const kvq_vq_cfg* cfg, const uint16_t* x, int64_t x_stride_t,
                         int64_t x_stride_b, int64_t x_stride_h, int seq_begin, int n_seq,
                         int n_tok, const float* cb, uint8_t* idx, int page_begin,
                         int g_begin, int g_count, int32_t* n_ties, kvq_stream stream);

/* Prefill of one layer (LoopVQ method step 4, Figure 5): for requests
 * [seq_begin, seq_begin + n_seq), each with L prompt tokens, keep positions [0, sink) and
 * the last recent + ((L - sink - recent) mod 8) positions in bf16 at every loop step, and
 * encode the positions in between into index pages (K and V, every loop block). Sets
 * seq_len = L and n_pages = max(0, (L - sink - recent) / 8) for those requests.
 * xk, xv: bf16 pre-RoPE keys / values of the layer, strides as in kvq_encode_vq, j < L.
 * Errors: KVQ_ERR_CAPACITY if L needs more than max_pages pages or L > max_ctx. */
kvq_status kvq_prefill_vq(const kvq_vq_cfg* cfg, const kvq_vq_cache* cache, int layer,
                          const uint16_t* xk, const uint16_t* xv, int64_t x_stride_t,
                          int64_t x_stride_b, int64_t x_stride_h, int seq_begin, int n_seq,
                          int L, int32_t* n_ties, kvq_stream stream);

/* Decode-time cache write (LoopVQ Figure 5: new keys and values are written in bf16; every
 * 8 generated tokens the oldest recent page is encoded into indices).
 * Call once per (layer, loop step) with that step's new pre-RoPE key and value, bf16
 * [n_seq][n_heads][D] for requests [0, n_seq). The first call of a token (layer 0,
 * loop_step 1) advances seq_len by one; when that makes the recent window hold
 * recent + 8 tokens, the same call first encodes the oldest recent page for every layer,
 * block, head, K and V (its tokens are complete at that point), adds it as page n_pages
 * and increments n_pages. Other calls only write the bf16 slot of the newest token.
 * Errors: KVQ_ERR_CAPACITY is reported through kvq_device_error() (the lengths live on the
 * device) if a request would exceed max_pages or max_ctx; such a request is left as is. */
kvq_status kvq_append_page(const kvq_vq_cfg* cfg, const kvq_vq_cache* cache, int layer,
                           int loop_step, const uint16_t* k_new, const uint16_t* v_new,
                           int n_seq, kvq_stream stream);

/* ---------------------------------------------------------------------------------- */
/* KIVI                                                                                */
/* ---------------------------------------------------------------------------------- */

typedef struct {
  int D;            /* head dimension (128)                                              */
  int n_heads;      /* KV heads                                                          */
  int n_q_heads;    /* query heads, a multiple of n_heads: query head h reads KV head     */
                    /* h / (n_q_heads / n_heads) (grouped-query attention, KIVI page,     */
                    /* implementation section); n_q_heads == n_heads is multi-head        */
  int k_bits;       /* 2 or 4: key code width   (implementation section: K and V bits     */
  int v_bits;       /* 2 or 4: value code width  are configured independently)            */
  int group;        /* 32: tokens per key group, channels per value group                */
  int residual;     /* R: fp16 residual capacity, a multiple of group (128 on the page);  */
                    /* 0 is allowed for attention-only caches with no residual           */
  int max_batch;
  int max_tokens;   /* quantized-token capacity per (request, KV head), multiple of group */
} kvq_kivi_cfg;

/* Device buffers of a KIVI cache (caller-owned, zero-filled before first use).
 * k_codes uint8 [max_batch][n_heads][max_tokens][D*k_bits/8], v_codes likewise with
 *     v_bits: 8/b codes per byte along channels, channel (8/b)k + i of a token in bits
 *     [b*i, b*i + b) of byte k.
 * k_scale, k_zero  fp16 [max_batch][n_heads][max_tokens/group][D]   (per channel)
 * v_scale, v_zero  fp16 [max_batch][n_heads][max_tokens][D/group]   (per token)
 * k_resid fp16 [max_batch][n_heads][residual][D]: key of token t at row t - n_quant_k[b]
 * v_resid fp16 [max_batch][n_heads][residual][D]: value of token t at row t % residual
 *     (a ring: the window drops one token at a time)
 * n_tok     int32 [max_batch]: tokens cached per request
 * n_quant_k int32 [max_batch]: keys of tokens [0, n_quant_k) are quantized (a multiple
 *     of group), the rest are in k_resid
 * n_quant_v int32 [max_batch]: values of tokens [0, n_quant_v) are quantized, the rest
 *     are in v_resid
 * sync      int32 [max_batch]: scratch of kvq_kivi_append (its blocks count their arrivals
 *     per request there); zero before the first call, every call leaves it zero
 * A valid state has n_quant_v <= n_quant_k <= n_tok, n_tok - n_quant_v <= residual and
 * n_quant_k <= max_tokens; kvq_kivi_prefill and kvq_kivi_append keep it valid. Attention
 * over an invalid state stays inside the buffers but its result is undefined.
 */
typedef struct {
  uint8_t* k_codes;
  uint16_t* k_scale;
  uint16_t* k_zero;
  uint8_t* v_codes;
  uint16_t* v_scale;
  uint16_t* v_zero;
  uint16_t* k_resid;
  uint16_t* v_resid;
  int32_t* n_tok;
  int32_t* n_quant_k;
  int32_t* n_quant_v;
  int32_t* sync;
} kvq_kivi_cache;

/* Group quantization (KIVI page, quantization-direction section and the group-quant
 * kernel of the implementation section). In fp32 per group: s = (max - min)/(2^b - 1),
 * s16 = fp16(s) (1 if that is 0), z16 = fp16(-min/s16),
 * q = clamp(rint(x/s16 + z16), 0, 2^b - 1) with IEEE division and no fused multiply-add,
 * so codes, scales and zero-points are reproducible bit for bit.
 * axis = KVQ_PER_CHANNEL: keys (b = k_bits), groups of `group` tokens per channel; n_tok
 *        and tok_begin multiples of group; writes k-style codes/scale/zero.
 * axis = KVQ_PER_TOKEN:   values (b = v_bits), groups of `group` channels per token.
 * x: fp16, element (b, h, j, ch) at x[b*x_stride_b + h*x_stride_h + j*D + ch], b < B.
 * codes / scale / zero: cache arrays (layouts in kvq_kivi_cache); token j of request b is
 *    written at token tok_begin + j.
 * Errors: KVQ_ERR_CAPACITY if tok_begin + n_tok > max_tokens or B > max_batch. */
kvq_status kvq_quantize_kivi(const kvq_kivi_cfg* cfg, int axis, const uint16_t* x,
                             int64_t x_stride_b, int64_t x_stride_h, int B, int n_tok,
                             uint8_t* codes, uint16_t* scale, uint16_t* zero, int tok_begin,
                             kvq_stream stream);

/* Prefill (KIVI page, core design section, Algorithm 1, prefill): requests b0 .. b0+B-1
 * of the cache receive the n_tok prompt tokens in k and v (fp16, element (b, h, j, ch) at
 * x[b*x_stride_b + h*x_stride_h + j*D + ch]). The first nq tokens are quantized (keys per
 * channel, values per token) and the rest are copied to the residuals, where
 * nq = 0 if n_tok <= residual, else n_tok - residual rounded up to a multiple of group (the
 * page's split l - R when that is a multiple of group). Sets n_tok, n_quant_k = n_quant_v
 * = nq on the device. Any earlier content of those requests is replaced.
 * Errors: KVQ_ERR_INVALID_ARG (residual not a positive multiple of group), KVQ_ERR_CAPACITY
 * (b0 + B > max_batch or nq > max_tokens). */
kvq_status kvq_kivi_prefill(const kvq_kivi_cfg* cfg, const kvq_kivi_cache* cache,
                            const uint16_t* k, const uint16_t* v, int64_t x_stride_b,
                            int64_t x_stride_h, int b0, int B, int n_tok, kvq_stream stream);

/* Decode append (KIVI page, Algorithm 1, decoding): one new token per request b < n_seq,
 * k_new and v_new fp16 [n_seq][n_heads][D].
 *  - keys: if the key residual already holds `residual` tokens, they are quantized per
 *    channel and appended to the quantized keys (n_quant_k += residual) and the new key
 *    starts a fresh residual; otherwise it is appended to the residual;
 *  - values: the new value enters the window; if the window then holds more than
 *    `residual` tokens, its oldest token is quantized per token (n_quant_v += 1);
 *  - n_tok += 1.
 * One kernel launch (a block per (request, KV head); the last block of a request to finish
 * advances its lengths); the lengths live on the device, so a whole decode loop can run in a
 * CUDA graph. Two appends to one cache must not run at the same time. A request whose state is invalid or whose key flush would exceed max_tokens
 * is left unchanged and KVQ_ERR_CAPACITY is raised through kvq_device_error().
 * Errors: KVQ_ERR_INVALID_ARG (residual not a positive multiple of group, n_seq < 0),
 * KVQ_ERR_CAPACITY (n_seq > max_batch). */
kvq_status kvq_kivi_append(const kvq_kivi_cfg* cfg, const kvq_kivi_cache* cache,
                           const uint16_t* k_new, const uint16_t* v_new, int n_seq,
                           kvq_stream stream);

/* ---------------------------------------------------------------------------------- */
/* Decode attention (both formats)                                                     */
/* ---------------------------------------------------------------------------------- */

/* One decode attention call: every request b < B attends with its query (bf16
 * [B][Hq][D], Hq = n_heads for LoopVQ and n_q_heads for KIVI; pre-RoPE for LoopVQ) to its
 * whole cache, split-K over the quantized
 * pages with partial softmax per split and an exact logsumexp merge (LoopVQ page:
 * Flash-Decoding background and method step 5; KIVI page: eq. (3), one softmax over the
 * quantized and residual segments). Scale 1/sqrt(D).
 * Arithmetic: scores and softmax in fp32. LoopVQ sums the values by codeword: per
 * (group, codeword) the weights p = exp2(s - M) <= 1 of the tokens using it (M the maximum
 * over a sub-piece of at most 3584 tokens) are added as integers in units of 2^-20 (each
 * weight rounded to the nearest unit once, an absolute error of at most 2^-21), then
 * multiplied by the fp16 value codebook in fp32. KIVI, when a block serves one query head
 * (n_q_heads / n_heads odd), rounds each token's weight to fp16 once in an fp16 x fp16 + fp32
 * FMA (relative error 2^-12); otherwise fp32 throughout.
 *
 * format KVQ_FMT_LOOPVQ: cfg is kvq_vq_cfg*, cache kvq_vq_cache*; layer and loop_step
 *   select the cache slice. The query sits at position seq_len[b] - 1; every key and the
 *   query are rotated by RoPE at their positions.
 * format KVQ_FMT_KIVI: cfg is kvq_kivi_cfg*, cache kvq_kivi_cache*; layer and loop_step
 *   are ignored; no RoPE (KIVI caches post-RoPE keys). Token t of request b uses the
 *   quantized key if t < n_quant_k[b] (else k_resid) and the quantized value if
 *   t < n_quant_v[b] (else v_resid), for t < n_tok[b].
 * out: [B][Hq][D], bf16 (KVQ_OUT_BF16) or fp32 (KVQ_OUT_FP32).
 * n_splits: how the quantized pages are split, 0 picks for the GPU.
 *   LoopVQ: thread blocks of the one persistent kernel. All index pages, in (head, request)
 *   segments, head-major, are cut into n_splits equal contiguous shares, one per block; the
 *   block holding a segment's first page also attends its bf16 window tokens (a block takes
 *   the windows of requests without index pages in turn). A segment split between blocks is
 *   merged exactly by the last of them to finish. 0 = one block per SM.
 *   KIVI: token splits per (request, KV head): split k takes an equal range of the
 *   quantized keys and the last split also the fp16 residual (its bytes counted in the
 *   ranges), merged by the last block of each (request, KV head) to finish; a block serves
 *   up to 4 query heads of its KV head, so their codes are read once.
 * ws: device workspace of at least kvq_decode_workspace_size() bytes (may be NULL when
 *   that size is 0; LoopVQ always needs one): merge counters (zero between calls) and
 *   partial softmaxes. A workspace must be zero-filled before its first use; every call
 *   that completes leaves it reusable (its counters back at zero). Two calls that run at the
 *   same time need two workspaces.
 * Errors: KVQ_ERR_INVALID_ARG, KVQ_ERR_WORKSPACE, KVQ_ERR_CAPACITY (B > max_batch),
 *   KVQ_ERR_UNSUPPORTED (LoopVQ: B > 8191). */
kvq_status kvq_decode_attn(int format, const void* cfg, const void* cache, int layer,
                           int loop_step, const uint16_t* q, int B, void* out, int out_dtype,
                           int n_splits, void* ws, size_t ws_bytes, kvq_stream stream);

/* Decode attention for callers that cannot allocate device memory: a serving engine that
 * gives all device memory to its own pool at start-up and forbids later allocations, or code
 * running inside another framework's callback that only sees the tensors it is handed.
 * The pages have no counterpart of this call; it is kvq_decode_attn with the workspace taken
 * from a fixed array inside the library (KVQ_NOALLOC_SCRATCH_BYTES per device) instead of
 * from the caller.
 * - Arguments and results are those of kvq_decode_attn without ws / ws_bytes; a call that
 *   kvq_decode_attn would refuse is refused with the same status before anything runs.
 * - CUDA loads the library's device code on a device lazily (first launch or symbol lookup
 *   there) and sets the array aside at that moment; it is then held until the process exits.
 *   The first call on a device looks the array's address up (cudaGetSymbolAddress), so make
 *   that first call before a memory pool takes the device's memory, and before any stream
 *   capture on that device.
 * - The address is kept per device: do not use the library across a cudaDeviceReset.
 * - Each call clears the part of the array it uses (cudaMemsetAsync on `stream`) and then
 *   launches; it never calls cudaMalloc or cudaFree.
 * - All calls on a device share the one array: calls that can run at the same time on the
 *   GPU (other streams, other host threads) race and must be serialised by the caller.
 * - A call that would need more scratch than the array holds returns KVQ_ERR_WORKSPACE
 *   without launching anything; use kvq_decode_attn with a workspace for it. */
#define KVQ_NOALLOC_SCRATCH_BYTES (8u << 20)
kvq_status kvq_decode_attn_noalloc(int format, const void* cfg, const void* cache, int layer,
                                   int loop_step, const uint16_t* q, int B, void* out,
                                   int out_dtype, int n_splits, kvq_stream stream);

/* Workspace bytes kvq_decode_attn needs for these arguments (0 if none). */
size_t kvq_decode_workspace_size(int format, const void* cfg, int B, int n_splits);

/* The split count kvq_decode_attn uses when n_splits = 0 (LoopVQ: the number of SMs). */
int kvq_decode_auto_splits(int format, const void* cfg, int B);

/* ---------------------------------------------------------------------------------- */
/* Diagnostics                                                                         */
/* ---------------------------------------------------------------------------------- */

const char* kvq_status_string(kvq_status s);
/* Detail of the last error on the calling host thread ("" if none). */
const char* kvq_last_error(void);
/* Reads and clears the device error word of the current device (synchronizes the device).
 * 0 = no device-side error; otherwise a KVQ_ERR_* code. The word's device address is looked
 * up once per device and kept, so the library must not be used across a cudaDeviceReset. */
int kvq_device_error(void);
/* Library version, major*10000 + minor*100 + patch. */
int kvq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
