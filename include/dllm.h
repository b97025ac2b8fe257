/*
 * dllm.h - C ABI of the GB300 (sm_103a) hot path of one LLaDA-style diffusion-LLM
 * denoising step: Q8_K activation quantization, Q4_K / Q6_K quantized GEMMs on the
 * tcgen05 tensor cores, the masked-rows-only LM head with softmax confidence and
 * top-k token commit, and the per-layer linear stream.
 *
 * Sources (mojo-dllm pages; cited by page title and section):
 *   [TS10]  Technical Specification, section 10 "Quantized Compute" (the entry point
 *           linear_q4k(x, weight, out): the product is formed from the packed blocks, each
 *           block expanded as it is used, with f32 accumulation; no dense weight copy)
 *   [TS9]   Technical Specification, section 9.2 (unknown types fail explicitly, no silent
 *           fallback) and section 27 (actionable errors).
 *   [TS28]  Technical Specification, section 28 (preallocated, reusable runtime buffers).
 *   [TS11]  Technical Specification, section 11 (LLaDA layer order) and 11.1 (bidirectional).
 *   [TS12]  Technical Specification, sections 12-14 (diffusion loop, scheduler select/update,
 *           softmax / argmax / top-k / scatter).
 *   [DP-CD] Development plan, "Compute design" (each token's activations become 8-bit codes
 *           with a float scale for every 256 of them and integer sums of every 16; each weight
 *           block expands to small unsigned integers with a scale and an offset for every 16;
 *           the output head runs only for the still-masked rows of the active block).
 *   [DP-MF] Development plan, "Model facts" (d 4096, 32 x 128 MHA, FFN 12288 SwiGLU,
 *           RMSNorm eps 1e-5, NORM RoPE theta 500000, vocab 126464, mask 126336).
 *   [DP-CO] Development plan, "Corrections to the spec" (Q4_K / Q6_K matrices, F32 norms).
 *   [RM-HW] README, "How it works" (logits for the positions the sampler reads, no others; LLaDA low-confidence
 *           remasking).
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers (global memory of the current device) unless a
 *     parameter says "host". The caller owns every buffer, including workspaces; no
 *     call allocates or frees device memory, and no call keeps a pointer after it
 *     returns.
 *   - Every call enqueues its kernels on `stream` and returns without synchronizing
 *     (asynchronous; stream-ordered). Calls enqueue no host callbacks and no
 *     allocations, so they may be captured into a CUDA graph by the caller.
 *   - Return value: DLLM_OK or a negative-free positive status below. On error nothing is
 *     launched and dllm_last_error() returns an actionable message (thread-local).
 *   - Device-side failures (a bounded wait that ran out) are recorded in a device error
 *     word; dllm_check(stream) synchronizes the stream and reports them.
 *   - Shapes: k (reduction length) must be a multiple of 256 (one super-block).
 *   - Host threads: calls may be made from several host threads at once, each with its own
 *     stream and buffers (the library's per-device caches are atomic, its error message is
 *     per thread). dllm_qgemm_noalloc is the exception: its calls share one device array. The
 *     device error word is one per device, so a device-side failure is reported by the next
 *     dllm_check on that device, whichever thread or stream makes it.
 */
#ifndef DLLM_H
#define DLLM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DLLM_API __attribute__((visibility("default")))
#else
#define DLLM_API
#endif

typedef struct CUstream_st* dllm_stream_t; /* same handle as cudaStream_t; NULL = legacy default */

/* ---- status codes ([TS9], [TS27]) ---------------------------------------------------------- */
enum {
  DLLM_OK = 0,
  DLLM_E_INVAL = 1,       /* NULL or non-device pointer, bad flag, bad range              */
  DLLM_E_SHAPE = 2,       /* k % 256 != 0, sizes <= 0, sizes above a stated limit          */
  DLLM_E_ALIGN = 3,       /* pointer not aligned as the call requires                      */
  DLLM_E_TYPE = 4,        /* unsupported block type (only Q4_K and Q6_K have kernels)      */
  DLLM_E_WORKSPACE = 5,   /* workspace smaller than the matching *_workspace_bytes()       */
  DLLM_E_CUDA = 6,        /* a CUDA runtime call failed (message names it)                 */
  DLLM_E_TIMEOUT = 7,     /* a device-side bounded wait ran out (reported by dllm_check)   */
  DLLM_E_DEVICE = 8,      /* current device is not sm_103 / lacks a feature               */
  DLLM_E_BOUNDS = 9       /* bounds-checked build only: a kernel access fell outside its
                             buffer and was skipped (reported by dllm_check with its site) */
};

/* GGML block type ids of the two matrix formats with kernels ([DP-CO]). */
enum { DLLM_Q4_K = 12, DLLM_Q6_K = 14 };

/* Thread-local message of the last failing call on this host thread ("" if none). */
DLLM_API const char* dllm_last_error(void);

/* Library ABI version (major * 100 + minor). */
DLLM_API int dllm_version(void);

/* Synchronize `stream`, then read and clear the device error word. Returns DLLM_OK,
 * DLLM_E_TIMEOUT (a kernel's bounded wait ran out; the message names the kernel role),
 * DLLM_E_INVAL (an input a kernel found invalid: an unfoldable Q4_K block, inconsistent plain
 * Q8_K sums), DLLM_E_BOUNDS (bounds-checked build only, see below) or DLLM_E_CUDA (a launch or
 * execution error, message from the runtime). */
DLLM_API int dllm_check(dllm_stream_t stream);

/* ---- weight packing ------------------------------------------------------------------------
 * The GEMMs read weights in a tile-major "packed" form made once at upload from the GGUF
 * blocks (the pages' one-time repack at load, README "How it works", re-shaped for the GPU):
 * rows are grouped in tiles of 128; for each (tile, super-block) the quant bytes and scale
 * bytes of the 128 rows form one contiguous blob (one bulk copy), and the f16 super-block
 * scales (d, and dmin for Q4_K) sit in a separate plane [tile][super-block][128 rows].
 * The packed form holds exactly the GGUF bytes, re-ordered (zero extra bytes per row);
 * rows beyond n up to the next multiple of 128 are zero.
 *
 * dllm_packed_bytes: bytes of the packed form of an n x k matrix (0 on bad arguments).
 * dllm_pack_weights: `blocks` = device copy of the GGUF row-major block array
 *   (n rows x k/256 blocks, 144 B per Q4_K block, 210 B per Q6_K block); `packed` must be
 *   256-byte aligned and hold dllm_packed_bytes(type, n, k) bytes. Errors: DLLM_E_TYPE,
 *   DLLM_E_SHAPE, DLLM_E_ALIGN, DLLM_E_INVAL, DLLM_E_WORKSPACE (packed_bytes too small). */
DLLM_API size_t dllm_packed_bytes(int type, int64_t n, int64_t k);
DLLM_API int dllm_pack_weights(int type, const void* blocks, int64_t n, int64_t k, void* packed,
                               size_t packed_bytes, dllm_stream_t stream);

/* ---- Q8_K activation quantization ([DP-CD]; RMSNorm [DP-MF]) -------------------------------
 * For each of `rows` rows of x (f32, row stride ldx elements), optionally RMSNorm first:
 *   xn = x / sqrt(mean(x^2) + eps) * norm_w          (norm_w == NULL: no normalization)
 * then per 256 values: amax = max|xn|; d = amax / 127; q = clamp(rint(xn * (127 / amax)),
 * -127, 127) (f32 multiply, round-half-even, IEEE division); amax == 0 gives d = 0, q = 0;
 * bsum[g] = sum of the 16 codes of group g.
 * Outputs (each optional, NULL = not written):
 *   q    int8  [rows][k]         d    f32 [rows][k/256]      bsum int16 [rows][k/16]
 *   act  the same codes in the tensor-core operand form read by the GEMMs, act_bytes
 *        >= dllm_act_bytes(rows, k), 256-byte aligned. Layout (Lp = dllm_act_rows(rows),
 *        planes at 1024-byte aligned offsets in this order):
 *          A-plane f16 [k/64][Lp][64]: the int8 codes as exact f16 values; within each
 *                  aligned group of 4 k-positions the order is (0, 2, 1, 3);
 *          J-plane f16 [k/256][Lp/8][2][8][8]: bsum (16 per super-block) as exact f16, in
 *                  8x8 core-matrix order (token-group, half, token, group);
 *          D-plane f32 [k/256][Lp]: the scales d.
 *        Rows rows..Lp-1 are written as zeros.
 * Errors: DLLM_E_SHAPE (k % 256, rows <= 0, rows > 65536), DLLM_E_INVAL, DLLM_E_ALIGN
 * (x not 16-byte aligned or ldx % 4), DLLM_E_WORKSPACE (act_bytes too small). */
DLLM_API int64_t dllm_act_rows(int64_t rows);
DLLM_API size_t dllm_act_bytes(int64_t rows, int64_t k);
DLLM_API int dllm_quantize_act(const float* x, int64_t rows, int64_t k, int64_t ldx,
                               const float* norm_w, float eps, int8_t* q, float* d, int16_t* bsum,
                               void* act, size_t act_bytes, dllm_stream_t stream);

/* ---- quantized GEMM ([TS10], [DP-CD]) --------------------------------------------------------
 * y[i][j] (+)= sum_k W[j][k] * d_act[i][k/256] * q_act[i][k]       i < m tokens, j < n rows
 * with W the exact decoded Q4_K (w = d*scale*q - dmin*min) or Q6_K (w = d*scale*(q-32))
 * weights of `w_packed` (from dllm_pack_weights) and the activations of `act` (from
 * dllm_quantize_act with the same m, k). Per super-block the integer sums run exactly on the
 * tensor cores (integer values carried in f16 operands, f32 accumulators in tensor memory)
 * and the f32 scale / offset epilogue applies d_act, d, dmin.
 * y: f32, row stride ldy >= n (elements, ldy % 4 == 0). accumulate = 0: y = result;
 * 1: y += result (residual add).
 * ws: scratch for split-K partial sums, ws_bytes >= dllm_qgemm_workspace_bytes(type, m, n,
 * k); may be NULL when that is 0. Deterministic: partials are summed in a fixed order.
 * Errors: DLLM_E_TYPE, DLLM_E_SHAPE, DLLM_E_ALIGN, DLLM_E_INVAL, DLLM_E_WORKSPACE. */
DLLM_API size_t dllm_qgemm_workspace_bytes(int type, int64_t m, int64_t n, int64_t k);
DLLM_API int dllm_qgemm(int type, const void* act, int64_t m, int64_t k, const void* w_packed,
                        int64_t n, float* y, int64_t ldy, int accumulate, void* ws, size_t ws_bytes,
                        dllm_stream_t stream);

/* The same GEMM on plain Q8_K activations, the form the pages' Q8_K blocks take ([DP-CD]: 8-bit
 * codes, an f32 scale for every 256 of them, int16 sums of every 16):
 *   q int8 [m][k], d f32 [m][k/256], bsum int16 [m][k/16] (e.g. dllm_quantize_act's q, d, bsum).
 * dllm_pack_act builds the operand form `act` (layout as in dllm_quantize_act, act_bytes >=
 *   dllm_act_bytes(rows, k), 256-byte aligned) from them; codes, scales and sums are copied
 *   exactly. bsum must hold the sums of the codes: a group whose sum differs is recorded in the
 *   device error word and dllm_check reports DLLM_E_INVAL (the outputs made from it are not
 *   valid). Alignment: q 8-byte, d 4-byte, bsum 2-byte.
 * dllm_qgemm_q4k / dllm_qgemm_q6k: dllm_pack_act into the start of ws, then dllm_qgemm with the
 *   rest of ws as its split-K workspace; ws >= dllm_qgemm_plain_workspace_bytes(type, m, n, k),
 *   256-byte aligned. Same results as dllm_qgemm on the operand form of the same codes.
 * Errors: as dllm_qgemm, plus those of dllm_pack_act. */
DLLM_API int dllm_pack_act(const int8_t* q, const float* d, const int16_t* bsum, int64_t rows, int64_t k, void* act,
                           size_t act_bytes, dllm_stream_t stream);
DLLM_API size_t dllm_qgemm_plain_workspace_bytes(int type, int64_t m, int64_t n, int64_t k);
DLLM_API int dllm_qgemm_q4k(const int8_t* q, const float* d, const int16_t* bsum, int64_t m, int64_t k,
                            const void* w_packed, int64_t n, float* y, int64_t ldy, int accumulate, void* ws,
                            size_t ws_bytes, dllm_stream_t stream);
DLLM_API int dllm_qgemm_q6k(const int8_t* q, const float* d, const int16_t* bsum, int64_t m, int64_t k,
                            const void* w_packed, int64_t n, float* y, int64_t ldy, int accumulate, void* ws,
                            size_t ws_bytes, dllm_stream_t stream);

/* Test hook ([DP-CD] integer sums): writes the exact per-super-block integer sums that the
 * tensor cores accumulate, as int32 sums[2][k/256][m][n]:
 *   Q4_K: sums[0] = sum_g scale * sum_i q4_i * a_i,      sums[1] = sum_g min * bsum_g
 *   Q6_K: sums[0] = sum_g s_hi * sum_i (q6_i-32) * a_i, sums[1] = sum_g s_lo * sum_i (q6_i-32) * a_i
 *         where the int8 group scale s = 16 * s_hi + s_lo, s_lo in [0, 15].
 * dllm_qgemm accumulates all parts of a super-block in one tensor-memory accumulator (Q4_K:
 * the integer chain uses re-centred quants, I' = sum_g scale * sum_i (q4_i - 8) * a_i, whose
 * partial sums stay below 2^24 for every input, and the offset 8 * scale and the min part
 * enter with f16 head and tail coefficients 8 * scale - min * dmin / d, 2^-22 relative;
 * Q6_K: the hi operand carries s_hi * (q6-32) and the lo operand s_lo * (q6-32) / 16, and the
 * epilogue applies 16 d). This hook runs the same kernel once per
 * part with one split, each time with one part isolated, and copies out its exact integers
 * (Q4_K: I', J, then the offset part added to I' to give sums[0] = I); intended for small
 * shapes. */
DLLM_API int dllm_qgemm_intsums(int type, const void* act, int64_t m, int64_t k, const void* w_packed,
                                int64_t n, int32_t* sums, dllm_stream_t stream);

/* ---- masked-rows-only LM head + softmax confidence + top-k commit ([RM-HW], [DP-CD], [TS12]) --
 * For the block positions p in [block_begin, block_end) (R = block_end - block_begin, 1..160):
 *   1. h_p = RMSNorm(hidden[p]) * out_norm_w (eps; out_norm_w f32 [d], required), Q8_K;
 *   2. logits_p = h_p x W_out^T over all `vocab` rows of the packed Q6_K head (the GEMM above);
 *      the logits are reduced on the fly (never stored): per row, argmax id (lowest id on ties)
 *      and confidence = softmax(logits_p)[argmax] = 1 / sum_v exp(logit_v - logit_max);
 *   3. among the positions with canvas[p] == mask_id, the k_commit with the highest confidence
 *      (ties: lowest position) get canvas[p] = argmax id.
 * hidden: f32 [L][ldh] (row stride ldh >= d, ldh % 4 == 0). canvas: int32 [L], updated in place.
 * out_pos / out_id (int32 [k_commit]) and out_conf (f32 [k_commit], may be NULL) receive the
 * commits in selection order (descending confidence); entries past the number of masked
 * positions are -1 / -1 / 0. row_id / row_conf (length R, may be NULL) receive every block row's
 * argmax id and confidence (masked or not). ws: >= dllm_lmhead_workspace_bytes(R, vocab, d),
 * 256-byte aligned. Errors: DLLM_E_SHAPE, DLLM_E_INVAL (block range, k_commit), DLLM_E_ALIGN,
 * DLLM_E_WORKSPACE. */
DLLM_API size_t dllm_lmhead_workspace_bytes(int64_t rows, int64_t vocab, int64_t d);

/* Confidence used to rank the masked positions (dllm_lmhead_select):
 *   DLLM_CONF_PMAX        softmax probability of the argmax token, 1 / sum_v exp(l_v - l_max)
 *                         (LLaDA's low-confidence remasking: mojo-dllm "Each model's own sampler");
 *   DLLM_CONF_NEG_ENTROPY minus the entropy of the row's softmax, sum_v p_v log p_v (natural log;
 *                         Dream's entropy ranking, same page, and the "entropy" primitive of the
 *                         sampling section). Committed tokens are the argmax in both (greedy).
 * Like p_max, the fused epilogue reduces it on the fly: per partial it also keeps
 * t = sum exp(l - m)(l - m), and -H = t / s - log s for the merged s = sum exp(l - l_max). */
enum { DLLM_CONF_PMAX = 0, DLLM_CONF_NEG_ENTROPY = 1 };

/* dllm_lmhead_select: dllm_lmhead_masked_select with the confidence chosen by conf_kind
 * (DLLM_CONF_PMAX or DLLM_CONF_NEG_ENTROPY; anything else is DLLM_E_INVAL) and an optional
 * temperature (the specification's sampling section: temperature, categorical sampling,
 * deterministic PRNG; its section 30, definition of done: a fixed seed gives the same run).
 * out_conf and row_conf hold the chosen confidence. The block may be the whole canvas (every
 * masked position, R up to 160).
 *   temperature == 0: greedy, the row's token is the argmax (as dllm_lmhead_masked_select).
 *   temperature  > 0: the row's token is a draw from softmax(logits / temperature) by the
 *       Gumbel-max rule, argmax_v (l_v / temperature + g_v), g_v = -log(-log u_v) (ties: lowest
 *       id). u_v comes from counter-based SplitMix64 (Steele, Lea and Flood, "Fast splittable
 *       pseudorandom number generators", OOPSLA 2014): z = mix(seed + (c + 1) 0x9E3779B97F4A7C15)
 *       for the counter c = step * 2^40 + p * 2^24 + v (p the canvas position, v the token id),
 *       u_v = ((z >> 41) + 1/2) / 2^23 (23 bits: exact in f32 and strictly inside (0, 1)).
 *       DLLM_CONF_PMAX is then the drawn token's probability under the untempered softmax,
 *       exp(l_draw - l_max) / sum_v exp(l_v - l_max); the entropy confidence does not depend on
 *       the draw. Same inputs give the same draws.
 * Errors as below, plus DLLM_E_INVAL for a negative or non-finite temperature, or (sampling
 * only) L > 65536 or step >= 2^24. */
DLLM_API int dllm_lmhead_select(const float* hidden, int64_t L, int64_t d, int64_t ldh, const float* out_norm_w,
                                float eps, const void* w_out_packed, int64_t vocab, int32_t* canvas, int32_t mask_id,
                                int32_t block_begin, int32_t block_end, int32_t k_commit, int32_t conf_kind,
                                float temperature, uint64_t seed, uint32_t step, int32_t* out_pos, int32_t* out_id,
                                float* out_conf, int32_t* row_id, float* row_conf, void* ws, size_t ws_bytes,
                                dllm_stream_t stream);
DLLM_API int dllm_lmhead_masked_select(const float* hidden, int64_t L, int64_t d, int64_t ldh, const float* out_norm_w,
                                       float eps, const void* w_out_packed, int64_t vocab, int32_t* canvas,
                                       int32_t mask_id, int32_t block_begin, int32_t block_end, int32_t k_commit,
                                       int32_t* out_pos, int32_t* out_id, float* out_conf, int32_t* row_id,
                                       float* row_conf, void* ws, size_t ws_bytes, dllm_stream_t stream);

/* ---- LLaDA layer stream and full denoising step ([TS11], [DP-MF], [TS12]) -------------------
 * Weights of one layer (device pointers). Q and K are packed as ONE Q4_K matrix of 2*d rows
 * (rows 0..d-1 = Q, d..2d-1 = K); gate and up as ONE Q4_K matrix of 2*d_ff rows (rows
 * 0..d_ff-1 = gate, d_ff..2*d_ff-1 = up); all from dllm_pack_weights. */
typedef struct dllm_layer {
  const void* wqk;         /* packed Q4_K [2d][d]      */
  const void* wv;          /* packed Q6_K [d][d]       */
  const void* wo;          /* packed Q4_K [d][d]       */
  const void* wgu;         /* packed Q4_K [2 d_ff][d]  */
  const void* wdown;       /* packed Q6_K [d][d_ff]    */
  const float* attn_norm;  /* f32 [d]                  */
  const float* ffn_norm;   /* f32 [d]                  */
} dllm_layer;

typedef struct dllm_model {
  int32_t n_layers, d_model, n_heads, head_dim, d_ff, vocab, mask_id;
  float eps, rope_theta;
  const dllm_layer* layers; /* HOST array of n_layers entries holding device pointers          */
  const void* tok_embd;     /* GGUF Q4_K blocks [vocab][d_model/256] (device, unpacked AoS)    */
  const float* out_norm;    /* f32 [d_model] (device)                                          */
  const void* w_out;        /* packed Q6_K [vocab][d_model] (device)                           */
} dllm_model;

enum { DLLM_STREAM_LINEAR = 0, DLLM_STREAM_FULL = 1 };

/* dllm_step_linear_stream: the per-layer stream over all model->n_layers layers on L canvas
 * rows; x is f32 [L][d_model] (row stride d_model, 16-byte aligned).
 *   DLLM_STREAM_FULL:   x = embedding of canvas (int32 [L] token ids); every layer runs
 *       x_n = RMSNorm(x) * attn_norm -> Q8_K -> [Q|K] (Q4_K), V (Q6_K) -> NORM RoPE on Q, K
 *       (theta, positions 0..L-1) -> non-causal attention (softmax(QK^T/sqrt(hd)) V) -> Q8_K
 *       -> O (Q4_K) -> x += O; RMSNorm(x) * ffn_norm -> Q8_K -> [gate|up] (Q4_K) ->
 *       silu(gate) * up -> Q8_K -> down (Q6_K) -> x += down. On return x holds the final
 *       residual stream (before the output norm).
 *   DLLM_STREAM_LINEAR: x is the input and is updated in place by the same stream without
 *       attention: the O projection consumes the V projection's output (canvas unused).
 * ws: >= dllm_step_workspace_bytes(m, L, flags), 1024-byte aligned; it holds the quantized
 * activations, the split-K partials of every projection and the attention buffers.
 * Limits: d_model and d_ff multiples of 256, d_model <= 16384, head_dim == 128, L <= 8192. */
DLLM_API size_t dllm_step_workspace_bytes(const dllm_model* m, int64_t L, int flags);
DLLM_API int dllm_step_linear_stream(const dllm_model* m, const int32_t* canvas, int64_t L, float* x, int flags,
                                     void* ws, size_t ws_bytes, dllm_stream_t stream);

/* Test hook: dllm_step_linear_stream that also copies out the intermediates of one layer, so
 * that each stage of the layer can be checked on its own input (the Development plan's
 * correctness ladder: RMSNorm, RoPE, softmax, attention, one layer). Every tap is optional
 * (NULL = not captured) and caller-owned device memory; "operand" taps are dllm_act_bytes(L, k)
 * bytes in the operand form of dllm_quantize_act. */
typedef struct dllm_taps {
  int32_t layer;   /* the layer whose intermediates are captured, 0 .. n_layers - 1              */
  float* x_in;     /* f32 [L][d]: the layer's input residual stream                                */
  void* act_attn;  /* operand of RMSNorm(x) * attn_norm (the Q|K and V projections' input), k = d */
  float* q;        /* f32 [L][d]: Q after RoPE, times 1/sqrt(head_dim) (DLLM_STREAM_FULL only)    */
  float* k;        /* f32 [L][d]: K after RoPE (DLLM_STREAM_FULL only)                            */
  float* v;        /* f32 [L][d]: V (DLLM_STREAM_FULL only)                                        */
  float* attn;     /* f32 [L][d], 16-byte aligned: the O projection's input before Q8_K (the
                      attention output; the V projection for DLLM_STREAM_LINEAR)                   */
  void* act_o;     /* operand of that input, k = d                                                 */
  float* x_mid;    /* f32 [L][d]: the residual stream after the O residual add                     */
  void* act_ffn;   /* operand of RMSNorm(x_mid) * ffn_norm (the gate|up input), k = d              */
  float* h;        /* f32 [L][d_ff], 16-byte aligned: silu(gate) * up before Q8_K                  */
  void* act_down;  /* operand of h (the down projection's input), k = d_ff                         */
  float* x_out;    /* f32 [L][d]: the residual stream after the down residual add                  */
} dllm_taps;
DLLM_API int dllm_step_taps(const dllm_model* m, const int32_t* canvas, int64_t L, float* x, int flags,
                            const dllm_taps* taps, void* ws, size_t ws_bytes, dllm_stream_t stream);

/* dllm_denoise_step: one full denoising step = DLLM_STREAM_FULL forward over the canvas,
 * then dllm_lmhead_masked_select on the block [block_begin, block_end) with k_commit
 * commits (canvas updated in place; out_* as there). hidden_out (f32 [L][d_model], may be
 * NULL) receives the final residual stream. ws: >= dllm_denoise_workspace_bytes(m, L,
 * block_end - block_begin), 1024-byte aligned. */
DLLM_API size_t dllm_denoise_workspace_bytes(const dllm_model* m, int64_t L, int32_t block_rows);
DLLM_API int dllm_denoise_step(const dllm_model* m, int32_t* canvas, int64_t L, int32_t block_begin,
                               int32_t block_end, int32_t k_commit, int32_t* out_pos, int32_t* out_id,
                               float* out_conf, float* hidden_out, void* ws, size_t ws_bytes,
                               dllm_stream_t stream);

/* ---- inter-step K/V cache ("--dual-cache": mojo-dllm README status table, opt-in and not
 * exact; specification section 23, "Future Caching Research": inter-step cache, which must report
 * speedup, memory and output divergence) ------------------------------------------------------
 * dllm_kv_cache_bytes: size of the cache, f32 [n_layers][2][L][d_model] (per layer K after RoPE,
 *   then V, for every canvas row); caller-owned device memory, 16-byte aligned.
 * dllm_denoise_step_cached: one denoising step with the cache.
 *   refresh = 1: exactly dllm_denoise_step, and every layer's K and V of all L rows are stored in
 *       kv_cache (the first step of a block);
 *   refresh = 0: only the block's rows [block_begin, block_end) (1..160 rows) run through the
 *       layers: embedding, projections, RoPE at their canvas positions, attention of their
 *       queries over all L keys and values taken from kv_cache (the block's own rows replaced by
 *       their fresh K and V, which are also written back), O, FFN; then the head and commit
 *       on the block as in dllm_denoise_step. Rows outside the block keep the K and V of the
 *       last refresh, so the result is an approximation of the uncached step.
 *   A cached step reads what the last refreshing step on this cache stored (same model, same L):
 *   the first step on a cache must refresh, and a cached step before any refresh computes from
 *   undefined cache contents (no fault: every access stays inside the buffer).
 *   hidden_out (may be NULL): f32 [L][d_model]; a cached step writes the block's rows only.
 *   ws: >= dllm_denoise_cached_workspace_bytes(m, L, block_end - block_begin), 1024-byte aligned.
 * Errors: as dllm_denoise_step, plus DLLM_E_WORKSPACE for a short kv_cache, DLLM_E_ALIGN for a
 * misaligned one and DLLM_E_INVAL for refresh not 0 or 1. */
DLLM_API size_t dllm_kv_cache_bytes(const dllm_model* m, int64_t L);
DLLM_API size_t dllm_denoise_cached_workspace_bytes(const dllm_model* m, int64_t L, int32_t block_rows);
DLLM_API int dllm_denoise_step_cached(const dllm_model* m, int32_t* canvas, int64_t L, int32_t block_begin,
                                      int32_t block_end, int32_t k_commit, int32_t refresh, float* kv_cache,
                                      size_t kv_bytes, int32_t* out_pos, int32_t* out_id, float* out_conf,
                                      float* hidden_out, void* ws, size_t ws_bytes, dllm_stream_t stream);

/* ---- transfer schedule (Development plan, "Benchmark protocol": 128 generated tokens in
 * blocks of 32 over 32 steps, 4 commits per step, transfer counts checked against the reference
 * generator; Technical Specification, section 13 "Scheduler Interface": select the positions
 * to commit, then update the canvas) -------------------------------------------------------
 * Host-only calls: no device work, no stream; outputs are HOST arrays owned by the caller.
 * dllm_transfer_counts: how many of a block's `masked` masked positions are committed at each
 *   of its `steps` steps: floor(masked / steps) at every step, plus one more at each of the
 *   first masked % steps steps. counts: int32 [steps]; the counts sum to `masked`.
 *   Errors: DLLM_E_INVAL (masked outside [0, 2^30], steps outside [1, 2^20], counts NULL).
 * dllm_schedule: the whole generation of gen_len positions after prompt_len, in blocks of
 *   block_len over `steps` steps: step s works on block b = s / (steps / blocks), the positions
 *   [prompt_len + b * block_len, prompt_len + (b + 1) * block_len), and commits k[s] tokens, the
 *   dllm_transfer_counts(block_len, steps / blocks) entry of its place in the block (every
 *   position of a block is masked when the block starts). block_begin, block_end, k: int32
 *   [steps]. Errors: DLLM_E_INVAL (a size out of range, gen_len not a multiple of block_len,
 *   steps not a multiple of the block count, a NULL output). */
DLLM_API int dllm_transfer_counts(int64_t masked, int64_t steps, int32_t* counts);
DLLM_API int dllm_schedule(int64_t prompt_len, int64_t gen_len, int64_t block_len, int64_t steps,
                           int32_t* block_begin, int32_t* block_end, int32_t* k);

/* Benchmark hooks.
 * dllm_launch_count: number of kernels this library has enqueued so far in this process (a
 *   host-side counter; launches recorded during stream capture count once, at capture).
 * dllm_qgemm_partials: the GEMM kernel alone, without the split-K reduction: writes the
 *   plan's split partials f32 [splits][m][n] (their sum is dllm_qgemm's result) and stores
 *   the number of splits in *splits (host pointer, may be NULL). partials_bytes >=
 *   dllm_qgemm_partials_bytes(type, m, n, k). Used to time the tensor-core kernel alone. */
DLLM_API long long dllm_launch_count(void);
DLLM_API size_t dllm_qgemm_partials_bytes(int type, int64_t m, int64_t n, int64_t k);
DLLM_API int dllm_qgemm_partials(int type, const void* act, int64_t m, int64_t k, const void* w_packed, int64_t n,
                                 float* partials, size_t partials_bytes, int32_t* splits, dllm_stream_t stream);

/* dllm_peak_mma_i8: measures the legacy int8 tensor path's dense rate (mma.sync m16n8k32,
 *   s8 x s8 -> s32, eight independent chains per warp, four 8-warp CTAs per SM) for the
 *   benchmark's second roofline: one launch of `iters` iterations; *ops_per_launch (host, may be
 *   NULL) receives the launch's algorithmic ops (2 * 16 * 8 * 32 per mma). sink: device int32,
 *   written only in a case that does not happen in practice. Time it with events on `stream`. */
DLLM_API int dllm_peak_mma_i8(int64_t iters, int32_t* sink, double* ops_per_launch, dllm_stream_t stream);

/* ---- allocation-free GEMM (the pages have no counterpart to this entry point) ----------------
 * For callers that cannot allocate device memory or hand over a workspace at call time (an
 * inference server that reserves all device memory at start-up, a plugin interface that
 * passes only inputs and outputs, a loop that must not call cudaMalloc because it can
 * synchronize the device). Same result as dllm_qgemm, but the split-K partial sums live in a
 * fixed 32 MiB array that the library holds in every GPU's memory until exit; m * n * 4 must
 * not exceed 32 MiB (larger shapes return DLLM_E_SHAPE; the split count is reduced to 1 when
 * the plan's partials would not fit). The first call on a device looks up that array's device
 * address (once per device, with the device current); make it before any stream capture.
 * Calls share the array: calls that overlap on the GPU race and must be serialized by the
 * caller. No device memory is allocated or freed. The looked-up address is kept for the life of
 * the process and does not survive a device reset: after cudaDeviceReset on a device, do not
 * call this entry point on that device again. */
DLLM_API int dllm_qgemm_noalloc(int type, const void* act, int64_t m, int64_t k, const void* w_packed, int64_t n,
                                float* y, int64_t ldy, int accumulate, dllm_stream_t stream);

/* Test hook for failure detection: launches one kernel whose mbarrier wait can never
 * complete, bounded by `limit_cycles` SM clock cycles; the kernel then records a timeout
 * in the device error word and returns. dllm_check() afterwards reports DLLM_E_TIMEOUT. */
DLLM_API int dllm_selftest_timeout(int64_t limit_cycles, dllm_stream_t stream);

/* ---- one step from host buffers ------------------------------------------------------------
 * The host side of one denoising step around a step the caller captured once into a CUDA graph
 * (e.g. dllm_denoise_step on `canvas` between cudaStreamBeginCapture and cudaStreamEndCapture,
 * instantiated): one call copies the host canvas in, runs the graph and reads the commits out
 * (README "How it works": each step commits k tokens into the canvas, which the next step
 * reads). `graph_exec` is the cudaGraphExec_t; `canvas_host` the host canvas (L int32, pinned
 * host memory for asynchronous copies), `canvas` the device canvas the graph was captured on;
 * `out` the device positions (int32 [k_commit] at out[0]) and ids (at out[out_stride]) the
 * graph's commit writes. The call copies the host canvas to `canvas`, launches the graph on
 * `stream`, copies the positions then the ids to out_host (host int32 [2 * k_commit]), waits
 * for the stream and writes each committed id into canvas_host (positions < 0, meaning no
 * commit, are skipped). It is synchronous (it returns after the step). Errors: DLLM_E_INVAL
 * (null host pointers or graph, k_commit > out_stride, L out of range, canvas / out not device
 * pointers), DLLM_E_CUDA. */
DLLM_API int dllm_step_graph_host(void* graph_exec, int32_t* canvas_host, int32_t* canvas, int64_t L,
                                  const int32_t* out, int32_t out_stride, int32_t k_commit, int32_t* out_host,
                                  dllm_stream_t stream);

/* ---- bounds-checked build --------------------------------------------------------------------
 * The same sources also build libdllm_checked.so (compiled with DLLM_BOUNDS_CHECK), a debug
 * library with the same entry points in which every global-memory access of every kernel is
 * first checked against the extent of the buffer it targets. The extents are computed on the
 * host from each call's shapes (the buffer sizes documented above); tensor-map copies are
 * checked by the hardware against their maps. An access outside its buffer is skipped instead
 * of performed, and dllm_check then returns DLLM_E_BOUNDS naming the source file and line of the
 * first such access (a skipped copy also makes the waits on it run out, so a GEMM launch may
 * report a timeout with it). Outputs of a launch that reported DLLM_E_BOUNDS are not valid. The
 * checked library is slower and is meant for tests and debugging, not for measurement.
 *
 * dllm_bounds_checked: 1 in the bounds-checked build, 0 in the regular one.
 * dllm_selftest_bounds: test hook; writes buf[i] = i for 0 <= i < n_write, each store checked
 *   against a span of the first n_declared floats of buf. The regular build performs every
 *   store; the checked build skips those with i >= n_declared and records DLLM_E_BOUNDS. `buf`
 *   must hold n_write floats, so no store ever leaves the real buffer. Errors: DLLM_E_INVAL
 *   (0 < n_write <= 2^20 and 0 <= n_declared <= n_write required). */
DLLM_API int dllm_bounds_checked(void);
DLLM_API int dllm_selftest_bounds(float* buf, int32_t n_write, int32_t n_declared, dllm_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DLLM_H */
