/*
 * gdpa.h -- C ABI of the GB300 (sm_103a) jagged attention library.
 *
 * The operation: attention over jagged (variable-length, unpadded) samples,
 * i.e. two matrix products with an elementwise activation between them.
 * Softmax as the activation is jagged flash attention (JFA); SiLU or GELU in
 * place of softmax is generalized dot-product attention (GDPA), one kernel
 * for self-attention, PMA and cross-attention.  Source: "GEM Training: How
 * Meta Doubled the Efficiency of Its LLM-Scale Ads Foundation Model", JFA
 * paragraph (jagged tensors, custom attention biases, asymmetric query /
 * key-value lengths, backward passes) and GDPA paragraph ("two matrix
 * multiplications with an element-wise activation in between").
 *
 * For sample b with Lq_b = q_offsets[b+1]-q_offsets[b] query rows and
 * Lkv_b = kv_offsets[b+1]-kv_offsets[b] key/value rows, head h, local row i
 * and local key j (mask: j <= i when causal, and |i - j| < window for the
 * sliding-window entry points; else all):
 *     s_ij  = scale * <q_i, k_j> + bias_h(i - j)      (or + a dense bias B_b[h][i][j])
 *     p_ij  = softmax_j(s_ij)       (GDPA_ACT_SOFTMAX, masked entries excluded)
 *           = act(s_ij)             (SiLU, GELU-tanh, GELU-erf, identity; no normalisation)
 *     out_i = sum_j p_ij v_j
 * SiLU(x) = x sigmoid(x); GELU-tanh(x) = 0.5 x (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3)));
 * GELU-erf(x) = 0.5 x (1 + erf(x / sqrt(2))).
 * A softmax row with no key gets out = 0 and lse = -inf; GDPA rows with no
 * key get 0.  Samples with no query rows write nothing.
 *
 * Conventions shared by every call:
 *  - Layouts: q, out, dout, dq: [Tq][H][d] bf16 row-major ("THD"); k, v, dk,
 *    dv: [Tkv][H][d] bf16; lse: [H][Tq] fp32; offsets: int32 [B+1] with
 *    offsets[0] = 0, non-decreasing, offsets[B] = Tq (or Tkv).  All tensors
 *    and offsets live in device memory; B, H, d, Tq, Tkv are host scalars,
 *    so no call reads anything back from the device.
 *  - d must be 64 or 128; H <= 256.  Tensor base addresses must be 16-byte
 *    aligned.
 *  - Ownership: the caller owns every buffer, including the workspace (size
 *    from the matching *_workspace_size query).  Calls enqueue work on
 *    `stream` (a cudaStream_t; NULL = legacy default stream) and return
 *    without synchronising.  They do not allocate device memory.
 *  - Errors: argument errors detectable on the host return immediately and
 *    launch nothing.  Errors only the device can see (malformed offsets,
 *    causal with Lq_b != Lkv_b, a pipeline wait that timed out) set a device
 *    status word; gdpa_get_device_status() synchronises the stream, returns
 *    it and clears it.  After such an error the outputs are undefined, but
 *    every write stays inside the caller's buffers.
 *  - Per-device state: on its first call on a device the library looks up
 *    the device addresses of its status word and of the gdpa_fwd_noalloc
 *    scratch array and keeps them for the life of the process.  A
 *    cudaDeviceReset() in the caller's process unloads the library's device
 *    code and makes those addresses stale: do not call the library on that
 *    device after a reset.
 *
 * Entry points: gdpa_fwd / gdpa_bwd (and their _window forms; gdpa_bwd_rope
 * adds the fused rotary backward), gdpa_fwd_noalloc, the block-aligned
 * gdpa_block_fwd / gdpa_block_bwd, the MXFP8 gdpa_quantize_mxfp8,
 * gdpa_fwd_mxfp8(_window) and gdpa_bwd_mxfp8(_window, _rope), the workspace-size
 * queries, and the status, launch-count, timing and self-test helpers.
 */
#ifndef GDPA_H_
#define GDPA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDPA_ACT_SOFTMAX = 0,   /* JFA */
  GDPA_ACT_SILU = 1,      /* GDPA */
  GDPA_ACT_GELU_TANH = 2, /* GDPA */
  GDPA_ACT_IDENTITY = 3,  /* GDPA, linear attention; useful for testing */
  GDPA_ACT_GELU_ERF = 4   /* GDPA, exact GELU 0.5 x (1 + erf(x / sqrt(2))) */
} gdpa_act;

typedef enum { GDPA_BIAS_NONE = 0, GDPA_BIAS_RELPOS = 1, GDPA_BIAS_DENSE = 2 } gdpa_bias_kind;

/* Additive attention bias ("custom attention biases", JFA paragraph).
 * GDPA_BIAS_RELPOS: per-head relative-position table, fp32 device memory
 * [H][2*max_rel-1]; bias_h(i-j) = table[h][clamp(i-j+max_rel-1, 0, 2*max_rel-2)]
 * with per-sample local positions i, j.  1 <= max_rel <= 65536.
 * GDPA_BIAS_DENSE: a dense jagged bias, one fp32 value per (head, query, key)
 * of each sample: `table` holds the samples' [H][Lq_b][Lkv_b] blocks one after
 * another, sample b's block starting at element offsets[b] (int64 device
 * array [B+1], offsets[0] = 0, offsets[b+1] - offsets[b] = H Lq_b Lkv_b;
 * a mismatch is reported as GDPA_ERR_BAD_OFFSETS through the device status).
 * max_rel is ignored.  The dense bias is read from global memory by the
 * kernels' activation warps; it is supported by gdpa_fwd, gdpa_bwd,
 * gdpa_fwd_noalloc, gdpa_fwd_window and gdpa_bwd_window / gdpa_bwd_rope
 * (these two also return its gradient), with or without a sliding window, by
 * gdpa_block_fwd / gdpa_block_bwd / gdpa_block_bwd_dbias (the last with its
 * gradient), by gdpa_fwd_mxfp8(_window) and by gdpa_bwd_mxfp8(_window,
 * _rope) (the last with its gradient). */
typedef struct {
  int kind;                /* gdpa_bias_kind */
  const float* table;      /* device pointer, ignored for GDPA_BIAS_NONE */
  int max_rel;
  const int64_t* offsets;  /* GDPA_BIAS_DENSE only (device pointer), else ignored */
} gdpa_bias;

typedef enum {
  GDPA_OK = 0,
  GDPA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned tensor */
  GDPA_ERR_UNSUPPORTED = 2,  /* d not in {64,128}, H > 256, ... */
  GDPA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than the query says */
  GDPA_ERR_CUDA = 4,         /* a CUDA runtime call failed */
  GDPA_ERR_TIMEOUT = 5,      /* device: a pipeline wait ran past its limit */
  GDPA_ERR_BAD_OFFSETS = 6   /* device: offsets malformed, or causal / window with Lq_b != Lkv_b */
} gdpa_status;

/* Bytes of workspace gdpa_fwd needs (the work list of the persistent
 * scheduler).  Depends only on the host scalars. */
size_t gdpa_fwd_workspace_size(int B, int H, int d, int64_t Tq, int64_t Tkv);

/* Forward pass.
 *   q [Tq][H][d] bf16, k/v [Tkv][H][d] bf16, offsets int32 [B+1] (device).
 *   bias: NULL or kind NONE for no bias.  act: gdpa_act.  causal: 0/1
 *   (top-left, j <= i; every sample must have Lq_b == Lkv_b).
 *   out [Tq][H][d] bf16 (written only at rows that belong to a sample).
 *   lse [H][Tq] fp32: natural-log row logsumexp for softmax (needed by the
 *   backward); may be NULL for the GDPA activations, where it is not written.
 *   workspace: device memory of at least gdpa_fwd_workspace_size() bytes. */
gdpa_status gdpa_fwd(const void* q, const int32_t* q_offsets, const void* k, const void* v,
                     const int32_t* kv_offsets, int B, int H, int d, int64_t Tq, int64_t Tkv,
                     const gdpa_bias* bias, int act, int causal, float scale, void* out,
                     float* lse, void* workspace, size_t ws_bytes, void* stream);

/* Bytes of workspace gdpa_bwd needs (work list, fp32 dQ accumulator and the
 * per-row D = rowsum(dO * O) of the softmax backward). */
size_t gdpa_bwd_workspace_size(int B, int H, int d, int64_t Tq, int64_t Tkv);

/* Backward pass: recomputes the scores per tile and writes dq [Tq][H][d],
 * dk and dv [Tkv][H][d] (bf16).  out and lse are the forward's outputs
 * (needed for softmax only; may be NULL for the GDPA activations).  dout
 * [Tq][H][d] bf16.  Rows of dk/dv of a sample with no query, and rows of dq
 * of a sample with no key, are written as zeros. */
gdpa_status gdpa_bwd(const void* q, const int32_t* q_offsets, const void* k, const void* v,
                     const int32_t* kv_offsets, int B, int H, int d, int64_t Tq, int64_t Tkv,
                     const gdpa_bias* bias, int act, int causal, float scale, const void* out,
                     const float* lse, const void* dout, void* dq, void* dk, void* dv,
                     void* workspace, size_t ws_bytes, void* stream);

/* Sliding-window attention ("GEM Training ..." SWA paragraph: each token
 * attends only to nearby events, O(L * window) work instead of O(L^2), and
 * the kernel skips the tiles outside the window).  window > 0 keeps the
 * pairs with |i - j| < window, intersected with j <= i when causal: a causal
 * row sees its `window` most recent keys (itself included), a non-causal row
 * also the window - 1 keys after it.  window == 0 is no window (the calls
 * then equal gdpa_fwd / gdpa_bwd).  A window needs Lq_b == Lkv_b for every
 * sample (device check, GDPA_ERR_BAD_OFFSETS); window < 0 returns
 * GDPA_ERR_INVALID_ARG.  Key / query tiles outside the band are never
 * loaded, and the scheduler's cost counts only the tiles inside it.  Every
 * other argument, output, workspace and error is that of gdpa_fwd /
 * gdpa_bwd; the backward must get the forward's window.
 * dbias (gdpa_bwd_window and gdpa_bwd_rope; NULL = not computed): the
 * gradient of a learnable bias ("custom attention biases", JFA paragraph),
 * fp32 device memory, ADDED to (so gradients of several calls accumulate;
 * zero it first for a fresh gradient); every activation.
 *   GDPA_BIAS_RELPOS: [H][2*max_rel-1]; entry t receives the sum of dS_ij
 *   over the unmasked pairs whose clamped table index (i - j + max_rel - 1)
 *   is t.  Its atomics make the sums' order, and so their last bits, vary
 *   between runs.
 *   GDPA_BIAS_DENSE: the dense bias's own layout (offsets[B] floats); the
 *   entry of each unmasked pair receives that pair's dS_ij (the bf16 value
 *   the softmax kernel feeds its products, the fp32 one for the other
 *   activations); masked pairs' entries are left as they are.
 * dS_ij is the gradient of the loss with respect to s_ij = scale q_i.k_j +
 * bias_ij.  Without a bias: GDPA_ERR_INVALID_ARG. */
gdpa_status gdpa_fwd_window(const void* q, const int32_t* q_offsets, const void* k,
                            const void* v, const int32_t* kv_offsets, int B, int H, int d,
                            int64_t Tq, int64_t Tkv, const gdpa_bias* bias, int act, int causal,
                            int window, float scale, void* out, float* lse, void* workspace,
                            size_t ws_bytes, void* stream);
gdpa_status gdpa_bwd_window(const void* q, const int32_t* q_offsets, const void* k,
                            const void* v, const int32_t* kv_offsets, int B, int H, int d,
                            int64_t Tq, int64_t Tkv, const gdpa_bias* bias, int act, int causal,
                            int window, float scale, const void* out, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, float* dbias,
                            void* workspace, size_t ws_bytes, void* stream);

/* Block-aligned attention ("GEM Training ..." SWA paragraph: with fixed
 * 64-token blocks each query block attends only to its own key/value block,
 * giving independent 64 x 64 problems without online softmax correction,
 * logsumexp traffic or a separate D pass).  Self-attention: q, k, v share
 * `offsets` (T rows).  The tokens of each sample are cut into blocks of 64
 * from the sample's first token (the last block may be shorter); row i sees
 * the keys of its own block (and only j <= i when causal).  Scores, bias
 * (the relative-position table or a dense jagged bias, of which only the
 * pairs inside a block are read), activations and layouts are those of
 * gdpa_fwd; a dense bias's offsets are checked on the device like the
 * offsets (GDPA_ERR_BAD_OFFSETS).  The forward writes `out`
 * only: no logsumexp (the backward recomputes each row's exact softmax from
 * its block).  workspace: gdpa_block_workspace_size() bytes of device memory
 * (the tile list), shared by gdpa_block_fwd and gdpa_block_bwd.  Malformed
 * offsets raise GDPA_ERR_BAD_OFFSETS on the device. */
size_t gdpa_block_workspace_size(int B, int H, int d, int64_t T);
gdpa_status gdpa_block_fwd(const void* q, const int32_t* offsets, const void* k, const void* v,
                           int B, int H, int d, int64_t T, const gdpa_bias* bias, int act,
                           int causal, float scale, void* out, void* workspace, size_t ws_bytes,
                           void* stream);

/* Backward of gdpa_block_fwd: writes dq, dk, dv [T][H][d] (bf16) from q, k,
 * v and dout alone.  Each 64-token block is one independent problem, so the
 * kernel recomputes the block's scores and exact softmax, forms D = sum_j P
 * dP inside the tile and writes every gradient row once (no atomics, no
 * logsumexp or forward output needed).  Rows of a sample never see another
 * sample's tokens.
 * rope_base > 0 fuses the rotary-embedding backward into the epilogue (the
 * same paragraph: "fusing RoPE backward into the attention epilogue"): q and
 * k are taken to be rotary-embedded (rotate-half form: channels c and c + d/2
 * rotated by pos * rope_base^(-2c/d), pos the token's position in its
 * sample), and dq, dk are returned with respect to the un-rotated q and k
 * (the transposed rotation applied to the fp32 gradients).  rope_base = 0:
 * no rotary embedding; negative or non-finite: GDPA_ERR_INVALID_ARG.
 * Other arguments, workspace and errors as gdpa_block_fwd. */
gdpa_status gdpa_block_bwd(const void* q, const int32_t* offsets, const void* k, const void* v,
                           int B, int H, int d, int64_t T, const gdpa_bias* bias, int act,
                           int causal, float scale, float rope_base, const void* dout, void* dq,
                           void* dk, void* dv, void* workspace, size_t ws_bytes, void* stream);

/* gdpa_block_bwd with the gradient of the bias (fp32 device memory, ADDED to,
 * as in gdpa_bwd_window):
 *   GDPA_BIAS_RELPOS: dbias [H][2*max_rel-1] receives, at entry
 *   clamp(i - j + max_rel - 1), the sum of dS_ij over the pairs each row sees
 *   in its block.  Each tile's sums are gathered in shared memory and added
 *   to the table with global atomics, so their order, and the sums' last
 *   bits, vary between runs.
 *   GDPA_BIAS_DENSE: dbias in the dense bias's own layout; the entry of each
 *   pair a row sees in its block receives that pair's dS_ij (the bf16 value
 *   the softmax products use, the fp32 one for the other activations); the
 *   entries of other pairs are left as they are.
 * dbias = NULL is gdpa_block_bwd; a dbias without a bias, or not 4-byte
 * aligned: GDPA_ERR_INVALID_ARG.  Every other argument, output and error is
 * that of gdpa_block_bwd. */
gdpa_status gdpa_block_bwd_dbias(const void* q, const int32_t* offsets, const void* k,
                                 const void* v, int B, int H, int d, int64_t T,
                                 const gdpa_bias* bias, int act, int causal, float scale,
                                 float rope_base, const void* dout, void* dq, void* dk, void* dv,
                                 float* dbias, void* workspace, size_t ws_bytes, void* stream);

/* gdpa_bwd_window with the rotary-embedding backward fused into the epilogue
 * ("GEM Training ..." SWA / block paragraph: RoPE backward in the attention
 * epilogue, gradients kept in fp32).  q and k are taken as already
 * rotary-embedded in the rotate-half form (channels c and c + d/2 rotated by
 * pos * rope_base^(-2c/d), pos = the token's position in its sample, queries
 * and keys each by their own offsets); dq and dk are returned for the
 * un-rotated q and k: the transposed rotation is applied to the fp32
 * gradients before rounding (dK in the kernel's epilogue, dQ in the
 * accumulator's conversion).  rope_base = 0: no rotary embedding (this is
 * gdpa_bwd_window); negative, infinite or NaN: GDPA_ERR_INVALID_ARG.  Every
 * other argument, output and error (biases and their gradients included) is
 * that of gdpa_bwd_window; not available for the MXFP8 backward. */
gdpa_status gdpa_bwd_rope(const void* q, const int32_t* q_offsets, const void* k, const void* v,
                          const int32_t* kv_offsets, int B, int H, int d, int64_t Tq,
                          int64_t Tkv, const gdpa_bias* bias, int act, int causal, int window,
                          float scale, float rope_base, const void* out, const float* lse,
                          const void* dout, void* dq, void* dk, void* dv, float* dbias,
                          void* workspace, size_t ws_bytes, void* stream);

/* MXFP8 block quantisation (OCP Microscaling Formats v1.0; "GEM Training ..."
 * low-precision paragraph: attention with MXFP8 block-scaled MMA).  Elements
 * become E4M3 codes (round to nearest even, saturated at +-448); each block of
 * 32 elements shares an E8M0 scale 2^(floor(log2 amax) - 8), biased by 127.
 * With GDPA_MX_NOSAT or-ed into `mode` the scale is instead the smallest power
 * of two X with amax / X <= 448, so no element saturates (the OCP rule clips a
 * block maximum whose mantissa is above 1.75 by up to 12.5%); this is the
 * recipe the MXFP8 forward is specified and tested with.
 *   GDPA_MX_ALONG_CHANNELS: blocks of 32 consecutive channels of one (token,
 *     head) row (for Q and K, whose product contracts over d).
 *     codes [T][H][d] u8, scales [T][H][d/32] u8.
 *   GDPA_MX_ALONG_TOKENS: blocks of 32 consecutive tokens of one sample, per
 *     (head, channel); the first block starts at the sample's first token and
 *     the last may be partial (for V, whose product contracts over keys).
 *     codes [T][H][d] u8; scales [B + T/32 + 1][H][d] u8 where block r of
 *     sample b is scale row b + floor(offsets[b]/32) + r (rows that belong to
 *     no block are not written).  Tokens outside every sample (before
 *     offsets[0] or from offsets[B] on) get code 0.  offsets are needed only
 *     in this mode.
 * x is [T][H][d] bf16, 16-byte aligned; all buffers are device memory.  Other
 * mode bits return GDPA_ERR_INVALID_ARG (gdpa_mxfp8_scale_bytes returns 0). */
enum { GDPA_MX_ALONG_CHANNELS = 0, GDPA_MX_ALONG_TOKENS = 1, GDPA_MX_NOSAT = 2 };
size_t gdpa_mxfp8_scale_bytes(int B, int H, int d, int64_t T, int mode);
gdpa_status gdpa_quantize_mxfp8(const void* x, const int32_t* offsets, int B, int H, int d,
                                int64_t T, int mode, void* codes, void* scales, void* stream);

/* Forward pass on MXFP8 operands: both products run on the block-scaled
 * tensor cores (E4M3 x E4M3 with E8M0 scales per 32 elements of the
 * contraction, fp32 accumulation), and P is quantised to E4M3 per 32 keys in
 * registers.  ("GEM Training ..." low-precision paragraph: attention with
 * end-to-end MXFP8 block-scaled MMA.)
 *   q_codes/q_scales, k_codes/k_scales: gdpa_quantize_mxfp8 output along
 *     channels ([T][H][128] u8, [T][H][4] u8).
 *   v_codes/v_scales: output along tokens ([Tkv][H][128] u8,
 *     [B + Tkv/32 + 1][H][128] u8), quantised with the same kv_offsets.
 * d must be 128 and act GDPA_ACT_SOFTMAX (an unnormalised GDPA sum of
 * thousands of E4M3-rounded terms would not keep the output's precision);
 * other values return GDPA_ERR_UNSUPPORTED.  The bias (a relative-position
 * table or a dense jagged bias) is added in fp32 to the fp32 scores.  Every
 * other argument, the outputs and the workspace (gdpa_fwd_workspace_size)
 * are those of gdpa_fwd. */
gdpa_status gdpa_fwd_mxfp8(const void* q_codes, const void* q_scales, const int32_t* q_offsets,
                           const void* k_codes, const void* k_scales, const void* v_codes,
                           const void* v_scales, const int32_t* kv_offsets, int B, int H, int d,
                           int64_t Tq, int64_t Tkv, const gdpa_bias* bias, int act, int causal,
                           float scale, void* out, float* lse, void* workspace, size_t ws_bytes,
                           void* stream);

/* gdpa_fwd_mxfp8 with a sliding window (semantics of gdpa_fwd_window). */
gdpa_status gdpa_fwd_mxfp8_window(const void* q_codes, const void* q_scales,
                                  const int32_t* q_offsets, const void* k_codes,
                                  const void* k_scales, const void* v_codes, const void* v_scales,
                                  const int32_t* kv_offsets, int B, int H, int d, int64_t Tq,
                                  int64_t Tkv, const gdpa_bias* bias, int act, int causal,
                                  int window, float scale, void* out, float* lse,
                                  void* workspace, size_t ws_bytes, void* stream);

/* Backward pass with every product on MXFP8 operands ("GEM Training ..."
 * low-precision paragraph: end-to-end MXFP8 block-scaled MMA in the forward
 * and the backward pass).  Takes the bf16 tensors of gdpa_bwd and quantises
 * them into the workspace first (gdpa_quantize_mxfp8's formats): Q, K and dO
 * along channels (for S = Q K^T and dP = dO V^T) and along tokens (for
 * dK = dS^T Q, dQ = dS K and dV = P^T dO), V along channels.  P and dS are
 * made in the kernel from fp32 S and dP and rounded to E4M3 in blocks of 32
 * keys x 32 queries (aligned to each sample's first key and first query)
 * sharing one E8M0 scale, the smallest power of two X with amax / X <= 448.
 * D = rowsum(dO * O) comes from the bf16 out and dout.  Products accumulate
 * in fp32; dq is written as bf16(scale * sum), dk and dv as bf16.
 * d must be 128 and act GDPA_ACT_SOFTMAX (else GDPA_ERR_UNSUPPORTED).  Every
 * other argument, output and error is that of gdpa_bwd_window; the workspace
 * is gdpa_bwd_mxfp8_workspace_size bytes (16-byte aligned). */
size_t gdpa_bwd_mxfp8_workspace_size(int B, int H, int d, int64_t Tq, int64_t Tkv);
gdpa_status gdpa_bwd_mxfp8(const void* q, const int32_t* q_offsets, const void* k, const void* v,
                           const int32_t* kv_offsets, int B, int H, int d, int64_t Tq,
                           int64_t Tkv, const gdpa_bias* bias, int act, int causal, float scale,
                           const void* out, const float* lse, const void* dout, void* dq, void* dk,
                           void* dv, void* workspace, size_t ws_bytes, void* stream);
/* gdpa_bwd_mxfp8 with a sliding window (semantics of gdpa_bwd_window). */
gdpa_status gdpa_bwd_mxfp8_window(const void* q, const int32_t* q_offsets, const void* k,
                                  const void* v, const int32_t* kv_offsets, int B, int H, int d,
                                  int64_t Tq, int64_t Tkv, const gdpa_bias* bias, int act,
                                  int causal, int window, float scale, const void* out,
                                  const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                  void* workspace, size_t ws_bytes, void* stream);
/* gdpa_bwd_mxfp8_window with the rotary-embedding backward (rope_base > 0:
 * dq, dk returned for the un-rotated q, k, as in gdpa_bwd_rope: dK rotated in
 * the kernel's epilogue, dQ in the accumulator's conversion; 0: none;
 * negative, infinite or NaN: GDPA_ERR_INVALID_ARG) and the gradient of the
 * bias (dbias, fp32, added to, from the fp32 dS before its E4M3 rounding: a
 * relative-position table's [H][2*max_rel-1] as in gdpa_bwd_window, or a
 * dense bias's own layout, each unmasked pair's entry receiving its dS;
 * NULL: not computed; without a bias or not 4-byte aligned:
 * GDPA_ERR_INVALID_ARG).  Every other argument, output and error is that of
 * gdpa_bwd_mxfp8_window. */
gdpa_status gdpa_bwd_mxfp8_rope(const void* q, const int32_t* q_offsets, const void* k,
                                const void* v, const int32_t* kv_offsets, int B, int H, int d,
                                int64_t Tq, int64_t Tkv, const gdpa_bias* bias, int act, int causal,
                                int window, float scale, float rope_base, const void* out,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                float* dbias, void* workspace, size_t ws_bytes, void* stream);

/* Reads the device status word set by earlier calls on this device,
 * synchronising `stream` first, then clears it.  Returns GDPA_OK,
 * GDPA_ERR_TIMEOUT, GDPA_ERR_BAD_OFFSETS or GDPA_ERR_CUDA. */
gdpa_status gdpa_get_device_status(void* stream);

/* Failure-detection self-test: launches one small kernel whose pipeline wait
 * (an mbarrier nothing arrives at) cannot complete, waited on with the
 * library's bounded wait for limit_us microseconds (1 .. 1e6).  The wait
 * gives up, the kernel sets GDPA_ERR_TIMEOUT in the device status word and
 * returns: the next gdpa_get_device_status() reports it, and the context
 * stays usable.  No fault is raised. */
gdpa_status gdpa_selftest_timeout(int limit_us, void* stream);

/* Static, human-readable name of a status code. */
const char* gdpa_status_string(int status);

/* Number of kernels the most recent gdpa_* call on this host thread
 * launched (for accounting in benchmarks). */
int gdpa_last_launch_count(void);

/* Kernel timing for benchmarks.  While enabled on a host thread, every
 * gdpa_fwd / gdpa_bwd call on that thread records a pair of CUDA events on
 * its stream around its main attention kernel (at most 4096 pairs; later
 * calls are not recorded).  gdpa_timing_enable(1) starts a fresh record,
 * gdpa_timing_enable(0) stops recording.  gdpa_timing_collect() waits for
 * the recorded events, writes up to `max` durations in milliseconds to
 * ms[] and the matching kinds (0 = forward, 1 = backward) to kind[], and
 * returns how many it wrote (or -1 on a CUDA error).  The events are
 * created on first use and kept for the life of the thread. */
gdpa_status gdpa_timing_enable(int enable);
int gdpa_timing_collect(float* ms, int* kind, int max);

/* Forward pass that allocates nothing and needs no workspace argument.  The
 * paper has no counterpart: this entry point exists for callers that cannot
 * allocate device memory -- for example a plugin running inside a framework
 * that has already reserved the GPU's memory for its own pool, or a service
 * whose memory plan forbids allocations after start-up -- and so cannot pass
 * the workspace gdpa_fwd asks for.
 *
 * Arguments and results are those of gdpa_fwd without workspace/ws_bytes.
 * The scratch comes from one 1 MiB array compiled into the library (every
 * GPU that loads the library holds it until the process exits).  Problems
 * whose gdpa_fwd_workspace_size() exceeds 1 MiB (about H * (Tq/256 + 2B) >
 * 131,000 work-list entries) are refused with GDPA_ERR_WORKSPACE before
 * anything is launched.  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress); make that first call before any stream
 * capture.  The address is kept for the life of the process: after a
 * cudaDeviceReset() on the device it is stale, so do not call this entry
 * point (or any other) on that device again.  All calls share the array:
 * calls whose kernels may overlap on the GPU (different streams or host
 * threads) race and give undefined results, so serialise them. */
gdpa_status gdpa_fwd_noalloc(const void* q, const int32_t* q_offsets, const void* k,
                             const void* v, const int32_t* kv_offsets, int B, int H, int d,
                             int64_t Tq, int64_t Tkv, const gdpa_bias* bias, int act, int causal,
                             float scale, void* out, float* lse, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDPA_H_ */
