/*
 * llama_block.h — C ABI of the GB300 (sm_103a) Llama decoder-block forward library.
 *
 * The block computed here (sources: "Llama Architecture: RMSNorm, SwiGLU, RoPE, GQA,
 * and PyTorch Implementation", Mathematical Foundations 1-4 and Production PyTorch
 * Implementation Steps 1-2; "LLaMA Architecture > Model Architecture", The Transformer
 * Block; "LLaMA-3 8B 现代 LLM 架构、计算规模与能耗", sections 四, 五, 九, 十):
 *
 *     u = RMSNorm(x; g_attn)                 x * rsqrt(mean(x^2) + eps) * g
 *     q = RoPE(u W_Q^T), k = RoPE(u W_K^T), v = u W_V^T
 *     o = softmax(q k^T / sqrt(head_dim) + causal mask) v,  query head h reads KV head h / (n_q/n_kv)
 *     h = x + o W_O^T
 *     y = h + W_down (SiLU(W_gate RMSNorm(h; g_ffn)) * W_up RMSNorm(h; g_ffn))
 *
 * Conventions shared by every call
 *   - All pointers are DEVICE pointers unless stated otherwise; the caller owns and allocates
 *     all memory (tensors, caches, workspace).  The library never allocates device memory.
 *   - All calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *     Argument and shape errors are returned synchronously and nothing is launched.  Errors
 *     found on the device (a wait that timed out) are latched in a device status word read by
 *     llama_get_device_status().
 *   - dtype: LLAMA_F32 or LLAMA_BF16 for activations, weights and gains alike.  Arithmetic
 *     accumulates in fp32 for both.
 *   - Weights are row-major [out, in] (the nn.Linear layout), so a projection is x W^T.
 *   - Activations are token-major: x [B, S, d_model] = [B*S rows, d_model];
 *     q [B, S, n_q, head_dim]; k, v [B, S, n_kv, head_dim]; caches [B, capacity, n_kv, head_dim].
 *   - Positions are 0-based absolute positions; token s of a call sits at pos0 + s, and a query
 *     at position m sees keys 0..m.  RoPE turns the interleaved pair (x_2k, x_2k+1) by
 *     m * theta_base^(-2k/head_dim).  Positions must be < 2^24; the angle is reduced exactly for
 *     positions below 2^19.
 *   - Device pointers must be 16-byte aligned; row widths must keep every row 16-byte aligned.
 *   - The bf16 path uses tcgen05 tensor cores and requires head_dim in {64, 128}, d_model,
 *     n_q*head_dim, n_kv*head_dim and d_ff multiples of 128, and 128 % (n_q/n_kv) == 0.
 *     Other bf16 shapes, and every f32 shape, run on CUDA-core kernels.
 *   - Accuracy, as tested against an exact fp64 evaluation of the same stored inputs: f32 calls
 *     to max|err| <= 1e-4 max|ref|; bf16 calls to max|err| <= 2e-2 RMS(ref row) on every row, for
 *     row widths (d_model) up to 4096.  Wider bf16 rows are not covered by that bar: the bf16
 *     storage of the intermediate activations alone reaches 2.2-3.0e-2 on the worst row at
 *     d_model 4352-5120 (the same inputs, exact arithmetic, rounded to bf16 where this library
 *     stores bf16).
 */
#ifndef LLAMA_BLOCK_H
#define LLAMA_BLOCK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The shape record every call takes.  Fields a call does not use must still be >= 0. */
typedef struct llama_dims {
  int64_t B;          /* batch (sequences) */
  int64_t S;          /* tokens per sequence in this call */
  int64_t d_model;    /* residual width */
  int64_t n_q;        /* query heads */
  int64_t n_kv;       /* key/value heads; n_q % n_kv == 0 */
  int64_t head_dim;   /* per-head width; even */
  int64_t d_ff;       /* SwiGLU hidden width */
  double theta_base;  /* RoPE base (1e4, 5e5, ...) */
  double eps;         /* RMSNorm epsilon, added inside the square root */
} llama_dims;

typedef enum llama_dtype { LLAMA_F32 = 0, LLAMA_BF16 = 1 } llama_dtype;

typedef enum llama_status {
  LLAMA_OK = 0,
  LLAMA_ERR_INVALID_ARG = 1,   /* null pointer, negative or inconsistent size */
  LLAMA_ERR_UNSUPPORTED = 2,   /* shape or dtype this library does not handle */
  LLAMA_ERR_ALIGNMENT = 3,     /* pointer not 16-byte aligned */
  LLAMA_ERR_WORKSPACE = 4,     /* workspace missing or smaller than llama_workspace_bytes() */
  LLAMA_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
  LLAMA_ERR_TIMEOUT = 6,       /* device side: a bounded wait ran out (kernel gave up cleanly) */
  LLAMA_ERR_BOUNDS = 7         /* device side, bounds-checking builds only: a kernel found a store
                                  or TMA box start outside its tensor, skipped it and returned */
} llama_status;

/* One block's parameters (device pointers, dtype of the call):
 *   attn_norm_g, ffn_norm_g [d_model]
 *   wq [n_q*hd, d_model], wk, wv [n_kv*hd, d_model], wo [d_model, n_q*hd]
 *   w_gate, w_up [d_ff, d_model], w_down [d_model, d_ff]                                     */
typedef struct llama_block_weights {
  const void* attn_norm_g;
  const void* wq;
  const void* wk;
  const void* wv;
  const void* wo;
  const void* ffn_norm_g;
  const void* w_gate;
  const void* w_up;
  const void* w_down;
} llama_block_weights;

/* Operation ids for llama_workspace_bytes. */
typedef enum llama_op {
  LLAMA_OP_RMSNORM = 0,
  LLAMA_OP_ROPE = 1,
  LLAMA_OP_GQA_ATTENTION = 2,
  LLAMA_OP_SWIGLU_FFN = 3,
  LLAMA_OP_BLOCK_FORWARD = 4,
  LLAMA_OP_STACK_DECODE_STEP = 5
} llama_op;

/* RMSNorm over the feature axis ("Llama Architecture ...", Mathematical Foundations 1, with eps
 * inside the root as in its Step 1 code; the RMSNorm study note, "How it works").
 * x, y: [B*S, d_model]; g: [d_model].  y = x * rsqrt(mean(x^2) + eps) * g, fp32 accumulation,
 * one rounding to dtype.  y may alias x.  Uses B, S, d_model, eps.                          */
int llama_rmsnorm(const llama_dims* dims, int dtype, const void* x, const void* g, void* y,
                  void* stream);

/* RoPE in place ("Llama Architecture ...", Mathematical Foundations 3; "LLaMA-3 8B ...",
 * section 四.3).  q: [B, S, n_q, hd], k: [B, S, n_kv, hd]; either may be NULL.  Token s of
 * every sequence is at position pos0 + s.  Uses B, S, n_q, n_kv, head_dim, theta_base.       */
int llama_rope(const llama_dims* dims, int dtype, void* q, void* k, int64_t pos0, void* stream);

/* Causal grouped-query attention on post-RoPE inputs ("Llama Architecture ...", Mathematical
 * Foundations 4; "LLaMA-3 8B ...", section 四.4 and its 8Q/2KV example).
 *   q: [B, S, n_q, hd], queries at positions pos0 .. pos0+S-1
 *   k, v: [B, kv_capacity, n_kv, hd], holding keys/values for positions 0 .. pos0+S-1
 *   o: [B, S, n_q, hd]
 * Query head h reads KV head h / (n_q/n_kv); a query at position m sees keys 0..m; scale
 * 1/sqrt(hd).  Requires pos0 + S <= kv_capacity.  ws: scratch of llama_workspace_bytes(
 * LLAMA_OP_GQA_ATTENTION, ...) bytes (may be 0; then ws may be NULL).                       */
int llama_gqa_attention(const llama_dims* dims, int dtype, const void* q, const void* k,
                        const void* v, int64_t kv_capacity, int64_t pos0, void* o, void* ws,
                        size_t ws_bytes, void* stream);

/* SwiGLU feed-forward ("Llama Architecture ...", Mathematical Foundations 2; "LLaMA-3 8B ...",
 * section 五).  x, y: [B*S, d_model]; y = W_down(SiLU(W_gate x) * W_up x), no residual.
 * ws holds the [B*S, d_ff] gated product.  y must not alias x.                              */
int llama_swiglu_ffn(const llama_dims* dims, int dtype, const void* x, const void* w_gate,
                     const void* w_up, const void* w_down, void* y, void* ws, size_t ws_bytes,
                     void* stream);

/* Residual-stream flags, OR-ed into the dtype argument of llama_block_forward only.  The
 * residual stream is what one block hands to the next (x in, y out); a stack of prefill blocks
 * keeps it in fp32 (as llama_stack_decode_step does) by giving its first block LLAMA_BF16 |
 * LLAMA_Y_F32 and every later block LLAMA_BF16 | LLAMA_X_F32 | LLAMA_Y_F32.  The GEMM and
 * attention operands, the weights and the KV cache keep the dtype; only x and y change.  With
 * LLAMA_Y_F32 the call computes the same values and skips the final bf16 rounding of y, which
 * alone is up to 2^-8 |y| (1.3e-2 of a row's RMS on the worst rows of the 4096-wide blocks).
 * Both flags are ignored for LLAMA_F32, where x and y are fp32 already.                      */
enum { LLAMA_X_F32 = 0x100, LLAMA_Y_F32 = 0x200 };

/* One decoder block over B sequences of S new tokens at positions pos0 .. pos0+S-1
 * ("Llama Architecture ...", Step 2 LlamaTransformerBlock; "LLaMA Architecture > Model
 * Architecture", The Transformer Block).  x, y: [B*S, d_model]; y must not alias x.
 * dtype: LLAMA_F32 or LLAMA_BF16, optionally OR-ed with LLAMA_X_F32 and LLAMA_Y_F32.
 * k_cache, v_cache: [B, cache_capacity, n_kv, hd]; on entry they hold positions 0..pos0-1,
 * and the call writes the rotated keys and the values of the new tokens at pos0..pos0+S-1.
 * Both NULL: pos0 must be 0 and the block's K/V live in the workspace.                       */
int llama_block_forward(const llama_dims* dims, int dtype, const llama_block_weights* w,
                        const void* x, void* y, int64_t pos0, void* k_cache, void* v_cache,
                        int64_t cache_capacity, void* ws, size_t ws_bytes, void* stream);

/* One decode step of an n_layers stack, one new token per sequence, then the final RMSNorm
 * and the untied LM head ("LLaMA-3 8B ...", sections 二, 九 and 十).  dims->S must be 1.
 *   layers: HOST array of n_layers weight records (device pointers inside)
 *   final_g [d_model]; w_lm [vocab, d_model]; x_emb [B, d_model] (the new tokens' embedding rows)
 *   k_cache, v_cache: [n_layers, B, cache_capacity, n_kv, hd]; positions 0..t_cache-1 are read,
 *   position t_cache of every layer is written (so t_cache < cache_capacity)
 *   logits: [B, vocab] float32, whatever dtype is.
 * The residual stream is kept in fp32 across layers (in ws).                                 */
int llama_stack_decode_step(const llama_dims* dims, int dtype, int n_layers,
                            const llama_block_weights* layers, const void* final_g,
                            const void* w_lm, int64_t vocab, const void* x_emb, void* k_cache,
                            void* v_cache, int64_t cache_capacity, int64_t t_cache, float* logits,
                            void* ws, size_t ws_bytes, void* stream);

/* Allocation-free one-token GQA attention (no counterpart in the method itself: this is a library entry
 * point for callers that cannot allocate device memory at the call site, e.g. code running under
 * an allocator that owns all of device memory, or loops where cudaMalloc/cudaFree would
 * synchronise the device).  Same arguments and result as llama_gqa_attention with dims->S == 1,
 * minus the workspace: its split-K partials live in a 12 MiB device array inside the library
 * (created when the library is loaded, resident on every device that loads it until exit).
 *   - bf16 only, head_dim 128, n_q / n_kv in {1, 2, 4, 8, 16}.
 *   - Size rule: the partials take B*n_kv + 256 slots of r = n_q/n_kv rows of 130 floats, stored as
 *     two arrays each rounded up to 256 bytes: round256(slots*r*512) + round256(slots*r*8) bytes,
 *     about (B*n_kv + 256)*r*520.  That does not depend on the number of keys, and the keys are
 *     never re-chunked to fit.  When it exceeds 12 MiB (12582912 bytes) the call returns
 *     LLAMA_ERR_WORKSPACE and launches nothing.  The Llama-3-8B decode shape (B 64, 32 query and
 *     8 KV heads) needs 1.6 MB; with 32 query and 8 KV heads the largest batch is B = 724.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress);
 *     make that first call before any stream capture.
 *   - Every call uses the same array: calls that overlap on the GPU (other streams, other host
 *     threads) race on it.  Each call overwrites every partial it reads, so nothing needs
 *     clearing between calls.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.                              */
int llama_gqa_attention_decode_noalloc(const llama_dims* dims, int dtype, const void* q,
                                       const void* k, const void* v, int64_t kv_capacity,
                                       int64_t pos0, void* o, void* stream);

/* Workspace bytes the call `op` needs for these arguments (0 if none).  kv_capacity is the
 * cache capacity for attention/decode and is ignored otherwise.                              */
size_t llama_workspace_bytes(int op, const llama_dims* dims, int dtype, int n_layers,
                             int64_t vocab, int64_t kv_capacity);

/* 8-bit KV cache.  The pages size the cache in bf16 and give no 8-bit format; this library's
 * format is OCP E4M3 ("e4m3fn") codes, one byte per element, with one fp32 scale per
 * (layer, K or V, KV head): the stored value is code * scale.  Encoding divides in fp32, rounds to
 * the nearest E4M3 value (ties to even) and saturates at +-448.  The cache layout is the bf16
 * one with 1-byte elements: [n_layers, B, capacity, n_kv, head_dim].                          */

/* codes[t, g, i] = E4M3(x[t, g, i] / scale[g]) for n_tokens rows of n_kv heads x head_dim bf16
 * values (x [n_tokens, n_kv, head_dim] bf16 and codes of the same shape, device; scale [n_kv]
 * fp32, device).  Errors: LLAMA_ERR_INVALID_ARG for n_tokens < 0, n_kv < 1, head_dim not a
 * positive multiple of 8, or NULL pointers with n_tokens > 0; LLAMA_ERR_ALIGNMENT unless x is
 * 16-byte, codes 8-byte and scale 4-byte aligned.                                              */
int llama_kv_quantize(const void* x, int64_t n_tokens, int64_t n_kv, int64_t head_dim,
                      const float* scale, void* codes, void* stream);

/* llama_gqa_attention for one new token per sequence (S = 1) over an 8-bit cache: k and v are
 * codes [B, kv_capacity, n_kv, head_dim] holding positions 0..pos0 (the new token's K/V already
 * written), k_scale / v_scale [n_kv] fp32 (device); q and o bf16 [B, n_q, head_dim].
 * Needs head_dim 128, n_q / n_kv in {1, 2, 4, 8, 16} (else LLAMA_ERR_UNSUPPORTED) and the
 * workspace llama_workspace_bytes(LLAMA_OP_GQA_ATTENTION, ...) gives for this shape.
 * Numerics: the products run on 8-bit tensor-core MMAs, so q and the softmax weights enter as
 * sums of two E4M3 values (about 8 significant bits, as in bf16); the result is attention over
 * the decoded cache (code * scale) to within the bf16 tolerance, accumulated in fp32.          */
int llama_gqa_attention_decode_kv8(const llama_dims* dims, const void* q, const void* k,
                                   const void* v, const float* k_scale, const float* v_scale,
                                   int64_t kv_capacity, int64_t pos0, void* o, void* ws,
                                   size_t ws_bytes, void* stream);

/* llama_stack_decode_step with bf16 weights and an 8-bit cache: k_cache / v_cache hold codes
 * [n_layers, B, cache_capacity, n_kv, head_dim]; kv_scales [n_layers][2][n_kv] fp32 (device),
 * index 0 for K and 1 for V.  The new token's K/V are encoded into the cache at t_cache and
 * attention reads the stored values.  Same workspace as the bf16 call; supported for the shapes
 * of its tensor-core path (bf16, B <= 128, head_dim 128, d_model, n_q*head_dim, n_kv*head_dim
 * and d_ff multiples of 128, n_q / n_kv in {1, 2, 4, 8, 16}), else LLAMA_ERR_UNSUPPORTED.     */
int llama_stack_decode_step_kv8(const llama_dims* dims, int n_layers,
                                const llama_block_weights* layers, const void* final_g,
                                const void* w_lm, int64_t vocab, const void* x_emb,
                                void* k_cache, void* v_cache, const float* kv_scales,
                                int64_t cache_capacity, int64_t t_cache, float* logits, void* ws,
                                size_t ws_bytes, void* stream);

/* Paged KV cache with per-sequence lengths (long contexts: the pages size the 8B cache at 4 GB for
 * 32K positions and 15.6 GB for 128K, "LLaMA-3 8B ...", section 七; "Llama Architecture ...",
 * Mathematical Foundations 4).  K and V of layer l live in a pool of 128-position pages,
 * [n_layers, n_pages, 128, n_kv, head_dim] bf16; sequence b's positions 128j .. 128j+127 are in
 * page block_table[b * max_pages + j].  seq_pos[b] is the position of b's new token, i.e. the
 * number of positions already cached (b attends to positions 0 .. seq_pos[b]); max_pos is an
 * upper bound of seq_pos over the batch (host value: it sizes the work split and the workspace,
 * llama_workspace_bytes(..., kv_capacity = max_pos + 1)).  block_table and seq_pos are int32
 * device arrays; every page that a sequence uses up to its new position must be listed.  Rows of
 * a sequence's last page past its new position are never used (their contents do not matter).
 * The page that receives a sequence's new K/V belongs to that sequence alone: the step writes it
 * while other sequences' attention may already be reading their earlier pages.                  */

/* llama_stack_decode_step over a paged cache: writes each sequence's new K/V into its page at
 * seq_pos[b] and runs RoPE at that position.  Same shapes as the tensor-core dense call (else
 * LLAMA_ERR_UNSUPPORTED).  LLAMA_ERR_INVALID_ARG for n_pages or max_pages < 1, max_pos < 0 or
 * max_pos + 1 > 128 * max_pages, or NULL pointers.                                              */
int llama_stack_decode_step_paged(const llama_dims* dims, int n_layers,
                                  const llama_block_weights* layers, const void* final_g,
                                  const void* w_lm, int64_t vocab, const void* x_emb,
                                  void* k_pool, void* v_pool, int64_t n_pages,
                                  const int32_t* block_table, int64_t max_pages,
                                  const int32_t* seq_pos, int64_t max_pos, float* logits, void* ws,
                                  size_t ws_bytes, void* stream);

/* One-token attention over a paged cache (S = 1, head_dim 128, n_q / n_kv in {1, 2, 4, 8, 16}):
 * q and o bf16 [B, n_q, head_dim]; k_pool / v_pool one layer's pools [n_pages, 128, n_kv,
 * head_dim] holding every sequence's positions 0 .. seq_pos[b].  Workspace:
 * llama_workspace_bytes(LLAMA_OP_GQA_ATTENTION, dims with S = 1, ..., kv_capacity = max_pos + 1). */
int llama_gqa_attention_decode_paged(const llama_dims* dims, const void* q, const void* k_pool,
                                     const void* v_pool, int64_t n_pages,
                                     const int32_t* block_table, int64_t max_pages,
                                     const int32_t* seq_pos, int64_t max_pos, void* o, void* ws,
                                     size_t ws_bytes, void* stream);

/* Next-token choice from the LM head's logits ("LLaMA-3 8B 现代 LLM 架构、计算规模与能耗", section 十:
 * softmax over the vocabulary, then argmax, or a draw shaped by temperature, top-k and top-p).
 *   logits  [B, ld] fp32 (device), row b's first `vocab` entries used; finite values or -inf,
 *           at least one finite per row
 *   temperature  T > 0 draws from softmax(z / T); T <= 0 returns the argmax
 *   top_k   keep the k most probable tokens (k <= 0 or k >= vocab: all; k = 1: argmax)
 *   top_p   then keep the shortest run of most probable tokens whose share of the top-k mass
 *           reaches p (p >= 1: all; p <= 0: the argmax)
 *   u       [B] fp32 (device): one uniform draw in [0, 1) per row, supplied by the caller (values
 *           outside are clamped into it)
 *   tokens  [B] int32 (device): the chosen token ids
 * Ranking is by logit, larger first, ties by the lower id.  The draw walks the kept tokens in
 * increasing id and returns the first whose cumulative probability exceeds u.  Probabilities are
 * exp((z - z_max) / T) in fp32 summed exactly in 2^-40 fixed point, so the result does not depend
 * on thread timing.  Errors: LLAMA_ERR_INVALID_ARG for B < 0, vocab < 1 or > 2^30, ld < vocab,
 * NaN temperature or top_p, or a NULL pointer with B > 0; LLAMA_ERR_ALIGNMENT for pointers not
 * 4-byte aligned.  B = 0 launches nothing.                                                      */
int llama_sample(const float* logits, int64_t B, int64_t vocab, int64_t ld, float temperature,
                 int64_t top_k, float top_p, const float* u, int32_t* tokens, void* stream);

/* Embedding lookup ("LLaMA-3 8B ...", section 三): x[i] = table[tokens[i]] for i < n.
 *   table  [vocab, d_model] of `dtype` (device), row-major
 *   tokens [n] int32 (device)
 *   x      [n, d_model] of `dtype` (device)
 * A token id outside [0, vocab) gives a zero row and latches LLAMA_ERR_INVALID_ARG in the device
 * status word (read with llama_get_device_status).  Errors returned synchronously:
 * LLAMA_ERR_INVALID_ARG for vocab < 1, d_model < 1, n < 0 or NULL pointers with n > 0.        */
int llama_embed(int dtype, const void* table, int64_t vocab, int64_t d_model, const int32_t* tokens,
                int64_t n, void* x, void* stream);

/* Synchronises `stream`, then reads and clears the device status word of the current device.
 * *out receives LLAMA_OK, LLAMA_ERR_TIMEOUT (a kernel's bounded wait ran out and it exited),
 * LLAMA_ERR_BOUNDS (bounds-checking builds: a kernel met an index outside its tensor) or
 * LLAMA_ERR_INVALID_ARG (llama_embed met a token id outside the table), in that order of
 * precedence when several were latched.
 * Returns LLAMA_OK, or LLAMA_ERR_CUDA if the synchronisation or the copy failed.             */
int llama_get_device_status(int* out, void* stream);

/* Build information: bit LLAMA_BUILD_BOUNDS_CHECKS is set when the library was compiled with
 * -DLLAMA_DEBUG.  In that build every kernel checks each global store's index range and each
 * TMA box (or tile) start against the extent of its tensor before issuing it.  A failed check
 * latches LLAMA_ERR_BOUNDS (read with llama_get_device_status) and skips the access; a TMA
 * producer that skips a load also raises its CTA's abort flag, so that the kernel's other roles
 * leave through their bounded waits.  No trap and no assert: the context stays usable.  Release
 * builds compile the checks away.  There is no counterpart on the source pages: it is a
 * debugging aid of this library, standing in for a memory checker.                           */
enum { LLAMA_BUILD_BOUNDS_CHECKS = 1 };
int llama_build_info(void);

/* Self-test of the bounds checks: one small kernel stores to element 40 of `scratch` (64 fp32
 * elements, device, 16-byte aligned) through the checked store path, declaring the tensor's
 * extent as 32 elements.  A bounds-checking build skips the store and latches LLAMA_ERR_BOUNDS;
 * a release build performs it (inside the 64 elements).  Asynchronous on `stream`; returns
 * LLAMA_OK, LLAMA_ERR_INVALID_ARG for a NULL or unaligned scratch, or LLAMA_ERR_CUDA if the
 * launch failed.                                                                              */
int llama_selftest_bounds(float* scratch, void* stream);

/* Self-test of the device-side failure path: one small kernel whose threads wait, through the
 * same bounded mbarrier wait every pipelined kernel uses, on phases that nothing completes.  The
 * waits give up after their limit (2 s of %globaltimer), latch LLAMA_ERR_TIMEOUT in the device
 * status word and the kernel exits: llama_get_device_status then reports LLAMA_ERR_TIMEOUT and
 * the context stays usable.  Asynchronous on `stream`; returns LLAMA_OK, or LLAMA_ERR_CUDA if the
 * launch failed.                                                                              */
int llama_selftest_bounded_wait(void* stream);

/* Benchmark timing.  While enabled, every kernel the library launches is bracketed by two CUDA
 * events recorded on the launching stream (the events are created on first use and reused;
 * no device memory is allocated).  Do not enable it while a stream is being captured. */
int llama_profile_enable(int on);

/* Synchronises the device, then reports the launches recorded since profiling was enabled or
 * last read, aggregated by kernel role: names[i] (static strings), launches[i], total_ms[i] for
 * i < *n_kinds (at most max_kinds).  Clears the record.                                      */
int llama_profile_read(int max_kinds, const char** names, int* launches, double* total_ms, int* n_kinds);

/* Static, human-readable name of a status code. */
const char* llama_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* LLAMA_BLOCK_H */
