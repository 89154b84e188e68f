/*
 * fp64 CPU oracle of the Llama decoder block forward: C interface.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of the build entry point and the
 * oracle legs of the benchmark (its CPU baseline and its reference arm) load this library.  The
 * CUDA library never calls it and shares no code, header, table or helper with it; the two sides
 * share only the seeded input generator, which holds none of the block's arithmetic.
 *
 * Every function is the plain definition written out in double precision, in the order the pages
 * state it, with plain loops (no BLAS, no tiling, no online softmax).  Inputs are the stored
 * bf16 / fp32 values widened exactly to double by the caller.
 *
 * Sources (page title, section):
 *   [P1] "Llama Architecture: RMSNorm, SwiGLU, RoPE, GQA, and PyTorch Implementation":
 *        Mathematical Foundations 1 (RMSNorm), 2 (SwiGLU and d_ff), 3 (RoPE), 4 (GQA, KV cache
 *        scaling); Production PyTorch Implementation, Steps 1-2.
 *   [P2] "RMSNorm" study note (LLaMA): "How it works".
 *   [P3] "LLaMA-3 8B 现代 LLM 架构、计算规模与能耗": sections 三 (embedding lookup), 四 (one block;
 *        4.3-4.6 the 8Q/2KV toy), 五 (SwiGLU), 六 (parameter counts), 七 (KV cache), 九 (decode),
 *        十 (final norm, LM head, next-token rules).
 *   [P4] "LLaMA Architecture > Model Architecture": The Transformer Block; Key Architectural Choices;
 *        the configuration table.
 *
 * Readings where the pages are silent or disagree (each one is pinned by a CPU test):
 *   - eps sits inside the square root ([P2], [P4], [P1] Step 1 code; [P1] section 1's displayed
 *     equation puts it outside);
 *   - RoPE: theta_k = theta_base^(-2k/head_dim) on interleaved pairs (x_2k, x_2k+1), rotated by
 *     +m*theta_k as [P1] section 3's matrix;
 *   - positions are 0-based and absolute; a query at position m sees keys 0..m;
 *   - query head h reads KV head floor(h / r), r = n_q / n_kv ([P1] section 4, [P3] 4.4);
 *   - softmax scale 1/sqrt(head_dim);
 *   - weights are stored [out][in] (nn.Linear), so y = x W^T;
 *   - no intermediate rounding: exact double arithmetic on the stored inputs.
 *
 * Conventions: row-major arrays, sizes in elements, the caller owns every buffer.  Each function
 * returns 0, or -1 for an argument it cannot take (a negative size, a NULL buffer that is needed,
 * n_q not a multiple of n_kv, an odd head_dim).  Parallel loops use OpenMP threads; the thread
 * count is whatever OpenMP gives (OMP_NUM_THREADS), reported by oracle_threads().
 */
#ifndef LLAMA_ORACLE_H
#define LLAMA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The shared shape record: (B, S, d_model, n_q, n_kv, head_dim, d_ff, theta_base, eps). */
typedef struct {
  int64_t B, S, d_model, n_q, n_kv, head_dim, d_ff;
  double theta_base, eps;
} oracle_dims;

/* One block's parameters: [out][in] matrices and [d_model] gains, in double. */
typedef struct {
  const double *attn_norm_g; /* [d] */
  const double *wq;          /* [n_q*hd][d] */
  const double *wk;          /* [n_kv*hd][d] */
  const double *wv;          /* [n_kv*hd][d] */
  const double *wo;          /* [d][n_q*hd] */
  const double *ffn_norm_g;  /* [d] */
  const double *w_gate;      /* [d_ff][d] */
  const double *w_up;        /* [d_ff][d] */
  const double *w_down;      /* [d][d_ff] */
} oracle_block_weights;

/* What one layer of a decode stack needs besides its weights: the cached keys and values of
 * positions 0..t_cache-1 ([B][past_stride][n_kv][hd], past_stride >= t_cache positions per
 * sequence), and, for an 8-bit cache, one fp32 scale per KV head for K and for V (NULL: the
 * cache holds the values exactly). */
typedef struct {
  oracle_block_weights w;
  const double *k_past, *v_past;
  int64_t past_stride;
  const float *k_scale, *v_scale;
} oracle_layer;

/* Fills *out for layer l of a stack; returns 0, or non-zero to abort the stack. */
typedef int (*oracle_layer_fn)(void *ctx, int64_t l, oracle_layer *out);

int oracle_threads(void);

/* ---- RMSNorm [P1 section 1; P2 "How it works"; P4 Key Architectural Choices] ----
 * y[r][i] = x[r][i] / sqrt(mean_j x[r][j]^2 + eps) * g[i], for each of `rows` rows of width d. */
int oracle_rmsnorm(const double *x, int64_t rows, int64_t d, const double *g, double eps, double *y);

/* ---- SwiGLU [P1 section 2; P3 section 五] ----
 * silu(z) = z / (1 + e^-z), elementwise over n values. */
int oracle_silu(const double *z, int64_t n, double *out);
/* y = W_down (SiLU(W_gate x) * W_up x) for `rows` rows x [rows][d]; y [rows][d]. */
int oracle_swiglu_ffn(const double *x, int64_t rows, int64_t d, int64_t d_ff, const double *w_gate,
                      const double *w_up, const double *w_down, double *y);
/* d_ff as [P1] section 2 prints the rule, floor(8d / (3 m)) * m; and 8d/3 rounded up to a
 * multiple of m (the rule that reproduces [P4]'s configuration table). */
int64_t oracle_ffn_dim_floor(int64_t d, int64_t multiple_of);
int64_t oracle_ffn_dim_ceil(int64_t d, int64_t multiple_of);

/* ---- RoPE [P1 section 3; P3 section 四.3] ----
 * x [T][H][hd] at absolute positions pos[T] (whole numbers held in double): each interleaved pair
 * (x_2k, x_2k+1) of every head is rotated by the angle pos[t] * theta_base^(-2k/hd).  y may be x. */
int oracle_rope(const double *x, int64_t T, int64_t H, int64_t hd, const double *pos, double theta_base,
                double *y);
/* theta_k = theta_base^(-2k/hd), k = 0 .. hd/2 - 1. */
int oracle_rope_theta(int64_t hd, double theta_base, double *theta);

/* ---- causal grouped-query attention [P1 section 4; P3 4.4-4.6] ----
 * The KV head read by query head h. */
int64_t oracle_kv_head_of(int64_t h, int64_t n_q, int64_t n_kv);
/* One head: p[s][j] = softmax_j(q[s] . k[j] / sqrt(hd)) over the keys j <= q_pos[s] (j < Tk),
 * and 0 for the keys a query does not see.  q [Sq][hd], k [Tk][hd], p [Sq][Tk]. */
int oracle_causal_probs(const double *q, int64_t Sq, const double *k, int64_t Tk, int64_t hd,
                        const double *q_pos, double *p);
/* o[b][s][h] = sum_j p_j v[b][j][g], p = the causal softmax of query head h of row s against KV head
 * g = floor(h / r).  q [B][Sq][n_q][hd] post-RoPE, k and v [B][Tk][n_kv][hd] for positions 0..Tk-1,
 * query row s at absolute position q_pos[s]; o [B][Sq][n_q][hd]. */
int oracle_gqa_attention(const double *q, const double *k, const double *v, int64_t B, int64_t Sq,
                         int64_t Tk, int64_t n_q, int64_t n_kv, int64_t hd, const double *q_pos, double *o);

/* ---- one decoder block [P1 Step 2; P3 sections 四-五; P4 The Transformer Block] ----
 * Post-RoPE K and V of every token of x [B][S][d] at positions pos0..pos0+S-1:
 * u = RMSNorm(x; g_attn), k = RoPE(u W_K^T), v = u W_V^T; k and v [B][S][n_kv][hd]. */
int oracle_project_kv(const oracle_dims *dims, const oracle_block_weights *w, const double *x, int64_t pos0,
                      double *k, double *v);
/* h = x + Attn(RMSNorm(x)); y = h + FFN(RMSNorm(h)) for the tokens of x [B][S][d] at positions
 * pos0..pos0+S-1.  k_past / v_past [B][past_stride][n_kv][hd] hold the keys and values of positions
 * 0..pos0-1 (NULL when pos0 == 0).  K and V are computed for every token; the query side and the
 * output only for the n_rows token rows listed in rows (NULL: every row, n_rows = S).
 * k_scale / v_scale (8-bit cache, one fp32 scale per KV head, else NULL): the new tokens' K and V
 * are replaced by the values the cache stores (E4M3 code times scale) before attention reads them.
 * Outputs: y [B][n_rows][d]; k_new, v_new [B][S][n_kv][hd] (the stored values), either may be NULL. */
int oracle_block_forward(const oracle_dims *dims, const oracle_block_weights *w, const double *x, int64_t pos0,
                         const double *k_past, const double *v_past, int64_t past_stride,
                         const int64_t *rows, int64_t n_rows, const float *k_scale, const float *v_scale,
                         double *y, double *k_new, double *v_new);
/* The query side of oracle_block_forward alone, given the keys and values of positions 0..Tk-1
 * (k_all, v_all [B][Tk][n_kv][hd], already stored form): y [B][n_rows][d] for the listed rows. */
int oracle_block_rows(const oracle_dims *dims, const oracle_block_weights *w, const double *x, int64_t pos0,
                      const double *k_all, const double *v_all, int64_t Tk, const int64_t *rows, int64_t n_rows,
                      double *y);

/* ---- the decode stack [P3 sections 二, 九, 十] ----
 * One new token per sequence (x_emb [B][d], position t_cache; dims->S must be 1) through n_layers
 * blocks, each described by layer(ctx, l, ...), with the residual stream in double across layers;
 * then z = RMSNorm(x; final_g) and logits = z W_lm^T (w_lm [vocab][d]); logits [B][vocab]. */
int oracle_stack_decode_step(const oracle_dims *dims, int64_t n_layers, oracle_layer_fn layer, void *ctx,
                             const double *x_emb, int64_t t_cache, const double *final_g, const double *w_lm,
                             int64_t vocab, double *logits);

/* ---- sizes [P3 sections 六, 七] ---- */
int64_t oracle_block_param_count(int64_t d, int64_t n_q, int64_t n_kv, int64_t hd, int64_t d_ff);
int64_t oracle_model_param_count(int64_t n_layers, int64_t d, int64_t n_q, int64_t n_kv, int64_t hd,
                                 int64_t d_ff, int64_t vocab, int tied);
int64_t oracle_kv_bytes_per_token(int64_t n_layers, int64_t n_kv, int64_t hd, int64_t bytes_per_elem);

/* ---- 8-bit KV cache: OCP E4M3 ("e4m3fn") codes with per-head scales ----
 * The pages size the cache in bf16 only ([P1] section 4, [P3] section 七); the format read here:
 * sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 holds subnormals 2^-6 * m/8;
 * S.1111.111 is NaN; no infinities; largest finite magnitude 448. */
int oracle_e4m3_decode(const uint8_t *code, int64_t n, double *out);
/* The nearest code to each value (ties to the even code), saturating at +-448; NaN -> 0x7F. */
int oracle_e4m3_encode(const double *q, int64_t n, uint8_t *out);
/* Codes of x [n_vec][n_kv][hd] with one scale per KV head: the quotient x / s is taken in fp32
 * (x first rounded to fp32), then encoded. */
int oracle_kv_quantize(const double *x, int64_t n_vec, int64_t n_kv, int64_t hd, const float *scale,
                       uint8_t *code);
/* code * s in double, codes [n_vec][n_kv][hd]. */
int oracle_kv_dequantize(const uint8_t *code, int64_t n_vec, int64_t n_kv, int64_t hd, const float *scale,
                         double *out);

/* ---- next-token choice and embedding lookup [P3 sections 三, 十] ----
 * The page names argmax, temperature, top-k and top-p without formulas.  Readings taken:
 *   T > 0 divides the logits before the softmax, T <= 0 means argmax; tokens are ranked by logit,
 *   larger first, ties to the lower id; top-k keeps the first k of that order (k <= 0 or k >= V keeps
 *   all); top-p, after top-k, keeps the shortest prefix of the order whose share of the top-k mass
 *   reaches p (p >= 1 keeps all); the draw walks the kept tokens in increasing id and returns the
 *   first whose cumulative mass exceeds u times the kept mass (u uniform in [0, 1)). */
int oracle_embed(const double *table, int64_t vocab, int64_t d, const int64_t *tokens, int64_t n, double *out);
int oracle_order_desc(const double *z, int64_t V, int64_t *ids);
int64_t oracle_argmax(const double *z, int64_t V);
/* The kept tokens in ranked order: ids[0 .. *n_kept-1] (ids holds V entries). */
int oracle_kept_set(const double *z, int64_t V, double temperature, int64_t top_k, double top_p, int64_t *ids,
                    int64_t *n_kept);
int64_t oracle_sample(const double *z, int64_t V, double temperature, int64_t top_k, double top_p, double u);
/* How far a draw is from changing: margins[0] = the relative gap between the top-p cut and its
 * target, margins[1] = between u times the kept mass and the nearest cumulative boundary
 * (infinity where the rule does not apply). */
int oracle_sample_margins(const double *z, int64_t V, double temperature, int64_t top_k, double top_p, double u,
                          double *margins);

#ifdef __cplusplus
}
#endif

#endif /* LLAMA_ORACLE_H */
