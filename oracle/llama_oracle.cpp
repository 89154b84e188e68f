// fp64 CPU oracle of the Llama decoder block forward: RMSNorm, SwiGLU, RoPE, causal GQA, one
// block, and the decode stack with its final norm and LM head.
//
// TEST INFRASTRUCTURE ONLY (see llama_oracle.h): the tests, the build entry point's smoke check and
// the benchmark's oracle legs load it; the CUDA library shares nothing with it.
//
// Each function writes out the definition the pages give, in their order, with plain loops in
// double precision.  The only liberty taken is that a dot product may be summed in SIMD lanes (the
// `omp simd reduction` below): the order of a floating-point sum is not part of its definition,
// and in double precision it moves results by ~1e-16 relative.  Independent outputs are spread
// over OpenMP threads.  Nothing is tiled, fused or reformulated: attention forms every score of a
// query, takes the maximum, exponentiates, normalises and sums the values, in that order.
#include "llama_oracle.h"

#include <omp.h>

#include <cmath>
#include <cstring>
#include <vector>

namespace {

// y[i][o] = sum_k x[i][k] * w[o][k]: y = x W^T with W stored [out][in], as nn.Linear keeps it
// ("Llama Architecture ...", Mathematical Foundations 2 and Step 2; the pages' weight orientation
// differs between pages, the [out][in] reading is the one every call here takes).
void linear(const double *x, int64_t rows, int64_t in, const double *w, int64_t out, double *y) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t i = 0; i < rows; ++i) {
    for (int64_t o = 0; o < out; ++o) {
      const double *xi = x + i * in;
      const double *wo = w + o * in;
      double s = 0.0;
#pragma omp simd reduction(+ : s)
      for (int64_t k = 0; k < in; ++k) s += xi[k] * wo[k];
      y[i * out + o] = s;
    }
  }
}

bool dims_ok(const oracle_dims *d) {
  return d && d->B >= 0 && d->S >= 0 && d->d_model > 0 && d->n_q > 0 && d->n_kv > 0 && d->head_dim > 0 &&
         d->head_dim % 2 == 0 && d->n_q % d->n_kv == 0 && d->d_ff > 0;
}

// The stored value of each new K or V element of an 8-bit cache: encode, then decode.
void store_8bit(double *kv, int64_t n_vec, int64_t n_kv, int64_t hd, const float *scale) {
  std::vector<uint8_t> code((size_t)(n_vec * n_kv * hd));
  oracle_kv_quantize(kv, n_vec, n_kv, hd, scale, code.data());
  oracle_kv_dequantize(code.data(), n_vec, n_kv, hd, scale, kv);
}

}  // namespace

extern "C" {

int oracle_threads(void) { return omp_get_max_threads(); }

// ------------------------------------------------------------------------------------------------
// RMSNorm ("Llama Architecture ...", Mathematical Foundations 1; "RMSNorm" study note, "How it
// works"): RMS(x) = sqrt(mean(x^2) + eps) over the feature axis, no centring, then the gain.
// ------------------------------------------------------------------------------------------------
int oracle_rmsnorm(const double *x, int64_t rows, int64_t d, const double *g, double eps, double *y) {
  if (rows < 0 || d <= 0 || !x || !g || !y) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const double *xr = x + r * d;
    double ss = 0.0;
    for (int64_t i = 0; i < d; ++i) ss += xr[i] * xr[i];
    const double rms = std::sqrt(ss / (double)d + eps);
    for (int64_t i = 0; i < d; ++i) y[r * d + i] = xr[i] / rms * g[i];
  }
  return 0;
}

// ------------------------------------------------------------------------------------------------
// SwiGLU ("Llama Architecture ...", Mathematical Foundations 2; "LLaMA-3 8B ...", section 五):
// FFN(x) = W_down (SiLU(W_gate x) * W_up x), SiLU(z) = z * sigmoid(z), no biases.
// ------------------------------------------------------------------------------------------------
int oracle_silu(const double *z, int64_t n, double *out) {
  if (n < 0 || (n > 0 && (!z || !out))) return -1;
  for (int64_t i = 0; i < n; ++i) out[i] = z[i] / (1.0 + std::exp(-z[i]));
  return 0;
}

int oracle_swiglu_ffn(const double *x, int64_t rows, int64_t d, int64_t d_ff, const double *w_gate,
                      const double *w_up, const double *w_down, double *y) {
  if (rows < 0 || d <= 0 || d_ff <= 0 || !x || !w_gate || !w_up || !w_down || !y) return -1;
  std::vector<double> gate((size_t)(rows * d_ff)), up((size_t)(rows * d_ff)), m((size_t)(rows * d_ff));
  linear(x, rows, d, w_gate, d_ff, gate.data());
  linear(x, rows, d, w_up, d_ff, up.data());
  oracle_silu(gate.data(), rows * d_ff, m.data());
  for (int64_t i = 0; i < rows * d_ff; ++i) m[i] *= up[i];
  linear(m.data(), rows, d_ff, w_down, d, y);
  return 0;
}

int64_t oracle_ffn_dim_floor(int64_t d, int64_t multiple_of) { return (8 * d) / (3 * multiple_of) * multiple_of; }

int64_t oracle_ffn_dim_ceil(int64_t d, int64_t multiple_of) {
  const int64_t den = 3 * multiple_of;
  return (8 * d + den - 1) / den * multiple_of;
}

// ------------------------------------------------------------------------------------------------
// RoPE ("Llama Architecture ...", Mathematical Foundations 3; "LLaMA-3 8B ...", section 四.3):
// the pair (x_2k, x_2k+1) at position m turns by m * theta_k, theta_k = theta_base^(-2k/head_dim):
// (x_2k, x_2k+1) -> (x_2k cos - x_2k+1 sin, x_2k sin + x_2k+1 cos).
// ------------------------------------------------------------------------------------------------
int oracle_rope_theta(int64_t hd, double theta_base, double *theta) {
  if (hd <= 0 || hd % 2 || !theta) return -1;
  for (int64_t k = 0; k < hd / 2; ++k) theta[k] = std::pow(theta_base, -2.0 * (double)k / (double)hd);
  return 0;
}

int oracle_rope(const double *x, int64_t T, int64_t H, int64_t hd, const double *pos, double theta_base,
                double *y) {
  if (T < 0 || H < 0 || hd <= 0 || hd % 2 || (T > 0 && (!x || !pos || !y))) return -1;
  std::vector<double> theta((size_t)(hd / 2));
  oracle_rope_theta(hd, theta_base, theta.data());
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t h = 0; h < H; ++h) {
      const double *xp = x + (t * H + h) * hd;
      double *yp = y + (t * H + h) * hd;
      for (int64_t k = 0; k < hd / 2; ++k) {
        const double ang = pos[t] * theta[(size_t)k];
        const double c = std::cos(ang), s = std::sin(ang);
        const double x0 = xp[2 * k], x1 = xp[2 * k + 1];
        yp[2 * k] = x0 * c - x1 * s;
        yp[2 * k + 1] = x0 * s + x1 * c;
      }
    }
  }
  return 0;
}

// ------------------------------------------------------------------------------------------------
// Causal grouped-query attention ("Llama Architecture ...", Mathematical Foundations 4;
// "LLaMA-3 8B ...", sections 4.4-4.6): query head h reads KV head floor(h / r); the scores
// q . k_j / sqrt(hd) of the keys j at or before the query's position go through a softmax (its
// maximum subtracted first, an identity of the softmax) and weight the values.
// ------------------------------------------------------------------------------------------------
int64_t oracle_kv_head_of(int64_t h, int64_t n_q, int64_t n_kv) { return h / (n_q / n_kv); }

namespace {
// Softmax weights of one query against keys k[0 .. n_vis-1] (row stride ks); returns them in p.
void causal_softmax_row(const double *q, const double *k, int64_t ks, int64_t n_vis, int64_t hd, double *p) {
  const double scale = 1.0 / std::sqrt((double)hd);
  double mx = -INFINITY;
  for (int64_t j = 0; j < n_vis; ++j) {
    double dot = 0.0;
    for (int64_t t = 0; t < hd; ++t) dot += q[t] * k[j * ks + t];
    p[j] = dot * scale;
    if (p[j] > mx) mx = p[j];
  }
  double sum = 0.0;
  for (int64_t j = 0; j < n_vis; ++j) {
    p[j] = std::exp(p[j] - mx);
    sum += p[j];
  }
  for (int64_t j = 0; j < n_vis; ++j) p[j] /= sum;
}

// Keys visible to a query at absolute position m among Tk keys at positions 0..Tk-1.
int64_t visible_keys(double m, int64_t Tk) {
  if (m < 0) return 0;
  const double n = std::floor(m) + 1.0;
  return n < (double)Tk ? (int64_t)n : Tk;
}
}  // namespace

int oracle_causal_probs(const double *q, int64_t Sq, const double *k, int64_t Tk, int64_t hd,
                        const double *q_pos, double *p) {
  if (Sq < 0 || Tk < 0 || hd <= 0 || (Sq > 0 && (!q || !q_pos || !p)) || (Tk > 0 && !k)) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t s = 0; s < Sq; ++s) {
    double *ps = p + s * Tk;
    for (int64_t j = 0; j < Tk; ++j) ps[j] = 0.0;
    causal_softmax_row(q + s * hd, k, hd, visible_keys(q_pos[s], Tk), hd, ps);
  }
  return 0;
}

int oracle_gqa_attention(const double *q, const double *k, const double *v, int64_t B, int64_t Sq,
                         int64_t Tk, int64_t n_q, int64_t n_kv, int64_t hd, const double *q_pos, double *o) {
  if (B < 0 || Sq < 0 || Tk < 0 || n_q <= 0 || n_kv <= 0 || n_q % n_kv || hd <= 0) return -1;
  if (B * Sq > 0 && (!q || !q_pos || !o || (Tk > 0 && (!k || !v)))) return -1;
#pragma omp parallel for collapse(3) schedule(dynamic, 4)
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t s = 0; s < Sq; ++s) {
      for (int64_t h = 0; h < n_q; ++h) {
        const int64_t g = oracle_kv_head_of(h, n_q, n_kv);
        const int64_t n_vis = visible_keys(q_pos[s], Tk);
        const double *kg = k + (b * Tk * n_kv + g) * hd;   // key j of head g at kg[j * n_kv * hd]
        const double *vg = v + (b * Tk * n_kv + g) * hd;
        std::vector<double> p((size_t)n_vis);
        causal_softmax_row(q + ((b * Sq + s) * n_q + h) * hd, kg, n_kv * hd, n_vis, hd, p.data());
        // o = sum_j p_j v_j, accumulated over j in increasing order for every component
        double *os = o + ((b * Sq + s) * n_q + h) * hd;
        for (int64_t t = 0; t < hd; ++t) os[t] = 0.0;
        for (int64_t j = 0; j < n_vis; ++j)
          for (int64_t t = 0; t < hd; ++t) os[t] += p[(size_t)j] * vg[j * n_kv * hd + t];
      }
    }
  }
  return 0;
}

// ------------------------------------------------------------------------------------------------
// One decoder block ("Llama Architecture ...", Step 2; "LLaMA-3 8B ...", sections 四-五;
// "LLaMA Architecture > Model Architecture", The Transformer Block):
//   u = RMSNorm(x; g_attn); q = RoPE(u W_Q^T); k = RoPE(u W_K^T); v = u W_V^T
//   h = x + Attn(q, k, v) W_O^T;  y = h + W_down(SiLU(W_gate w) * W_up w), w = RMSNorm(h; g_ffn)
// ------------------------------------------------------------------------------------------------
int oracle_project_kv(const oracle_dims *dims, const oracle_block_weights *w, const double *x, int64_t pos0,
                      double *k, double *v) {
  if (!dims_ok(dims) || !w || pos0 < 0) return -1;
  const int64_t T = dims->B * dims->S, d = dims->d_model, kvw = dims->n_kv * dims->head_dim;
  if (T == 0) return 0;
  if (!x || !k || !v) return -1;
  std::vector<double> u((size_t)(T * d)), kr((size_t)(T * kvw)), pos((size_t)T);
  oracle_rmsnorm(x, T, d, w->attn_norm_g, dims->eps, u.data());
  linear(u.data(), T, d, w->wk, kvw, kr.data());
  linear(u.data(), T, d, w->wv, kvw, v);
  for (int64_t t = 0; t < T; ++t) pos[(size_t)t] = (double)(pos0 + t % dims->S);
  oracle_rope(kr.data(), T, dims->n_kv, dims->head_dim, pos.data(), dims->theta_base, k);
  return 0;
}

int oracle_block_rows(const oracle_dims *dims, const oracle_block_weights *w, const double *x, int64_t pos0,
                      const double *k_all, const double *v_all, int64_t Tk, const int64_t *rows, int64_t n_rows,
                      double *y) {
  if (!dims_ok(dims) || !w || pos0 < 0 || Tk < 0) return -1;
  const int64_t B = dims->B, S = dims->S, d = dims->d_model, hd = dims->head_dim;
  const int64_t n_q = dims->n_q, n_kv = dims->n_kv, qw = n_q * hd;
  const int64_t R = rows ? n_rows : S;
  if (R < 0) return -1;
  if (B * R == 0) return 0;
  if (!x || !y || (Tk > 0 && (!k_all || !v_all))) return -1;
  for (int64_t i = 0; rows && i < R; ++i)
    if (rows[i] < 0 || rows[i] >= S) return -1;
  // the selected rows of x, and their absolute positions
  std::vector<double> xs((size_t)(B * R * d)), pos((size_t)R);
  for (int64_t i = 0; i < R; ++i) pos[(size_t)i] = (double)(pos0 + (rows ? rows[i] : i));
  for (int64_t b = 0; b < B; ++b)
    for (int64_t i = 0; i < R; ++i)
      std::memcpy(&xs[(size_t)((b * R + i) * d)], x + (b * S + (rows ? rows[i] : i)) * d, sizeof(double) * d);
  // attention sublayer
  std::vector<double> u((size_t)(B * R * d)), q((size_t)(B * R * qw)), o((size_t)(B * R * qw));
  oracle_rmsnorm(xs.data(), B * R, d, w->attn_norm_g, dims->eps, u.data());
  linear(u.data(), B * R, d, w->wq, qw, q.data());
  for (int64_t b = 0; b < B; ++b)
    oracle_rope(&q[(size_t)(b * R * qw)], R, n_q, hd, pos.data(), dims->theta_base, &q[(size_t)(b * R * qw)]);
  if (oracle_gqa_attention(q.data(), k_all, v_all, B, R, Tk, n_q, n_kv, hd, pos.data(), o.data())) return -1;
  std::vector<double> h((size_t)(B * R * d));
  linear(o.data(), B * R, qw, w->wo, d, h.data());
  for (int64_t i = 0; i < B * R * d; ++i) h[(size_t)i] += xs[(size_t)i];
  // feed-forward sublayer
  std::vector<double> z((size_t)(B * R * d)), f((size_t)(B * R * d));
  oracle_rmsnorm(h.data(), B * R, d, w->ffn_norm_g, dims->eps, z.data());
  oracle_swiglu_ffn(z.data(), B * R, d, dims->d_ff, w->w_gate, w->w_up, w->w_down, f.data());
  for (int64_t i = 0; i < B * R * d; ++i) y[i] = h[(size_t)i] + f[(size_t)i];
  return 0;
}

int oracle_block_forward(const oracle_dims *dims, const oracle_block_weights *w, const double *x, int64_t pos0,
                         const double *k_past, const double *v_past, int64_t past_stride,
                         const int64_t *rows, int64_t n_rows, const float *k_scale, const float *v_scale,
                         double *y, double *k_new, double *v_new) {
  if (!dims_ok(dims) || !w || pos0 < 0) return -1;
  if (pos0 > 0 && (!k_past || !v_past || past_stride < pos0)) return -1;
  const int64_t B = dims->B, S = dims->S, n_kv = dims->n_kv, hd = dims->head_dim, row = n_kv * hd;
  const int64_t Tk = pos0 + S;
  // K and V of the new tokens, in the form the cache holds them
  std::vector<double> kn((size_t)(B * S * row)), vn((size_t)(B * S * row));
  if (oracle_project_kv(dims, w, x, pos0, kn.data(), vn.data())) return -1;
  if (k_scale) store_8bit(kn.data(), B * S, n_kv, hd, k_scale);
  if (v_scale) store_8bit(vn.data(), B * S, n_kv, hd, v_scale);
  // every key and value the queries may see: positions 0..pos0-1 from the cache, then the new ones
  std::vector<double> ka((size_t)(B * Tk * row)), va((size_t)(B * Tk * row));
  for (int64_t b = 0; b < B; ++b) {
    if (pos0 > 0) {
      std::memcpy(&ka[(size_t)(b * Tk * row)], k_past + b * past_stride * row, sizeof(double) * pos0 * row);
      std::memcpy(&va[(size_t)(b * Tk * row)], v_past + b * past_stride * row, sizeof(double) * pos0 * row);
    }
    std::memcpy(&ka[(size_t)((b * Tk + pos0) * row)], &kn[(size_t)(b * S * row)], sizeof(double) * S * row);
    std::memcpy(&va[(size_t)((b * Tk + pos0) * row)], &vn[(size_t)(b * S * row)], sizeof(double) * S * row);
  }
  if (y && oracle_block_rows(dims, w, x, pos0, ka.data(), va.data(), Tk, rows, n_rows, y)) return -1;
  if (k_new) std::memcpy(k_new, kn.data(), sizeof(double) * B * S * row);
  if (v_new) std::memcpy(v_new, vn.data(), sizeof(double) * B * S * row);
  return 0;
}

// ------------------------------------------------------------------------------------------------
// The decode stack ("LLaMA-3 8B ...", section 二 data flow, section 九 decode, section 十 final
// RMSNorm and untied LM head): the new token of each sequence at position t_cache goes through
// every block against that layer's cache, then z = RMSNorm(x; g_final), logits = z W_lm^T.
// ------------------------------------------------------------------------------------------------
int oracle_stack_decode_step(const oracle_dims *dims, int64_t n_layers, oracle_layer_fn layer, void *ctx,
                             const double *x_emb, int64_t t_cache, const double *final_g, const double *w_lm,
                             int64_t vocab, double *logits) {
  if (!dims_ok(dims) || dims->S != 1 || n_layers < 0 || !layer || t_cache < 0 || vocab < 0) return -1;
  const int64_t B = dims->B, d = dims->d_model;
  if (B == 0) return 0;
  if (!x_emb || !final_g || !logits || (vocab > 0 && !w_lm)) return -1;
  std::vector<double> x(x_emb, x_emb + B * d), y((size_t)(B * d));
  for (int64_t l = 0; l < n_layers; ++l) {
    oracle_layer L;
    std::memset(&L, 0, sizeof(L));
    if (layer(ctx, l, &L)) return -1;
    if (oracle_block_forward(dims, &L.w, x.data(), t_cache, L.k_past, L.v_past, L.past_stride, nullptr, 0,
                             L.k_scale, L.v_scale, y.data(), nullptr, nullptr))
      return -1;
    x.swap(y);
  }
  std::vector<double> z((size_t)(B * d));
  oracle_rmsnorm(x.data(), B, d, final_g, dims->eps, z.data());
  linear(z.data(), B, d, w_lm, vocab, logits);
  return 0;
}

// ------------------------------------------------------------------------------------------------
// Sizes ("LLaMA-3 8B ...", section 六 parameter counts, section 七 KV cache per token).
// ------------------------------------------------------------------------------------------------
int64_t oracle_block_param_count(int64_t d, int64_t n_q, int64_t n_kv, int64_t hd, int64_t d_ff) {
  // W_Q + W_K + W_V + W_O, three FFN matrices, two RMSNorm gains
  return d * n_q * hd + 2 * d * n_kv * hd + n_q * hd * d + 3 * d * d_ff + 2 * d;
}

int64_t oracle_model_param_count(int64_t n_layers, int64_t d, int64_t n_q, int64_t n_kv, int64_t hd,
                                 int64_t d_ff, int64_t vocab, int tied) {
  // blocks, the embedding table, the LM head unless tied to it, the final RMSNorm gain
  const int64_t emb = vocab * d;
  return n_layers * oracle_block_param_count(d, n_q, n_kv, hd, d_ff) + emb + (tied ? 0 : emb) + d;
}

int64_t oracle_kv_bytes_per_token(int64_t n_layers, int64_t n_kv, int64_t hd, int64_t bytes_per_elem) {
  return n_layers * 2 * n_kv * hd * bytes_per_elem;  // K and V of every layer
}

}  // extern "C"
