// fp64 CPU oracle of the steps either side of the decode stack: the embedding lookup that turns
// token ids into input rows, and the choice of the next token from the LM head's logits.
// TEST INFRASTRUCTURE ONLY (see llama_oracle.h).
//
// "LLaMA-3 8B ...", section 三: the embedding is a row lookup in the [vocab, d_model] table;
// section 十: a softmax over the vocabulary, then argmax, or a draw shaped by temperature, top-k
// and top-p; the drawn token goes back to the embedding for the next step.  The page gives no
// formulas; the readings taken are listed in llama_oracle.h beside these functions.  Logits may
// hold -infinity (a masked token); NaN logits are not taken.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <numeric>
#include <vector>

#include "llama_oracle.h"

namespace {

// Token ids ranked by logit, larger first, ties to the lower id (a stable sort of increasing ids).
std::vector<int64_t> ranked(const double *z, int64_t V) {
  std::vector<int64_t> ids((size_t)V);
  std::iota(ids.begin(), ids.end(), 0);
  std::stable_sort(ids.begin(), ids.end(), [z](int64_t a, int64_t b) { return z[a] > z[b]; });
  return ids;
}

// The tokens kept by top-k and then top-p, in ranked order.
std::vector<int64_t> kept(const double *z, int64_t V, double T, int64_t top_k, double top_p) {
  std::vector<int64_t> order = ranked(z, V);
  if (T <= 0 || top_k == 1) {
    order.resize(1);
    return order;
  }
  const int64_t n = (top_k <= 0 || top_k >= V) ? V : top_k;
  order.resize((size_t)n);
  if (top_p < 1.0) {
    // softmax over the top-k set at temperature T, unnormalised (the shift by the maximum cancels)
    std::vector<double> cum((size_t)n);
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i) {
      acc += std::exp((z[order[(size_t)i]] - z[order[0]]) / T);
      cum[(size_t)i] = acc;
    }
    const double need = top_p * cum[(size_t)(n - 1)];
    int64_t n_p = 1;
    while (cum[(size_t)(n_p - 1)] < need) ++n_p;
    order.resize((size_t)n_p);
  }
  return order;
}

double max_logit(const double *z, int64_t V) {
  double m = -INFINITY;
  for (int64_t i = 0; i < V; ++i) m = std::max(m, z[i]);
  return m;
}

}  // namespace

extern "C" {

int oracle_embed(const double *table, int64_t vocab, int64_t d, const int64_t *tokens, int64_t n, double *out) {
  if (vocab < 0 || d <= 0 || n < 0 || (n > 0 && (!table || !tokens || !out))) return -1;
  for (int64_t i = 0; i < n; ++i) {
    if (tokens[i] < 0 || tokens[i] >= vocab) return -1;
    std::memcpy(out + i * d, table + tokens[i] * d, sizeof(double) * d);
  }
  return 0;
}

int oracle_order_desc(const double *z, int64_t V, int64_t *ids) {
  if (V < 0 || (V > 0 && (!z || !ids))) return -1;
  std::vector<int64_t> o = ranked(z, V);
  std::copy(o.begin(), o.end(), ids);
  return 0;
}

int64_t oracle_argmax(const double *z, int64_t V) {
  if (V <= 0 || !z) return -1;
  return ranked(z, V)[0];
}

int oracle_kept_set(const double *z, int64_t V, double temperature, int64_t top_k, double top_p, int64_t *ids,
                    int64_t *n_kept) {
  if (V <= 0 || !z || !ids || !n_kept) return -1;
  std::vector<int64_t> k = kept(z, V, temperature, top_k, top_p);
  std::copy(k.begin(), k.end(), ids);
  *n_kept = (int64_t)k.size();
  return 0;
}

int64_t oracle_sample(const double *z, int64_t V, double temperature, int64_t top_k, double top_p, double u) {
  if (V <= 0 || !z) return -1;
  std::vector<int64_t> ids = kept(z, V, temperature, top_k, top_p);
  if (ids.size() == 1) return ids[0];
  std::sort(ids.begin(), ids.end());   // the draw walks the kept tokens in increasing id
  const double zmax = max_logit(z, V);
  std::vector<double> mass(ids.size());
  double total = 0.0;
  for (size_t i = 0; i < ids.size(); ++i) {
    mass[i] = std::exp((z[ids[i]] - zmax) / temperature);
    total += mass[i];
  }
  double acc = 0.0;
  for (size_t i = 0; i < ids.size(); ++i) {
    acc += mass[i];
    if (acc > u * total) return ids[i];
  }
  return ids.back();
}

int oracle_sample_margins(const double *z, int64_t V, double temperature, int64_t top_k, double top_p, double u,
                          double *margins) {
  if (V <= 0 || !z || !margins) return -1;
  margins[0] = margins[1] = INFINITY;
  if (temperature <= 0 || top_k == 1) return 0;
  std::vector<int64_t> order = ranked(z, V);
  const int64_t n = (top_k <= 0 || top_k >= V) ? V : top_k;
  if (top_p < 1.0) {
    double acc = 0.0;
    std::vector<double> cum((size_t)n);
    for (int64_t i = 0; i < n; ++i) {
      acc += std::exp((z[order[(size_t)i]] - z[order[0]]) / temperature);
      cum[(size_t)i] = acc;
    }
    const double need = top_p * acc;
    double m = INFINITY;
    for (int64_t i = 0; i < n; ++i) m = std::min(m, std::fabs(cum[(size_t)i] - need));
    margins[0] = m / acc;
  }
  std::vector<int64_t> ids = kept(z, V, temperature, top_k, top_p);
  if (ids.size() == 1) return 0;
  std::sort(ids.begin(), ids.end());
  const double zmax = max_logit(z, V);
  std::vector<double> cum(ids.size());
  double acc = 0.0;
  for (size_t i = 0; i < ids.size(); ++i) {
    acc += std::exp((z[ids[i]] - zmax) / temperature);
    cum[i] = acc;
  }
  double m = INFINITY;
  for (size_t i = 0; i < ids.size(); ++i) m = std::min(m, std::fabs(cum[i] - u * acc));
  margins[1] = m / acc;
  return 0;
}

}  // extern "C"
