// fp64 CPU oracle of the 8-bit KV cache: OCP E4M3 ("e4m3fn") codes with one fp32 scale per
// (layer, K or V, KV head).  TEST INFRASTRUCTURE ONLY (see llama_oracle.h).
//
// The pages size the KV cache in bf16 and note that it dominates decode memory ("Llama
// Architecture ...", Mathematical Foundations 4; "LLaMA-3 8B ...", section 七); they give no 8-bit
// format.  Readings taken: the format is E4M3 as OCP defines it (bias 7, subnormals 2^-6 * m/8 in
// exponent field 0, S.1111.111 the only NaN, no infinities, largest finite magnitude 448); a cached
// element is code * s; encoding rounds the fp32 quotient x / s to the nearest code (ties to the
// even code) and saturates at +-448, so the integer decision is taken in the precision a GPU
// kernel takes it; attention reads the decoded values, the new token's own K/V included.
#include <cmath>

#include "llama_oracle.h"

namespace {

double e4m3_value(uint8_t c) {
  const double sign = (c & 0x80) ? -1.0 : 1.0;
  const int e = (c >> 3) & 0xF, m = c & 0x7;
  if (e == 15 && m == 7) return NAN;
  const double mag = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return sign * mag;
}

uint8_t e4m3_code(double q) {
  if (std::isnan(q)) return 0x7F;
  const double a = std::fmin(std::fabs(q), 448.0);
  // codes 0x00..0x7E are every finite non-negative value, in increasing order
  int hi = 0;
  while (hi < 126 && e4m3_value((uint8_t)hi) < a) ++hi;   // first code whose value is >= a
  const int lo = hi > 0 ? hi - 1 : 0;
  const double d_lo = a - e4m3_value((uint8_t)lo), d_hi = e4m3_value((uint8_t)hi) - a;
  const bool take_hi = d_hi < d_lo || (d_hi == d_lo && (hi & 1) == 0);
  const uint8_t code = (uint8_t)(take_hi ? hi : lo);
  return std::signbit(q) ? (uint8_t)(code | 0x80) : code;
}

}  // namespace

extern "C" {

int oracle_e4m3_decode(const uint8_t *code, int64_t n, double *out) {
  if (n < 0 || (n > 0 && (!code || !out))) return -1;
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(code[i]);
  return 0;
}

int oracle_e4m3_encode(const double *q, int64_t n, uint8_t *out) {
  if (n < 0 || (n > 0 && (!q || !out))) return -1;
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_code(q[i]);
  return 0;
}

int oracle_kv_quantize(const double *x, int64_t n_vec, int64_t n_kv, int64_t hd, const float *scale,
                       uint8_t *code) {
  if (n_vec < 0 || n_kv <= 0 || hd <= 0 || (n_vec > 0 && (!x || !scale || !code))) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n_vec; ++t)
    for (int64_t g = 0; g < n_kv; ++g)
      for (int64_t i = 0; i < hd; ++i) {
        const int64_t at = (t * n_kv + g) * hd + i;
        const float x32 = (float)x[at];
        const float quot = x32 / scale[g];   // the quotient rounded to fp32
        code[at] = e4m3_code((double)quot);
      }
  return 0;
}

int oracle_kv_dequantize(const uint8_t *code, int64_t n_vec, int64_t n_kv, int64_t hd, const float *scale,
                         double *out) {
  if (n_vec < 0 || n_kv <= 0 || hd <= 0 || (n_vec > 0 && (!code || !scale || !out))) return -1;
  for (int64_t t = 0; t < n_vec; ++t)
    for (int64_t g = 0; g < n_kv; ++g)
      for (int64_t i = 0; i < hd; ++i) {
        const int64_t at = (t * n_kv + g) * hd + i;
        out[at] = e4m3_value(code[at]) * (double)scale[g];
      }
  return 0;
}

}  // extern "C"
