/*
 * Seeded synthetic inputs, host side.
 *
 * This file holds no arithmetic of the Llama block: it only draws the seeded
 * numbers that both the CPU oracle and the GPU tests/bench feed in.  The device
 * side (synth_dev.cu) implements the same definition, so a tensor drawn on the
 * GPU is bit-identical to the one drawn here.
 *
 * Definition (counter-based, integer-exact):
 *   mix64(z)   : the SplitMix64 output finaliser (Steele, Lea, Flood,
 *                "Fast splittable pseudorandom number generators", OOPSLA 2014):
 *                z ^= z>>30; z *= 0xBF58476D1CE4E5B9; z ^= z>>27;
 *                z *= 0x94D049BB133111EB; z ^= z>>31.
 *   key        = mix64(mix64(seed + G) + tid * G),  G = 0x9E3779B97F4A7C15
 *   h_j        = mix64(key + (3*i + j + 1) * G),     j = 0,1,2
 *   S          = sum of the twelve 16-bit fields of h_0, h_1, h_2
 *   z          = (S - 393210) / 65536               (Irwin-Hall, 12 uniforms:
 *                                                    mean 0, variance 1, |z| <= 6)
 *   x          = (std * z) + mean, two fp64 roundings, no fused multiply-add
 *   f32 output = x rounded to nearest float
 *   bf16 output= that float rounded to nearest-even bf16 (integer rounding)
 * All 64-bit arithmetic wraps modulo 2^64.
 */
#include <stdint.h>
#include <string.h>

#define SYNTH_G 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27; z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

static inline uint64_t stream_key(uint64_t seed, uint64_t tid) {
  return mix64(mix64(seed + SYNTH_G) + tid * SYNTH_G);
}

static inline double draw(uint64_t key, uint64_t i, double mean, double stdv) {
  uint64_t s = 0;
  for (uint64_t j = 0; j < 3; ++j) {
    uint64_t h = mix64(key + (3 * i + j + 1) * SYNTH_G);
    s += (h & 0xFFFF) + ((h >> 16) & 0xFFFF) + ((h >> 32) & 0xFFFF) + (h >> 48);
  }
  double z = (double)((int64_t)s - 393210) / 65536.0;
  volatile double t = stdv * z;   /* keep the product rounded on its own */
  return t + mean;
}

static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFF) ? 0x40 : 0));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* out[k] = draw(offset + k) for k in [0, n), as float32 */
void synth_fill_f32(float* out, int64_t n, uint64_t seed, uint64_t tid, int64_t offset,
                    double mean, double stdv) {
  const uint64_t key = stream_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < n; ++k)
    out[k] = (float)draw(key, (uint64_t)(offset + k), mean, stdv);
}

/* out[k] = bf16 bits of draw(offset + k) */
void synth_fill_bf16(uint16_t* out, int64_t n, uint64_t seed, uint64_t tid, int64_t offset,
                     double mean, double stdv) {
  const uint64_t key = stream_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < n; ++k)
    out[k] = f32_to_bf16_rne((float)draw(key, (uint64_t)(offset + k), mean, stdv));
}

/* Same draws, widened exactly to fp64 after rounding to the stored type
 * (dtype 0 = f32, 1 = bf16): what a consumer of the stored tensor sees. */
void synth_fill_f64_as(double* out, int dtype, int64_t n, uint64_t seed, uint64_t tid,
                       int64_t offset, double mean, double stdv) {
  const uint64_t key = stream_key(seed, tid);
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < n; ++k) {
    float f = (float)draw(key, (uint64_t)(offset + k), mean, stdv);
    if (dtype == 1) {
      uint32_t u = (uint32_t)f32_to_bf16_rne(f) << 16;
      memcpy(&f, &u, 4);
    }
    out[k] = (double)f;
  }
}
