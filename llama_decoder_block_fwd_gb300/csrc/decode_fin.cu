// Decode-step finishers: each reduces the fp32 split-K partial sums of one weight-streaming GEMM
// and applies what follows that GEMM in the block, writing the next GEMM's input as two bf16
// parts (hi + lo) so that the activation carries ~16 mantissa bits into the tensor cores.
//
//   fin_norm   : x (+)= sum_s partial_s (O or down projection) in the fp32 residual stream, then
//                RMSNorm in split form: rs = rsqrt(mean(x^2) + eps), a = x * g as hi + lo.
//   fin_qkv    : (q, k, v) = rs * sum_s partial_s; RoPE on q and k at position t; q to its buffer,
//                k and v into the caches at position t (bf16, or E4M3 codes of x / scale).
//   fin_swiglu : m = SiLU(rs * gate) * (rs * up) as hi + lo.
// ("Llama Architecture ...", Mathematical Foundations 1-3; "LLaMA-3 8B ...", section 九.)
#include "epilogue.cuh"
#include "kernels.h"

namespace llama {
namespace {

__device__ __forceinline__ void split_bf16(float v, uint16_t& hi, uint16_t& lo) {
  hi = f2bf(v);
  lo = f2bf(v - bf2f(hi));
}

constexpr int FN_THREADS = 256;
constexpr int FN_MAX_PER_THREAD = 32;   // d_model <= 8192

// One CTA per row.
__global__ void __launch_bounds__(FN_THREADS) fin_norm_kernel(float* __restrict__ x, const uint16_t* __restrict__ init,
                                                              const float* __restrict__ part, int n_split,
                                                              const uint16_t* __restrict__ g, uint16_t* __restrict__ a_hi,
                                                              uint16_t* __restrict__ a_lo, float* __restrict__ rs_out,
                                                              int B, int d, float eps) {
  __shared__ float red[FN_THREADS / 32];
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  float v[FN_MAX_PER_THREAD];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < FN_MAX_PER_THREAD; ++j) {
    const int i = threadIdx.x + j * FN_THREADS;
    v[j] = 0.f;
    if (i < d) {
      float t = init ? bf2f(init[(int64_t)r * d + i]) : x[(int64_t)r * d + i];
      for (int s = 0; s < n_split; ++s) t += part[((int64_t)s * B + r) * d + i];
      x[(int64_t)r * d + i] = t;
      v[j] = t;
      ss = fmaf(t, t, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < FN_THREADS / 32; ++w) tot += red[w];
  const float rs = rsqrtf(tot / (float)d + eps);
  if (threadIdx.x == 0) rs_out[r] = rs;
#pragma unroll
  for (int j = 0; j < FN_MAX_PER_THREAD; ++j) {
    const int i = threadIdx.x + j * FN_THREADS;
    if (i < d) {
      uint16_t hi, lo;
      split_bf16(v[j] * bf2f(g[i]), hi, lo);
      a_hi[(int64_t)r * d + i] = hi;
      a_lo[(int64_t)r * d + i] = lo;
    }
  }
}

struct FinQkvParams {
  const float* part;     // [n_split, B, n_cols]
  const float* rs;       // [B]
  uint16_t* q;           // [B, nq_cols]
  void* kc;              // layer cache [B, cap, nkv_cols]: bf16, or E4M3 codes with k_scale set
  void* vc;
  const float* k_scale;  // [n_kv] or null
  const float* v_scale;
  int n_split, B, nq_cols, nkv_cols, hd;
  int64_t cap, t;
  RopeFreq freq[kMaxRopePairs];
};

// One thread per (row, column pair).
__global__ void fin_qkv_kernel(const __grid_constant__ FinQkvParams p) {
  pdl_trigger();
  pdl_wait();
  const int n_cols = p.nq_cols + 2 * p.nkv_cols;
  const int pairs = n_cols / 2;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)p.B * pairs) return;
  const int r = (int)(idx / pairs);
  const int c = (int)(idx % pairs) * 2;
  float v0 = 0.f, v1 = 0.f;
  for (int s = 0; s < p.n_split; ++s) {
    const float2 w = *reinterpret_cast<const float2*>(p.part + ((int64_t)s * p.B + r) * n_cols + c);
    v0 += w.x;
    v1 += w.y;
  }
  const float rs = p.rs[r];
  v0 *= rs;
  v1 *= rs;
  const float pos = (float)p.t;
  if (c < p.nq_cols + p.nkv_cols) {       // RoPE on q and k
    const int cc = c < p.nq_cols ? c : c - p.nq_cols;
    float sn, cs;
    rope_sincos(pos, p.freq[(cc % p.hd) >> 1], sn, cs);
    const float x0 = v0, x1 = v1;
    v0 = x0 * cs - x1 * sn;
    v1 = x0 * sn + x1 * cs;
  }
  if (c < p.nq_cols) {
    *reinterpret_cast<uint32_t*>(p.q + (int64_t)r * p.nq_cols + c) = pack_bf2(v0, v1);
    return;
  }
  const bool is_k = c < p.nq_cols + p.nkv_cols;
  const int cc = is_k ? c - p.nq_cols : c - p.nq_cols - p.nkv_cols;
  const int64_t off = ((int64_t)r * p.cap + p.t) * p.nkv_cols + cc;
  if (p.k_scale) {   // 8-bit cache: code = E4M3(fl32(x) / scale), rounded to nearest even, saturating
    const float s = (is_k ? p.k_scale : p.v_scale)[cc / p.hd];
    uint16_t code;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(code) : "f"(v1 / s), "f"(v0 / s));
    *reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(is_k ? p.kc : p.vc) + off) = code;
  } else {
    *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(is_k ? p.kc : p.vc) + off) = pack_bf2(v0, v1);
  }
}

// One thread per (row, hidden unit): gate in columns [0, d_ff), up in [d_ff, 2 d_ff).
__global__ void fin_swiglu_kernel(const float* __restrict__ part, const float* __restrict__ rs, uint16_t* __restrict__ m_hi,
                                  uint16_t* __restrict__ m_lo, int n_split, int B, int dff) {
  pdl_trigger();
  pdl_wait();
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)B * dff) return;
  const int r = (int)(idx / dff), j = (int)(idx % dff);
  float gsum = 0.f, usum = 0.f;
  for (int s = 0; s < n_split; ++s) {
    const float* row = part + ((int64_t)s * B + r) * 2 * dff;
    gsum += row[j];
    usum += row[dff + j];
  }
  const float sc = rs[r];
  const float m = silu_f(gsum * sc) * (usum * sc);
  uint16_t hi, lo;
  split_bf16(m, hi, lo);
  m_hi[idx] = hi;
  m_lo[idx] = lo;
}

}  // namespace

int launch_fin_norm(float* x, const void* init_bf16, const float* part, int n_split, const void* g, void* a_hi,
                    void* a_lo, float* rs, int B, int d, float eps, cudaStream_t st) {
  if (d > FN_THREADS * FN_MAX_PER_THREAD) return -1;
  return launch_k(fin_norm_kernel, dim3(B), dim3(FN_THREADS), 0, st, x, static_cast<const uint16_t*>(init_bf16), part,
                  n_split, static_cast<const uint16_t*>(g), static_cast<uint16_t*>(a_hi), static_cast<uint16_t*>(a_lo),
                  rs, B, d, eps) == cudaSuccess ? 0 : -1;
}

int launch_fin_qkv(const float* part, int n_split, const float* rs, void* q, void* kc, void* vc, int B, int nq_cols,
                   int nkv_cols, int hd, int64_t cap, int64_t t, const RopeFreq* freq, const float* k_scale,
                   const float* v_scale, cudaStream_t st) {
  FinQkvParams p;
  p.part = part; p.rs = rs;
  p.q = static_cast<uint16_t*>(q); p.kc = kc; p.vc = vc;
  p.k_scale = k_scale; p.v_scale = v_scale;
  p.n_split = n_split; p.B = B; p.nq_cols = nq_cols; p.nkv_cols = nkv_cols; p.hd = hd; p.cap = cap; p.t = t;
  for (int i = 0; i < hd / 2; ++i) p.freq[i] = freq[i];
  const int64_t n = (int64_t)B * (nq_cols + 2 * nkv_cols) / 2;
  return launch_k(fin_qkv_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, p) == cudaSuccess ? 0 : -1;
}

int launch_fin_swiglu(const float* part, int n_split, const float* rs, void* m_hi, void* m_lo, int B, int dff,
                      cudaStream_t st) {
  const int64_t n = (int64_t)B * dff;
  return launch_k(fin_swiglu_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, part, rs,
                  static_cast<uint16_t*>(m_hi), static_cast<uint16_t*>(m_lo), n_split, B, dff) == cudaSuccess ? 0 : -1;
}

}  // namespace llama
