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
#include <algorithm>

#include "epilogue.cuh"
#include "kernels.h"

namespace llama {
namespace {

__device__ __forceinline__ void split_bf16(float v, uint16_t& hi, uint16_t& lo) {
  hi = f2bf(v);
  lo = f2bf(v - bf2f(hi));
}

constexpr int FN_THREADS = 256;
constexpr int FN_MAX_VEC = 8;   // float4 chunks per thread: d_model <= 8192

// One CTA per row; every load of the row is issued before the first use (the loads come from L2
// right after the producing GEMM, so their latency dominates).  x is written back only when it
// changes (embedding rows on the first layer, or split-K partials added).
__global__ void __launch_bounds__(FN_THREADS) fin_norm_kernel(float* __restrict__ x, const uint16_t* __restrict__ init,
                                                              const float* __restrict__ part, int n_split,
                                                              const uint16_t* __restrict__ g, uint16_t* __restrict__ a_hi,
                                                              uint16_t* __restrict__ a_lo, float* __restrict__ rs_out,
                                                              int B, int d, float eps) {
  __shared__ float red[FN_THREADS / 32];
  pdl_trigger();
  const int r = blockIdx.x;
  const int nv = d / 4;
  // the gain is a weight (no kernel writes it): loaded before the dependency wait
  uint2 gw[FN_MAX_VEC];
#pragma unroll
  for (int j = 0; j < FN_MAX_VEC; ++j) {
    const int i = threadIdx.x + j * FN_THREADS;
    gw[j] = i < nv ? *reinterpret_cast<const uint2*>(g + 4 * i) : make_uint2(0, 0);
  }
  pdl_wait();
  float4 v[FN_MAX_VEC];
#pragma unroll
  for (int j = 0; j < FN_MAX_VEC; ++j) {
    const int i = threadIdx.x + j * FN_THREADS;
    v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < nv) {
      if (init) {
        const uint2 w = *reinterpret_cast<const uint2*>(init + (int64_t)r * d + 4 * i);
        v[j] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                           __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
      } else {
        v[j] = *reinterpret_cast<const float4*>(x + (int64_t)r * d + 4 * i);
      }
    }
  }
  const bool write_x = init != nullptr || n_split > 0;
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < FN_MAX_VEC; ++j) {
    const int i = threadIdx.x + j * FN_THREADS;
    if (i < nv) {
      for (int s = 0; s < n_split; ++s) {
        const float4 w = *reinterpret_cast<const float4*>(part + ((int64_t)s * B + r) * d + 4 * i);
        v[j].x += w.x; v[j].y += w.y; v[j].z += w.z; v[j].w += w.w;
      }
      if (write_x && in_extent((int64_t)r * d + 4 * i, 4, (int64_t)B * d))
        *reinterpret_cast<float4*>(x + (int64_t)r * d + 4 * i) = v[j];
      ss = fmaf(v[j].x, v[j].x, ss);
      ss = fmaf(v[j].y, v[j].y, ss);
      ss = fmaf(v[j].z, v[j].z, ss);
      ss = fmaf(v[j].w, v[j].w, ss);
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
  if (threadIdx.x == 0 && in_extent(r, 1, B)) rs_out[r] = rs;
#pragma unroll
  for (int j = 0; j < FN_MAX_VEC; ++j) {
    const int i = threadIdx.x + j * FN_THREADS;
    if (i < nv) {
      const float y[4] = {v[j].x * __uint_as_float(gw[j].x << 16), v[j].y * __uint_as_float(gw[j].x & 0xFFFF0000u),
                          v[j].z * __uint_as_float(gw[j].y << 16), v[j].w * __uint_as_float(gw[j].y & 0xFFFF0000u)};
      uint16_t hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) split_bf16(y[k], hi[k], lo[k]);
      if (!in_extent((int64_t)r * d + 4 * i, 4, (int64_t)B * d)) continue;   // a_hi, a_lo: [B, d] each
      *reinterpret_cast<uint2*>(a_hi + (int64_t)r * d + 4 * i) =
          make_uint2((uint32_t)hi[0] | ((uint32_t)hi[1] << 16), (uint32_t)hi[2] | ((uint32_t)hi[3] << 16));
      *reinterpret_cast<uint2*>(a_lo + (int64_t)r * d + 4 * i) =
          make_uint2((uint32_t)lo[0] | ((uint32_t)lo[1] << 16), (uint32_t)lo[2] | ((uint32_t)lo[3] << 16));
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
  const int* block_table;  // paged cache: [B, max_pages]; position t goes to page t / 128, row t % 128
  const int* seq_pos;      // paged cache: per-row position of the new token (else all rows at t)
  int max_pages;
  int n_split, B, nq_cols, nkv_cols, hd;
  int64_t cap, t;
  int64_t cache_rows;      // rows of each cache: B * cap, or n_pages * 128 (bounds checks)
  RopeFreq freq[kMaxRopePairs];
};

// One thread per (row, column pair).
__global__ void fin_qkv_kernel(const __grid_constant__ FinQkvParams p) {
  pdl_trigger();
  pdl_wait();
  const int n_cols = p.nq_cols + 2 * p.nkv_cols;
  const int pairs = n_cols / 2;
  const int64_t total = (int64_t)p.B * pairs;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
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
  const int64_t tpos = p.seq_pos ? (int64_t)__ldg(p.seq_pos + r) : p.t;
  const float pos = (float)tpos;
  if (c < p.nq_cols + p.nkv_cols) {       // RoPE on q and k
    const int cc = c < p.nq_cols ? c : c - p.nq_cols;
    float sn, cs;
    rope_sincos(pos, p.freq[(cc % p.hd) >> 1], sn, cs);
    const float x0 = v0, x1 = v1;
    v0 = x0 * cs - x1 * sn;
    v1 = x0 * sn + x1 * cs;
  }
  if (c < p.nq_cols) {
    if (in_extent((int64_t)r * p.nq_cols + c, 2, (int64_t)p.B * p.nq_cols))
      *reinterpret_cast<uint32_t*>(p.q + (int64_t)r * p.nq_cols + c) = pack_bf2(v0, v1);
    continue;
  }
  const bool is_k = c < p.nq_cols + p.nkv_cols;
  const int cc = is_k ? c - p.nq_cols : c - p.nq_cols - p.nkv_cols;
  const int64_t slot = p.block_table ? (int64_t)__ldg(p.block_table + (int64_t)r * p.max_pages + tpos / 128) * 128 + tpos % 128
                                     : (int64_t)r * p.cap + tpos;
  const int64_t off = slot * p.nkv_cols + cc;
  if (!in_extent(off, 2, p.cache_rows * p.nkv_cols)) continue;
  if (p.k_scale) {   // 8-bit cache: code = E4M3(fl32(x) / scale), rounded to nearest even, saturating
    const float s = (is_k ? p.k_scale : p.v_scale)[cc / p.hd];
    uint16_t code;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(code) : "f"(v1 / s), "f"(v0 / s));
    *reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(is_k ? p.kc : p.vc) + off) = code;
  } else {
    *reinterpret_cast<uint32_t*>(static_cast<uint16_t*>(is_k ? p.kc : p.vc) + off) = pack_bf2(v0, v1);
  }
  }
}

// Four hidden units per thread (grid-stride): gate in columns [0, d_ff), up in [d_ff, 2 d_ff).
__global__ void fin_swiglu_kernel(const float* __restrict__ part, const float* __restrict__ rs, uint16_t* __restrict__ m_hi,
                                  uint16_t* __restrict__ m_lo, int n_split, int B, int dff) {
  pdl_trigger();
  pdl_wait();
  const int q4 = dff / 4;
  const int64_t total = (int64_t)B * q4;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(idx / q4), j = (int)(idx % q4) * 4;
    float4 gs = make_float4(0.f, 0.f, 0.f, 0.f), us = gs;
    for (int s = 0; s < n_split; ++s) {
      const float* row = part + ((int64_t)s * B + r) * 2 * dff;
      const float4 gv = *reinterpret_cast<const float4*>(row + j);
      const float4 uv = *reinterpret_cast<const float4*>(row + dff + j);
      gs.x += gv.x; gs.y += gv.y; gs.z += gv.z; gs.w += gv.w;
      us.x += uv.x; us.y += uv.y; us.z += uv.z; us.w += uv.w;
    }
    const float sc = rs[r];
    uint16_t h0, h1, h2, h3, l0, l1, l2, l3;
    split_bf16(silu_f(gs.x * sc) * (us.x * sc), h0, l0);
    split_bf16(silu_f(gs.y * sc) * (us.y * sc), h1, l1);
    split_bf16(silu_f(gs.z * sc) * (us.z * sc), h2, l2);
    split_bf16(silu_f(gs.w * sc) * (us.w * sc), h3, l3);
    const int64_t o = (int64_t)r * dff + j;
    if (!in_extent(o, 4, (int64_t)B * dff)) continue;   // m_hi, m_lo: [B, d_ff] each
    *reinterpret_cast<uint2*>(m_hi + o) = make_uint2((uint32_t)h0 | ((uint32_t)h1 << 16), (uint32_t)h2 | ((uint32_t)h3 << 16));
    *reinterpret_cast<uint2*>(m_lo + o) = make_uint2((uint32_t)l0 | ((uint32_t)l1 << 16), (uint32_t)l2 | ((uint32_t)l3 << 16));
  }
}

}  // namespace

int launch_fin_norm(float* x, const void* init_bf16, const float* part, int n_split, const void* g, void* a_hi,
                    void* a_lo, float* rs, int B, int d, float eps, cudaStream_t st) {
  if (d % 4 || d > FN_THREADS * FN_MAX_VEC * 4) return -1;
  return launch_k(fin_norm_kernel, dim3(B), dim3(FN_THREADS), 0, st, x, static_cast<const uint16_t*>(init_bf16), part,
                  n_split, static_cast<const uint16_t*>(g), static_cast<uint16_t*>(a_hi), static_cast<uint16_t*>(a_lo),
                  rs, B, d, eps) == cudaSuccess ? 0 : -1;
}

int launch_fin_qkv(const float* part, int n_split, const float* rs, void* q, void* kc, void* vc, int B, int nq_cols,
                   int nkv_cols, int hd, int64_t cap, int64_t t, const RopeFreq* freq, const float* k_scale,
                   const float* v_scale, const int* block_table, int max_pages, const int* seq_pos,
                   int64_t n_pages, cudaStream_t st) {
  FinQkvParams p;
  p.part = part; p.rs = rs;
  p.q = static_cast<uint16_t*>(q); p.kc = kc; p.vc = vc;
  p.k_scale = k_scale; p.v_scale = v_scale;
  p.block_table = block_table; p.max_pages = max_pages; p.seq_pos = seq_pos;
  p.n_split = n_split; p.B = B; p.nq_cols = nq_cols; p.nkv_cols = nkv_cols; p.hd = hd; p.cap = cap; p.t = t;
  p.cache_rows = block_table ? n_pages * 128 : (int64_t)B * cap;
  for (int i = 0; i < hd / 2; ++i) p.freq[i] = freq[i];
  const int64_t n = (int64_t)B * (nq_cols + 2 * nkv_cols) / 2;
  // one thread per pair: B * 3 * 1024 threads at most for the shapes of the decode path, which
  // are resident at once (the next kernel of the stream can launch early)
  return launch_k(fin_qkv_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, p) == cudaSuccess ? 0 : -1;
}

int launch_fin_swiglu(const float* part, int n_split, const float* rs, void* m_hi, void* m_lo, int B, int dff,
                      cudaStream_t st) {
  if (dff % 4) return -1;
  const int64_t n = (int64_t)B * dff / 4;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, 2 * num_sms()));
  return launch_k(fin_swiglu_kernel, dim3(grid), dim3(256), 0, st, part, rs,
                  static_cast<uint16_t*>(m_hi), static_cast<uint16_t*>(m_lo), n_split, B, dff) == cudaSuccess ? 0 : -1;
}

LLAMA_DEFINE_BOUNDS_READER(decode_fin)

}  // namespace llama
