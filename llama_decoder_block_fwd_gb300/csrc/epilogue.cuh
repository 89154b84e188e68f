// GEMM epilogues shared by the CUDA-core and tcgen05 GEMMs.
//
// RoPE ("Llama Architecture ...", Mathematical Foundations 3): the pair (x_2k, x_2k+1) of a
// head turns by m*theta_k:  (x_2k c - x_2k+1 s,  x_2k s + x_2k+1 c),  c, s = cos, sin(m theta_k).
// SwiGLU (same page, Mathematical Foundations 2): SiLU(g) * u with SiLU(z) = z / (1 + e^-z).
#pragma once

#include "kernels.h"

namespace llama {

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

// Store n consecutive values (c % n == 0 for vector paths) of row r into a [*, ld] matrix of
// `extent` elements (checked in -DLLAMA_DEBUG builds: a run outside it is skipped).
template <int n>
__device__ __forceinline__ void store_run(void* base, int is_f32, int64_t ld, int64_t r, int64_t c,
                                          const float* v, int64_t extent) {
  if (!in_extent(r * ld + c, n, extent)) return;
  if (is_f32) {
    float* p = static_cast<float*>(base) + r * ld + c;
    if constexpr (n % 4 == 0) {
#pragma unroll
      for (int i = 0; i < n; i += 4) *reinterpret_cast<float4*>(p + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < n; ++i) p[i] = v[i];
    }
  } else {
    uint16_t* p = static_cast<uint16_t*>(base) + r * ld + c;
    if constexpr (n % 8 == 0) {
#pragma unroll
      for (int i = 0; i < n; i += 8) {
        uint4 w;
        w.x = pack_bf2(v[i], v[i + 1]);
        w.y = pack_bf2(v[i + 2], v[i + 3]);
        w.z = pack_bf2(v[i + 4], v[i + 5]);
        w.w = pack_bf2(v[i + 6], v[i + 7]);
        *reinterpret_cast<uint4*>(p + i) = w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < n; ++i) p[i] = f2bf(v[i]);
    }
  }
}

template <int n>
__device__ __forceinline__ void load_run(const void* base, int is_f32, int64_t ld, int64_t r, int64_t c,
                                         float* v) {
  if (is_f32) {
    const float* p = static_cast<const float*>(base) + r * ld + c;
    if constexpr (n % 4 == 0) {
#pragma unroll
      for (int i = 0; i < n; i += 4) {
        float4 w = *reinterpret_cast<const float4*>(p + i);
        v[i] = w.x; v[i + 1] = w.y; v[i + 2] = w.z; v[i + 3] = w.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < n; ++i) v[i] = p[i];
    }
  } else {
    const uint16_t* p = static_cast<const uint16_t*>(base) + r * ld + c;
    if constexpr (n % 8 == 0) {
#pragma unroll
      for (int i = 0; i < n; i += 8) {
        uint4 w = *reinterpret_cast<const uint4*>(p + i);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[i + 2 * j] = __uint_as_float(u[j] << 16);
          v[i + 2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < n; ++i) v[i] = bf2f(p[i]);
    }
  }
}

// Rotate n/2 consecutive pairs starting at column c (c even) of a head-major row at position pos
// (token s of the call).  With a table, (cos, sin) are read from it; otherwise computed.
template <int n>
__device__ __forceinline__ void rope_run(const Epi& e, int64_t c_in_seg, float pos, int64_t s, float* v) {
  static_assert(n % 2 == 0 || n == 1, "runs of pairs");
  if constexpr (n == 1) return;   // a lone column never carries RoPE (head_dim is even)
  if (n <= e.hd && e.hd % n == 0) {   // the run lies inside one head
    const int k0 = (int)(c_in_seg % e.hd) >> 1;
    if (e.rope_tab) {
      const float2* t = e.rope_tab + s * (e.hd >> 1) + k0;
#pragma unroll
      for (int i = 0; i + 1 < n; i += 2) {
        const float2 cs = __ldg(t + (i >> 1));
        const float x0 = v[i], x1 = v[i + 1];
        v[i] = x0 * cs.x - x1 * cs.y;
        v[i + 1] = x0 * cs.y + x1 * cs.x;
      }
      return;
    }
#pragma unroll
    for (int i = 0; i + 1 < n; i += 2) {
      float sn, co;
      rope_sincos(pos, e.freq[k0 + (i >> 1)], sn, co);
      const float x0 = v[i], x1 = v[i + 1];
      v[i] = x0 * co - x1 * sn;
      v[i + 1] = x0 * sn + x1 * co;
    }
    return;
  }
#pragma unroll
  for (int i = 0; i + 1 < n; i += 2) {
    const int k = (int)((c_in_seg + i) % e.hd) >> 1;
    float sn, co;
    rope_sincos(pos, e.freq[k], sn, co);
    const float x0 = v[i], x1 = v[i + 1];
    v[i] = x0 * co - x1 * sn;
    v[i + 1] = x0 * sn + x1 * co;
  }
}

// Apply the epilogue to n consecutive columns c .. c+n-1 of row r (n even; for EPI_QKV the run
// lies inside one of the Q/K/V column ranges; for EPI_SWIGLU `v` holds gate values and `u` the
// matching up values and c indexes the d_ff output).
// `rs_in` is the row factor when e.ss_in is set (computed once per row by the caller).  Returns
// the sum of squares of the run's output values when e.norm_u is set (else 0).
template <int n>
__device__ __forceinline__ float epi_run(const Epi& e, int64_t r, int64_t c, float* v, float* u, float rs_in = 1.f) {
  float ssq = 0.f;
  if (e.row_scale || e.ss_in) {   // RMSNorm's per-row factor, applied to the fp32 accumulator
    const float rs = e.row_scale ? __ldg(e.row_scale + r) : rs_in;
#pragma unroll
    for (int i = 0; i < n; ++i) v[i] *= rs;
    if (e.kind == EPI_SWIGLU) {
#pragma unroll
      for (int i = 0; i < n; ++i) u[i] *= rs;
    }
  }
  switch (e.kind) {
    case EPI_STORE:
      store_run<n>(e.out, e.out_f32, e.ldo, r, c, v, e.out_rows * e.ldo);
      break;
    case EPI_RESID: {
      float t[n];
      load_run<n>(e.resid, e.resid_f32, e.ldr, r, c, t);
#pragma unroll
      for (int i = 0; i < n; ++i) v[i] += t[i];
      store_run<n>(e.out, e.out_f32, e.ldo, r, c, v, e.out_rows * e.ldo);
      if (e.norm_u) {   // the next RMSNorm's x * g and sum of squares, from the fp32 h
        float gg[n], sq = 0.f;
        load_run<n>(e.norm_g, 0, 0, 0, c, gg);
#pragma unroll
        for (int i = 0; i < n; ++i) {
          sq = fmaf(v[i], v[i], sq);
          gg[i] *= v[i];
        }
        store_run<n>(e.norm_u, 0, e.ldo, r, c, gg, e.M * e.ldo);
        ssq = sq;
      }
      break;
    }
    case EPI_SWIGLU: {
#pragma unroll
      for (int i = 0; i < n; ++i) v[i] = silu_f(v[i]) * u[i];
      store_run<n>(e.out, e.out_f32, e.ldo, r, c, v, e.out_rows * e.ldo);
      break;
    }
    case EPI_ATOMIC: {   // partial sums of a split K range, added into an fp32 buffer
      if (!in_extent(r * e.ldo + c, n, e.out_rows * e.ldo)) break;
      float* p = static_cast<float*>(e.out) + r * e.ldo + c;
      if constexpr (n % 4 == 0) {
#pragma unroll
        for (int i = 0; i < n; i += 4) atomicAdd(reinterpret_cast<float4*>(p + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
      } else {
#pragma unroll
        for (int i = 0; i < n; ++i) atomicAdd(p + i, v[i]);
      }
      break;
    }
    case EPI_QKV: {
      const int64_t s = r % e.S;
      const float pos = (float)(e.pos0 + s);
      if (c < e.nq_cols) {
        rope_run<n>(e, c, pos, s, v);
        store_run<n>(e.out, e.out_f32, e.nq_cols, r, c, v, e.M * e.nq_cols);
      } else {
        const int64_t krow = (r / e.S) * e.cap + e.pos0 + s;
        if (c < e.nq_cols + e.nkv_cols) {
          const int64_t cc = c - e.nq_cols;
          rope_run<n>(e, cc, pos, s, v);
          store_run<n>(e.k_out, e.out_f32, e.nkv_cols, krow, cc, v, (e.M / e.S) * e.cap * e.nkv_cols);
        } else {
          store_run<n>(e.v_out, e.out_f32, e.nkv_cols, krow, c - e.nq_cols - e.nkv_cols, v,
                       (e.M / e.S) * e.cap * e.nkv_cols);
        }
      }
      break;
    }
    default:
      break;
  }
  return ssq;
}

}  // namespace llama
