// CUDA-core kernels: RMSNorm (the one used on every path), RoPE, and the generic GEMM and
// attention used for float32 and for bf16 shapes the tcgen05 kernels do not take.
#include <algorithm>
#include <cstring>

#include "epilogue.cuh"
#include "kernels.h"

namespace llama {
namespace {

// ------------------------------------------------------------------------------------------
// RMSNorm: y = x * rsqrt(mean(x^2) + eps) * g  ("Llama Architecture ...", Mathematical
// Foundations 1 with eps inside the root as its Step 1 code has it; RMSNorm study note, "How
// it works").  One warp per row, fp32 sum of squares, 128-bit loads; the row stays in
// registers between the reduction and the scaling pass (CH 16-byte chunks per lane).
// ------------------------------------------------------------------------------------------
// N consecutive elements <-> floats, one vector access (p aligned to N * sizeof(T)).
template <typename T, int N> struct VecIO;
template <> struct VecIO<float, 4> {
  static __device__ __forceinline__ void ld(const float* p, float* f) {
    const float4 w = __ldg(reinterpret_cast<const float4*>(p));
    f[0] = w.x; f[1] = w.y; f[2] = w.z; f[3] = w.w;
  }
  static __device__ __forceinline__ void st(float* p, const float* f) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(f[0], f[1], f[2], f[3]));
  }
};
template <> struct VecIO<uint16_t, 8> {
  static __device__ __forceinline__ void ld(const uint16_t* p, float* f) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = __uint_as_float(u[j] << 16);
      f[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
    }
  }
  static __device__ __forceinline__ void st(uint16_t* p, const float* f) {
    __stcs(reinterpret_cast<uint4*>(p),
           make_uint4(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]), pack_bf2(f[4], f[5]), pack_bf2(f[6], f[7])));
  }
};
template <> struct VecIO<uint16_t, 4> {
  static __device__ __forceinline__ void ld(const uint16_t* p, float* f) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
    f[0] = __uint_as_float(w.x << 16); f[1] = __uint_as_float(w.x & 0xFFFF0000u);
    f[2] = __uint_as_float(w.y << 16); f[3] = __uint_as_float(w.y & 0xFFFF0000u);
  }
  static __device__ __forceinline__ void st(uint16_t* p, const float* f) {
    __stcs(reinterpret_cast<uint2*>(p), make_uint2(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3])));
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// The N = 16 / sizeof(T) elements of a 16-byte value (held in registers) as floats.
__device__ __forceinline__ void unpack16(const uint4& w, float* f, float) {
  f[0] = __uint_as_float(w.x); f[1] = __uint_as_float(w.y); f[2] = __uint_as_float(w.z); f[3] = __uint_as_float(w.w);
}
__device__ __forceinline__ void unpack16(const uint4& w, float* f, uint16_t) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(u[j] << 16);
    f[2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
  }
}

// One warp per row; the row is held in registers (CH 16-byte chunks per lane) between the
// sum of squares and the scaling pass.  SPLIT: write a = x * g and rs[row] = rsqrt(mean(x^2)+eps)
// instead of y = x * rs * g, for a consumer GEMM that applies rs to its fp32 accumulator.
// (rows 8 * bid .. 8 * bid + 7 for a block of 256 threads)
template <typename TX, typename TG, typename TY, int CH, bool SPLIT>
__device__ __forceinline__ void rmsnorm_reg_rows(const TX* __restrict__ x, const TG* __restrict__ g,
                                                 TY* __restrict__ y, float* __restrict__ rs_out, int64_t rows, int d,
                                                 float eps, int64_t bid) {
  constexpr int N = 16 / (int)sizeof(TX);
  const int lane = threadIdx.x & 31;
  const int64_t row = bid * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int nch = d / N;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * d);
  uint4 buf[CH];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    const int c = lane + 32 * i;
    if (c < nch) {
      buf[i] = __ldcs(xr + c);   // streamed once: keep it out of L1
      float f[N];
      unpack16(buf[i], f, TX());
#pragma unroll
      for (int j = 0; j < N; ++j) ss = fmaf(f[j], f[j], ss);
    }
  }
  ss = warp_sum(ss);
  const float rs = rsqrtf(ss / (float)d + eps);
  if (SPLIT && lane == 0 && in_extent(row, 1, rows)) rs_out[row] = rs;
  const float mul = SPLIT ? 1.f : rs;
  TY* yr = y + row * d;
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    const int c = lane + 32 * i;
    if (c < nch && in_extent(row * d + c * N, N, rows * d)) {
      float f[N], w[N];
      unpack16(buf[i], f, TX());
      VecIO<TG, N>::ld(g + c * N, w);
#pragma unroll
      for (int j = 0; j < N; ++j) f[j] = f[j] * mul * w[j];
      VecIO<TY, N>::st(yr + c * N, f);
    }
  }
}

template <typename TX, typename TG, typename TY, int CH, bool SPLIT>
__global__ void __launch_bounds__(256) rmsnorm_reg_kernel(const TX* __restrict__ x, const TG* __restrict__ g,
                                                          TY* __restrict__ y, float* __restrict__ rs_out,
                                                          int64_t rows, int d, float eps) {
  rmsnorm_reg_rows<TX, TG, TY, CH, SPLIT>(x, g, y, rs_out, rows, d, eps, blockIdx.x);
}

// Any width, any alignment.  Two passes over the row.
template <typename TX, typename TG, typename TY, bool SPLIT>
__global__ void __launch_bounds__(256) rmsnorm_generic_kernel(const TX* __restrict__ x, const TG* __restrict__ g,
                                                              TY* __restrict__ y, float* __restrict__ rs_out,
                                                              int64_t rows, int64_t d, float eps) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const TX* xr = x + row * d;
  float ss = 0.f;
  for (int64_t c = lane; c < d; c += 32) {
    const float f = Elt<TX>::ld(xr + c);
    ss = fmaf(f, f, ss);
  }
  ss = warp_sum(ss);
  const float rs = rsqrtf(ss / (float)d + eps);
  if (SPLIT && lane == 0 && in_extent(row, 1, rows)) rs_out[row] = rs;
  const float mul = SPLIT ? 1.f : rs;
  TY* yr = y + row * d;
  for (int64_t c = lane; c < d; c += 32)
    if (in_extent(row * d + c, 1, rows * d)) Elt<TY>::st(yr + c, Elt<TX>::ld(xr + c) * mul * Elt<TG>::ld(g + c));
}

// Streaming RMSNorm for bf16 rows of 1024..4096 elements (multiples of 8): two CTAs per SM, CTA b
// walks rows b, b + G, b + 2G, ...  In each CTA a producer thread keeps a ring of row buffers in
// shared memory filled with bulk TMA copies (one copy per row), and eight consumer warps each take a
// row, form its sum of squares from shared memory, then read it again to write the normalised row
// with streaming stores, and hand the buffer back.  The arithmetic runs on packed fp32 pairs (FFMA2 /
// FMUL2) and a paired bf16 convert, which halves its instruction count: with one instruction per
// element more, the consumers and not HBM set the pace.  Two CTAs (two producers) per SM rather
// than one CTA with a ring twice as deep: measured on this part, one producer per SM left even a
// plain copy ~15% short of HBM bandwidth.  The gain is staged once in shared memory.  Every
// mbarrier wait is bounded (status word, no trap).
constexpr int kRnWarps = 8, kRnThreads = (kRnWarps + 1) * 32;

__device__ __forceinline__ void bulk_load_row(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ float2 bf16x2_lo_hi(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float2 v) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The RoPE table of a block's positions, written by one extra warp of the block's first norm
// (TAB): tab[s][k] = (cos, sin) of (pos0 + s) * theta_k for s < S, k < half.
struct RnTab {
  float2* tab;
  int64_t S, pos0;
  int half;
  RopeFreq freq[kMaxRopePairs];
};

template <int CH, bool SPLIT, bool TAB>
__global__ void __launch_bounds__(kRnThreads + 32, 2) rmsnorm_stream_kernel(const uint16_t* __restrict__ x,
                                                                           const uint16_t* __restrict__ g,
                                                                           uint16_t* __restrict__ y,
                                                                           float* __restrict__ rs_out, int64_t rows,
                                                                           int d, float eps, int nbuf, unsigned* status,
                                                                           const __grid_constant__ RnTab tp) {
  extern __shared__ __align__(128) uint8_t rn_smem[];
  pdl_trigger();
  pdl_wait();   // x may come from the previous kernel; the table is read by the previous call's GEMM
  const uint32_t row_bytes = (uint32_t)d * 2;
  uint4* gs = reinterpret_cast<uint4*>(rn_smem + (size_t)nbuf * row_bytes);   // the gain, d bf16
  uint64_t* full = reinterpret_cast<uint64_t*>(rn_smem + (size_t)(nbuf + 1) * row_bytes);
  uint64_t* empty = full + nbuf;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + nbuf);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t G = gridDim.x, b = blockIdx.x;
  const int64_t my_rows = rows > b ? (rows - b + G - 1) / G : 0;   // rows b, b + G, ...
  if (threadIdx.x == 0) {
    for (int s = 0; s < nbuf; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (TAB && warp == kRnWarps + 1) {   // the RoPE table, beside the norm's memory traffic
    __shared__ RopeFreq fq[kMaxRopePairs];
    for (int k = lane; k < tp.half; k += 32) fq[k] = tp.freq[k];
    __syncwarp();
    const int64_t total = tp.S * tp.half;
    for (int64_t i = (int64_t)blockIdx.x * 32 + lane; i < total; i += (int64_t)gridDim.x * 32) {
      const int64_t sp = i / tp.half;
      const int k = (int)(i - sp * tp.half);
      float sn, cs;
      rope_sincos((float)(tp.pos0 + sp), fq[k], sn, cs);
      if (in_extent(i, 1, total)) tp.tab[i] = make_float2(cs, sn);
    }
    return;
  }
  if (warp == kRnWarps) {
    if (lane == 0) {   // producer
      int64_t issued = 0;
      for (; issued < my_rows; ++issued) {
        const int s = (int)(issued % nbuf);
        const uint32_t ph = (uint32_t)((issued / nbuf) & 1);
        if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, status)) break;
        if (!in_extent((b + issued * G) * (int64_t)d, d, rows * (int64_t)d)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(&full[s], row_bytes);
        bulk_load_row(smem_u32(rn_smem + (size_t)s * row_bytes), x + (b + issued * G) * (int64_t)d, row_bytes,
                      &full[s]);
      }
      // After an abort, let the copies still in flight land (bounded) before the CTA exits.
      volatile int never = 0;
      for (int64_t i = std::max<int64_t>(0, issued - nbuf); i < issued; ++i)
        mbar_wait(&full[i % nbuf], (uint32_t)((i / nbuf) & 1), &never, status);
    }
    return;
  }
  // The producer is already streaming rows while the consumer warps stage the gain (named barrier 1
  // spans the consumer warps only).
  for (int c = threadIdx.x; c < d / 8; c += kRnWarps * 32) gs[c] = __ldg(reinterpret_cast<const uint4*>(g) + c);
  asm volatile("bar.sync 1, %0;" ::"n"(kRnWarps * 32) : "memory");
  const int nch = d / 8;   // 16-byte chunks of a row; lane takes chunks lane, lane + 32, ...
  for (int64_t i = warp; i < my_rows; i += kRnWarps) {
    const int s = (int)(i % nbuf);
    const uint32_t ph = (uint32_t)((i / nbuf) & 1);
    if (!mbar_wait(&full[s], ph, abort_flag, status)) break;
    const uint4* srow = reinterpret_cast<const uint4*>(rn_smem + (size_t)s * row_bytes);
    float2 acc = make_float2(0.f, 0.f);   // even and odd elements
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int c = lane + 32 * k;
      const uint4 v = c < nch ? srow[c] : make_uint4(0, 0, 0, 0);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 t = bf16x2_lo_hi(u[j]);
        acc = __ffma2_rn(t, t, acc);
      }
    }
    const float ss = warp_sum(acc.x + acc.y);
    const float rs = rsqrtf(ss / (float)d + eps);
    const int64_t row = b + i * G;
    if (SPLIT && lane == 0 && in_extent(row, 1, rows)) rs_out[row] = rs;
    const float mul = SPLIT ? 1.f : rs;
    const float2 mul2 = make_float2(mul, mul);
    uint16_t* yr = y + row * (int64_t)d;
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int c = lane + 32 * k;
      if (c < nch && in_extent(row * d + c * 8, 8, rows * (int64_t)d)) {
        const uint4 v = srow[c], w = gs[c];
        const uint32_t u[4] = {v.x, v.y, v.z, v.w}, gw[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = pack_bf16x2(__fmul2_rn(__fmul2_rn(bf16x2_lo_hi(u[j]), mul2), bf16x2_lo_hi(gw[j])));
        __stcs(reinterpret_cast<uint4*>(yr + c * 8), make_uint4(o[0], o[1], o[2], o[3]));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);   // both reads of the buffer are done: it can be refilled
  }
}

template <bool SPLIT, bool TAB>
int rmsnorm_stream_launch(const void* x, const void* g, void* y, float* rs, int64_t rows, int d, float eps,
                          cudaStream_t st, const RnTab& tp) {
  unsigned* status = status_ptr();
  if (!status) return -1;
  const uint32_t row_bytes = (uint32_t)d * 2;
  // Ring depth: a multiple of the consumer warp count, so that row i always lands in a slot that
  // warp i % kRnWarps owns and every slot's phases are awaited, in order, by that one warp.  With any other
  // depth a warp could test a slot whose previous fill, meant for another warp, is still in flight,
  // and the parity wait would pass on that older phase.
  const int nbuf = (int)std::min<uint32_t>(32, (104u * 1024u) / row_bytes - 1) / kRnWarps * kRnWarps;
  if (nbuf < kRnWarps) return -1;
  const size_t smem = (size_t)(nbuf + 1) * row_bytes + (size_t)2 * nbuf * 8 + 16;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(rows, 2 * (int64_t)num_sms()));
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64][3] = {};
  auto go = [&](auto kernel, int idx) -> int {
    if (dev < 0 || dev >= 64) return -1;
    if (!attr_set[dev][idx]) {
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 106 * 1024) != cudaSuccess)
        return -1;
      attr_set[dev][idx] = true;
    }
    return launch_k(kernel, dim3(grid), dim3(kRnThreads + (TAB ? 32 : 0)), smem, st,
                    static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(g), static_cast<uint16_t*>(y), rs,
                    rows, d, eps, nbuf, status, tp) == cudaSuccess ? 0 : -1;
  };
  const int ch = (d / 8 + 31) / 32;
  if (ch <= 4) return go(rmsnorm_stream_kernel<4, SPLIT, TAB>, 0);
  if (ch <= 8) return go(rmsnorm_stream_kernel<8, SPLIT, TAB>, 1);
  return go(rmsnorm_stream_kernel<16, SPLIT, TAB>, 2);
}

// bf16 rows the streaming kernel takes: 16-byte aligned, 1024..4096 wide, at least two per SM
bool rmsnorm_stream_ok(const void* x, const void* g, const void* y, int64_t rows, int64_t d) {
  const bool aligned = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(g) |
                         reinterpret_cast<uintptr_t>(y)) & 15) == 0;
  return aligned && d % 8 == 0 && d >= 1024 && d <= 4096 && rows >= 2 * 152;
}

template <typename TX, typename TG, typename TY, bool SPLIT>
int rmsnorm_dispatch(const void* xv, const void* gv, void* yv, float* rs, int64_t rows, int64_t d, float eps,
                     cudaStream_t st) {
  constexpr int N = 16 / (int)sizeof(TX);
  const TX* x = static_cast<const TX*>(xv);
  const TG* g = static_cast<const TG*>(gv);
  TY* y = static_cast<TY*>(yv);
  const unsigned grid = (unsigned)((rows + 7) / 8);
  const bool aligned = ((reinterpret_cast<uintptr_t>(xv) | reinterpret_cast<uintptr_t>(gv) |
                         reinterpret_cast<uintptr_t>(yv)) & 15) == 0;
  const int64_t per_lane = (d / N + 31) / 32;
  if (aligned && d % N == 0 && per_lane <= 32) {
    if (per_lane <= 1) rmsnorm_reg_kernel<TX, TG, TY, 1, SPLIT><<<grid, 256, 0, st>>>(x, g, y, rs, rows, (int)d, eps);
    else if (per_lane <= 2) rmsnorm_reg_kernel<TX, TG, TY, 2, SPLIT><<<grid, 256, 0, st>>>(x, g, y, rs, rows, (int)d, eps);
    else if (per_lane <= 4) rmsnorm_reg_kernel<TX, TG, TY, 4, SPLIT><<<grid, 256, 0, st>>>(x, g, y, rs, rows, (int)d, eps);
    else if (per_lane <= 8) rmsnorm_reg_kernel<TX, TG, TY, 8, SPLIT><<<grid, 256, 0, st>>>(x, g, y, rs, rows, (int)d, eps);
    else if (per_lane <= 16) rmsnorm_reg_kernel<TX, TG, TY, 16, SPLIT><<<grid, 256, 0, st>>>(x, g, y, rs, rows, (int)d, eps);
    else rmsnorm_reg_kernel<TX, TG, TY, 32, SPLIT><<<grid, 256, 0, st>>>(x, g, y, rs, rows, (int)d, eps);
  } else {
    rmsnorm_generic_kernel<TX, TG, TY, SPLIT><<<grid, 256, 0, st>>>(x, g, y, rs, rows, d, eps);
  }
  return 0;
}

// ------------------------------------------------------------------------------------------
// RoPE in place on q [B,S,n_q,hd] and k [B,S,n_kv,hd]; one thread per pair.
// ------------------------------------------------------------------------------------------
struct RopeParams {
  void* q;
  void* k;
  int64_t B, S, n_q, n_kv, pos0;
  int hd;
  RopeFreq freq[kMaxRopePairs];
};

template <typename T>
__global__ void rope_kernel(const __grid_constant__ RopeParams p) {
  __shared__ RopeFreq freq[kMaxRopePairs];
  stage_freq(p.freq, p.hd / 2, freq);
  const int64_t half = p.hd / 2;
  const int64_t nq_pairs = p.B * p.S * p.n_q * half;
  const int64_t nk_pairs = p.B * p.S * p.n_kv * half;
  const int64_t total = nq_pairs + (p.k ? nk_pairs : 0);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    T* base;
    int64_t idx, heads, pairs;
    if (i < nq_pairs && p.q) { base = static_cast<T*>(p.q); idx = i; heads = p.n_q; pairs = nq_pairs; }
    else if (i >= nq_pairs) { base = static_cast<T*>(p.k); idx = i - nq_pairs; heads = p.n_kv; pairs = nk_pairs; }
    else continue;
    const int kk = (int)(idx % half);
    const int64_t token = idx / half / heads;
    const float pos = (float)(p.pos0 + token % p.S);
    float s, c;
    rope_sincos(pos, freq[kk], s, c);
    T* e = base + 2 * idx;
    if (!in_extent(2 * idx, 2, 2 * pairs)) continue;
    const float x0 = Elt<T>::ld(e), x1 = Elt<T>::ld(e + 1);
    Elt<T>::st(e, x0 * c - x1 * s);
    Elt<T>::st(e + 1, x0 * s + x1 * c);
  }
}

// ------------------------------------------------------------------------------------------
// Generic GEMM D = A B^T (fp32 accumulation), 64x64 tiles, 256 threads, 4x4 per thread.
// ------------------------------------------------------------------------------------------
constexpr int SB = 64, SK = 16;

template <typename T>
__device__ __forceinline__ const T* b_row(const GemmDesc& g, int64_t n) {
  int64_t off = n;
  for (int s = 0; s < g.nseg; ++s) {
    if (off < g.nB[s]) return static_cast<const T*>(g.B[s]) + off * g.K;
    off -= g.nB[s];
  }
  return nullptr;
}

template <typename T, bool SWIGLU>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const __grid_constant__ GemmDesc g) {
  __shared__ float As[SK][SB];
  __shared__ float Bs[SK][SB];
  __shared__ float Us[SK][SB];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t m0 = (int64_t)blockIdx.y * SB, n0 = (int64_t)blockIdx.x * SB;
  const int64_t Nout = SWIGLU ? g.nB[0] : g.N;
  float acc[4][4] = {}, accu[4][4] = {};
  const T* A = static_cast<const T*>(g.A);
  for (int64_t k0 = 0; k0 < g.K; k0 += SK) {
    for (int i = threadIdx.x; i < SB * SK; i += 256) {
      const int mm = i / SK, kk = i % SK;
      const int64_t r = m0 + mm, k = k0 + kk;
      As[kk][mm] = (r < g.M && k < g.K) ? Elt<T>::ld(A + r * g.lda + k) : 0.f;
      const int64_t n = n0 + mm;
      float bv = 0.f, uv = 0.f;
      if (n < Nout && k < g.K) {
        if (SWIGLU) {
          bv = Elt<T>::ld(static_cast<const T*>(g.B[0]) + n * g.K + k);
          uv = Elt<T>::ld(static_cast<const T*>(g.B[1]) + n * g.K + k);
        } else {
          bv = Elt<T>::ld(b_row<T>(g, n) + k);
        }
      }
      Bs[kk][mm] = bv;
      if (SWIGLU) Us[kk][mm] = uv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SK; ++kk) {
      float a[4], b[4], u[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Bs[kk][tx * 4 + i]; if (SWIGLU) u[i] = Us[kk][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if (SWIGLU) accu[i][j] = fmaf(a[i], u[j], accu[i][j]);
        }
    }
    __syncthreads();
  }
  for (int i = 0; i < 4; ++i) {
    const int64_t r = m0 + ty * 4 + i;
    if (r >= g.M) continue;
    for (int j = 0; j < 4; j += 2) {
      const int64_t c = n0 + tx * 4 + j;
      if (c + 1 < Nout) {
        float v[2] = {acc[i][j], acc[i][j + 1]};
        float u[2] = {accu[i][j], accu[i][j + 1]};
        epi_run<2>(g.epi, r, c, v, u);
      } else if (c < Nout) {     // odd tail column (no RoPE pair can straddle: hd is even)
        float v[1] = {acc[i][j]};
        float u[1] = {accu[i][j]};
        epi_run<1>(g.epi, r, c, v, u);
      }
    }
  }
}

// ------------------------------------------------------------------------------------------
// Generic causal GQA attention: one warp per (b, s, h) query row, 32 keys per step (one per
// lane), online softmax (running max and sum), output dims split across lanes.
// ------------------------------------------------------------------------------------------
// Block (half, rows): thread (k, y) writes pair k of position blockIdx.x * rows + y.
__global__ void rope_table_kernel(float2* __restrict__ tab, int64_t S, int half, int64_t pos0,
                                  const __grid_constant__ RopeParams p) {
  __shared__ RopeFreq freq[kMaxRopePairs];
  stage_freq(p.freq, half, freq);
  const int k = threadIdx.x;
  const int64_t s = (int64_t)blockIdx.x * blockDim.y + threadIdx.y;
  if (s >= S) return;
  float sn, cs;
  rope_sincos((float)(pos0 + s), freq[k], sn, cs);
  if (in_extent(s * half + k, 1, S * half)) tab[s * half + k] = make_float2(cs, sn);
}

// The split-form RMSNorm of bf16 rows (CH 16-byte chunks per lane) and the RoPE table of the
// same call in one launch, so that the table's arithmetic runs beside the norm's memory traffic
// instead of in a launch of its own.  Blocks come in groups of K norm blocks (8 rows each, as in
// rmsnorm_reg_kernel) and one table block (kTabPasses x 256 / half positions), so table blocks
// are dispatched throughout the norm; the norm blocks left over follow the groups.
constexpr int kTabPasses = 8;
template <int CH>
__global__ void __launch_bounds__(256) rmsnorm_rope_table_kernel(const uint16_t* __restrict__ x,
                                                                 const uint16_t* __restrict__ g,
                                                                 uint16_t* __restrict__ y, float* __restrict__ rs_out,
                                                                 int64_t rows, int d, float eps, int K, int tab_blocks,
                                                                 float2* __restrict__ tab, int64_t S, int half,
                                                                 int64_t pos0, const __grid_constant__ RopeParams p) {
  pdl_trigger();
  pdl_wait();   // x may come from the previous kernel; the table is read by the previous call's GEMM
  const int b = blockIdx.x;
  const int lead = tab_blocks * (K + 1);
  int norm_idx = -1, tab_idx = -1;
  if (b < lead) {
    const int grp = b / (K + 1), pos = b - grp * (K + 1);
    if (pos == K) tab_idx = grp;
    else norm_idx = grp * K + pos;
  } else {
    norm_idx = tab_blocks * K + (b - lead);
  }
  if (norm_idx >= 0) {   // block-uniform
    rmsnorm_reg_rows<uint16_t, uint16_t, uint16_t, CH, true>(x, g, y, rs_out, rows, d, eps, norm_idx);
    return;
  }
  __shared__ RopeFreq freq[kMaxRopePairs];
  stage_freq(p.freq, half, freq);
  const int per = 256 / half;
  const int k = (int)threadIdx.x % half, j = (int)threadIdx.x / half;
  if (j >= per) return;
  for (int pass = 0; pass < kTabPasses; ++pass) {
    const int64_t s = ((int64_t)tab_idx * kTabPasses + pass) * per + j;
    if (s >= S) return;
    float sn, cs;
    rope_sincos((float)(pos0 + s), freq[k], sn, cs);
    if (in_extent(s * half + k, 1, S * half)) tab[s * half + k] = make_float2(cs, sn);
  }
}

__global__ void widen_bf16_kernel(const uint16_t* __restrict__ src, float* __restrict__ dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    if (in_extent(i, 1, n)) dst[i] = bf2f(src[i]);
}

template <typename T>
__global__ void __launch_bounds__(128) attn_simt_kernel(const __grid_constant__ AttnDesc a) {
  extern __shared__ float qs[];                       // [4 warps][hd]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 4 + warp;  // (b*S + s)*n_q + h
  const int64_t rows = a.B * a.S * a.n_q;
  if (row >= rows) return;
  const int hd = (int)a.hd;
  const int64_t h = row % a.n_q, bs = row / a.n_q, s = bs % a.S, b = bs / a.S;
  const int64_t grp = h / (a.n_q / a.n_kv);
  const int64_t pos = a.pos0 + s;
  float* q = qs + warp * hd;
  const T* qrow = static_cast<const T*>(a.q) + row * hd;
  for (int i = lane; i < hd; i += 32) q[i] = Elt<T>::ld(qrow + i) * a.scale;
  __syncwarp();
  const T* K = static_cast<const T*>(a.k) + (b * a.cap * a.n_kv + grp) * hd;
  const T* V = static_cast<const T*>(a.v) + (b * a.cap * a.n_kv + grp) * hd;
  const int64_t kstride = a.n_kv * hd;
  float m = -INFINITY, l = 0.f;
  float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // dims lane + 32*i
  for (int64_t j0 = 0; j0 <= pos; j0 += 32) {
    const int64_t j = j0 + lane;
    float sc = -INFINITY;
    if (j <= pos) {
      const T* kr = K + j * kstride;
      float acc = 0.f;
      for (int t = 0; t < hd; ++t) acc = fmaf(q[t], Elt<T>::ld(kr + t), acc);
      sc = acc;
    }
    const float mnew = fmaxf(m, warp_max(sc));
    const float alpha = __expf(m - mnew);             // m = -inf on the first block -> 0
    const float p = (j <= pos) ? expf(sc - mnew) : 0.f;
    l = l * alpha + warp_sum(p);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] *= alpha;
    const int nk = (pos + 1 - j0) < 32 ? (int)(pos + 1 - j0) : 32;
    for (int jj = 0; jj < nk; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      const T* vr = V + (j0 + jj) * kstride;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int t = lane + 32 * i;
        if (t < hd) o[i] = fmaf(pj, Elt<T>::ld(vr + t), o[i]);
      }
    }
    m = mnew;
  }
  const float inv = 1.f / l;
  T* orow = static_cast<T*>(a.o) + row * hd;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = lane + 32 * i;
    if (t < hd && in_extent(row * hd + t, 1, rows * hd)) Elt<T>::st(orow + t, o[i] * inv);
  }
}

}  // namespace

int launch_rmsnorm(int dtype, int x_f32, int y_f32, const void* x, const void* g, void* y, float* rs_out,
                   int64_t rows, int64_t d, float eps, cudaStream_t st) {
  if (rows <= 0) return 0;
  using bf = uint16_t;
  const bool split = rs_out != nullptr;
  if (dtype == LLAMA_F32) {
    if (!x_f32 || !y_f32) return -1;
    return split ? rmsnorm_dispatch<float, float, float, true>(x, g, y, rs_out, rows, d, eps, st)
                 : rmsnorm_dispatch<float, float, float, false>(x, g, y, rs_out, rows, d, eps, st);
  }
  if (y_f32) return -1;
  if (x_f32)
    return split ? rmsnorm_dispatch<float, bf, bf, true>(x, g, y, rs_out, rows, d, eps, st)
                 : rmsnorm_dispatch<float, bf, bf, false>(x, g, y, rs_out, rows, d, eps, st);
  // bf16 rows of 1024..4096 elements with 16-byte aligned rows: the streaming kernel
  if (rmsnorm_stream_ok(x, g, y, rows, d)) {
    RnTab none;
    memset(&none, 0, sizeof(none));
    return split ? rmsnorm_stream_launch<true, false>(x, g, y, rs_out, rows, (int)d, eps, st, none)
                 : rmsnorm_stream_launch<false, false>(x, g, y, rs_out, rows, (int)d, eps, st, none);
  }
  return split ? rmsnorm_dispatch<bf, bf, bf, true>(x, g, y, rs_out, rows, d, eps, st)
               : rmsnorm_dispatch<bf, bf, bf, false>(x, g, y, rs_out, rows, d, eps, st);
}

int launch_rope(int dtype, void* q, void* k, int64_t B, int64_t S, int64_t n_q, int64_t n_kv, int hd, int64_t pos0,
                const RopeFreq* freq, cudaStream_t st) {
  RopeParams p;
  p.q = q; p.k = k; p.B = B; p.S = S; p.n_q = n_q; p.n_kv = n_kv; p.pos0 = pos0; p.hd = hd;
  for (int i = 0; i < hd / 2; ++i) p.freq[i] = freq[i];
  const int64_t total = B * S * (n_q + n_kv) * (hd / 2);
  if (total <= 0) return 0;
  const unsigned grid = (unsigned)std::min<int64_t>((total + 255) / 256, 152 * 32);
  if (dtype == LLAMA_F32) rope_kernel<float><<<grid, 256, 0, st>>>(p);
  else rope_kernel<uint16_t><<<grid, 256, 0, st>>>(p);
  return 0;
}

int launch_gemm_simt(const GemmDesc& g, cudaStream_t st) {
  const int64_t nout = g.epi.kind == EPI_SWIGLU ? g.nB[0] : g.N;
  if (g.M <= 0 || nout <= 0) return 0;
  dim3 grid((unsigned)((nout + SB - 1) / SB), (unsigned)((g.M + SB - 1) / SB));
  const bool sw = g.epi.kind == EPI_SWIGLU;
  GemmDesc gd = g;
  epi_set_extents(gd.epi, g.M, g.M);
  if (g.dtype == LLAMA_F32) {
    if (sw) gemm_simt_kernel<float, true><<<grid, 256, 0, st>>>(gd);
    else gemm_simt_kernel<float, false><<<grid, 256, 0, st>>>(gd);
  } else {
    if (sw) gemm_simt_kernel<uint16_t, true><<<grid, 256, 0, st>>>(gd);
    else gemm_simt_kernel<uint16_t, false><<<grid, 256, 0, st>>>(gd);
  }
  return 0;
}

bool rmsnorm_rope_table_ok(const void* x, const void* g, const void* y, int64_t rows, int64_t d, int64_t S, int hd) {
  const int half = hd / 2;
  const bool aligned = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(g) |
                         reinterpret_cast<uintptr_t>(y)) & 15) == 0;
  const int64_t per_lane = (d / 8 + 31) / 32;   // 16-byte chunks (8 bf16) per lane
  return aligned && d % 8 == 0 && per_lane >= 1 && per_lane <= 16 && rows > 0 && S > 0 && half >= 1 &&
         half <= kMaxRopePairs && (rows + 7) / 8 + S < INT32_MAX;
}

int launch_rmsnorm_rope_table(const void* x, const void* g, void* y, float* rs, int64_t rows, int64_t d, float eps,
                              float2* tab, int64_t S, int hd, int64_t pos0, const RopeFreq* freq, cudaStream_t st) {
  if (!rmsnorm_rope_table_ok(x, g, y, rows, d, S, hd)) return -1;
  if (rmsnorm_stream_ok(x, g, y, rows, d)) {   // rows streamed through shared memory, table by a 10th warp
    RnTab tp;
    memset(&tp, 0, sizeof(tp));
    tp.tab = tab;
    tp.S = S;
    tp.pos0 = pos0;
    tp.half = hd / 2;
    for (int i = 0; i < tp.half; ++i) tp.freq[i] = freq[i];
    return rmsnorm_stream_launch<true, true>(x, g, y, rs, rows, (int)d, eps, st, tp);
  }
  const int half = hd / 2;
  const int64_t per_lane = (d / 8 + 31) / 32;
  RopeParams p;
  memset(&p, 0, sizeof(p));
  p.hd = hd;
  for (int i = 0; i < half; ++i) p.freq[i] = freq[i];
  const int norm_blocks = (int)((rows + 7) / 8);
  const int per = 256 / half;
  const int tab_blocks = (int)((S + (int64_t)per * kTabPasses - 1) / ((int64_t)per * kTabPasses));
  const int K = norm_blocks / tab_blocks;   // 0: the table blocks come first
  const dim3 grid((unsigned)(norm_blocks + tab_blocks));
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  const uint16_t* gb = static_cast<const uint16_t*>(g);
  uint16_t* yb = static_cast<uint16_t*>(y);
  if (per_lane <= 4)
    return launch_k(rmsnorm_rope_table_kernel<4>, grid, dim3(256), 0, st, xb, gb, yb, rs, rows, (int)d, eps, K,
                    tab_blocks, tab, S, half, pos0, p) == cudaSuccess ? 0 : -1;
  else if (per_lane <= 8)
    return launch_k(rmsnorm_rope_table_kernel<8>, grid, dim3(256), 0, st, xb, gb, yb, rs, rows, (int)d, eps, K,
                    tab_blocks, tab, S, half, pos0, p) == cudaSuccess ? 0 : -1;
  else
    return launch_k(rmsnorm_rope_table_kernel<16>, grid, dim3(256), 0, st, xb, gb, yb, rs, rows, (int)d, eps, K,
                    tab_blocks, tab, S, half, pos0, p) == cudaSuccess ? 0 : -1;
  return 0;
}

int launch_rope_table(float2* tab, int64_t S, int hd, int64_t pos0, const RopeFreq* freq, cudaStream_t st) {
  RopeParams p;
  memset(&p, 0, sizeof(p));
  p.hd = hd;
  for (int i = 0; i < hd / 2; ++i) p.freq[i] = freq[i];
  const int half = hd / 2;
  if (S <= 0 || half <= 0) return 0;
  const int rows = std::max(1, 256 / half);
  rope_table_kernel<<<(unsigned)((S + rows - 1) / rows), dim3(half, rows), 0, st>>>(tab, S, half, pos0, p);
  return 0;
}

int launch_widen_bf16(const void* src, float* dst, int64_t n, cudaStream_t st) {
  if (n <= 0) return 0;
  const unsigned grid = (unsigned)std::min<int64_t>((n + 255) / 256, 152 * 16);
  widen_bf16_kernel<<<grid, 256, 0, st>>>(static_cast<const uint16_t*>(src), dst, n);
  return 0;
}

int launch_attn_simt(const AttnDesc& a, cudaStream_t st) {
  const int64_t rows = a.B * a.S * a.n_q;
  if (rows <= 0) return 0;
  const unsigned grid = (unsigned)((rows + 3) / 4);
  const size_t smem = 4 * a.hd * sizeof(float);
  if (a.dtype == LLAMA_F32) attn_simt_kernel<float><<<grid, 128, smem, st>>>(a);
  else attn_simt_kernel<uint16_t><<<grid, 128, smem, st>>>(a);
  return 0;
}

LLAMA_DEFINE_BOUNDS_READER(kernels_simt)

}  // namespace llama
