// Split-K GQA decode attention over an 8-bit KV cache: K and V are stored as E4M3 codes with one
// fp32 scale per KV head (x = code * scale), which halves the bytes that bound decode ("LLaMA-3
// 8B ...", section 七 sizes the cache; section 九 has decode read all of it per token).
//
// Same work split as the bf16 kernel (decode_attn.cu): persistent CTAs take (sequence, KV head,
// chunk of 128-key tiles) items, S^T = K Q^T and O^T += V^T P^T run on tcgen05 with the r query
// heads of the group padded to N = 16, and each item leaves an unnormalised partial (m, l, O) for
// the combine pass.  What differs:
//   * TMA brings 128 keys x 128 codes (16 KB) per K or V tile into a 4-stage ring;
//   * the codes are expanded to f16 (exact: every E4M3 value is an f16 value): K by four warps,
//     one key row per thread, straight into tensor memory, where S^T = K Q^T reads its A operand;
//     V by two warps into the 128-byte-swizzled shared-memory layout the P V MMA reads.  Both
//     are double-buffered, so the expansion of tile j + 1 overlaps the MMAs of tile j;
//   * the MMAs run in f16 (kind::f16 with f16 A and B): q is converted from bf16 in place when
//     it lands, P is written as f16;
//   * the K scale multiplies the scores, the V scale the partial O.
#include <algorithm>
#include <cmath>
#include <cstring>

#include <cuda_fp16.h>

#include "kernels.h"

namespace llama {
namespace {

constexpr int D8_THREADS = 384;   // warp 0 TMA, 1 MMA, 2-5 softmax, 6-9 expand K, 10-11 expand V (+ q)
constexpr int D8_STAGES = 4;
constexpr int D8_HD = 128;
constexpr int D8_NPAD = 16;
constexpr uint32_t D8_TMEM_COLS = 256;   // S^T 2 x 16, O^T 16, K (f16, A operand) 2 x 64
constexpr float kD8RescaleLog2 = 8.0f;

struct __align__(64) DecodeAttn8Params {
  CUtensorMap tmK;   // codes [B, kv_len, n_kv, hd] (bytes), box (128, 1, 128, 1)
  CUtensorMap tmV;
  CUtensorMap tmQ;   // bf16 [B, n_q, hd], box (64, r, 1)
  const float* k_scale;   // [n_kv]
  const float* v_scale;   // [n_kv]
  float* part_o;
  float* part_ml;
  int B, n_q, n_kv, r, kv_len, kv_tiles, chunk_tiles, n_chunks, n_items;
  float scale_log2;
  unsigned* status;
};

struct D8Smem {
  static constexpr uint32_t F8 = 128 * D8_HD;              // one code tile: 16 KB
  static constexpr uint32_t H16 = 128 * D8_HD * 2;         // one f16 tile: 32 KB (two 64-column halves)
  static constexpr uint32_t QB = D8_NPAD * D8_HD * 2;      // 4 KB
  static constexpr uint32_t PB = D8_NPAD * 128 * 2;        // 4 KB
  static constexpr uint32_t OFF_K8 = 0;
  static constexpr uint32_t OFF_V8 = OFF_K8 + D8_STAGES * F8;
  static constexpr uint32_t OFF_V16 = OFF_V8 + D8_STAGES * F8;    // 2 buffers
  static constexpr uint32_t OFF_Q = OFF_V16 + 2 * H16;            // 2 buffers
  static constexpr uint32_t OFF_P = OFF_Q + 2 * QB;         // 2 buffers
  static constexpr uint32_t OFF_RED = OFF_P + 2 * PB;       // [3][4][16] floats
  static constexpr uint32_t OFF_BAR = OFF_RED + 3 * 4 * 16 * 4;
  static constexpr uint32_t TOTAL = OFF_BAR + 512 + 1024;
};
static_assert(D8Smem::TOTAL <= 232448, "shared memory");

// barrier slots
enum : int {
  B_K8F = 0, B_V8F = 4, B_K8E = 8, B_V8E = 12, B_K16F = 16, B_K16E = 18, B_V16F = 20, B_V16E = 22,
  B_QF = 24, B_QR = 26, B_QE = 28, B_SF = 30, B_SFREE = 32, B_PF = 34, B_OD = 36, B_OFREE = 38, B_DRAIN = 39,
  B_COUNT = 40
};

__device__ __forceinline__ void tma_load_4d_d8(uint32_t dst, const CUtensorMap* m, uint64_t* bar, int x, int y,
                                               int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_ld16_d8(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void softmax_sync8() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ float warp_max_f32_d8(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// f16 instruction descriptor: D f32, A and B f16 (format 0), K-major unless stated.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool b_mn_major = false, bool a_mn_major = false) {
  return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Four E4M3 codes (one 32-bit word, lowest byte first) to four f16 values (two 32-bit words).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Expand one 128 x 128 code tile (TMA 128-byte swizzle: the 16-byte chunk c of key row k sits at
// chunk c ^ (k & 7)) into the f16 operand layout (two 64-column halves, same swizzle), with the
// 64 threads of the two V warps.
__device__ __forceinline__ void expand_tile(const uint8_t* src, uint8_t* dst, int t64) {
#pragma unroll 4
  for (int u = t64; u < 1024; u += 64) {
    const int k = u >> 3, c = u & 7, sw = k & 7;
    const uint4 w = *reinterpret_cast<const uint4*>(src + k * 128 + ((c ^ sw) << 4));
    uint4 a, b;
    e4m3x4_to_f16x4(w.x, a.x, a.y);
    e4m3x4_to_f16x4(w.y, a.z, a.w);
    e4m3x4_to_f16x4(w.z, b.x, b.y);
    e4m3x4_to_f16x4(w.w, b.z, b.w);
    uint8_t* row = dst + (c >> 2) * 16384 + k * 128;
    const int c0 = 2 * (c & 3);
    *reinterpret_cast<uint4*>(row + ((c0 ^ sw) << 4)) = a;
    *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ sw) << 4)) = b;
  }
}

__device__ __forceinline__ void item_coords8(const DecodeAttn8Params& p, int item, int& b, int& g, int& t_begin,
                                             int& t_end, int& chunk) {
  chunk = item % p.n_chunks;
  const int bg = item / p.n_chunks;
  b = bg / p.n_kv;
  g = bg % p.n_kv;
  t_begin = chunk * p.chunk_tiles;
  t_end = min(t_begin + p.chunk_tiles, p.kv_tiles);
}

template <int R>
__global__ void __launch_bounds__(D8_THREADS, 1) decode_attn8_kernel(const __grid_constant__ DecodeAttn8Params p) {
  using L = D8Smem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(smem + L::OFF_RED);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      int cnt = 1;
      if ((i >= B_V8E && i < B_V8E + D8_STAGES) || i == B_V16F || i == B_V16F + 1 || i == B_QR || i == B_QR + 1)
        cnt = 64;
      if ((i >= B_K8E && i < B_K8E + D8_STAGES) || i == B_K16F || i == B_K16F + 1 || i == B_SFREE ||
          i == B_SFREE + 1 || i == B_PF || i == B_PF + 1 || i == B_OFREE)
        cnt = 128;
      mbar_init(&bars[i], cnt);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmK);
    tma_prefetch_desc(&p.tmV);
    tma_prefetch_desc(&p.tmQ);
  }
  // Q operand rows r..15 and the padded P^T rows stay zero for the whole kernel.
  for (int i = threadIdx.x; i < (int)(2 * L::QB + 2 * L::PB) / 16; i += D8_THREADS)
    reinterpret_cast<uint4*>(smem + L::OFF_Q)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 1) { tmem_alloc(tmem_slot, D8_TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;          // S^T buffers: columns 0..15 and 16..31
  const uint32_t tO = tmem + 32;     // O^T: columns 32..47
  const uint32_t tK = tmem + 64;     // K tiles (f16 pairs): columns 64..127 and 128..191
  const uint32_t sbase = smem_u32(smem);

  pdl_wait();
  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------------- TMA producer
      int tile = 0, it = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x, ++it) {
        int b, g, t0, t1, chunk;
        item_coords8(p, item, b, g, t0, t1, chunk);
        const int qb = it & 1;
        if (!mbar_wait(&bars[B_QE + qb], ((it >> 1) & 1) ^ 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(&bars[B_QF + qb], 2 * 64 * p.r * 2);
        for (int hh = 0; hh < 2; ++hh)
          tma_load_3d(sbase + L::OFF_Q + qb * L::QB + hh * (L::QB / 2), &p.tmQ, &bars[B_QF + qb], hh * 64, g * p.r, b);
        for (int t = t0; t < t1; ++t, ++tile) {
          const int st = tile % D8_STAGES;
          const uint32_t ph = (tile / D8_STAGES) & 1;
          if (!mbar_wait(&bars[B_K8E + st], ph ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&bars[B_K8F + st], L::F8);
          tma_load_4d_d8(sbase + L::OFF_K8 + st * L::F8, &p.tmK, &bars[B_K8F + st], 0, g, t * 128, b);
          if (!mbar_wait(&bars[B_V8E + st], ph ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&bars[B_V8F + st], L::F8);
          tma_load_4d_d8(sbase + L::OFF_V8 + st * L::F8, &p.tmV, &bars[B_V8F + st], 0, g, t * 128, b);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------------------------------------------- MMA issuer
      const uint32_t idesc_s = idesc_f16(128, D8_NPAD);
      const uint32_t idesc_o = idesc_f16(128, D8_NPAD, /*b_mn_major=*/false, /*a_mn_major=*/true);
      const uint32_t va0 = sbase + L::OFF_V16;
      int tile = 0, it = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x, ++it) {
        int b, g, t0, t1, chunk;
        item_coords8(p, item, b, g, t0, t1, chunk);
        const int qb = it & 1;
        if (!mbar_wait(&bars[B_QR + qb], (it >> 1) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t qa = sbase + L::OFF_Q + qb * L::QB;
        const int n = t1 - t0;
        auto issue_s = [&](int j) -> bool {
          const int gt = tile + j;
          const int sb = gt & 1;
          if (!mbar_wait(&bars[B_K16F + sb], (gt >> 1) & 1, abort_flag, p.status)) return false;
          if (!mbar_wait(&bars[B_SFREE + sb], ((gt >> 1) & 1) ^ 1, abort_flag, p.status)) return false;
          tc_fence_after();
          const uint64_t bd0 = sdesc_sw128(qa, 16, 1024);
#pragma unroll
          for (int k = 0; k < D8_HD / 16; ++k)   // A = K from tensor memory, 16 hd per step
            tc_mma_ts(tS + sb * 16, tK + sb * 64 + k * 8,
                      bd0 + (uint64_t)(((k >> 2) * (L::QB / 2) + (k & 3) * 32) >> 4), idesc_s, k > 0 ? 1u : 0u);
          tc_commit(&bars[B_SF + sb]);
          tc_commit(&bars[B_K16E + sb]);
          return true;
        };
        auto issue_pv = [&](int j) -> bool {
          const int gt = tile + j;
          const int pb = gt & 1;
          if (!mbar_wait(&bars[B_PF + pb], (gt >> 1) & 1, abort_flag, p.status)) return false;
          if (!mbar_wait(&bars[B_V16F + pb], (gt >> 1) & 1, abort_flag, p.status)) return false;
          const uint32_t va = va0 + pb * L::H16;
          if (j == 0 && !mbar_wait(&bars[B_OFREE], (it & 1) ^ 1, abort_flag, p.status)) return false;
          tc_fence_after();
          const uint32_t pa = sbase + L::OFF_P + pb * L::PB;
          const uint64_t ad0 = sdesc_sw128(va, 16384, 1024);   // V^T, MN-major
          const uint64_t bd0 = sdesc_sw128(pa, 16, 1024);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            tc_mma(tO, ad0 + (uint64_t)(k * 2048 >> 4), bd0 + (uint64_t)(((k >> 2) * (L::PB / 2) + (k & 3) * 32) >> 4),
                   idesc_o, (j > 0 || k > 0) ? 1u : 0u);
          tc_commit(&bars[B_OD + pb]);
          tc_commit(&bars[B_V16E + pb]);
          return true;
        };
        for (int j = 0; j < n; ++j) {
          if (!issue_s(j)) { ok = false; break; }
          if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
        }
        if (!ok) break;
        tc_commit(&bars[B_QE + qb]);
        if (!issue_pv(n - 1)) break;
        tile += n;
      }
      int no_abort = 0;
      tc_commit(&bars[B_DRAIN]);
      mbar_wait(&bars[B_DRAIN], 0, &no_abort, p.status);
    }
  } else if (warp >= 6 && warp < 10) {  // -------------------------------- K codes -> f16 in TMEM
    const int key = (warp & 3) * 32 + lane;          // this thread's TMEM lane = key row of the tile
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    int tile = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
      int b, g, t0, t1, chunk;
      item_coords8(p, item, b, g, t0, t1, chunk);
      for (int tt = t0; tt < t1; ++tt, ++tile) {
        const int st = tile % D8_STAGES;
        const int hb = tile & 1;
        if (!mbar_wait(&bars[B_K8F + st], (tile / D8_STAGES) & 1, abort_flag, p.status)) { ok = false; break; }
        if (!mbar_wait(&bars[B_K16E + hb], ((tile >> 1) & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint8_t* row = smem + L::OFF_K8 + st * L::F8 + key * 128;
        const int sw = key & 7;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t w[32];
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int c = half * 4 + cc;
            const uint4 v = *reinterpret_cast<const uint4*>(row + ((c ^ sw) << 4));
            e4m3x4_to_f16x4(v.x, w[cc * 8 + 0], w[cc * 8 + 1]);
            e4m3x4_to_f16x4(v.y, w[cc * 8 + 2], w[cc * 8 + 3]);
            e4m3x4_to_f16x4(v.z, w[cc * 8 + 4], w[cc * 8 + 5]);
            e4m3x4_to_f16x4(v.w, w[cc * 8 + 6], w[cc * 8 + 7]);
          }
          tmem_st32(tK + hb * 64 + half * 32 + lane_off, w);
        }
        tc_wait_st();
        tc_fence_before();
        mbar_arrive(&bars[B_K16F + hb]);
        mbar_arrive(&bars[B_K8E + st]);
      }
    }
  } else if (warp >= 10) {  // ------------------------------------ V codes -> f16 in shared memory; q
    const int t64 = (warp & 1) * 32 + lane;
    int tile = 0, it = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x, ++it) {
      int b, g, t0, t1, chunk;
      item_coords8(p, item, b, g, t0, t1, chunk);
      {   // q: bf16 -> f16 in place (same 2-byte layout)
        const int qb = it & 1;
        if (!mbar_wait(&bars[B_QF + qb], (it >> 1) & 1, abort_flag, p.status)) break;
        uint4* q = reinterpret_cast<uint4*>(smem + L::OFF_Q + qb * L::QB);
        for (int i = t64; i < (int)(L::QB / 16); i += 64) {
          uint4 w = q[i];
          uint32_t* e = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(e[j] << 16), hi = __uint_as_float(e[j] & 0xFFFF0000u);
            const __half2 h = __floats2half2_rn(lo, hi);
            e[j] = *reinterpret_cast<const uint32_t*>(&h);
          }
          q[i] = w;
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars[B_QR + qb]);
      }
      for (int tt = t0; tt < t1; ++tt, ++tile) {
        const int st = tile % D8_STAGES;
        const int hb = tile & 1;
        if (!mbar_wait(&bars[B_V8F + st], (tile / D8_STAGES) & 1, abort_flag, p.status)) { ok = false; break; }
        if (!mbar_wait(&bars[B_V16E + hb], ((tile >> 1) & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
        expand_tile(smem + L::OFF_V8 + st * L::F8, smem + L::OFF_V16 + hb * L::H16, t64);
        fence_proxy_async_smem();
        mbar_arrive(&bars[B_V16F + hb]);
        mbar_arrive(&bars[B_V8E + st]);
      }
    }
  } else {  // ------------------------------------------------------------ softmax warps 2..5
    const int qw = warp & 3;
    const int t = qw * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    constexpr int r = R;
    int tile = 0, it = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x, ++it) {
      int b, g, t0, t1, chunk;
      item_coords8(p, item, b, g, t0, t1, chunk);
      const float sc = p.scale_log2 * p.k_scale[g];
      float m_ref[R], lsum[R];
#pragma unroll
      for (int h = 0; h < R; ++h) { m_ref[h] = -INFINITY; lsum[h] = 0.f; }
      for (int tt = t0; tt < t1; ++tt, ++tile) {
        const int sb = tile & 1;
        if (!mbar_wait(&bars[B_SF + sb], (tile >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[16];
        tmem_ld16_d8(tS + sb * 16 + lane_off, sv);
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars[B_SFREE + sb]);
        const bool valid = tt * 128 + t < p.kv_len;
        float s[R];
#pragma unroll
        for (int h = 0; h < R; ++h) s[h] = valid ? __uint_as_float(sv[h]) * sc : -INFINITY;
        float* rbuf = red + (tile & 1) * 64;
#pragma unroll
        for (int h = 0; h < R; ++h) {
          const float v = warp_max_f32_d8(s[h]);
          if (lane == h) rbuf[qw * 16 + h] = v;
        }
        softmax_sync8();
        float alpha[R];
        bool resc = false;
#pragma unroll
        for (int h = 0; h < R; ++h) {
          const float tm = fmaxf(fmaxf(rbuf[h], rbuf[16 + h]), fmaxf(rbuf[32 + h], rbuf[48 + h]));
          alpha[h] = 1.f;
          if (m_ref[h] == -INFINITY) {
            m_ref[h] = tm;
          } else if (tm > m_ref[h] + kD8RescaleLog2) {
            alpha[h] = exp2f(m_ref[h] - tm);
            m_ref[h] = tm;
            resc = true;
          }
        }
        const int pb = tile & 1;
        if (tile >= 2) {
          if (!mbar_wait(&bars[B_OD + pb], ((tile - 2) >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
        }
        if (resc) {
          if (!mbar_wait(&bars[B_OD + ((tile - 1) & 1)], ((tile - 1) >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          uint32_t ov[16];
          tmem_ld16_d8(tO + lane_off, ov);
          tc_wait_ld();
#pragma unroll
          for (int h = 0; h < R; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
          tmem_st16(tO + lane_off, ov);
          tc_wait_st();
#pragma unroll
          for (int h = 0; h < R; ++h) lsum[h] *= alpha[h];
        }
        uint8_t* pbase = smem + L::OFF_P + pb * L::PB + (t >> 6) * (L::PB / 2);
        const int kin = t & 63;
#pragma unroll
        for (int h = 0; h < R; ++h) {
          const float pv = exp2f(s[h] - m_ref[h]);
          const __half pq = __float2half_rn(pv);
          lsum[h] += pv;
          const int chunk16 = (kin >> 3) ^ (h & 7);
          *reinterpret_cast<__half*>(pbase + h * 128 + chunk16 * 16 + (kin & 7) * 2) = pq;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[B_PF + pb]);
      }
      if (!ok) break;
      if (!mbar_wait(&bars[B_OD + ((tile - 1) & 1)], ((tile - 1) >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      uint32_t ov[16];
      tmem_ld16_d8(tO + lane_off, ov);
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars[B_OFREE]);
      const float vs = p.v_scale[g];
      const int64_t base = ((int64_t)b * p.n_chunks + chunk) * p.n_q + (int64_t)g * r;
#pragma unroll
      for (int h = 0; h < R; ++h) p.part_o[(base + h) * D8_HD + t] = __uint_as_float(ov[h]) * vs;
      float* lbuf = red + 128;
#pragma unroll
      for (int h = 0; h < R; ++h) {
        float v = lsum[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == h) lbuf[qw * 16 + h] = v;
      }
      softmax_sync8();
      if (t < r) {
        const float l = lbuf[t] + lbuf[16 + t] + lbuf[32 + t] + lbuf[48 + t];
        float mm = -INFINITY;
#pragma unroll
        for (int h = 0; h < R; ++h) if (h == t) mm = m_ref[h];
        p.part_ml[(base + t) * 2 + 0] = mm;
        p.part_ml[(base + t) * 2 + 1] = l;
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, D8_TMEM_COLS);
  }
}

int launch_decode8_kernel(const DecodeAttn8Params& p, int grid, cudaStream_t st) {
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return -1;
  if (!attr_set[dev]) {
    const void* fns[5] = {(const void*)decode_attn8_kernel<1>, (const void*)decode_attn8_kernel<2>,
                          (const void*)decode_attn8_kernel<4>, (const void*)decode_attn8_kernel<8>,
                          (const void*)decode_attn8_kernel<16>};
    for (const void* f : fns)
      if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, D8Smem::TOTAL) != cudaSuccess) return -1;
    attr_set[dev] = true;
  }
  cudaError_t e;
  switch (p.r) {
    case 1: e = launch_k(decode_attn8_kernel<1>, dim3(grid), dim3(D8_THREADS), D8Smem::TOTAL, st, p); break;
    case 2: e = launch_k(decode_attn8_kernel<2>, dim3(grid), dim3(D8_THREADS), D8Smem::TOTAL, st, p); break;
    case 4: e = launch_k(decode_attn8_kernel<4>, dim3(grid), dim3(D8_THREADS), D8Smem::TOTAL, st, p); break;
    case 8: e = launch_k(decode_attn8_kernel<8>, dim3(grid), dim3(D8_THREADS), D8Smem::TOTAL, st, p); break;
    case 16: e = launch_k(decode_attn8_kernel<16>, dim3(grid), dim3(D8_THREADS), D8Smem::TOTAL, st, p); break;
    default: return -1;
  }
  return e == cudaSuccess ? 0 : -1;
}

__global__ void kv_quantize_kernel(const uint16_t* __restrict__ x, const float* __restrict__ scale, uint8_t* __restrict__ out,
                                   int64_t n8, int n_kv, int hd) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // one group of 8 elements
  if (i >= n8) return;
  const int64_t e0 = i * 8;
  const int head = (int)((e0 / hd) % n_kv);
  const float s = scale[head];
  const uint4 w = *reinterpret_cast<const uint4*>(x + e0);
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  uint32_t packed[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint16_t c[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t pair = in[2 * j + k];
      const float a = __uint_as_float(pair << 16) / s, bb = __uint_as_float(pair & 0xFFFF0000u) / s;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c[k]) : "f"(bb), "f"(a));
    }
    packed[j] = (uint32_t)c[0] | ((uint32_t)c[1] << 16);
  }
  *reinterpret_cast<uint2*>(out + e0) = make_uint2(packed[0], packed[1]);
}

}  // namespace

bool decode_attn8_supported(const AttnDesc& a) {
  if (a.hd != D8_HD || a.S != 1 || a.n_kv <= 0 || a.n_q % a.n_kv != 0) return false;
  const int64_t r = a.n_q / a.n_kv;
  if (r != 1 && r != 2 && r != 4 && r != 8 && r != 16) return false;
  if (a.pos0 + 1 > ((int64_t)1 << 30)) return false;
  const uintptr_t al = reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k) |
                       reinterpret_cast<uintptr_t>(a.v) | reinterpret_cast<uintptr_t>(a.o);
  return (al & 15) == 0;
}

int launch_decode_attn8(const AttnDesc& a, void* ws, int num_sms, unsigned* status, cudaStream_t st) {
  DecodeAttn8Params p;
  memset(&p, 0, sizeof(p));
  const int r = (int)(a.n_q / a.n_kv);
  const int64_t kv_len = a.pos0 + 1;
  int kv_tiles, chunk_tiles, n_chunks;
  decode_attn_plan(kv_len, kv_tiles, chunk_tiles, n_chunks);
  const uint64_t dims[4] = {(uint64_t)D8_HD, (uint64_t)a.n_kv, (uint64_t)kv_len, (uint64_t)a.B};
  const uint64_t strides[3] = {(uint64_t)D8_HD, (uint64_t)a.n_kv * D8_HD, (uint64_t)a.cap * a.n_kv * D8_HD};
  const uint32_t box[4] = {128, 1, 128, 1};
  if (!encode_tmap_4d_u8(&p.tmK, a.k, dims, strides, box)) return -1;
  if (!encode_tmap_4d_u8(&p.tmV, a.v, dims, strides, box)) return -1;
  if (!encode_tmap_3d_bf16(&p.tmQ, a.q, D8_HD, (uint64_t)a.n_q, (uint64_t)a.B, D8_HD * 2,
                           (uint64_t)a.n_q * D8_HD * 2, 64, (uint32_t)r, 1))
    return -1;
  const size_t o_bytes = (((size_t)a.B * n_chunks * a.n_q * D8_HD * 4) + 255) & ~size_t(255);
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.part_o = static_cast<float*>(ws);
  p.part_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + o_bytes);
  p.B = (int)a.B; p.n_q = (int)a.n_q; p.n_kv = (int)a.n_kv; p.r = r;
  p.kv_len = (int)kv_len;
  p.kv_tiles = kv_tiles;
  p.chunk_tiles = chunk_tiles;
  p.n_chunks = n_chunks;
  p.n_items = (int)(a.B * a.n_kv * n_chunks);
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = status;
  const int grid = std::max(1, std::min(p.n_items, num_sms));
  if (launch_decode8_kernel(p, grid, st) != 0) return -1;
  return launch_decode_combine(p.part_o, p.part_ml, a.o, a.o_lo, a.B, a.n_q, n_chunks, st);
}

int launch_kv_quantize(const void* x, const float* scale, void* codes, int64_t n, int n_kv, int hd, cudaStream_t st) {
  const int64_t n8 = n / 8;
  if (n8 == 0) return 0;
  kv_quantize_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, st>>>(static_cast<const uint16_t*>(x), scale,
                                                                   static_cast<uint8_t*>(codes), n8, n_kv, hd);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace llama
