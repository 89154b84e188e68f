// Split-K GQA decode attention over an 8-bit KV cache: K and V are stored as E4M3 codes with one
// fp32 scale per KV head (x = code * scale), which halves the bytes that bound decode ("LLaMA-3
// 8B ...", section 七 sizes the cache; section 九 has decode read all of it per token).
//
// Same work split as the bf16 kernel (decode_attn.cu): persistent CTAs take (sequence, KV head,
// chunk of 128-key tiles) items, S^T = K Q^T and O^T += V^T P^T run on tcgen05, and each item
// leaves an unnormalised partial (m, l, O) for the combine pass.  What differs:
//   * the MMAs read the codes as TMA lands them (kind::f8f6f4, E4M3 A and B, K = 32 per
//     instruction): 4 MMAs for S^T and 4 for O^T per 128-key tile, nothing expanded;
//   * the other operand is E4M3 too, so q and P enter as hi + lo pairs: x = hi + lo with
//     hi = e4m3(x) and lo = e4m3(x - hi), about 8 significant bits, in the N rows 0..r-1 (hi) and
//     r..2r-1 (lo) of an operand padded to N = 16 (32 for r = 16).  An MMA with N = 16 costs as
//     much to issue as one with N = 8, so the lo rows are free; the two column groups of S^T and
//     O^T are summed when read;
//   * q is scaled by a power of two per item so its largest magnitude lands in [128, 256) (E4M3
//     saturates at 448); P is taken as exp2(s - m + 6) with a rescale threshold of 2, so it lies
//     in [0, 256] and keeps ~8 bits down to 2^-7 of the maximum;
//   * the K scale and the inverse q scale multiply the scores, the V scale the partial O.
#include <algorithm>
#include <cmath>
#include <cstring>

#include <cuda_fp16.h>

#include "kernels.h"

namespace llama {
namespace {

constexpr int D8_THREADS = 224;   // warp 0 TMA, 1 MMA, 2-5 softmax, 6 q -> E4M3 hi/lo
// TMA rings, sized so that two CTAs fit on an SM (2 x 100.6 KB of shared memory): with one CTA
// per SM the per-tile hand-offs between the TMA, MMA and softmax roles set the pace, and a second
// CTA overlaps them (3 + 2 stages per CTA moved 6.25 TB/s against 5.32 for 6 + 7 stages in one CTA)
constexpr int D8_KSTAGES = 3;
constexpr int D8_VSTAGES = 2;
constexpr int D8_CTAS_PER_SM = 2;
constexpr int D8_HD = 128;
constexpr uint32_t D8_TMEM_COLS = 128;   // S^T 2 x NP (cols 0..63), O^T NP (cols 64..)
// Lazy rescale: O and l keep the reference maximum until a tile's maximum exceeds it by 2 (log2
// units), so P <= 4 before the 2^6 scale below and P * 2^6 <= 256 stays under E4M3's 448, while
// P down to 2^-7 keeps ~8 significant bits as hi + lo (the scale cancels in O / l).
constexpr float kD8RescaleLog2 = 2.0f;
constexpr float kD8PScaleLog2 = 6.0f;

struct DecodeAttn8Params {   // 128-byte aligned by its tensor maps
  CUtensorMap tmK;   // codes [B, kv_len, n_kv, hd] (bytes), box (128, 1, 128, 1), 128-byte swizzle
  CUtensorMap tmV;
  const uint16_t* q;      // bf16 [B, n_q, hd]
  const float* k_scale;   // [n_kv]
  const float* v_scale;   // [n_kv]
  float* part_o;
  float* part_ml;
  int B, n_q, n_kv, r, kv_len, kv_tiles, chunk_tiles, n_chunks, n_items;
  float scale_log2;
  unsigned* status;
};

struct D8Smem {
  static constexpr uint32_t F8 = 128 * D8_HD;   // one code tile: 128 keys x 128 bytes = 16 KB
  static constexpr uint32_t OPB = 32 * 128;     // q or P operand: up to 32 rows of 128 codes
  static constexpr uint32_t OFF_K8 = 0;
  static constexpr uint32_t OFF_V8 = OFF_K8 + D8_KSTAGES * F8;
  static constexpr uint32_t OFF_Q = OFF_V8 + D8_VSTAGES * F8;  // 2 buffers
  static constexpr uint32_t OFF_P = OFF_Q + 2 * OPB;           // 2 buffers
  static constexpr uint32_t OFF_RED = OFF_P + 2 * OPB;         // [3][4][16] floats
  static constexpr uint32_t OFF_QS = OFF_RED + 3 * 4 * 16 * 4; // inverse q scale per q buffer
  static constexpr uint32_t OFF_BAR = OFF_QS + 16;
  static constexpr uint32_t TOTAL = OFF_BAR + 512 + 1024;
};
static_assert(D8Smem::TOTAL <= 232448, "shared memory");
// the CTAs of an SM share its 228 KB of shared memory (1 KB of it reserved per CTA)
static_assert(D8_CTAS_PER_SM * (D8Smem::TOTAL + 1024) <= 233472, "two CTAs per SM");

// barrier slots
enum : int {
  B_K8F = 0, B_V8F = 6, B_K8E = 13, B_V8E = 19, B_QR = 26, B_QE = 28, B_SF = 30, B_SFREE = 32, B_PF = 34,
  B_OD = 36, B_OFREE = 38, B_DRAIN = 39, B_QC = 40, B_COUNT = 42
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

// Instruction descriptor for kind::f8f6f4 with E4M3 A and B (format 0) and an fp32 accumulator;
// K-major unless stated.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool a_mn_major = false) {
  return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D[tmem] (+)= A[smem] * B[smem]^T on 8-bit operands (K = 32 per instruction), one thread.
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Two floats to two E4M3 codes (round to nearest even, saturating): a in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(b), "f"(a));
  return c;
}
// Two E4M3 codes (low byte first) back to floats.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t c) {
  uint32_t h;
  asm("{\n\t.reg .b16 a;\n\tcvt.u16.u32 a, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\t}" : "=r"(h) : "r"(c));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}
// x = hi + lo in E4M3 (both codes of each pair in one byte, a first): returns hi codes, sets lo codes.
__device__ __forceinline__ uint32_t split_e4m3x2(float a, float b, uint32_t& lo) {
  const uint32_t hi = e4m3x2(a, b);
  const float2 h = e4m3x2_to_f2(hi);
  lo = e4m3x2(a - h.x, b - h.y);
  return hi;
}

// Byte offset of (row n, byte c) in a K-major operand of 128-byte rows with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_off(int n, int c) {
  return (uint32_t)(n * 128 + ((((c >> 4) ^ (n & 7))) << 4) + (c & 15));
}

__device__ __forceinline__ void item_coords8(const DecodeAttn8Params& p, int item, int& b, int& g, int& t_begin,
                                             int& t_end, int& chunk) {
  // heads innermost: the CTAs working at the same time read the n_kv heads of the same keys, so
  // each key's n_kv * 128 contiguous code bytes are fetched together
  g = item % p.n_kv;
  const int bc = item / p.n_kv;
  chunk = bc % p.n_chunks;
  b = bc / p.n_chunks;
  t_begin = chunk * p.chunk_tiles;
  t_end = min(t_begin + p.chunk_tiles, p.kv_tiles);
}

template <int R>
__global__ void __launch_bounds__(D8_THREADS, D8_CTAS_PER_SM) decode_attn8_kernel(const __grid_constant__ DecodeAttn8Params p) {
  using L = D8Smem;
  constexpr int NP = R <= 8 ? 16 : 32;   // operand rows: hi 0..R-1, lo R..2R-1, zero padding
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(smem + L::OFF_RED);
  float* qinv = reinterpret_cast<float*>(smem + L::OFF_QS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      int cnt = 1;
      if (i == B_QR || i == B_QR + 1) cnt = 32;
      if (i == B_SFREE || i == B_SFREE + 1 || i == B_PF || i == B_PF + 1 || i == B_OFREE || i == B_QC ||
          i == B_QC + 1)
        cnt = 128;
      mbar_init(&bars[i], cnt);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmK);
    tma_prefetch_desc(&p.tmV);
  }
  // the padding rows (2R..NP-1) of the q and P operands stay zero for the whole kernel
  for (int i = threadIdx.x; i < (int)(4 * L::OPB) / 16; i += D8_THREADS)
    reinterpret_cast<uint4*>(smem + L::OFF_Q)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 1) { tmem_alloc(tmem_slot, D8_TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;          // S^T buffers: columns 0..NP-1 and NP..2NP-1
  const uint32_t tO = tmem + 64;     // O^T: columns 64..64+NP-1
  const uint32_t sbase = smem_u32(smem);

  // Before the dependency wait the producer starts on the first K stages: the codes of a
  // sequence's tiles before its last are not written by the kernel before this one (the decode
  // step writes only the new position, which lies in the last tile).
  int pre = 0;
  if (warp == 0 && lane == 0) {
    bool stop = false;
    for (int item = blockIdx.x; !stop && pre < D8_KSTAGES && item < p.n_items; item += gridDim.x) {
      int b, g, t0, t1, chunk;
      item_coords8(p, item, b, g, t0, t1, chunk);
      for (int t = t0; t < t1 && pre < D8_KSTAGES; ++t) {
        if (t >= p.kv_tiles - 1) { stop = true; break; }
        if (!box_in(0, D8_HD, g, p.n_kv, (int64_t)t * 128, p.kv_len, b, p.B)) { *abort_flag = 1; stop = true; break; }
        mbar_arrive_expect_tx(&bars[B_K8F + pre], L::F8);
        tma_load_4d_d8(sbase + L::OFF_K8 + pre * L::F8, &p.tmK, &bars[B_K8F + pre], 0, g, t * 128, b);
        ++pre;
      }
    }
  }
  pdl_wait();
  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------------- TMA producer
      // V(j) is requested one tile after K(j): P V needs it only after S^T and the softmax of
      // its tile, so it spends less time resident in its stage and more in flight
      int tile = 0;
      bool ok = true;
      int vb = 0, vg = 0, vt = 0;   // the V tile still to be requested
      auto issue_v = [&](int gt) -> bool {
        const int vs = gt % D8_VSTAGES;
        if (!mbar_wait(&bars[B_V8E + vs], ((gt / D8_VSTAGES) & 1) ^ 1, abort_flag, p.status)) return false;
        if (!box_in(0, D8_HD, vg, p.n_kv, (int64_t)vt * 128, p.kv_len, vb, p.B)) { *abort_flag = 1; return false; }
        mbar_arrive_expect_tx(&bars[B_V8F + vs], L::F8);
        tma_load_4d_d8(sbase + L::OFF_V8 + vs * L::F8, &p.tmV, &bars[B_V8F + vs], 0, vg, vt * 128, vb);
        return true;
      };
      for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x) {
        int b, g, t0, t1, chunk;
        item_coords8(p, item, b, g, t0, t1, chunk);
        for (int t = t0; t < t1; ++t, ++tile) {
          if (tile >= pre) {   // (tiles below pre were issued before the dependency wait)
            const int ks = tile % D8_KSTAGES;
            if (!mbar_wait(&bars[B_K8E + ks], ((tile / D8_KSTAGES) & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
            if (!box_in(0, D8_HD, g, p.n_kv, (int64_t)t * 128, p.kv_len, b, p.B)) { *abort_flag = 1; ok = false; break; }
            mbar_arrive_expect_tx(&bars[B_K8F + ks], L::F8);
            tma_load_4d_d8(sbase + L::OFF_K8 + ks * L::F8, &p.tmK, &bars[B_K8F + ks], 0, g, t * 128, b);
          }
          if (tile > 0 && !issue_v(tile - 1)) { ok = false; break; }
          vb = b; vg = g; vt = t;
        }
      }
      if (ok && tile > 0) issue_v(tile - 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------------------------------------------- MMA issuer
      const uint32_t idesc_s = idesc_e4m3(128, NP);
      const uint32_t idesc_o = idesc_e4m3(128, NP, /*a_mn_major=*/true);
      int tile = 0, it = 0;
      bool ok = true;
      for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x, ++it) {
        int b, g, t0, t1, chunk;
        item_coords8(p, item, b, g, t0, t1, chunk);
        const int qb = it & 1;
        if (!mbar_wait(&bars[B_QR + qb], (it >> 1) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint64_t qd0 = sdesc_sw128(sbase + L::OFF_Q + qb * L::OPB, 16, 1024);
        const int n = t1 - t0;
        auto issue_s = [&](int j) -> bool {
          const int gt = tile + j;
          const int st = gt % D8_KSTAGES, sb = gt & 1;
          if (!mbar_wait(&bars[B_K8F + st], (gt / D8_KSTAGES) & 1, abort_flag, p.status)) return false;
          if (!mbar_wait(&bars[B_SFREE + sb], ((gt >> 1) & 1) ^ 1, abort_flag, p.status)) return false;
          tc_fence_after();
          const uint64_t kd0 = sdesc_sw128(sbase + L::OFF_K8 + st * L::F8, 16, 1024);
#pragma unroll
          for (int k = 0; k < D8_HD / 32; ++k)   // 32 hd (bytes) per step
            tc_mma_f8(tS + sb * NP, kd0 + (uint64_t)(2 * k), qd0 + (uint64_t)(2 * k), idesc_s, k > 0 ? 1u : 0u);
          tc_commit(&bars[B_SF + sb]);
          tc_commit(&bars[B_K8E + st]);
          return true;
        };
        auto issue_pv = [&](int j) -> bool {
          const int gt = tile + j;
          const int st = gt % D8_VSTAGES, pb = gt & 1;
          if (!mbar_wait(&bars[B_PF + pb], (gt >> 1) & 1, abort_flag, p.status)) return false;
          if (!mbar_wait(&bars[B_V8F + st], (gt / D8_VSTAGES) & 1, abort_flag, p.status)) return false;
          if (j == 0 && !mbar_wait(&bars[B_OFREE], (it & 1) ^ 1, abort_flag, p.status)) return false;
          tc_fence_after();
          // V^T: M = hd runs along each 128-byte key row (MN-major), 8-key groups 1024 bytes apart
          const uint64_t vd0 = sdesc_sw128(sbase + L::OFF_V8 + st * L::F8, 16384, 1024);
          const uint64_t pd0 = sdesc_sw128(sbase + L::OFF_P + pb * L::OPB, 16, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k)   // 32 keys per step
            tc_mma_f8(tO, vd0 + (uint64_t)(k * 4096 >> 4), pd0 + (uint64_t)(2 * k), idesc_o,
                      (j > 0 || k > 0) ? 1u : 0u);
          tc_commit(&bars[B_OD + pb]);
          tc_commit(&bars[B_V8E + st]);
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
  } else if (warp == 6) {  // ------------------------------------------- q -> E4M3 hi / lo operand
    constexpr int NCH = R * D8_HD / 8;          // 8-element chunks of the group's q rows
    constexpr int PER = (NCH + 31) / 32;
    int it = 0;
    for (int item = blockIdx.x; item < p.n_items; item += gridDim.x, ++it) {
      int b, g, t0, t1, chunk;
      item_coords8(p, item, b, g, t0, t1, chunk);
      const int qb = it & 1;
      // the buffer is free once the MMAs of item it - 2 have read it and the softmax warps its scale
      if (!mbar_wait(&bars[B_QE + qb], ((it >> 1) & 1) ^ 1, abort_flag, p.status)) break;
      if (!mbar_wait(&bars[B_QC + qb], ((it >> 1) & 1) ^ 1, abort_flag, p.status)) break;
      const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.n_q + (int64_t)g * R) * D8_HD);
      uint4 w[PER];
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int c = lane + 32 * j;
        w[j] = c < NCH ? src[c] : make_uint4(0, 0, 0, 0);
        const uint32_t e[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
          amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(e[k] << 16)), fabsf(__uint_as_float(e[k] & 0xFFFF0000u))));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      // power-of-two scale: amax * qs in [128, 256)
      int ex = 0;
      frexpf(amax, &ex);
      ex = amax > 0.f ? min(max(ex, -100), 100) : 0;
      const float qs = ldexpf(1.f, 8 - ex);
      uint8_t* qop = smem + L::OFF_Q + qb * L::OPB;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int c = lane + 32 * j;
        if (c < NCH) {
          const int h = c / (D8_HD / 8), d = (c % (D8_HD / 8)) * 8;
          const uint32_t e[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            hi[k] = split_e4m3x2(__uint_as_float(e[k] << 16) * qs, __uint_as_float(e[k] & 0xFFFF0000u) * qs, lo[k]);
          *reinterpret_cast<uint2*>(qop + sw128_off(h, d)) =
              make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
          *reinterpret_cast<uint2*>(qop + sw128_off(R + h, d)) =
              make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
        }
      }
      if (lane == 0) qinv[qb] = 1.f / qs;
      fence_proxy_async_smem();
      __syncwarp();
      mbar_arrive(&bars[B_QR + qb]);
    }
  } else if (warp >= 2 && warp < 6) {  // ------------------------------------ softmax warps 2..5
    const int qw = warp & 3;   // a warp reaches TMEM lanes 32 * (warp % 4) ..
    const int t = qw * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    int tile = 0, it = 0;
    bool ok = true;
    for (int item = blockIdx.x; ok && item < p.n_items; item += gridDim.x, ++it) {
      int b, g, t0, t1, chunk;
      item_coords8(p, item, b, g, t0, t1, chunk);
      const int qb = it & 1;
      if (!mbar_wait(&bars[B_QR + qb], (it >> 1) & 1, abort_flag, p.status)) break;
      const float sc = p.scale_log2 * p.k_scale[g] * qinv[qb];
      mbar_arrive(&bars[B_QC + qb]);
      float m_ref[R], lsum[R];
#pragma unroll
      for (int h = 0; h < R; ++h) { m_ref[h] = -INFINITY; lsum[h] = 0.f; }
      for (int tt = t0; tt < t1; ++tt, ++tile) {
        const int sb = tile & 1;
        if (!mbar_wait(&bars[B_SF + sb], (tile >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[NP];
#pragma unroll
        for (int c = 0; c < NP / 16; ++c) tmem_ld16_d8(tS + sb * NP + c * 16 + lane_off, *reinterpret_cast<uint32_t(*)[16]>(sv + 16 * c));
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars[B_SFREE + sb]);
        const bool valid = tt * 128 + t < p.kv_len;
        float s[R];
#pragma unroll
        for (int h = 0; h < R; ++h) s[h] = valid ? (__uint_as_float(sv[h]) + __uint_as_float(sv[R + h])) * sc : -INFINITY;
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
#pragma unroll
          for (int c = 0; c < NP / 16; ++c) {
            uint32_t ov[16];
            tmem_ld16_d8(tO + c * 16 + lane_off, ov);
            tc_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const int col = c * 16 + k;
              if (col < 2 * R) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha[col % R]);
            }
            tmem_st16(tO + c * 16 + lane_off, ov);
          }
          tc_wait_st();
#pragma unroll
          for (int h = 0; h < R; ++h) lsum[h] *= alpha[h];
        }
        // P^T rows: h (hi) and R + h (lo), this thread's key in byte t of each row
        uint8_t* pbase = smem + L::OFF_P + pb * L::OPB;
#pragma unroll
        for (int h = 0; h < R; ++h) {
          const float pv = exp2f(s[h] - (m_ref[h] - kD8PScaleLog2));
          uint32_t lo;
          const uint32_t hi = split_e4m3x2(pv, 0.f, lo);
          const float2 hf = e4m3x2_to_f2(hi), lf = e4m3x2_to_f2(lo);
          lsum[h] += hf.x + lf.x;   // the weights the MMA applies
          pbase[sw128_off(h, t)] = (uint8_t)(hi & 0xFFu);
          pbase[sw128_off(R + h, t)] = (uint8_t)(lo & 0xFFu);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[B_PF + pb]);
      }
      if (!ok) break;
      if (!mbar_wait(&bars[B_OD + ((tile - 1) & 1)], ((tile - 1) >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      uint32_t ov[NP];
#pragma unroll
      for (int c = 0; c < NP / 16; ++c) tmem_ld16_d8(tO + c * 16 + lane_off, *reinterpret_cast<uint32_t(*)[16]>(ov + 16 * c));
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars[B_OFREE]);
      const float vs = p.v_scale[g];
      const int64_t base = ((int64_t)b * p.n_chunks + chunk) * p.n_q + (int64_t)g * R;
      const bool slot_in = in_extent(base, R, (int64_t)p.B * p.n_chunks * p.n_q);   // checking builds
#pragma unroll
      for (int h = 0; h < R; ++h)
        if (slot_in) p.part_o[(base + h) * D8_HD + t] = (__uint_as_float(ov[h]) + __uint_as_float(ov[R + h])) * vs;
      float* lbuf = red + 128;
#pragma unroll
      for (int h = 0; h < R; ++h) {
        float v = lsum[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == h) lbuf[qw * 16 + h] = v;
      }
      softmax_sync8();
      if (t < R && slot_in) {
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
  if (i >= n8 || !in_extent(i * 8, 8, n8 * 8)) return;
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
  p.q = static_cast<const uint16_t*>(a.q);
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
  const int grid = std::max(1, std::min(p.n_items, D8_CTAS_PER_SM * num_sms));
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

LLAMA_DEFINE_BOUNDS_READER(decode_attn8)

}  // namespace llama
