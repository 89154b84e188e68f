// tcgen05 causal GQA flash attention (prefill, and chunked prefill against a cache).
//
// What it computes ("Llama Architecture ...", Mathematical Foundations 4; "LLaMA-3 8B ...",
// section 四.4): for query head h at absolute position m and its KV head g = h / r,
//     o = sum_j softmax_j(q . k_j / sqrt(hd)) v_j   over keys j <= m.
// The softmax is taken blockwise over 128-key tiles with a running maximum and sum (the
// FlashAttention reformulation the "LLaMA-3 8B" page describes in section 四.4): the result is
// the same up to the order of floating-point additions.
//
// Layout of the work (sm_103a):
//   * A Q tile is 128 rows = (128/r) consecutive tokens x the r query heads of one KV group (one
//     3-D TMA box of Q [B*S, n_q, hd]).  A CTA owns TWO Q tiles of the same group (adjacent token
//     blocks), so each K/V tile staged in shared memory serves 2 x r query heads, and two softmax
//     warp groups take turns with the tensor core.
//   * warp 0 (one thread): TMA loads of both Q tiles once, then K/V tiles (128 keys x hd) into a
//     2-stage ring.  K/V use a 4-D tensor map whose position extent is the number of valid keys.
//   * warp 1 (one thread): per Q tile X and key tile j it issues S_X = Q_X K_j^T (M=128, N=128,
//     K=hd) into TMEM, then, once the softmax has written P_X, O_X += P_X V_j with P_X read from
//     TMEM (it overwrites S_X's columns) and V the MN-major operand, then S_X for tile j+1.
//   * warps 2-5 / 6-9 (one thread per row = TMEM lane, one group per Q tile): read S in two
//     passes (row max, then P = exp2(S*scale*log2e - m)), write P back to TMEM as bf16, keep the
//     running sum, and rescale O in TMEM only when the row max grew by more than 2^8.  At the end
//     they divide O by the sum and store bf16 rows.
// TMEM: S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512).
#include <algorithm>
#include <cstring>

#include "kernels.h"

namespace llama {
namespace {

constexpr int AT_THREADS = 320;
constexpr uint32_t TMEM_COLS_ATTN = 512;
constexpr float kRescaleLog2 = 8.0f;

struct AttnParams {   // 128-byte aligned by its tensor maps
  CUtensorMap tmQ;   // [B*S, n_q, hd], box (64, r, 128/r)
  CUtensorMap tmK;   // [B, kv_len, n_kv, hd], box (64, 1, 128, 1)
  CUtensorMap tmV;
  uint16_t* o;       // [B, S, n_q, hd]
  int B, S, n_q, n_kv, hd, r, tokens_per_tile, t_blocks, pairs;
  int pos0;
  float scale_log2;  // log2(e) / sqrt(hd)
  unsigned* status;
};

template <int HD>
struct Smem {
  static constexpr uint32_t QT = 128 * HD * 2;      // one Q tile
  static constexpr uint32_t KV = 128 * HD * 2;      // one K or V tile
  static constexpr uint32_t OFF_Q = 0;              // 2 Q tiles
  static constexpr uint32_t OFF_K = OFF_Q + 2 * QT; // 2 stages
  static constexpr uint32_t OFF_V = OFF_K + 2 * KV; // 2 stages
  static constexpr uint32_t OFF_BAR = OFF_V + 2 * KV;
  static constexpr uint32_t TOTAL = OFF_BAR + 256 + 1024;
};

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z,
                                            int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x with one MUFU instruction (PTX ex2.approx.ftz: relative error about 2^-22, subnormal
// results flushed to zero -- exact enough for P, which is rounded to bf16).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void tmem_ld16_at(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}

// Packed pairs of fp32 (sm_100 and later): (d0, d1) = (a0 b0 + c0, a1 b1 + c1) in one instruction,
// and (s0, s1) += (a0, a1).
__device__ __forceinline__ void fma_f32x2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                          float c1) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add_f32x2(float& s0, float& s1, float a0, float a1) {
  asm("{\n\t.reg .b64 ra, rs;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rs, {%0, %1};\n\t"
      "add.rn.f32x2 rs, rs, ra;\n\tmov.b64 {%0, %1}, rs;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
}

// 32 scores of a row -> 16 bf16 pairs of P = 2^(s * scale - m) stored at TMEM column `col`; the
// fp32 values are added to the row sums.  The scaling and the sums run on packed pairs.
__device__ __forceinline__ void exp_chunk(const uint32_t (&v)[32], uint32_t col, float scale, float m, float& ls0,
                                          float& ls1) {
  uint32_t w[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    float a0, a1;
    fma_f32x2(a0, a1, __uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]), scale, scale, -m, -m);
    const float p0 = ex2(a0);
    const float p1 = ex2(a1);
    add_f32x2(ls0, ls1, p0, p1);
    w[e] = pack_bf16x2(p0, p1);
  }
  tmem_st16(col, w);
}

template <int HD>
__global__ void __launch_bounds__(AT_THREADS, 1) attn_tc_kernel(const __grid_constant__ AttnParams p) {
  using L = Smem<HD>;
  constexpr int HALVES = HD / 64;          // 64-wide (128-byte) column blocks of Q, K, V
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;     // [2] per stage
  uint64_t* v_full = bars + 3;     // [2]
  uint64_t* kv_empty = bars + 5;   // [2]
  uint64_t* s_full = bars + 7;     // [2] per Q tile
  uint64_t* p_full = bars + 9;     // [2] per Q tile (128 arrivals)
  uint64_t* o_done = bars + 11;    // [2] per Q tile
  uint64_t* drain = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // ---- the two Q tiles: token blocks 2*pair+1 (X=0, the later one, with at least as many key
  //      tiles) and 2*pair (X=1); pairs with the most work run first
  const int groups = p.B * p.n_kv;
  const int pair = p.pairs - 1 - (int)(blockIdx.x / groups);
  const int bg = (int)(blockIdx.x % groups);
  const int b = bg / p.n_kv, g = bg % p.n_kv;
  int t0[2], ntile[2], full_tiles[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int tb = 2 * pair + 1 - x;
    t0[x] = tb * p.tokens_per_tile;
    if (tb >= p.t_blocks) { ntile[x] = 0; full_tiles[x] = 0; continue; }
    const int t_end = min(t0[x] + p.tokens_per_tile, p.S);
    ntile[x] = (p.pos0 + t_end - 1) / 128 + 1;          // key tiles any valid row of the tile sees
    full_tiles[x] = (p.pos0 + t0[x] + 1) / 128;          // tiles entirely visible to every row
  }
  const int nmax = max(ntile[0], ntile[1]);
  const int nq_tiles = (ntile[0] > 0) + (ntile[1] > 0);

  pdl_trigger();   // the next kernel may be scheduled once every CTA of this one has started
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 14; ++i) mbar_init(&bars[i], (i == 9 || i == 10) ? 128 : 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmQ);
    tma_prefetch_desc(&p.tmK);
    tma_prefetch_desc(&p.tmV);
  }
  if (warp == 1) { tmem_alloc(tmem_slot, TMEM_COLS_ATTN); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_u32(smem);
  pdl_wait();   // q, K and V come from the previous kernel

  if (warp == 0) {
    if (lane == 0) {  // ------------------------------------------------ TMA producer
      // bounds-checking builds: every box start inside Q [B*S, n_q, hd] and K/V [B, kv_len, n_kv, hd]
      bool inb = true;
      for (int x = 0; x < 2; ++x)
        if (ntile[x] > 0) inb = inb && box_in(0, HD, (int64_t)g * p.r, p.n_q, (int64_t)b * p.S + t0[x], (int64_t)p.B * p.S);
      if (!inb) *abort_flag = 1;
      if (inb) mbar_arrive_expect_tx(q_full, nq_tiles * L::QT);
      for (int x = 0; x < 2 && inb; ++x) {
        if (ntile[x] == 0) continue;
        for (int hh = 0; hh < HALVES; ++hh)
          tma_load_3d(sbase + L::OFF_Q + x * L::QT + hh * 16384, &p.tmQ, q_full, hh * 64, g * p.r, b * p.S + t0[x]);
      }
      for (int j = 0; j < nmax && inb; ++j) {
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        if (!mbar_wait(&kv_empty[st], ph ^ 1, abort_flag, p.status)) break;
        if (!box_in(0, HD, g, p.n_kv, (int64_t)j * 128, (int64_t)p.pos0 + p.S, b, p.B)) { *abort_flag = 1; break; }
        mbar_arrive_expect_tx(&k_full[st], L::KV);
        for (int hh = 0; hh < HALVES; ++hh)
          tma_load_4d(sbase + L::OFF_K + st * L::KV + hh * 16384, &p.tmK, &k_full[st], hh * 64, g, j * 128, b);
        mbar_arrive_expect_tx(&v_full[st], L::KV);
        for (int hh = 0; hh < HALVES; ++hh)
          tma_load_4d(sbase + L::OFF_V + st * L::KV + hh * 16384, &p.tmV, &v_full[st], hh * 64, g, j * 128, b);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ------------------------------------------------ MMA issuer
      const uint32_t idesc_s = idesc_bf16(128, 128);
      const uint32_t idesc_o = idesc_bf16(128, HD, /*b_mn_major=*/true);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status);
      tc_fence_after();
      auto issue_s = [&](int x, int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait(&k_full[st], (j >> 1) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        // descriptors of k-step 0; k-step k starts (k >> 2) * 16384 + (k & 3) * 32 bytes further,
        // which is added to the address field (bits 0-13, in 16-byte units) directly
        const uint64_t ad0 = sdesc_sw128(sbase + L::OFF_Q + x * L::QT, 16, 1024);
        const uint64_t bd0 = sdesc_sw128(sbase + L::OFF_K + st * L::KV, 16, 1024);
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint64_t off = (uint64_t)(((k >> 2) * 16384 + (k & 3) * 32) >> 4);
          tc_mma(tmem + x * 128, ad0 + off, bd0 + off, idesc_s, k > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[x]);
        return true;
      };
      auto issue_pv = [&](int x, int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait(&p_full[x], j & 1, abort_flag, p.status)) return false;
        if (!mbar_wait(&v_full[st], (j >> 1) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint64_t bd0 = sdesc_sw128(sbase + L::OFF_V + st * L::KV, 16384, 1024);
#pragma unroll
        for (int k = 0; k < 8; ++k)   // 16 keys per step; P_X k-step k is TMEM columns 8k..8k+7
          tc_mma_ts(tmem + 256 + x * 128, tmem + x * 128 + k * 8, bd0 + (uint64_t)(k * 2048 >> 4), idesc_o,
                    (j > 0 || k > 0) ? 1u : 0u);
        tc_commit(&o_done[x]);
        return true;
      };
      for (int x = 0; ok && x < 2; ++x)
        if (ntile[x] > 0) ok = issue_s(x, 0);
      for (int j = 0; ok && j < nmax; ++j) {
        for (int x = 0; ok && x < 2; ++x) {
          if (j >= ntile[x]) continue;
          if (!issue_pv(x, j)) { ok = false; break; }
          // the last user of key tile j releases its stage
          const bool last_user = (x == 1) || (j >= ntile[1]);
          if (last_user) tc_commit(&kv_empty[j & 1]);
          if (j + 1 < ntile[x] && !issue_s(x, j + 1)) { ok = false; break; }
        }
      }
      int no_abort = 0;
      tc_commit(drain);
      mbar_wait(drain, 0, &no_abort, p.status);
    }
  } else {  // ------------------------------------------------------------ softmax groups
    const int x = (warp - 2) >> 2;                      // warps 2-5: Q tile 0, warps 6-9: Q tile 1
    const int qw = warp & 3;
    const int row = qw * 32 + lane;                     // TMEM lane = Q tile row
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    const uint32_t tS = tmem + x * 128 + lane_off;
    const uint32_t tO = tmem + 256 + x * 128 + lane_off;
    const int n = ntile[x];
    const int tok = t0[x] + row / p.r;                  // token within the sequence
    const int qpos = p.pos0 + tok;                      // absolute position of this row
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!mbar_wait(&s_full[x], j & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      const bool mask = j >= full_tiles[x];
      const int kbase = j * 128;
      // the row of S (128 scores) is read from TMEM once, into registers
      uint32_t v0[32], v1[32], v2[32], v3[32];
      tmem_ld32(tS + 0, v0);
      tmem_ld32(tS + 32, v1);
      tmem_ld32(tS + 64, v2);
      tmem_ld32(tS + 96, v3);
      tc_wait_ld();
      if (mask) {   // key positions past the query's, only on the diagonal tiles
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (kbase + i > qpos) v0[i] = __float_as_uint(-INFINITY);
          if (kbase + 32 + i > qpos) v1[i] = __float_as_uint(-INFINITY);
          if (kbase + 64 + i > qpos) v2[i] = __float_as_uint(-INFINITY);
          if (kbase + 96 + i > qpos) v3[i] = __float_as_uint(-INFINITY);
        }
      }
      float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        m0 = max3(m0, __uint_as_float(v0[i]), __uint_as_float(v0[i + 1]));
        m1 = max3(m1, __uint_as_float(v1[i]), __uint_as_float(v1[i + 1]));
        m2 = max3(m2, __uint_as_float(v2[i]), __uint_as_float(v2[i + 1]));
        m3 = max3(m3, __uint_as_float(v3[i]), __uint_as_float(v3[i + 1]));
      }
      const float mt = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * p.scale_log2;
      float alpha = 1.f;
      bool resc = false;
      if (j == 0) {
        m_ref = mt;
      } else if (mt > m_ref + kRescaleLog2) {
        alpha = ex2(m_ref - mt);
        m_ref = mt;
        resc = true;
      }
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        // O holds the P V of tiles < j only once P_{j-1} V_{j-1} has completed
        if (!mbar_wait(&o_done[x], (j - 1) & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        l *= alpha;
#pragma unroll 1
        for (int c = 0; c < HD / 16; ++c) {
          uint32_t ov[16];
          tmem_ld16_at(tO + c * 16, ov);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tmem_st16(tO + c * 16, ov);
        }
        tc_wait_st();
      }
      // P = exp2(S * scale_log2 - m) as bf16 pairs into TMEM columns [0, 64) of S_X.  The row sum
      // is taken over the fp32 values.
      const float mb = m_ref;
      float ls0 = 0.f, ls1 = 0.f;
      exp_chunk(v0, tS + 0, p.scale_log2, mb, ls0, ls1);
      exp_chunk(v1, tS + 16, p.scale_log2, mb, ls0, ls1);
      exp_chunk(v2, tS + 32, p.scale_log2, mb, ls0, ls1);
      exp_chunk(v3, tS + 48, p.scale_log2, mb, ls0, ls1);
      const float lsum = ls0 + ls1;
      tc_wait_st();
      l += lsum;
      tc_fence_before();
      mbar_arrive(&p_full[x]);
    }
    if (ok && n > 0 && mbar_wait(&o_done[x], (n - 1) & 1, abort_flag, p.status)) {
      tc_fence_after();
      const float inv = 1.f / l;
      const bool live = tok < p.S;
      const int h = g * p.r + row % p.r;
      uint16_t* orow = p.o + (((int64_t)b * p.S + tok) * p.n_q + h) * HD;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tO + c * 32, v);
        tc_wait_ld();
        if (live && in_extent((((int64_t)b * p.S + tok) * p.n_q + h) * HD + c * 32, 32, (int64_t)p.B * p.S * p.n_q * HD)) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[i]) * inv, __uint_as_float(v[i + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(v[i + 2]) * inv, __uint_as_float(v[i + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(v[i + 4]) * inv, __uint_as_float(v[i + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(v[i + 6]) * inv, __uint_as_float(v[i + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + i) = w;
          }
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS_ATTN);
  }
}

template <int HD>
int launch_hd(const AttnDesc& a, unsigned* status, cudaStream_t st) {
  AttnParams p;
  memset(&p, 0, sizeof(p));
  const int r = (int)(a.n_q / a.n_kv);
  const int tpt = 128 / r;
  const int64_t kv_len = a.pos0 + a.S;
  if (!encode_tmap_3d_bf16(&p.tmQ, a.q, (uint64_t)HD, (uint64_t)a.n_q, (uint64_t)(a.B * a.S), HD * 2,
                           (uint64_t)a.n_q * HD * 2, 64, (uint32_t)r, (uint32_t)tpt))
    return -1;
  // K/V: dims (hd, n_kv, kv_len, B), strides in bytes for dims 1..3
  const uint64_t dims[4] = {(uint64_t)HD, (uint64_t)a.n_kv, (uint64_t)kv_len, (uint64_t)a.B};
  const uint64_t strides[3] = {(uint64_t)HD * 2, (uint64_t)a.n_kv * HD * 2, (uint64_t)a.cap * a.n_kv * HD * 2};
  const uint32_t box[4] = {64, 1, 128, 1};
  if (!encode_tmap_4d_bf16(&p.tmK, a.k, dims, strides, box) || !encode_tmap_4d_bf16(&p.tmV, a.v, dims, strides, box))
    return -1;
  p.o = static_cast<uint16_t*>(a.o);
  p.B = (int)a.B; p.S = (int)a.S; p.n_q = (int)a.n_q; p.n_kv = (int)a.n_kv; p.hd = HD; p.r = r;
  p.tokens_per_tile = tpt;
  p.t_blocks = (int)((a.S + tpt - 1) / tpt);
  p.pairs = (p.t_blocks + 1) / 2;
  p.pos0 = (int)a.pos0;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = status;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return -1;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(attn_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<HD>::TOTAL) !=
        cudaSuccess)
      return -1;
    attr_set[dev] = true;
  }
  const int64_t grid = (int64_t)p.pairs * a.B * a.n_kv;
  if (launch_k(attn_tc_kernel<HD>, dim3((unsigned)grid), dim3(AT_THREADS), Smem<HD>::TOTAL, st, p) != cudaSuccess)
    return -1;
  return 0;
}

}  // namespace

bool attn_tc_supported(const AttnDesc& a) {
  if (a.dtype != LLAMA_BF16 || (a.hd != 64 && a.hd != 128)) return false;
  if (a.n_kv <= 0 || a.n_q % a.n_kv != 0) return false;
  const int64_t r = a.n_q / a.n_kv;
  if (r > 128 || 128 % r != 0) return false;
  if (a.S < 16) return false;                         // one-token steps use the decode kernel
  if (a.pos0 + a.S > ((int64_t)1 << 30) || a.B * a.S > ((int64_t)1 << 30)) return false;
  const uintptr_t al = reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k) |
                       reinterpret_cast<uintptr_t>(a.v) | reinterpret_cast<uintptr_t>(a.o);
  return (al & 15) == 0;
}

int launch_attn_tc(const AttnDesc& a, int, unsigned* status, cudaStream_t st) {
  return a.hd == 128 ? launch_hd<128>(a, status, st) : launch_hd<64>(a, status, st);
}

LLAMA_DEFINE_BOUNDS_READER(attn_tc)

}  // namespace llama
