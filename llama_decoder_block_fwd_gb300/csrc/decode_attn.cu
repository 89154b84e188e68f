// Split-K GQA decode attention over a bf16 KV cache: one new query token per sequence attends
// to every cached key plus its own ("LLaMA-3 8B ...", section 九: the 8193rd token sees the 8192
// cached keys and itself; "Llama Architecture ...", Mathematical Foundations 4 for GQA).
//
//   phase 1 (decode_attn_kernel): the 128-key tiles of all (sequence b, KV group g) pairs, in
//     (b, g, tile) order, are cut into one equal contiguous range per CTA, so every CTA streams
//     the same number of tiles; a pair is split only where a range ends, and the CTA c's piece of
//     pair q leaves its partial in slot q + c (unique: along the sequence q and c never decrease
//     and one of them grows at each new piece, so B n_kv + grid slots suffice).  Per tile, tcgen05 computes S^T = K Q^T (M = 128 keys, N = 16: the r <= 16 query
//     heads of KV group g, zero-padded; K = hd) and O^T += V^T P^T (M = hd, N = 16, K = 128 keys;
//     V is read as the MN-major A operand straight from the TMA tile).  One thread per key does
//     the softmax for the r heads; the running max is shared per head through shared memory and
//     O^T is rescaled in TMEM only when a head's max grows by more than 2^8.  Each piece writes its
//     unnormalised partial (m, l, O) to the workspace.
//   phase 2 (decode_combine_seg_kernel): o = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c over the
//     pieces of the pair, found from the same range arithmetic.
// The result equals softmax(q K^T / sqrt(hd)) V up to the order of additions.
//
// Paged cache (block_table set): K and V live in a pool of 128-position pages [n_pages, 128, n_kv,
// hd]; sequence b's tile t is page block_table[b * max_pages + t], and b holds seq_pos[b] + 1
// keys, so sequences may have different lengths (a pair has ceil((seq_pos[b] + 1) / 128) tiles).
// Positions past a sequence's last key in its last page are not read: their V rows are zeroed
// in shared memory before the P V MMA (P is 0 there).
#include <algorithm>
#include <cmath>
#include <cstring>

#include "kernels.h"

namespace llama {
namespace {

constexpr int DA_THREADS = 192;          // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr int DA_STAGES = 3;
constexpr int DA_HD = 128;
constexpr int DA_NPAD = 16;              // MMA N: query heads of the group, zero-padded
constexpr uint32_t DA_TMEM_COLS = 64;
constexpr float kDaRescaleLog2 = 8.0f;

constexpr int DA_MAX_GRID = 256;         // CTAs at most (sizes the partial slots)

struct DecodeAttnParams {   // 128-byte aligned by its tensor maps
  CUtensorMap tmK;   // [B, kv_len, n_kv, hd], box (64, 1, 128, 1)
  CUtensorMap tmV;
  CUtensorMap tmQ;   // [B, n_q, hd], box (64, r, 1)
  float* part_o;     // [B n_kv + grid slots, r, hd]
  float* part_ml;    // [B n_kv + grid slots, r, 2]  (m in log2 units, l)
  int B, n_q, n_kv, r, kv_len, kv_tiles;
  float scale_log2;
  unsigned* status;
  const int* block_table;   // paged cache: [B, max_pages] page ids; null: dense [B, cap, n_kv, hd]
  const int* seq_pos;       // paged cache: [B] position of the new token (keys 0..seq_pos[b])
  int max_pages;
  int n_pages;              // paged cache: pages in each pool (bounds checks)
  int64_t n_slots;          // partial slots part_o / part_ml hold (bounds checks)
};

struct DaSmem {
  static constexpr uint32_t KV = 128 * DA_HD * 2;          // one K or V tile: 32 KB
  static constexpr uint32_t QB = DA_NPAD * DA_HD * 2;      // one Q operand: 4 KB
  static constexpr uint32_t PB = DA_NPAD * 128 * 2;        // P^T operand: 4 KB
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + DA_STAGES * KV;
  static constexpr uint32_t OFF_Q = OFF_V + DA_STAGES * KV;   // 2 buffers
  static constexpr uint32_t OFF_P = OFF_Q + 2 * QB;           // 2 buffers
  static constexpr uint32_t OFF_RED = OFF_P + 2 * PB;         // [3][4 warps][16] floats
  static constexpr uint32_t OFF_BAR = OFF_RED + 3 * 4 * 16 * 4;
  static constexpr uint32_t TOTAL = OFF_BAR + 256 + 1024;
};

__device__ __forceinline__ void tma_load_4d_da(uint32_t dst, const CUtensorMap* m, uint64_t* bar, int x, int y,
                                               int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
// Named barrier over the 128 softmax threads (warps 2..5).
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// ---- the work split: one contiguous range of the (b, g, tile) sequence per CTA
__device__ __forceinline__ int seq_tiles(const int* seq_pos, int kv_tiles, int b) {
  return seq_pos ? (__ldg(seq_pos + b) + 1 + 127) / 128 : kv_tiles;
}
__device__ __forceinline__ int64_t all_tiles(const int* seq_pos, int kv_tiles, int B, int n_kv) {
  if (!seq_pos) return (int64_t)B * n_kv * kv_tiles;
  int64_t s = 0;
  for (int b = 0; b < B; ++b) s += seq_tiles(seq_pos, kv_tiles, b);
  return s * n_kv;
}
__device__ __forceinline__ int64_t range_begin(int64_t T, int G, int c) { return (int64_t)c * T / G; }
// The CTA whose range holds tile x (the last of several with the same start: ranges may be empty
// when there are fewer tiles than CTAs).
__device__ __forceinline__ int cta_of(int64_t T, int G, int64_t x) {
  int c = (int)min((int64_t)G - 1, x * G / T);
  while (c + 1 < G && range_begin(T, G, c + 1) <= x) ++c;
  while (c > 0 && range_begin(T, G, c) > x) --c;
  return c;
}
// First tile of pair (b, g) in the sequence and its tile count.
__device__ __forceinline__ void pair_span(const int* seq_pos, int kv_tiles, int n_kv, int b, int g, int64_t& off,
                                          int& nt) {
  if (!seq_pos) {
    off = ((int64_t)b * n_kv + g) * kv_tiles;
    nt = kv_tiles;
    return;
  }
  int64_t s = 0;
  for (int bb = 0; bb < b; ++bb) s += seq_tiles(seq_pos, kv_tiles, bb);
  nt = seq_tiles(seq_pos, kv_tiles, b);
  off = s * n_kv + (int64_t)g * nt;
}

// The pieces of this CTA's range, one pair at a time, in order.
struct SegIter {
  int64_t x, end, pair_off;
  int b, g, nt;
};
__device__ __forceinline__ void seg_begin(const DecodeAttnParams& p, int64_t T, SegIter& s) {
  s.x = range_begin(T, gridDim.x, blockIdx.x);
  s.end = range_begin(T, gridDim.x, blockIdx.x + 1);
  if (s.x >= s.end) return;
  if (!p.seq_pos) {
    const int64_t pair = s.x / p.kv_tiles;
    s.b = (int)(pair / p.n_kv);
    s.g = (int)(pair % p.n_kv);
    s.nt = p.kv_tiles;
    s.pair_off = pair * p.kv_tiles;
  } else {
    int64_t off = 0;
    int b = 0, nt = 0;
    for (;; ++b) {
      nt = seq_tiles(p.seq_pos, p.kv_tiles, b);
      if (s.x < off + (int64_t)p.n_kv * nt) break;
      off += (int64_t)p.n_kv * nt;
    }
    s.b = b;
    s.nt = nt;
    s.g = (int)((s.x - off) / nt);
    s.pair_off = off + (int64_t)s.g * nt;
  }
}
// Next piece: pair (b, g), its tiles [t0, t1), the pair's key count and its partial slot.
__device__ __forceinline__ bool seg_next(const DecodeAttnParams& p, SegIter& s, int& b, int& g, int& t0, int& t1,
                                         int& kv_len, int64_t& slot) {
  if (s.x >= s.end) return false;
  b = s.b;
  g = s.g;
  t0 = (int)(s.x - s.pair_off);
  t1 = (int)min((int64_t)s.nt, s.end - s.pair_off);
  kv_len = p.seq_pos ? __ldg(p.seq_pos + b) + 1 : p.kv_len;
  slot = (int64_t)b * p.n_kv + g + blockIdx.x;
  s.x = s.pair_off + t1;
  if (t1 == s.nt) {   // the pair is done: the next one starts here
    s.pair_off += s.nt;
    if (++s.g == p.n_kv) {
      s.g = 0;
      if (++s.b < p.B) s.nt = seq_tiles(p.seq_pos, p.kv_tiles, s.b);
    }
  }
  return true;
}

// Warp-wide maximum of a float (one instruction).
__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// R = n_q / n_kv query heads per KV group (1, 2, 4, 8 or 16), a compile-time constant so that the
// softmax touches only the R real columns of the padded N = 16 operands.
template <int R>
__global__ void __launch_bounds__(DA_THREADS, 1) decode_attn_kernel(const __grid_constant__ DecodeAttnParams p) {
  using L = DaSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* k_full = bars + 0;              // [3]
  uint64_t* v_full = bars + 3;              // [3]
  uint64_t* kv_empty = bars + 6;            // [3]
  uint64_t* q_full = bars + 9;              // [2]
  uint64_t* q_empty = bars + 11;            // [2]
  uint64_t* s_full = bars + 13;             // [2]
  uint64_t* s_free = bars + 15;             // [2]  (128 arrivals)
  uint64_t* p_full = bars + 17;             // [2]  (128 arrivals), one per P buffer
  uint64_t* o_done = bars + 19;             // [2]  one per P buffer
  uint64_t* o_free = bars + 21;             //      (128 arrivals)
  uint64_t* drain = bars + 22;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 23);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(smem + L::OFF_RED);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < 23; ++i) {
      const bool many = (i == 15 || i == 16 || i == 17 || i == 18 || i == 21);
      mbar_init(&bars[i], many ? 128 : 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmK);
    tma_prefetch_desc(&p.tmV);
    tma_prefetch_desc(&p.tmQ);
  }
  // Q operand rows r..15 and the padded P^T rows stay zero for the whole kernel.
  for (int i = threadIdx.x; i < (int)(2 * L::QB + 2 * L::PB) / 16; i += DA_THREADS)
    reinterpret_cast<uint4*>(smem + L::OFF_Q)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 1) { tmem_alloc(tmem_slot, DA_TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;          // S^T buffers: columns 0..15 and 16..31
  const uint32_t tO = tmem + 32;     // O^T: columns 32..47
  const uint32_t sbase = smem_u32(smem);

  const int64_t T = all_tiles(p.seq_pos, p.kv_tiles, p.B, p.n_kv);
  // K and V of tile t of pair (b, g) into ring stage st (false: a box outside the cache, which
  // bounds-checking builds report)
  auto load_kv = [&](int b, int g, int t, int st) -> bool {
    const int zc = p.block_table ? 0 : t * 128;
    const int wc = p.block_table ? __ldg(p.block_table + (int64_t)b * p.max_pages + t) : b;
    if (!box_in(0, DA_HD, g, p.n_kv, zc, p.block_table ? 128 : p.kv_len, wc, p.block_table ? p.n_pages : p.B))
      return false;
    mbar_arrive_expect_tx(&k_full[st], L::KV);
    for (int hh = 0; hh < 2; ++hh)
      tma_load_4d_da(sbase + L::OFF_K + st * L::KV + hh * 16384, &p.tmK, &k_full[st], hh * 64, g, zc, wc);
    mbar_arrive_expect_tx(&v_full[st], L::KV);
    for (int hh = 0; hh < 2; ++hh)
      tma_load_4d_da(sbase + L::OFF_V + st * L::KV + hh * 16384, &p.tmV, &v_full[st], hh * 64, g, zc, wc);
    return true;
  };
  // Before the dependency wait the producer starts on the first ring stages: the cached keys and
  // values of a pair's tiles before its last are not written by the kernel before this one (the
  // decode step writes only the new position, which lies in the pair's last tile).
  int pre = 0;
  bool pre_ok = true;
  if (warp == 0 && lane == 0) {
    SegIter si;
    seg_begin(p, T, si);
    int b, g, t0, t1, kv_len;
    int64_t slot;
    bool stop = false;
    while (!stop && pre < DA_STAGES && seg_next(p, si, b, g, t0, t1, kv_len, slot)) {
      const int nt = seq_tiles(p.seq_pos, p.kv_tiles, b);
      for (int t = t0; t < t1 && pre < DA_STAGES; ++t) {
        if (t >= nt - 1) { stop = true; break; }
        if (!load_kv(b, g, t, pre)) { *abort_flag = 1; pre_ok = false; stop = true; break; }
        ++pre;
      }
    }
  }
  pdl_wait();   // q and the newest K/V come from the previous kernel; the partials may still be read
  if (warp == 0) {
    if (lane == 0 && pre_ok) {  // ---------------------------------------------------- TMA producer
      int tile = 0, it = 0;
      bool ok = true;
      SegIter si;
      seg_begin(p, T, si);
      int b, g, t0, t1, kv_len;
      int64_t slot;
      while (ok && seg_next(p, si, b, g, t0, t1, kv_len, slot)) {
        const int qb = it & 1;
        ++it;
        if (!mbar_wait(&q_empty[qb], (((it - 1) >> 1) & 1) ^ 1, abort_flag, p.status)) break;
        if (!box_in(0, DA_HD, (int64_t)g * p.r, p.n_q, b, p.B)) { *abort_flag = 1; break; }   // checking builds
        mbar_arrive_expect_tx(&q_full[qb], 2 * 64 * p.r * 2);
        for (int hh = 0; hh < 2; ++hh)
          tma_load_3d(sbase + L::OFF_Q + qb * L::QB + hh * (L::QB / 2), &p.tmQ, &q_full[qb], hh * 64, g * p.r, b);
        for (int t = t0; t < t1; ++t, ++tile) {
          if (tile < pre) continue;   // issued before the dependency wait
          const int st = tile % DA_STAGES;
          const uint32_t ph = (tile / DA_STAGES) & 1;
          if (!mbar_wait(&kv_empty[st], ph ^ 1, abort_flag, p.status)) { ok = false; break; }
          if (!load_kv(b, g, t, st)) { *abort_flag = 1; ok = false; break; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------------------------------------------- MMA issuer
      const uint32_t idesc_s = idesc_bf16(128, DA_NPAD);
      const uint32_t idesc_o = idesc_bf16(128, DA_NPAD, /*b_mn_major=*/false, /*a_mn_major=*/true);
      int tile = 0, it = 0;
      bool ok = true;
      SegIter si;
      seg_begin(p, T, si);
      int b, g, t0, t1, kv_len;
      int64_t slot;
      for (; ok && seg_next(p, si, b, g, t0, t1, kv_len, slot); ++it) {
        const int qb = it & 1;
        if (!mbar_wait(&q_full[qb], (it >> 1) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t qa = sbase + L::OFF_Q + qb * L::QB;
        const int n = t1 - t0;
        auto issue_s = [&](int j) -> bool {    // tile j of this item (global tile index tile + j)
          const int gt = tile + j;
          const int st = gt % DA_STAGES;
          const int sb = gt & 1;
          if (!mbar_wait(&k_full[st], (gt / DA_STAGES) & 1, abort_flag, p.status)) return false;
          if (!mbar_wait(&s_free[sb], ((gt >> 1) & 1) ^ 1, abort_flag, p.status)) return false;
          tc_fence_after();
          const uint32_t ka = sbase + L::OFF_K + st * L::KV;
          const uint64_t ad0 = sdesc_sw128(ka, 16, 1024), bd0 = sdesc_sw128(qa, 16, 1024);
#pragma unroll
          for (int k = 0; k < DA_HD / 16; ++k)   // k-step offsets added to the address field (16-byte units)
            tc_mma(tS + sb * 16, ad0 + (uint64_t)(((k >> 2) * 16384 + (k & 3) * 32) >> 4),
                   bd0 + (uint64_t)(((k >> 2) * (L::QB / 2) + (k & 3) * 32) >> 4), idesc_s, k > 0 ? 1u : 0u);
          tc_commit(&s_full[sb]);
          return true;
        };
        auto issue_pv = [&](int j) -> bool {
          const int gt = tile + j;
          const int st = gt % DA_STAGES;
          const int pb = gt & 1;
          if (!mbar_wait(&p_full[pb], (gt >> 1) & 1, abort_flag, p.status)) return false;
          if (!mbar_wait(&v_full[st], (gt / DA_STAGES) & 1, abort_flag, p.status)) return false;
          // the first P V of a piece overwrites O^T: the previous piece's O^T must have been read
          if (j == 0 && !mbar_wait(o_free, (it & 1) ^ 1, abort_flag, p.status)) return false;
          tc_fence_after();
          const uint32_t va = sbase + L::OFF_V + st * L::KV;
          const uint32_t pa = sbase + L::OFF_P + pb * L::PB;
          const uint64_t ad0 = sdesc_sw128(va, 16384, 1024);   // V^T, MN-major
          const uint64_t bd0 = sdesc_sw128(pa, 16, 1024);
#pragma unroll
          for (int k = 0; k < 8; ++k)       // 16 keys per step
            tc_mma(tO, ad0 + (uint64_t)(k * 2048 >> 4), bd0 + (uint64_t)(((k >> 2) * (L::PB / 2) + (k & 3) * 32) >> 4),
                   idesc_o, (j > 0 || k > 0) ? 1u : 0u);
          tc_commit(&o_done[pb]);
          tc_commit(&kv_empty[st]);
          return true;
        };
        for (int j = 0; j < n; ++j) {
          if (!issue_s(j)) { ok = false; break; }
          if (j > 0 && !issue_pv(j - 1)) { ok = false; break; }
        }
        if (!ok) break;
        tc_commit(&q_empty[qb]);
        if (!issue_pv(n - 1)) break;
        tile += n;
      }
      int no_abort = 0;
      tc_commit(drain);
      mbar_wait(drain, 0, &no_abort, p.status);
    }
  } else {  // ------------------------------------------------------------ softmax warps 2..5
    const int qw = warp & 3;
    const int t = qw * 32 + lane;                 // TMEM lane: key of the tile / hd index of O^T
    const uint32_t lane_off = (uint32_t)(qw * 32) << 16;
    constexpr int r = R;
    int tile = 0, it = 0;
    bool ok = true;
    SegIter si;
    seg_begin(p, T, si);
    int b, g, t0, t1, kv_len;
    int64_t slot;
    for (; ok && seg_next(p, si, b, g, t0, t1, kv_len, slot); ++it) {
      float m_ref[R], lsum[R];
#pragma unroll
      for (int h = 0; h < R; ++h) { m_ref[h] = -INFINITY; lsum[h] = 0.f; }
      for (int tt = t0; tt < t1; ++tt, ++tile) {
        const int sb = tile & 1;
        if (!mbar_wait(&s_full[sb], (tile >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[16];
        tmem_ld16(tS + sb * 16 + lane_off, sv);
        tc_wait_ld();
        tc_fence_before();
        mbar_arrive(&s_free[sb]);
        const bool valid = tt * 128 + t < kv_len;
        float s[R];
#pragma unroll
        for (int h = 0; h < R; ++h) s[h] = valid ? __uint_as_float(sv[h]) * p.scale_log2 : -INFINITY;
        // per-head max over the 128 keys of the tile: warp maxima, then across the four warps
        float* rbuf = red + (tile & 1) * 64;    // alternate halves: one barrier per tile suffices
#pragma unroll
        for (int h = 0; h < R; ++h) {
          const float v = warp_max_f32(s[h]);
          if (lane == h) rbuf[qw * 16 + h] = v;
        }
        softmax_sync();
        float alpha[R];
        bool resc = false;
#pragma unroll
        for (int h = 0; h < R; ++h) {
          const float tm = fmaxf(fmaxf(rbuf[h], rbuf[16 + h]), fmaxf(rbuf[32 + h], rbuf[48 + h]));
          alpha[h] = 1.f;
          if (m_ref[h] == -INFINITY) {
            m_ref[h] = tm;
          } else if (tm > m_ref[h] + kDaRescaleLog2) {
            alpha[h] = exp2f(m_ref[h] - tm);
            m_ref[h] = tm;
            resc = true;
          }
        }
        const int pb = tile & 1;
        // P buffer pb is free once the P V of tile - 2 (the same buffer) has completed
        if (tile >= 2) {
          if (!mbar_wait(&o_done[pb], ((tile - 2) >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
        }
        // a rescale of O^T (rare; uniform across the 128 threads, which saw the same maxima) needs
        // every P V issued so far to have completed
        if (resc) {
          if (!mbar_wait(&o_done[(tile - 1) & 1], ((tile - 1) >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          {
            uint32_t ov[16];
            tmem_ld16(tO + lane_off, ov);
            tc_wait_ld();
#pragma unroll
            for (int h = 0; h < R; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
            tmem_st16(tO + lane_off, ov);
            tc_wait_st();
#pragma unroll
            for (int h = 0; h < R; ++h) lsum[h] *= alpha[h];
          }
        }
        // paged cache, a sequence's last page: the rows past its last key hold whatever the pool
        // held there; zero them so that P = 0 times them stays 0
        if (p.block_table && (tt + 1) * 128 > kv_len) {
          const int st = tile % DA_STAGES;
          if (!mbar_wait(&v_full[st], (tile / DA_STAGES) & 1, abort_flag, p.status)) { ok = false; break; }
          if (!valid) {
            uint8_t* vrow = smem + L::OFF_V + st * L::KV + t * 128;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
              for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + hh * 16384 + c * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        // P^T rows = heads, columns = keys (K-major, 128B swizzle, two 64-key atoms)
        uint8_t* pbase = smem + L::OFF_P + pb * L::PB + (t >> 6) * (L::PB / 2);
        const int kin = t & 63;
#pragma unroll
        for (int h = 0; h < R; ++h) {
          const float pv = exp2f(s[h] - m_ref[h]);
          const __nv_bfloat16 pq = __float2bfloat16_rn(pv);
          lsum[h] += pv;
          const int chunk16 = (kin >> 3) ^ (h & 7);
          *reinterpret_cast<__nv_bfloat16*>(pbase + h * 128 + chunk16 * 16 + (kin & 7) * 2) = pq;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[pb]);
      }
      if (!ok) break;
      // ---- piece done: write the unnormalised partial (m, l, O) to its slot
      if (!mbar_wait(&o_done[(tile - 1) & 1], ((tile - 1) >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      uint32_t ov[16];
      tmem_ld16(tO + lane_off, ov);
      tc_wait_ld();
      tc_fence_before();
      mbar_arrive(o_free);
      const int64_t base = slot * r;
      const bool slot_in = in_extent(base, r, p.n_slots * r);   // checking builds: the slot exists
#pragma unroll
      for (int h = 0; h < R; ++h)
        if (slot_in) p.part_o[(base + h) * DA_HD + t] = __uint_as_float(ov[h]);
      // l: sum the per-thread partial sums over the 128 keys of each head
      float* lbuf = red + 128;
#pragma unroll
      for (int h = 0; h < R; ++h) {
        float v = lsum[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == h) lbuf[qw * 16 + h] = v;
      }
      softmax_sync();
      if (t < r && slot_in) {
        const float l = lbuf[t] + lbuf[16 + t] + lbuf[32 + t] + lbuf[48 + t];
        float mm = -INFINITY;
#pragma unroll
        for (int h = 0; h < R; ++h) if (h == t) mm = m_ref[h];
        p.part_ml[(base + t) * 2 + 0] = mm;
        p.part_ml[(base + t) * 2 + 1] = l;
      }
      // lbuf is written again only after the next piece's first tile barrier, which every thread
      // passes after reading it here
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, DA_TMEM_COLS);
  }
}

// o[b, h, :] = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c; one warp per (b, h).
// With o_lo set, o receives the bf16 rounding of the result and o_lo the bf16 rounding of what it
// missed (hi + lo carries ~16 mantissa bits into the next GEMM).
__global__ void decode_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                                      uint16_t* __restrict__ o, uint16_t* __restrict__ o_lo, int B, int n_q,
                                      int n_chunks) {
  pdl_trigger();
  pdl_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= B * n_q) return;
  const int b = warp / n_q, h = warp % n_q;
  float M = -INFINITY;
  for (int c = 0; c < n_chunks; ++c) M = fmaxf(M, part_ml[(((int64_t)b * n_chunks + c) * n_q + h) * 2]);
  float l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int c = 0; c < n_chunks; ++c) {
    const int64_t idx = ((int64_t)b * n_chunks + c) * n_q + h;
    const float w = exp2f(part_ml[idx * 2] - M);
    l += w * part_ml[idx * 2 + 1];
    const float4 v = *reinterpret_cast<const float4*>(part_o + idx * DA_HD + lane * 4);
    acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
  }
  const float inv = 1.f / l;
  float r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) r[i] = acc[i] * inv;
  uint2 out;
  out.x = pack_bf2(r[0], r[1]);
  out.y = pack_bf2(r[2], r[3]);
  const int64_t off = ((int64_t)b * n_q + h) * DA_HD + lane * 4;
  if (!in_extent(off, 4, (int64_t)B * n_q * DA_HD)) return;
  *reinterpret_cast<uint2*>(o + off) = out;
  if (o_lo) {
    uint2 lo;
    lo.x = pack_bf2(r[0] - __uint_as_float(out.x << 16), r[1] - __uint_as_float(out.x & 0xFFFF0000u));
    lo.y = pack_bf2(r[2] - __uint_as_float(out.y << 16), r[3] - __uint_as_float(out.y & 0xFFFF0000u));
    *reinterpret_cast<uint2*>(o_lo + off) = lo;
  }
}

// The same merge over the pieces of pair (b, g = h / r): the CTAs c0..c1 whose ranges hold the
// pair's first and last tiles (a CTA with an empty range wrote nothing and is skipped).
__global__ void decode_combine_seg_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                                          uint16_t* __restrict__ o, uint16_t* __restrict__ o_lo, int B, int n_q,
                                          int n_kv, int kv_tiles, const int* __restrict__ seq_pos, int G) {
  pdl_trigger();
  pdl_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= B * n_q) return;
  const int b = warp / n_q, h = warp % n_q;
  const int r = n_q / n_kv, g = h / r, hh = h % r;
  const int64_t T = all_tiles(seq_pos, kv_tiles, B, n_kv);
  int64_t off;
  int nt;
  pair_span(seq_pos, kv_tiles, n_kv, b, g, off, nt);
  const int c0 = cta_of(T, G, off), c1 = cta_of(T, G, off + nt - 1);
  const int64_t pair = (int64_t)b * n_kv + g;
  float M = -INFINITY;
  for (int c = c0; c <= c1; ++c)
    if (range_begin(T, G, c) < range_begin(T, G, c + 1)) M = fmaxf(M, part_ml[((pair + c) * r + hh) * 2]);
  float l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int c = c0; c <= c1; ++c) {
    if (range_begin(T, G, c) >= range_begin(T, G, c + 1)) continue;
    const int64_t idx = (pair + c) * r + hh;
    const float w = exp2f(part_ml[idx * 2] - M);
    l += w * part_ml[idx * 2 + 1];
    const float4 v = *reinterpret_cast<const float4*>(part_o + idx * DA_HD + lane * 4);
    acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
  }
  const float inv = 1.f / l;
  float rr[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) rr[i] = acc[i] * inv;
  uint2 out;
  out.x = pack_bf2(rr[0], rr[1]);
  out.y = pack_bf2(rr[2], rr[3]);
  const int64_t o_off = ((int64_t)b * n_q + h) * DA_HD + lane * 4;
  if (!in_extent(o_off, 4, (int64_t)B * n_q * DA_HD)) return;
  *reinterpret_cast<uint2*>(o + o_off) = out;
  if (o_lo) {
    uint2 lo;
    lo.x = pack_bf2(rr[0] - __uint_as_float(out.x << 16), rr[1] - __uint_as_float(out.x & 0xFFFF0000u));
    lo.y = pack_bf2(rr[2] - __uint_as_float(out.y << 16), rr[3] - __uint_as_float(out.y & 0xFFFF0000u));
    *reinterpret_cast<uint2*>(o_lo + o_off) = lo;
  }
}

int launch_combine_seg(const DecodeAttnParams& p, void* o, void* o_lo, int G, cudaStream_t st) {
  const int warps = p.B * p.n_q;
  return launch_k(decode_combine_seg_kernel, dim3((warps * 32 + 255) / 256), dim3(256), 0, st, (const float*)p.part_o,
                  (const float*)p.part_ml, static_cast<uint16_t*>(o), static_cast<uint16_t*>(o_lo), p.B, p.n_q,
                  p.n_kv, p.kv_tiles, p.seq_pos, G) == cudaSuccess
             ? 0
             : -1;
}

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

// Partial slots of the range split: B n_kv + grid, each r x (hd + 2) floats.
size_t seg_ws_bytes(int64_t B, int64_t n_kv, int64_t r, int64_t grid) {
  const size_t slots = (size_t)(B * n_kv + grid);
  return round256(slots * r * DA_HD * 4) + round256(slots * r * 2 * 4);
}

// Launch phase 1 for the params' head ratio (attributes set once per device).
int launch_decode_kernel(const DecodeAttnParams& p, int grid, cudaStream_t st) {
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return -1;
  if (!attr_set[dev]) {
    const void* fns[5] = {(const void*)decode_attn_kernel<1>, (const void*)decode_attn_kernel<2>,
                          (const void*)decode_attn_kernel<4>, (const void*)decode_attn_kernel<8>,
                          (const void*)decode_attn_kernel<16>};
    for (const void* f : fns)
      if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, DaSmem::TOTAL) != cudaSuccess) return -1;
    attr_set[dev] = true;
  }
  cudaError_t e;
  switch (p.r) {
    case 1: e = launch_k(decode_attn_kernel<1>, dim3(grid), dim3(DA_THREADS), DaSmem::TOTAL, st, p); break;
    case 2: e = launch_k(decode_attn_kernel<2>, dim3(grid), dim3(DA_THREADS), DaSmem::TOTAL, st, p); break;
    case 4: e = launch_k(decode_attn_kernel<4>, dim3(grid), dim3(DA_THREADS), DaSmem::TOTAL, st, p); break;
    case 8: e = launch_k(decode_attn_kernel<8>, dim3(grid), dim3(DA_THREADS), DaSmem::TOTAL, st, p); break;
    case 16: e = launch_k(decode_attn_kernel<16>, dim3(grid), dim3(DA_THREADS), DaSmem::TOTAL, st, p); break;
    default: return -1;
  }
  return e == cudaSuccess ? 0 : -1;
}

struct DecodePlan {
  int kv_tiles, chunk_tiles, n_chunks;
};

DecodePlan plan(int64_t B, int64_t n_kv, int64_t kv_len) {
  DecodePlan d;
  d.kv_tiles = (int)((kv_len + 127) / 128);
  d.chunk_tiles = std::max(1, std::min(d.kv_tiles, 8));
  d.n_chunks = (d.kv_tiles + d.chunk_tiles - 1) / d.chunk_tiles;
  (void)B; (void)n_kv;
  return d;
}

}  // namespace

bool decode_attn_supported(const AttnDesc& a) {
  if (a.dtype != LLAMA_BF16 || a.hd != DA_HD || a.S != 1) return false;
  if (a.n_kv <= 0 || a.n_q % a.n_kv != 0) return false;
  const int64_t r = a.n_q / a.n_kv;
  if (r != 1 && r != 2 && r != 4 && r != 8 && r != 16) return false;
  if (a.pos0 + 1 > ((int64_t)1 << 30)) return false;
  const uintptr_t al = reinterpret_cast<uintptr_t>(a.q) | reinterpret_cast<uintptr_t>(a.k) |
                       reinterpret_cast<uintptr_t>(a.v) | reinterpret_cast<uintptr_t>(a.o);
  return (al & 15) == 0;
}

size_t decode_attn_ws_bytes(const AttnDesc& a) {
  if (a.n_kv <= 0 || a.n_q % a.n_kv != 0) return 0;
  const size_t seg = seg_ws_bytes(a.B, a.n_kv, a.n_q / a.n_kv, DA_MAX_GRID);
  // the 8-bit kernel keeps fixed chunks of up to 8 tiles per (b, g) and uses the same workspace
  const DecodePlan d = plan(a.B, a.n_kv, a.pos0 + 1);
  const size_t chunked = round256((size_t)a.B * d.n_chunks * a.n_q * DA_HD * 4) +
                         round256((size_t)a.B * d.n_chunks * a.n_q * 2 * 4);
  return std::max(seg, chunked);
}

int launch_decode_attn(const AttnDesc& a, void* ws, int num_sms, unsigned* status, cudaStream_t st) {
  DecodeAttnParams p;
  memset(&p, 0, sizeof(p));
  const int r = (int)(a.n_q / a.n_kv);
  const int64_t kv_len = a.pos0 + 1;
  const DecodePlan d = plan(a.B, a.n_kv, kv_len);
  const bool paged = a.block_table != nullptr;
  const uint64_t dims[4] = {(uint64_t)DA_HD, (uint64_t)a.n_kv, paged ? 128u : (uint64_t)kv_len,
                            paged ? (uint64_t)a.n_pages : (uint64_t)a.B};
  const uint64_t strides[3] = {(uint64_t)DA_HD * 2, (uint64_t)a.n_kv * DA_HD * 2,
                               (paged ? (uint64_t)128 : (uint64_t)a.cap) * a.n_kv * DA_HD * 2};
  const uint32_t box[4] = {64, 1, 128, 1};
  if (!encode_tmap_4d_bf16(&p.tmK, a.k, dims, strides, box)) return -1;
  if (!encode_tmap_4d_bf16(&p.tmV, a.v, dims, strides, box)) return -1;
  p.block_table = a.block_table;
  p.seq_pos = a.seq_pos;
  p.max_pages = (int)a.max_pages;
  p.n_pages = (int)a.n_pages;
  if (!encode_tmap_3d_bf16(&p.tmQ, a.q, DA_HD, (uint64_t)a.n_q, (uint64_t)a.B, DA_HD * 2,
                           (uint64_t)a.n_q * DA_HD * 2, 64, (uint32_t)r, 1))
    return -1;
  const int64_t slots = a.B * a.n_kv + DA_MAX_GRID;
  p.n_slots = slots;
  p.part_o = static_cast<float*>(ws);
  p.part_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + round256((size_t)slots * r * DA_HD * 4));
  p.B = (int)a.B; p.n_q = (int)a.n_q; p.n_kv = (int)a.n_kv; p.r = r;
  p.kv_len = (int)kv_len;
  p.kv_tiles = d.kv_tiles;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = status;
  // one CTA per SM; with a dense cache no more CTAs than tiles (a paged cache's tile count is on
  // the device: CTAs past it get empty ranges)
  int grid = std::min(num_sms, DA_MAX_GRID);
  if (!paged) grid = (int)std::min<int64_t>(grid, a.B * a.n_kv * d.kv_tiles);
  grid = std::max(1, grid);
  if (launch_decode_kernel(p, grid, st) != 0) return -1;
  return launch_combine_seg(p, a.o, a.o_lo, grid, st);
}

void decode_attn_plan(int64_t kv_len, int& kv_tiles, int& chunk_tiles, int& n_chunks) {
  const DecodePlan d = plan(0, 0, kv_len);
  kv_tiles = d.kv_tiles;
  chunk_tiles = d.chunk_tiles;
  n_chunks = d.n_chunks;
}

int launch_decode_combine(const float* part_o, const float* part_ml, void* o, void* o_lo, int64_t B, int64_t n_q,
                          int n_chunks, cudaStream_t st) {
  const int warps = (int)(B * n_q);
  return launch_k(decode_combine_kernel, dim3((warps * 32 + 255) / 256), dim3(256), 0, st, part_o, part_ml,
                  static_cast<uint16_t*>(o), static_cast<uint16_t*>(o_lo), (int)B, (int)n_q, n_chunks) == cudaSuccess
             ? 0
             : -1;
}

// ------------------------------------------------------------------------------------------
// Allocation-free variant of the decode attention call.  Its split-K partials live in one
// file-scope device array instead of a caller workspace, so callers that cannot allocate device
// memory where they call (code running under an allocator that owns all of device memory, such
// as a fixed-budget arena or a caching allocator, where a stray cudaMalloc would fail or split
// the pool; latency-bound loops where cudaMalloc/cudaFree would synchronise the device) can run
// it with only their inputs and output.  The array is created when the library is loaded and
// stays resident on every device that loads it until the process exits.
// ------------------------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)12 << 20;   // 12 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up on first use per device.
// (In host code the array's name is only a host-side stand-in, not a device address.)
void* noalloc_scratch_ptr() {
  static void* cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cached[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
    cached[dev] = ptr;
  }
  return cached[dev];
}


}  // namespace

LLAMA_DEFINE_BOUNDS_READER(decode_attn)

}  // namespace llama

using namespace llama;

extern "C" int llama_gqa_attention_decode_noalloc(const llama_dims* dims, int dtype, const void* q, const void* k,
                                                   const void* v, int64_t kv_capacity, int64_t pos0, void* o,
                                                   void* stream) {
  if (!dims || dtype != LLAMA_BF16) return dtype == LLAMA_BF16 ? LLAMA_ERR_INVALID_ARG : LLAMA_ERR_UNSUPPORTED;
  if (dims->B < 0 || dims->S != 1 || dims->n_q <= 0 || dims->n_kv <= 0 || dims->n_q % dims->n_kv != 0)
    return LLAMA_ERR_INVALID_ARG;
  {
    const int64_t rr = dims->n_q / dims->n_kv;
    if (dims->head_dim != DA_HD || (rr != 1 && rr != 2 && rr != 4 && rr != 8 && rr != 16)) return LLAMA_ERR_UNSUPPORTED;
  }
  if (pos0 < 0 || kv_capacity < pos0 + 1 || pos0 + 1 > ((int64_t)1 << 30)) return LLAMA_ERR_INVALID_ARG;
  if (dims->B == 0) return LLAMA_OK;
  if (!q || !k || !v || !o) return LLAMA_ERR_INVALID_ARG;
  const uintptr_t al = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if (al & 15) return LLAMA_ERR_ALIGNMENT;
  const int64_t rr = dims->n_q / dims->n_kv;
  // The partials need B n_kv + grid slots of r (hd + 2) floats, whatever the number of keys.  The
  // size rule takes the largest grid (DA_MAX_GRID), so whether a shape fits does not depend on the
  // device's SM count.
  if (seg_ws_bytes(dims->B, dims->n_kv, rr, DA_MAX_GRID) > kNoAllocScratchBytes)
    return LLAMA_ERR_WORKSPACE;
  const DecodePlan d = plan(dims->B, dims->n_kv, pos0 + 1);
  const int grid = std::max(1, (int)std::min<int64_t>(std::min(num_sms(), DA_MAX_GRID),
                                                      dims->B * dims->n_kv * d.kv_tiles));
  void* scratch = noalloc_scratch_ptr();
  unsigned* status = status_ptr();
  if (!scratch || !status) return LLAMA_ERR_CUDA;

  DecodeAttnParams p;
  memset(&p, 0, sizeof(p));
  const int r = (int)(dims->n_q / dims->n_kv);
  const int64_t kv_len = pos0 + 1;
  const uint64_t tdims[4] = {(uint64_t)DA_HD, (uint64_t)dims->n_kv, (uint64_t)kv_len, (uint64_t)dims->B};
  const uint64_t strides[3] = {(uint64_t)DA_HD * 2, (uint64_t)dims->n_kv * DA_HD * 2,
                               (uint64_t)kv_capacity * dims->n_kv * DA_HD * 2};
  const uint32_t box[4] = {64, 1, 128, 1};
  if (!encode_tmap_4d_bf16(&p.tmK, k, tdims, strides, box) || !encode_tmap_4d_bf16(&p.tmV, v, tdims, strides, box) ||
      !encode_tmap_3d_bf16(&p.tmQ, q, DA_HD, (uint64_t)dims->n_q, (uint64_t)dims->B, DA_HD * 2,
                           (uint64_t)dims->n_q * DA_HD * 2, 64, (uint32_t)r, 1))
    return LLAMA_ERR_CUDA;
  // Every partial slot the combine reads is written by its piece: nothing has to start at zero.
  p.n_slots = dims->B * dims->n_kv + grid;
  p.part_o = static_cast<float*>(scratch);
  p.part_ml = reinterpret_cast<float*>(static_cast<char*>(scratch) +
                                       round256((size_t)(dims->B * dims->n_kv + grid) * rr * DA_HD * 4));
  p.B = (int)dims->B; p.n_q = (int)dims->n_q; p.n_kv = (int)dims->n_kv; p.r = r;
  p.kv_len = (int)kv_len;
  p.kv_tiles = d.kv_tiles;
  p.scale_log2 = (float)(1.0 / std::sqrt((double)DA_HD)) * 1.4426950408889634f;
  p.status = status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_decode_kernel(p, grid, st) != 0) return LLAMA_ERR_CUDA;
  if (launch_combine_seg(p, o, nullptr, grid, st) != 0) return LLAMA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? LLAMA_OK : LLAMA_ERR_CUDA;
}
