// Weight-streaming tcgen05 GEMM for few token rows (the decode step): out = X W^T with
// W [N, K] (the projection, bf16) and X [M <= 128, K] given as two bf16 parts, hi + lo.
//
// The roles are swapped against gemm_tc.cu: 128 weight rows are the MMA's M operand and the
// token rows the N operand, stacked as X2 = [hi rows 0..M-1 | lo rows Mp..Mp+M-1] (Mp = 64 or 128,
// so N = 2 Mp), so one MMA per k-step yields W X_hi^T and W X_lo^T side by side in TMEM and the
// epilogue adds column c and column Mp + c.  Per stage the shared memory holds 16 KB of weights
// and 16 KB (Mp = 64) of activations; six stages keep ~96 KB of weights in flight per SM.
// Work units are (128 weight rows, K range).  Split-K partials are either written as fp32
// out[split * M + c, n] (fixed splits, units dealt round robin), or added atomically into
// out[c, n] -- the residual stream, or a zeroed buffer the next kernel reads -- in which case the
// (weight tile, k-block) items are cut into equal contiguous ranges, one per CTA, so every SM
// streams the same number of weight bytes.  With one split and a row scale the result is stored
// scaled (the LM head after the final RMSNorm).
#include <algorithm>
#include <cstring>

#include "kernels.h"

namespace llama {
namespace {

constexpr int SK_TK = 64, SK_THREADS = 192;
constexpr uint32_t SK_A_BYTES = 128 * SK_TK * 2;     // 128 weight rows x 64: 16 KB
constexpr uint32_t SK_TMEM_COLS = 512;

struct SkParams {   // 128-byte aligned by its tensor maps
  CUtensorMap tmW[3];   // weight segments [n_i, K], box (64, 128)
  CUtensorMap tmX;      // stacked activations [2 Mp, K], box (64, 2 Mp)
  int M, Mp, K, N;
  int seg_tile_end[3];  // cumulative 128-row tiles per segment
  int nseg;
  int n_tiles, k_splits, kb_per_split, num_units, stages;
  int mode;             // 0: partials [split*M + c, n]; 1: atomic add into out[c, n]; 2: store (x row scale)
  int streamk;          // mode 1: equal item ranges per CTA instead of fixed units
  int64_t total_items;  // n_tiles * k-blocks
  float* out;
  int64_t ldo;
  const float* row_scale;
  unsigned* status;
};

__device__ __forceinline__ void sk_unit(const SkParams& p, int u, int nkb, int& nt, int& split, int& kb0, int& kb1) {
  nt = u / p.k_splits;
  split = u - nt * p.k_splits;
  kb0 = split * p.kb_per_split;
  kb1 = min(nkb, kb0 + p.kb_per_split);
}

__device__ __forceinline__ void sk_seg(const SkParams& p, int nt, int& seg, int& row) {
  seg = 0;
  int start = 0;
  while (seg < p.nseg - 1 && nt >= p.seg_tile_end[seg]) { start = p.seg_tile_end[seg]; ++seg; }
  row = (nt - start) * 128;
}

// Rows of weight segment s.
__device__ __forceinline__ int sk_seg_rows(const SkParams& p, int s) {
  return (p.seg_tile_end[s] - (s ? p.seg_tile_end[s - 1] : 0)) * 128;
}

// The units of this CTA, in order.
struct UnitIter {
  int64_t pos, end;   // stream-K: the CTA's range of (tile, k-block) items, tile-major
  int u;              // fixed units: the next unit index
};
__device__ __forceinline__ UnitIter unit_begin(const SkParams& p) {
  UnitIter it;
  it.pos = (int64_t)blockIdx.x * p.total_items / gridDim.x;
  it.end = (int64_t)(blockIdx.x + 1) * p.total_items / gridDim.x;
  it.u = blockIdx.x;
  return it;
}
__device__ __forceinline__ bool unit_next(const SkParams& p, UnitIter& it, int nkb, int& nt, int& split, int& kb0,
                                          int& kb1) {
  if (p.streamk) {
    if (it.pos >= it.end) return false;
    nt = (int)(it.pos / nkb);
    kb0 = (int)(it.pos - (int64_t)nt * nkb);
    kb1 = (int)min((int64_t)nkb, (int64_t)kb0 + (it.end - it.pos));
    split = 0;
    it.pos += kb1 - kb0;
    return true;
  }
  if (it.u >= p.num_units) return false;
  sk_unit(p, it.u, nkb, nt, split, kb0, kb1);
  it.u += gridDim.x;
  return true;
}

template <int MODE>   // 0: split-K partials; 1: atomic add; 2: store (x row scale)
__global__ void __launch_bounds__(SK_THREADS, 1) gemm_skinny_kernel(const __grid_constant__ SkParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t b_bytes = (uint32_t)(2 * p.Mp) * SK_TK * 2;
  const uint32_t stage_bytes = SK_A_BYTES + b_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.stages * stage_bytes);
  uint64_t* empty = full + p.stages;
  uint64_t* acc_full = empty + p.stages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 128); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmX);
    for (int s = 0; s < p.nseg; ++s) tma_prefetch_desc(&p.tmW[s]);
  }
  if (warp == 1) { tmem_alloc(tmem_slot, SK_TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nkb = (p.K + SK_TK - 1) / SK_TK;
  const uint32_t smem_base = smem_u32(smem);
  const int nmma = 2 * p.Mp;

  if (warp == 0) {
    if (lane == 0) {  // ---------------- TMA producer
      // The weights are never written by an earlier kernel: the first unit's first stages are
      // loaded before waiting for the kernel that produced the activations.
      int pre = 0;
      bool bad = false;   // bounds-checking builds: a box start outside its tensor
      UnitIter first = unit_begin(p);
      int nt, split, kb0, kb1, seg, row;
      if (unit_next(p, first, nkb, nt, split, kb0, kb1)) {
        sk_seg(p, nt, seg, row);
        pre = min(p.stages, kb1 - kb0);
        for (int i = 0; i < pre; ++i) {
          if (!box_in((kb0 + i) * SK_TK, p.K, row, sk_seg_rows(p, seg))) { *abort_flag = 1; bad = true; break; }
          mbar_arrive_expect_tx(&full[i], stage_bytes);
          tma_load_2d(smem_base + i * stage_bytes, &p.tmW[seg], &full[i], (kb0 + i) * SK_TK, row);
        }
      }
      pdl_wait();
      int stage = 0;
      uint32_t phase = 0;
      bool first_unit = true;
      UnitIter ui = unit_begin(p);
      while (!bad && unit_next(p, ui, nkb, nt, split, kb0, kb1)) {
        sk_seg(p, nt, seg, row);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          const uint32_t sa = smem_base + stage * stage_bytes;
          if (!box_in(kb * SK_TK, p.K, row, sk_seg_rows(p, seg))) { *abort_flag = 1; ok = false; break; }
          if (first_unit && kb - kb0 < pre) {   // weights already on their way
            tma_load_2d(sa + SK_A_BYTES, &p.tmX, &full[stage], kb * SK_TK, 0);
          } else {
            if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
            mbar_arrive_expect_tx(&full[stage], stage_bytes);
            tma_load_2d(sa, &p.tmW[seg], &full[stage], kb * SK_TK, row);
            tma_load_2d(sa + SK_A_BYTES, &p.tmX, &full[stage], kb * SK_TK, 0);
          }
          if (++stage == p.stages) { stage = 0; phase ^= 1; }
        }
        first_unit = false;
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------- MMA issuer
      const uint32_t idesc = idesc_bf16(128, nmma);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      int nt, split, kb0, kb1;
      UnitIter ui = unit_begin(p);
      for (; unit_next(p, ui, nkb, nt, split, kb0, kb1); ++it) {
        const int buf = it & 1;
        if (!mbar_wait(&acc_empty[buf], ((it >> 1) & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * 256;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_base + stage * stage_bytes;
          const uint32_t sb = sa + SK_A_BYTES;
          const uint64_t ad0 = sdesc_sw128(sa, 16, 1024), bd0 = sdesc_sw128(sb, 16, 1024);
#pragma unroll
          for (int k = 0; k < SK_TK / 16; ++k)   // +32 bytes per k-step = +2 in the address field
            tc_mma(d, ad0 + 2 * k, bd0 + 2 * k, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
          tc_commit(&empty[stage]);
          if (++stage == p.stages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
      }
      int no_abort = 0;
      tc_commit(drain);
      mbar_wait(drain, 0, &no_abort, p.status);
    }
  } else {  // ---------------- epilogue warps 2..5: one weight row per thread
    pdl_wait();   // outputs may still be read by an earlier kernel
    const int q = warp & 3;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int it = 0;
    int nt, split, kb0, kb1;
    UnitIter ui = unit_begin(p);
    for (; unit_next(p, ui, nkb, nt, split, kb0, kb1); ++it) {
      const int buf = it & 1;
      if (!mbar_wait(&acc_full[buf], (it >> 1) & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const int64_t n = (int64_t)nt * 128 + q * 32 + lane;     // output column (virtual N)
      const bool live = n < p.N;
      const uint32_t tb = tmem + buf * 256 + lane_base;
      // Four token rows per step, rolled: this code runs once per unit, at the end of the CTA's
      // weight stream, and a short loop keeps its instruction fetches few while the memory system
      // is still saturated by the other SMs' streams.
#pragma unroll 1
      for (int c0 = 0; c0 < p.M; c0 += 4) {
        uint32_t hi[4], lo[4];
        tmem_ld4(tb + c0, hi);
        tmem_ld4(tb + p.Mp + c0, lo);
        tc_wait_ld();
        if (!live) continue;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int64_t c = c0 + i;
          if (c >= p.M) break;
          const float v = __uint_as_float(hi[i]) + __uint_as_float(lo[i]);
          if (MODE == 0) {
            const int64_t at = ((int64_t)split * p.M + c) * p.ldo + n;
            if (in_extent(at, 1, (int64_t)p.k_splits * p.M * p.ldo)) p.out[at] = v;
          } else if (in_extent(c * p.ldo + n, 1, (int64_t)p.M * p.ldo)) {
            if (MODE == 1) atomicAdd(p.out + c * p.ldo + n, v);
            else p.out[c * p.ldo + n] = p.row_scale ? v * __ldg(p.row_scale + c) : v;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, SK_TMEM_COLS);
  }
}

}  // namespace

int gemm_skinny_splits(int64_t K, int requested) {
  const int nkb = (int)((K + SK_TK - 1) / SK_TK);
  const int ks = std::max(1, std::min(requested, nkb));
  const int kbps = (nkb + ks - 1) / ks;
  return (nkb + kbps - 1) / kbps;
}

int launch_gemm_skinny(const SkinnyDesc& g, int num_sms, unsigned* status, cudaStream_t st) {
  if (g.M < 1 || g.M > 128 || g.K < 1 || g.K % 8 || g.nseg < 1 || g.nseg > 3) return -1;
  SkParams p;
  memset(&p, 0, sizeof(p));
  p.Mp = g.M <= 64 ? 64 : 128;
  int tiles = 0;
  for (int s = 0; s < g.nseg; ++s) {
    if (g.nW[s] % 128 || (reinterpret_cast<uintptr_t>(g.W[s]) & 15)) return -1;
    if (!encode_tmap_2d_bf16(&p.tmW[s], g.W[s], (uint64_t)g.K, (uint64_t)g.nW[s], (uint64_t)g.K * 2, SK_TK, 128))
      return -1;
    tiles += (int)(g.nW[s] / 128);
    p.seg_tile_end[s] = tiles;
  }
  if (!encode_tmap_2d_bf16(&p.tmX, g.X2, (uint64_t)g.K, (uint64_t)(2 * p.Mp), (uint64_t)g.K * 2, SK_TK,
                           (uint32_t)(2 * p.Mp)))
    return -1;
  p.M = (int)g.M;
  p.K = (int)g.K;
  p.N = tiles * 128;
  p.nseg = g.nseg;
  p.n_tiles = tiles;
  const int nkb = (int)((g.K + SK_TK - 1) / SK_TK);
  const int ks = std::max(1, std::min(g.k_splits, nkb));
  p.kb_per_split = (nkb + ks - 1) / ks;
  p.k_splits = (nkb + p.kb_per_split - 1) / p.kb_per_split;
  p.num_units = p.n_tiles * p.k_splits;
  p.mode = g.mode;
  p.streamk = g.mode == 1;
  p.total_items = (int64_t)p.n_tiles * nkb;
  p.out = g.out;
  p.ldo = g.ldo;
  p.row_scale = g.row_scale;
  p.status = status;
  const uint32_t stage_bytes = SK_A_BYTES + (uint32_t)(2 * p.Mp) * SK_TK * 2;
  const uint32_t budget = 200 * 1024;
  p.stages = (int)std::min<uint32_t>(8, budget / stage_bytes);
  const uint32_t smem = p.stages * stage_bytes + 1024 + 256;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return -1;
  if (!attr_set[dev]) {
    const void* fns[3] = {(const void*)gemm_skinny_kernel<0>, (const void*)gemm_skinny_kernel<1>,
                          (const void*)gemm_skinny_kernel<2>};
    for (const void* f : fns)
      if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, budget + 1280) != cudaSuccess) return -1;
    attr_set[dev] = true;
  }
  const int grid = p.streamk ? (int)std::max<int64_t>(1, std::min<int64_t>(p.total_items, num_sms))
                             : std::max(1, std::min(p.num_units, num_sms));
  cudaError_t e;
  switch (p.mode) {
    case 0: e = launch_k(gemm_skinny_kernel<0>, dim3(grid), dim3(SK_THREADS), smem, st, p); break;
    case 1: e = launch_k(gemm_skinny_kernel<1>, dim3(grid), dim3(SK_THREADS), smem, st, p); break;
    case 2: e = launch_k(gemm_skinny_kernel<2>, dim3(grid), dim3(SK_THREADS), smem, st, p); break;
    default: return -1;
  }
  return e == cudaSuccess ? 0 : -1;
}

LLAMA_DEFINE_BOUNDS_READER(gemm_skinny)

}  // namespace llama
