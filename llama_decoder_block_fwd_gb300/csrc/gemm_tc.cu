// tcgen05 GEMM for the block's projections: D[M, N] = A[M, K] * B[N, K]^T in bf16 with an fp32
// accumulator in tensor memory, followed by one of the epilogues in epilogue.cuh (plain store,
// residual add, SiLU(gate)*up, or RoPE + KV-cache write for the fused Q/K/V projection).
//
// Design (sm_103a):
//   * persistent CTAs, one per SM, walking 128 x 256 output tiles in bands of 8 column tiles so
//     that the tiles in flight at once share their A rows and B rows in L2;
//   * warp 0: one thread issues TMA loads (128B-swizzled 128x64 boxes) into a 4-stage ring;
//   * warp 1: one thread issues tcgen05.mma (M=128, N=256, K=16) into one of two TMEM
//     accumulators (2 x 256 columns), committing each stage back to the producer;
//   * warps 2-5: read the finished accumulator with tcgen05.ld (each warp owns its 32-lane
//     quarter of TMEM), apply the epilogue and store 16-byte runs, while the MMA warp already
//     fills the other accumulator.
// B is a virtual row-concatenation of up to three weight matrices, each a multiple of 128 rows,
// loaded per 128-row half tile: Q|K|V for the fused projection, or, for SwiGLU, gate rows
// 128t..128t+127 followed by the same rows of up, so one tile holds matching gate/up columns.
#include <algorithm>
#include <cstring>

#include "epilogue.cuh"
#include "kernels.h"

namespace llama {
namespace {

constexpr int TM = 128, TK = 64, STAGES = 4, BAND = 8;   // tiles of 128 rows x 256 columns
constexpr uint32_t A_BYTES = TM * TK * 2;        // 16 KB
constexpr uint32_t BH_BYTES = 128 * TK * 2;      // 16 KB per 128-row half of B
constexpr uint32_t STAGE_BYTES = A_BYTES + 2 * BH_BYTES;
constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;

struct TcParams {   // 128-byte aligned by its tensor maps
  CUtensorMap tmA;
  CUtensorMap tmA_lo;    // dual: low bf16 part of A (A = hi + lo)
  CUtensorMap tmB[3];
  int M, K;
  int dual;              // two MMAs per k-step (A hi and A lo) into one accumulator; N tiles of 128
  int max_halves;        // 128-column halves per tile: 2, or 1 (dual / skinny)
  int k_splits, kb_per_split, num_units;
  int split_rows;        // 1: split s writes rows s*M + r (fp32 partials); 0: all splits write row r
  int n_halves;          // 128-column halves of the virtual N
  int seg_half_end[3];   // cumulative halves per B segment
  int nseg;
  int swiglu;
  int m_tiles, n_tiles, num_tiles;
  unsigned* status;
  Epi epi;
};

__device__ __forceinline__ void tile_coords(const TcParams& p, int t, int& mb, int& nb) {
  const int band_tiles = p.m_tiles * BAND;
  const int band = t / band_tiles;
  const int rem = t - band * band_tiles;
  const int gw = min(BAND, p.n_tiles - band * BAND);
  nb = band * BAND + rem % gw;
  mb = rem / gw;
}

__device__ __forceinline__ int tile_halves(const TcParams& p, int nb) {
  return p.swiglu ? 2 : min(p.max_halves, p.n_halves - p.max_halves * nb);
}

// Work unit u -> output tile and K range [kb0, kb1) in 64-wide k-blocks.
__device__ __forceinline__ void unit_coords(const TcParams& p, int u, int nkb, int& mb, int& nb, int& split, int& kb0,
                                            int& kb1) {
  const int t = u / p.k_splits;
  split = u - t * p.k_splits;
  tile_coords(p, t, mb, nb);
  kb0 = split * p.kb_per_split;
  kb1 = min(nkb, kb0 + p.kb_per_split);
}

// Rows of B segment s.
__device__ __forceinline__ int seg_rows(const TcParams& p, int s) {
  return (p.seg_half_end[s] - (s ? p.seg_half_end[s - 1] : 0)) * 128;
}

// Which B segment, and which row of it, supplies half hh of column tile nb.
__device__ __forceinline__ void half_source(const TcParams& p, int nb, int hh, int& seg, int& row) {
  if (p.swiglu) { seg = hh; row = nb * 128; return; }
  const int gh = p.max_halves * nb + hh;
  seg = 0;
  int start = 0;
  while (seg < p.nseg - 1 && gh >= p.seg_half_end[seg]) { start = p.seg_half_end[seg]; ++seg; }
  row = (gh - start) * 128;
}

__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 128); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmA);
    for (int s = 0; s < p.nseg; ++s) tma_prefetch_desc(&p.tmB[s]);
  }
  if (warp == 1) { tmem_alloc(tmem_slot, TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nkb = (p.K + TK - 1) / TK;
  const uint32_t smem_base = smem_u32(smem);

  if (warp == 0) {
    if (lane == 0) {  // ---------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
        int mb, nb, split, kb0, kb1;
        unit_coords(p, u, nkb, mb, nb, split, kb0, kb1);
        const int nvh = tile_halves(p, nb);
        int seg[2], row[2];
        for (int hh = 0; hh < nvh; ++hh) half_source(p, nb, hh, seg[hh], row[hh]);
        // stage layout: [A | B half 0 | B half 1], or with dual A: [A hi | A lo | B half 0]
        const uint32_t bytes = A_BYTES * (p.dual ? 2 : 1) + nvh * BH_BYTES;
        const uint32_t boff = p.dual ? 2 * A_BYTES : A_BYTES;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          bool inb = box_in(kb * TK, p.K, (int64_t)mb * TM, p.M);   // bounds-checking builds only
          for (int hh = 0; hh < nvh; ++hh) inb = inb && box_in(kb * TK, p.K, row[hh], seg_rows(p, seg[hh]));
          if (!inb) { *abort_flag = 1; ok = false; break; }
          mbar_arrive_expect_tx(&full[stage], bytes);
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          tma_load_2d(sa, &p.tmA, &full[stage], kb * TK, mb * TM);
          if (p.dual) tma_load_2d(sa + A_BYTES, &p.tmA_lo, &full[stage], kb * TK, mb * TM);
          for (int hh = 0; hh < nvh; ++hh)
            tma_load_2d(sa + boff + hh * BH_BYTES, &p.tmB[seg[hh]], &full[stage], kb * TK, row[hh]);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++it) {
        int mb, nb, split, kb0, kb1;
        unit_coords(p, u, nkb, mb, nb, split, kb0, kb1);
        const int nvh = tile_halves(p, nb);
        const uint32_t idesc = idesc_bf16(TM, nvh * 128);
        const int buf = it & 1;
        const uint32_t aphase = (it >> 1) & 1;
        if (!mbar_wait(&acc_empty[buf], aphase ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * 256;
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_base + stage * STAGE_BYTES;
          const uint32_t sb = sa + (p.dual ? 2 * A_BYTES : A_BYTES);
          const uint64_t ad0 = sdesc_sw128(sa, 16, 1024), bd0 = sdesc_sw128(sb, 16, 1024);
          const uint64_t ad1 = sdesc_sw128(sa + A_BYTES, 16, 1024);
#pragma unroll
          for (int k = 0; k < TK / 16; ++k) {   // +32 bytes per k-step = +2 in the address field
            tc_mma(d, ad0 + 2 * k, bd0 + 2 * k, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
            if (p.dual) tc_mma(d, ad1 + 2 * k, bd0 + 2 * k, idesc, 1u);
          }
          tc_commit(&empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
      }
      // Every MMA this thread issued has finished before TMEM is released.
      int no_abort = 0;
      tc_commit(drain);
      mbar_wait(drain, 0, &no_abort, p.status);
    }
  } else {  // ---------------- epilogue warps 2..5
    const int q = warp & 3;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int it = 0;
    for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++it) {
      int mb, nb, split, kb0, kb1;
      unit_coords(p, u, nkb, mb, nb, split, kb0, kb1);
      const int nvh = tile_halves(p, nb);
      const int buf = it & 1;
      const uint32_t aphase = (it >> 1) & 1;
      if (!mbar_wait(&acc_full[buf], aphase, abort_flag, p.status)) break;
      tc_fence_after();
      const int64_t r = (int64_t)mb * TM + q * 32 + lane;
      const bool live = r < p.M;
      const int64_t r_out = p.split_rows ? r + (int64_t)split * p.M : r;   // partials: [k_splits, M, N]
      const uint32_t tb = tmem + buf * 256 + lane_base;
      if (p.swiglu) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(tb + c * 32, g);
          tmem_ld32(tb + 128 + c * 32, u);
          tc_wait_ld();
          if (live) {
            float gv[32], uv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) { gv[i] = __uint_as_float(g[i]); uv[i] = __uint_as_float(u[i]); }
            epi_run<32>(p.epi, r, (int64_t)nb * 128 + c * 32, gv, uv);
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < nvh * 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tb + c * 32, v);
          tc_wait_ld();
          if (live) {
            float fv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) fv[i] = __uint_as_float(v[i]);
            epi_run<32>(p.epi, r_out, (int64_t)nb * 128 * p.max_halves + c * 32, fv, fv);
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
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

int gemm_tc_effective_splits(int64_t K, int requested) {
  const int nkb = (int)((K + TK - 1) / TK);
  const int ks = std::max(1, std::min(requested, nkb));
  const int kbps = (nkb + ks - 1) / ks;
  return (nkb + kbps - 1) / kbps;
}

bool gemm_tc_supported(const GemmDesc& g) {
  if (g.dtype != LLAMA_BF16 || g.M <= 0 || g.K <= 0 || g.K % 8 != 0 || g.lda != g.K) return false;
  if (g.A_lo && ((reinterpret_cast<uintptr_t>(g.A_lo) & 15) || g.epi.kind == EPI_SWIGLU)) return false;
  if (g.k_splits > 1 && ((g.epi.kind != EPI_STORE && g.epi.kind != EPI_ATOMIC) || !g.epi.out_f32 || g.epi.row_scale))
    return false;
  if (g.K > (int64_t)1 << 30 || g.M > (int64_t)1 << 30) return false;
  if (reinterpret_cast<uintptr_t>(g.A) & 15) return false;
  const int ns = g.epi.kind == EPI_SWIGLU ? 2 : g.nseg;
  if (ns < 1 || ns > 3) return false;
  for (int s = 0; s < ns; ++s) {
    if (g.nB[s] <= 0 || g.nB[s] % 128 != 0 || (reinterpret_cast<uintptr_t>(g.B[s]) & 15)) return false;
  }
  if (g.epi.kind == EPI_SWIGLU && g.nB[0] != g.nB[1]) return false;
  const Epi& e = g.epi;
  // 16-byte runs of the output (and the residual) must stay aligned
  const int osz = e.out_f32 ? 4 : 2;
  if (e.kind != EPI_QKV && ((e.ldo * osz) % 16 != 0 || (reinterpret_cast<uintptr_t>(e.out) & 15))) return false;
  if (e.kind == EPI_RESID && (((e.ldr * (e.resid_f32 ? 4 : 2)) % 16) != 0 || (reinterpret_cast<uintptr_t>(e.resid) & 15)))
    return false;
  if (e.kind == EPI_ATOMIC && !e.out_f32) return false;
  if (e.kind == EPI_QKV && (e.nq_cols % 128 != 0 || e.nkv_cols % 128 != 0 || e.out_f32)) return false;
  return true;
}

int launch_gemm_tc(const GemmDesc& g, int num_sms, unsigned* status, cudaStream_t st) {
  TcParams p;
  memset(&p, 0, sizeof(p));
  const int ns = g.epi.kind == EPI_SWIGLU ? 2 : g.nseg;
  if (!encode_tmap_2d_bf16(&p.tmA, g.A, (uint64_t)g.K, (uint64_t)g.M, (uint64_t)g.lda * 2, TK, TM)) return -1;
  p.dual = g.A_lo != nullptr;
  if (p.dual && !encode_tmap_2d_bf16(&p.tmA_lo, g.A_lo, (uint64_t)g.K, (uint64_t)g.M, (uint64_t)g.lda * 2, TK, TM))
    return -1;
  p.max_halves = (p.dual || g.narrow) ? 1 : 2;
  int64_t halves = 0;
  for (int s = 0; s < ns; ++s) {
    if (!encode_tmap_2d_bf16(&p.tmB[s], g.B[s], (uint64_t)g.K, (uint64_t)g.nB[s], (uint64_t)g.K * 2, TK, 128))
      return -1;
    halves += g.nB[s] / 128;
    p.seg_half_end[s] = (int)halves;
  }
  p.M = (int)g.M;
  p.K = (int)g.K;
  p.nseg = ns;
  p.swiglu = g.epi.kind == EPI_SWIGLU;
  p.n_halves = (int)halves;
  p.m_tiles = (int)((g.M + TM - 1) / TM);
  p.n_tiles = p.swiglu ? (int)(g.nB[0] / 128) : (int)((halves + p.max_halves - 1) / p.max_halves);
  p.num_tiles = p.m_tiles * p.n_tiles;
  const int nkb = (int)((g.K + TK - 1) / TK);
  const int ks = std::max(1, std::min(g.k_splits, nkb));
  p.kb_per_split = (nkb + ks - 1) / ks;
  p.k_splits = (nkb + p.kb_per_split - 1) / p.kb_per_split;
  p.num_units = p.num_tiles * p.k_splits;
  p.split_rows = (p.k_splits > 1 && g.epi.kind == EPI_STORE) ? 1 : 0;
  p.status = status;
  p.epi = g.epi;
  epi_set_extents(p.epi, g.M, p.split_rows ? g.M * p.k_splits : g.M);
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return -1;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess)
      return -1;
    attr_set[dev] = true;
  }
  const int grid = std::max(1, std::min(p.num_units, num_sms));
  gemm_tc_kernel<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(p);
  return 0;
}

LLAMA_DEFINE_BOUNDS_READER(gemm_tc)

}  // namespace llama
