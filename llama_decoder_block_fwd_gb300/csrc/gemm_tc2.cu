// tcgen05 GEMM on SM pairs (cta_group::2) for the prefill projections:
// D[M, N] = A[M, K] * B[N, K]^T, bf16 operands, fp32 accumulation, same epilogues as gemm_tc.cu.
//
// A cluster of two CTAs owns a 256 x 256 output tile.  CTA r (r = 0, 1) stages rows
// 128r..128r+127 of the A tile and the r-th 128-row half of the B tile; the leader (r = 0) issues
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16), which reads both CTAs' shared memory and
// leaves rows 128r.. of the accumulator in CTA r's tensor memory.  Per SM and k-step this moves
// half the B bytes of the one-SM 128 x 256 tile through shared memory, which is what lets the
// tensor pipe run near its rate.
//   * TMA loads of both CTAs complete on the leader's stage barrier (.cta_group::2 form);
//   * the leader's commits are multicast to the stage and accumulator barriers of both CTAs;
//   * both CTAs' epilogue threads release an accumulator on the leader's barrier.
// Tiles are walked in bands of column tiles (kBandBytes below); the grid holds as many clusters
// as can be resident at once (persistent).
#include <algorithm>
#include <cstring>

#include "epilogue.cuh"
#include "kernels.h"

namespace llama {
namespace {

constexpr int T2M = 256, T2N = 256, T2K = 64, S2 = 6;
// Tile order.  Tiles are walked in bands so that one operand's band stays in L2 while the other
// operand streams past it once per band:
//   * column bands (the default): a band of column tiles, row tiles inside it; the weight rows of
//     the band stay resident and the activations are read once per band.  The band is as wide as
//     kBandBytes of weights allows, and at least 8 tiles.
//   * row bands, when the weights are more than twice the activations (the gate/up projection):
//     a band of row tiles whose activation rows stay resident, column tiles inside it (the row
//     tiles of the band take each column tile together, so its weights come from DRAM once per
//     band); the weights are read once per band of kRowBandBytes of activations.
constexpr int64_t kBandBytes = 48ll << 20;
constexpr int64_t kRowBandBytes = 32ll << 20;
constexpr uint32_t A2_BYTES = 128 * T2K * 2;    // this CTA's 128 rows of A: 16 KB
constexpr uint32_t B2_BYTES = 128 * T2K * 2;    // this CTA's 128-row half of B: 16 KB
constexpr uint32_t STAGE2 = A2_BYTES + B2_BYTES;
constexpr uint32_t SMEM2 = S2 * STAGE2 + 1024 + 256;
constexpr int THREADS2 = 320;   // TMA warp, MMA warp, 8 epilogue warps
constexpr uint32_t TMEM2_COLS = 512;

struct Tc2Params {   // 128-byte aligned by its tensor maps
  CUtensorMap tmA;
  CUtensorMap tmB[3];
  int M, K;
  int n_halves;
  int seg_half_end[3];
  int nseg;
  int swiglu;
  int m_tiles, n_tiles, num_tiles;
  int band;             // column tiles per band (column bands)
  int row_band;         // > 0: row tiles per band (row bands)
  unsigned* status;
  Epi epi;
};

__device__ __forceinline__ void tile2_coords(const Tc2Params& p, int t, int& mb, int& nb) {
  if (p.row_band > 0) {
    const int band_tiles = p.n_tiles * p.row_band;
    const int band = t / band_tiles;
    const int rem = t - band * band_tiles;
    const int gh = min(p.row_band, p.m_tiles - band * p.row_band);
    mb = band * p.row_band + rem % gh;
    nb = rem / gh;
    return;
  }
  const int band_tiles = p.m_tiles * p.band;
  const int band = t / band_tiles;
  const int rem = t - band * band_tiles;
  const int gw = min(p.band, p.n_tiles - band * p.band);
  nb = band * p.band + rem % gw;
  mb = rem / gw;
}

__device__ __forceinline__ void half2_source(const Tc2Params& p, int nb, int hh, int& seg, int& row) {
  if (p.swiglu) { seg = hh; row = nb * 128; return; }
  const int gh = 2 * nb + hh;
  seg = 0;
  int start = 0;
  while (seg < p.nseg - 1 && gh >= p.seg_half_end[seg]) { start = p.seg_half_end[seg]; ++seg; }
  row = (gh - start) * 128;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait with cluster-scope acquire (for barriers that receive the peer CTA's arrivals).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  unsigned* status) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait_cluster(a, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(a, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicOr(status, STATUS_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* m, uint32_t leader_bar, int x,
                                                 int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(leader_bar)
      : "memory");
}
__device__ __forceinline__ void tc2_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the barrier at this shared-memory offset in every CTA of `mask` once all tcgen05
// operations issued so far by this thread have completed.
__device__ __forceinline__ void tc2_commit_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS2, 1)
    gemm_tc2_kernel(const __grid_constant__ Tc2Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S2 * STAGE2);   // used in the leader
  uint64_t* empty = full + S2;                                         // both CTAs
  uint64_t* acc_full = empty + S2;                                     // both CTAs
  uint64_t* acc_empty = acc_full + 2;                                  // used in the leader
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  // programmatic dependent launch: the next kernel may be scheduled as soon as every CTA of this
  // one has started (it waits in its own pdl_wait until this grid has completed)
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int cluster_id = (int)(blockIdx.x >> 1), n_clusters = (int)(gridDim.x >> 1);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S2; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 2 * 256); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmA);
    for (int s = 0; s < p.nseg; ++s) tma_prefetch_desc(&p.tmB[s]);
  }
  if (warp == 1) {   // one warp in each CTA of the pair allocates, jointly
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM2_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync_all();     // barriers of both CTAs initialised before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int nkb = (p.K + T2K - 1) / T2K;
  const uint32_t smem_base = smem_u32(smem);
  // The set-up above overlapped the previous kernel's tail; past pdl_wait its outputs are visible.
  // The producer first issues the weight halves of its first stages (no kernel writes weights),
  // then waits.
  if (warp != 0 || lane != 0) pdl_wait();

  if (warp == 0) {
    if (lane == 0) {  // ---------------- TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      int pre = 0;   // stages of the first tile whose weights went out before pdl_wait
      if (cluster_id < p.num_tiles) {
        int mb, nb, seg, row;
        tile2_coords(p, cluster_id, mb, nb);
        half2_source(p, nb, (int)rank, seg, row);
        const int seg_rows = (p.seg_half_end[seg] - (seg ? p.seg_half_end[seg - 1] : 0)) * 128;
        for (; pre < min(S2, nkb); ++pre) {   // fresh stages: nothing to wait for
          if (!box_in(pre * T2K, p.K, row, seg_rows)) break;   // bounds-checking builds
          if (leader) mbar_arrive_expect_tx(&full[pre], 2 * STAGE2);   // both CTAs' bytes
          tma_load_2d_pair(smem_base + pre * STAGE2 + A2_BYTES, &p.tmB[seg], map_to_rank(smem_u32(&full[pre]), 0),
                           pre * T2K, row);
        }
      }
      pdl_wait();
      bool first_tile = true;
      for (int t = cluster_id; t < p.num_tiles; t += n_clusters) {
        int mb, nb, seg, row;
        tile2_coords(p, t, mb, nb);
        half2_source(p, nb, (int)rank, seg, row);
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (first_tile && kb < pre) {   // its weights are on their way: the activations only
            if (!box_in(kb * T2K, p.K, (int64_t)mb * T2M, p.M)) { *abort_flag = 1; ok = false; break; }
            tma_load_2d_pair(smem_base + stage * STAGE2, &p.tmA, map_to_rank(smem_u32(&full[stage]), 0), kb * T2K,
                             mb * T2M + (int)rank * 128);
            if (++stage == S2) { stage = 0; phase ^= 1; }
            continue;
          }
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          // bounds-checking builds: the tile's start in A (the second CTA's 128-row half of a ragged
          // last tile may lie past M by design: the load fills zeros) and this CTA's B half
          if (!box_in(kb * T2K, p.K, (int64_t)mb * T2M, p.M) ||
              !box_in(kb * T2K, p.K, row, (p.seg_half_end[seg] - (seg ? p.seg_half_end[seg - 1] : 0)) * 128)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          const uint32_t lbar = map_to_rank(smem_u32(&full[stage]), 0);
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * STAGE2);   // both CTAs' bytes
          const uint32_t sa = smem_base + stage * STAGE2;
          tma_load_2d_pair(sa, &p.tmA, lbar, kb * T2K, mb * T2M + (int)rank * 128);
          tma_load_2d_pair(sa + A2_BYTES, &p.tmB[seg], lbar, kb * T2K, row);
          if (++stage == S2) { stage = 0; phase ^= 1; }
        }
        first_tile = false;
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {  // ---------------- MMA issuer (leader CTA only)
      const uint32_t idesc = idesc_bf16(T2M, T2N);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int t = cluster_id; t < p.num_tiles; t += n_clusters, ++it) {
        const int buf = it & 1;
        const uint32_t aphase = (it >> 1) & 1;
        if (!mbar_wait_cluster(&acc_empty[buf], aphase ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + buf * 256;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_cluster(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_base + stage * STAGE2;
          const uint32_t sb = sa + A2_BYTES;
          const uint64_t ad0 = sdesc_sw128(sa, 16, 1024), bd0 = sdesc_sw128(sb, 16, 1024);
#pragma unroll
          for (int k = 0; k < T2K / 16; ++k)   // +32 bytes per k-step = +2 in the address field
            tc2_mma(d, ad0 + 2 * k, bd0 + 2 * k, idesc, (kb | k) != 0);
          tc2_commit_mc(&empty[stage], 0x3);
          if (++stage == S2) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc2_commit_mc(&acc_full[buf], 0x3);
      }
      int no_abort = 0;
      tc2_commit_mc(drain, 0x1);
      mbar_wait(drain, 0, &no_abort, p.status);
    }
  } else {  // ---------------- epilogue warps 2..9 (both CTAs)
    // Warp w reads TMEM lanes 32 (w % 4) .. +31 (the lane quarter a warp may access) and column
    // half (w - 2) / 4 of the tile: two warps per lane quarter halve each warp's serial chain of
    // TMEM loads, global loads and stores per tile.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int it = 0;
    for (int t = cluster_id; t < p.num_tiles; t += n_clusters, ++it) {
      int mb, nb;
      tile2_coords(p, t, mb, nb);
      const int buf = it & 1;
      const uint32_t aphase = (it >> 1) & 1;
      if (!mbar_wait(&acc_full[buf], aphase, abort_flag, p.status)) break;
      tc_fence_after();
      const int64_t r = (int64_t)mb * T2M + rank * 128 + q * 32 + lane;
      const bool live = r < p.M;
      const uint32_t tb = tmem + buf * 256 + lane_base;
      if (p.swiglu) {
        float rs = 1.f;
        if (p.epi.ss_in && live) {   // the row's RMSNorm factor from the producing GEMM's partial sums
          float ss = 0.f;
          const float* sp = p.epi.ss_in + r * p.epi.ss_n;
          if ((p.epi.ss_n & 3) == 0) {
            for (int j = 0; j < p.epi.ss_n; j += 4) {
              const float4 t4 = __ldg(reinterpret_cast<const float4*>(sp + j));
              ss += (t4.x + t4.y) + (t4.z + t4.w);
            }
          } else {
            for (int j = 0; j < p.epi.ss_n; ++j) ss += __ldg(sp + j);
          }
          rs = rsqrtf(ss * p.epi.ss_inv_d + p.epi.ss_eps);
        }
#pragma unroll 1
        for (int c = 2 * half; c < 2 * half + 2; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(tb + c * 32, g);
          tmem_ld32(tb + 128 + c * 32, u);
          tc_wait_ld();
          if (live) {
            float gv[32], uv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) { gv[i] = __uint_as_float(g[i]); uv[i] = __uint_as_float(u[i]); }
            epi_run<32>(p.epi, r, (int64_t)nb * 128 + c * 32, gv, uv, rs);
          }
        }
      } else {
        float ssq = 0.f;
#pragma unroll 1
        for (int c = 4 * half; c < 4 * half + 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tb + c * 32, v);
          tc_wait_ld();
          if (live) {
            float fv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) fv[i] = __uint_as_float(v[i]);
            ssq += epi_run<32>(p.epi, r, (int64_t)nb * T2N + c * 32, fv, fv);
          }
        }
        if (p.epi.ss_out && live && in_extent(r * p.epi.ss_n + 2 * nb + half, 1, p.epi.M * p.epi.ss_n))
          p.epi.ss_out[r * p.epi.ss_n + 2 * nb + half] = ssq;
      }
      tc_fence_before();
      mbar_arrive_cluster(map_to_rank(smem_u32(&acc_empty[buf]), 0));
    }
  }
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();    // the pair is done with tensor memory and with each other's barriers
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM2_COLS) : "memory");
  }
}

}  // namespace

bool gemm_tc2_supported(const GemmDesc& g) {
  if (!gemm_tc_supported(g) || g.A_lo || g.k_splits > 1 || g.narrow) return false;
  if (g.M < 256) return false;
  const int ns = g.epi.kind == EPI_SWIGLU ? 2 : g.nseg;
  int64_t halves = 0;
  for (int s = 0; s < ns; ++s) halves += g.nB[s] / 128;
  return g.epi.kind == EPI_SWIGLU || halves % 2 == 0;   // every tile has both 128-row halves
}

int launch_gemm_tc2(const GemmDesc& g, unsigned* status, cudaStream_t st) {
  Tc2Params p;
  memset(&p, 0, sizeof(p));
  const int ns = g.epi.kind == EPI_SWIGLU ? 2 : g.nseg;
  if (!encode_tmap_2d_bf16(&p.tmA, g.A, (uint64_t)g.K, (uint64_t)g.M, (uint64_t)g.lda * 2, T2K, 128)) return -1;
  int64_t halves = 0;
  for (int s = 0; s < ns; ++s) {
    if (!encode_tmap_2d_bf16(&p.tmB[s], g.B[s], (uint64_t)g.K, (uint64_t)g.nB[s], (uint64_t)g.K * 2, T2K, 128))
      return -1;
    halves += g.nB[s] / 128;
    p.seg_half_end[s] = (int)halves;
  }
  p.M = (int)g.M;
  p.K = (int)g.K;
  p.nseg = ns;
  p.swiglu = g.epi.kind == EPI_SWIGLU;
  p.n_halves = (int)halves;
  p.m_tiles = (int)((g.M + T2M - 1) / T2M);
  p.n_tiles = p.swiglu ? (int)(g.nB[0] / 128) : (int)(halves / 2);
  p.num_tiles = p.m_tiles * p.n_tiles;
  // bytes of one column tile's weights (256 rows; gate and up: 128 rows of each) and of one row
  // tile's activations (256 rows), both K bf16
  const int64_t tile_bytes = 256 * g.K * 2;
  const int64_t w_bytes = (int64_t)p.n_tiles * tile_bytes, a_bytes = (int64_t)p.m_tiles * tile_bytes;
  p.band = (int)std::min<int64_t>(p.n_tiles, std::max<int64_t>(8, kBandBytes / tile_bytes));
  p.row_band = w_bytes > 2 * a_bytes ? (int)std::max<int64_t>(1, std::min<int64_t>(p.m_tiles, kRowBandBytes / tile_bytes)) : 0;
  p.status = status;
  p.epi = g.epi;
  epi_set_extents(p.epi, g.M, g.M);
  int dev = 0;
  cudaGetDevice(&dev);
  static int max_clusters[64] = {};
  if (dev < 0 || dev >= 64) return -1;
  if (!max_clusters[dev]) {
    if (cudaFuncSetAttribute(gemm_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM2) != cudaSuccess)
      return -1;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(2 * 128, 1, 1);
    cfg.blockDim = dim3(THREADS2, 1, 1);
    cfg.dynamicSmemBytes = SMEM2;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc2_kernel, &cfg) != cudaSuccess || n <= 0) return -1;
    max_clusters[dev] = n;
  }
  const int clusters = std::max(1, std::min(p.num_tiles, max_clusters[dev]));
  return launch_k(gemm_tc2_kernel, dim3(2 * clusters), dim3(THREADS2), SMEM2, st, p) == cudaSuccess ? 0 : -1;
}

LLAMA_DEFINE_BOUNDS_READER(gemm_tc2)

}  // namespace llama
