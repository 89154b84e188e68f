// The two steps either side of the decode stack ("LLaMA-3 8B 现代 LLM 架构、计算规模与能耗",
// sections 三 and 十): the embedding lookup x[b] = E[token_b], and the choice of the next token
// from the LM head's logits by argmax, or by a draw from softmax(z / T) restricted by top-k and
// top-p.
//
// Ranking: tokens are ordered by logit (larger first), ties by the lower token id; top-k keeps
// the first k of that order; top-p (after top-k) keeps the shortest prefix whose share of the
// top-k mass reaches p; the draw walks the kept tokens in increasing id and stops at the first
// whose cumulative mass exceeds u times the kept mass (u in [0, 1) is supplied by the caller).
//
// A cluster of P CTAs per row (P up to 8, chosen so that the B x P CTAs cover the SMs; P = 1 for
// rows that are not 16-byte aligned or for the general path below).  Each CTA takes 1/P of the row
// for the argmax pass; the partial maxima are exchanged through distributed shared memory.
// Top-k up to 1024 (the usual case): the argmax pass also keeps every thread's two largest logits;
// the k-th largest of those bounds the k-th largest logit of the CTA's part of the row from below,
// so a second pass over that part (from L2) gathers the few tokens at or above the bound into the
// CTA's shared memory.  Every token of the row's top k is among the top k of its own part, hence
// gathered; the cluster's leader CTA copies the other CTAs' candidates into its own shared memory
// and ranks them all by a bitonic sort.  Otherwise (or when too many tokens tie near the bound) the
// thresholds are found by radix selection on an order-preserving 32-bit key of the logit, four
// 8-bit digits from the top: by count for top-k, by probability mass for top-p, one pass over the
// row (from L2) per digit.  Masses are exp((z - z_max) / T) in fp32, held as 2^-40 fixed point in
// 64-bit integers so that every sum is exact and independent of the order of the atomic adds: the
// same logits always give the same token.  Terms below 2^-40 of the largest count as zero.
#include <cooperative_groups.h>

#include <climits>

#include "kernels.h"

namespace llama {
namespace {

constexpr int SP_THREADS = 1024;
constexpr int SP_WARPS = SP_THREADS / 32;
constexpr float kMassOne = 1099511627776.0f;   // 2^40
using u64 = unsigned long long;

__device__ __forceinline__ uint32_t order_key(float z) {
  const uint32_t b = __float_as_uint(z == 0.f ? 0.f : z);   // -0 ranks as +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

constexpr int SP_SMALL_K = 1024;   // top-k up to this: ranked in shared memory
constexpr int SP_CAP = 4096;       // candidates gathered into shared memory at most
constexpr int SP_BUCKETS = 256;    // top-p buckets of (z_max - z) / T, 1/8 wide: [0, 32) holds every nonzero mass
// dynamic shared memory: candidate keys, their logits and ranked masses; the per-warp top-p
// bucket mass histograms use the same bytes before any candidate is gathered
constexpr size_t SP_CAND_SMEM = SP_CAP * 8 + SP_CAP * 4 + SP_SMALL_K * 8;
constexpr size_t SP_BUCKET_SMEM = (size_t)SP_WARPS * SP_BUCKETS * 8;
constexpr size_t SP_DYN_SMEM = SP_CAND_SMEM > SP_BUCKET_SMEM ? SP_CAND_SMEM : SP_BUCKET_SMEM;

struct SampleShared {
  u64 hmass[256];
  unsigned hcnt[256];
  unsigned ccount;
  unsigned cbin, ctotal;
  u64 wsum[SP_WARPS];
  float wval[SP_WARPS];
  int widx[SP_WARPS];
  u64 b64[4];
  unsigned b32[4];
  int bidx;
  float cval;   // this CTA's part of the row: its largest logit and that logit's lowest id
  int cidx;
};

// Exclusive prefix sum of v over the threads in id order; *total gets the block's sum.
__device__ u64 block_scan_excl(u64 v, SampleShared& sh, u64* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  u64 x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const u64 y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh.wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    u64 w = sh.wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const u64 y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh.wsum[lane] = w;
  }
  __syncthreads();
  const u64 before = warp ? sh.wsum[warp - 1] : 0ull;
  *total = sh.wsum[SP_WARPS - 1];
  __syncthreads();
  return before + x - v;
}

// Warp 0: walking the 256 digit bins from the largest digit down, find the bin in which the
// running sum first reaches `target` (>= 1).  Returns through sh.b32[0] (digit), sh.b64[0] (the
// sum of the bins above it), sh.b32[1] (its count) and sh.b64[1] (its mass).
template <bool MASS>
__device__ void select_digit(SampleShared& sh, u64 target) {
  const int lane = threadIdx.x & 31;
  u64 mine = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int dg = 255 - (lane * 8 + j);
    mine += MASS ? sh.hmass[dg] : (u64)sh.hcnt[dg];
  }
  u64 incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const u64 y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const u64 before = incl - mine;
  if (before < target && target <= incl) {
    u64 acc = before;
    for (int j = 0; j < 8; ++j) {
      const int dg = 255 - (lane * 8 + j);
      const u64 c = MASS ? sh.hmass[dg] : (u64)sh.hcnt[dg];
      if (acc + c >= target) {
        sh.b32[0] = (unsigned)dg;
        sh.b64[0] = acc;
        sh.b32[1] = sh.hcnt[dg];
        sh.b64[1] = sh.hmass[dg];
        break;
      }
      acc += c;
    }
  }
}

// Call f(i, z_i, valid) for every element of the float4 units [q_lo, q_hi) of the row, and, when
// `tail`, for its last V % 4 elements: 16-byte loads, two in flight per thread, the same trip count
// on every lane of a warp (f may use warp-collective operations); `valid` is false on the padding
// calls.  z must be 16-byte aligned.
template <typename F>
__device__ __forceinline__ void row_pass4(const float* __restrict__ z, int V, int q_lo, int q_hi, bool tail, F&& f) {
  const int lane = threadIdx.x & 31;
  const int nv4 = V >> 2;
  const float4* z4 = reinterpret_cast<const float4*>(z);
  for (int base = q_lo + (int)(threadIdx.x & ~31u); base < q_hi; base += 2 * SP_THREADS) {
    const int q0 = base + lane, q1 = base + SP_THREADS + lane;
    const bool ok0 = q0 < q_hi, ok1 = q1 < q_hi;
    const float4 w0 = ok0 ? __ldg(z4 + q0) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 w1 = ok1 ? __ldg(z4 + q1) : make_float4(0.f, 0.f, 0.f, 0.f);
    f(4 * q0, w0.x, ok0); f(4 * q0 + 1, w0.y, ok0); f(4 * q0 + 2, w0.z, ok0); f(4 * q0 + 3, w0.w, ok0);
    if (base + SP_THREADS < q_hi) {   // warp-uniform
      f(4 * q1, w1.x, ok1); f(4 * q1 + 1, w1.y, ok1); f(4 * q1 + 2, w1.z, ok1); f(4 * q1 + 3, w1.w, ok1);
    }
  }
  if (tail && threadIdx.x < 32) {   // the last V % 4 elements
    const int i = 4 * nv4 + lane;
    const bool ok = i < V;
    f(i, ok ? z[i] : 0.f, ok);
  }
}

// A walk over the float4 units [q_lo, q_hi) with U loads in flight per thread: one call
// f4(q, w, valid) per unit q, a thread's units in increasing q, the same calls on every lane of a
// warp (f4 may use warp-collective operations).  U x 16 KB per CTA in flight keeps a pass from being
// bound by load latency (a row part is only a few such rounds).
template <int U, typename F4>
__device__ __forceinline__ void row_pass_f4(const float* __restrict__ z, int q_lo, int q_hi, F4&& f4) {
  const int lane = threadIdx.x & 31;
  const float4* z4 = reinterpret_cast<const float4*>(z);
  for (int base = q_lo + (int)(threadIdx.x & ~31u); base < q_hi; base += U * SP_THREADS) {
    float4 w[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int q = base + j * SP_THREADS + lane;
      w[j] = q < q_hi ? __ldg(z4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int q = base + j * SP_THREADS + lane;
      if (base + j * SP_THREADS < q_hi) f4(q, w[j], q < q_hi);   // warp-uniform
    }
  }
}

__device__ __forceinline__ float max4(const float4& w) { return fmaxf(fmaxf(w.x, w.y), fmaxf(w.z, w.w)); }

// row_pass4 over the whole of a 16-byte aligned row, else one element per thread and step (same
// contract).
template <typename F>
__device__ __forceinline__ void row_each(const float* __restrict__ z, int V, bool vec, F&& f) {
  if (vec) {
    row_pass4(z, V, 0, V >> 2, true, f);
  } else {
    for (int base = (int)(threadIdx.x & ~31u); base < V; base += SP_THREADS) {
      const int i = base + (int)(threadIdx.x & 31);
      f(i, i < V ? z[i] : 0.f, i < V);
    }
  }
}

// Bitonic sort of ckey[0, n2) into descending order (n2 a power of two), cz moved alongside.
__device__ void sort_desc(u64* ckey, float* cz, int n2) {
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < n2; t += SP_THREADS) {
        const int o = t ^ stride;
        if (o > t) {
          const bool desc = (t & size) == 0;
          const u64 a = ckey[t], c = ckey[o];
          if (desc ? (a < c) : (a > c)) {
            ckey[t] = c; ckey[o] = a;
            const float fz = cz[t]; cz[t] = cz[o]; cz[o] = fz;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Sort of n <= SP_THREADS distinct keys by rank: thread t counts the keys that go before its own and
// moves its entry there (one barrier, against a bitonic network's log^2 n).  Worth it for short
// lists only, since every thread reads all n keys.  DESC: larger keys first.  cz (may be null) moves
// alongside.
template <bool DESC>
__device__ void sort_by_rank(u64* ckey, float* cz, int n) {
  const int t = threadIdx.x;
  const u64 mine = t < n ? ckey[t] : 0ull;
  const float mz = (cz && t < n) ? cz[t] : 0.f;
  int r = 0;
  if (t < n)
    for (int j = 0; j < n; ++j) r += DESC ? (ckey[j] > mine) : (ckey[j] < mine);
  __syncthreads();
  if (t < n) {
    ckey[r] = mine;
    if (cz) cz[r] = mz;
  }
  __syncthreads();
}
constexpr int SP_RANK_SORT_MAX = 256;

// The id of the n-th (1-based) token, in increasing id, for which pred(i, z_i) holds.
template <typename Pred>
__device__ int nth_index(const float* z, int V, int n, Pred pred, SampleShared& sh) {
  const int seg = (V + SP_THREADS - 1) / SP_THREADS;
  const int lo = min(V, (int)threadIdx.x * seg), hi = min(V, lo + seg);
  unsigned c = 0;
  for (int i = lo; i < hi; ++i) c += pred(i, z[i]) ? 1u : 0u;
  u64 total;
  const u64 before = block_scan_excl(c, sh, &total);
  if (before < (u64)n && (u64)n <= before + c) {
    u64 acc = before;
    for (int i = lo; i < hi; ++i) {
      if (pred(i, z[i]) && ++acc == (u64)n) { sh.bidx = i; break; }
    }
  }
  __syncthreads();
  const int r = sh.bidx;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(SP_THREADS) sample_kernel(const float* __restrict__ logits, int64_t ld, int V,
                                                            float temperature, int top_k, float top_p,
                                                            const float* __restrict__ uniforms, int* __restrict__ tokens) {
  __shared__ SampleShared sh;
  namespace cg = cooperative_groups;
  const cg::cluster_group cl = cg::this_cluster();
  const int P = (int)cl.num_blocks(), cr = (int)cl.block_rank();   // P = 1 without a cluster launch
  const int row = blockIdx.x / P, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* z = logits + (int64_t)row * ld;

  // ---- the largest logit and its lowest id (argmax); CTA cr of the cluster takes the float4
  //      units [q_lo, q_hi) and, the last one, the V % 4 tail (P > 1 only for aligned rows)
  const bool vec = (reinterpret_cast<uintptr_t>(z) & 15) == 0;
  const int nv4 = V >> 2, per_cta = (nv4 + P - 1) / P;
  const int q_lo = min(nv4, cr * per_cta), q_hi = min(nv4, q_lo + per_cta);
  const bool tail = cr == P - 1;

  // small top-k: the argmax pass also keeps each thread's two largest logits; the k-th largest
  // of those 2 x SP_THREADS values bounds the k-th largest logit from below, so one more pass
  // gathers every token at or above it and the ranking is finished in shared memory
  const bool small_k = vec && temperature > 0.f && top_k >= 2 && top_k <= SP_SMALL_K && top_k < V && top_p > 0.f;
  extern __shared__ uint8_t dyn[];
  u64* ckey = reinterpret_cast<u64*>(dyn);
  float* cz = reinterpret_cast<float*>(dyn + SP_CAP * 8);
  u64* cmass = reinterpret_cast<u64*>(dyn + SP_CAP * 8 + SP_CAP * 4);
  float best = -INFINITY, second = -INFINITY;
  int bi = INT_MAX;
  if (vec) {
    auto upd = [&](int i, float v, bool ok) {
      if (!ok) return;
      if (v > best || (v == best && i < bi)) { second = best; best = v; bi = i; }
      else if (v > second) { second = v; }
    };
    // a unit whose largest value is not above the thread's second largest changes nothing (the
    // thread visits ids in increasing order, so an equal maximum found later keeps the lower id)
    row_pass_f4<8>(z, q_lo, q_hi, [&](int q, const float4& w, bool ok) {
      if (!ok || !(max4(w) > second)) return;
      upd(4 * q, w.x, true); upd(4 * q + 1, w.y, true); upd(4 * q + 2, w.z, true); upd(4 * q + 3, w.w, true);
    });
    row_pass4(z, V, q_hi, q_hi, tail, upd);   // the V % 4 tail
  } else {
    for (int i = tid; i < V; i += SP_THREADS) {
      const float v = z[i];
      if (v > best || (v == best && i < bi)) { best = v; bi = i; }
    }
  }
  const uint32_t top2_key[2] = {order_key(best), order_key(second)};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
  }
  if (lane == 0) { sh.wval[warp] = best; sh.widx[warp] = bi; }
  __syncthreads();
  best = sh.wval[0];
  bi = sh.widx[0];
  for (int w = 1; w < SP_WARPS; ++w) {
    if (sh.wval[w] > best || (sh.wval[w] == best && sh.widx[w] < bi)) { best = sh.wval[w]; bi = sh.widx[w]; }
  }
  if (P > 1) {   // the row's maximum from the CTAs' maxima (each CTA reads them all)
    if (tid == 0) { sh.cval = best; sh.cidx = bi; }
    cl.sync();
    for (int r = 0; r < P; ++r) {
      const float ov = *cl.map_shared_rank(&sh.cval, r);
      const int oi = *cl.map_shared_rank(&sh.cidx, r);
      if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
    }
    cl.sync();   // no CTA leaves, or overwrites sh, while another still reads it
  }
  const float zmax = best;
  if (!(temperature > 0.f) || top_k == 1 || !(top_p > 0.f) || !isfinite(zmax) || V == 1) {
    if (tid == 0 && cr == 0 && in_extent(row, 1, gridDim.x / P)) tokens[row] = bi == INT_MAX ? 0 : bi;
    return;
  }
  auto mass = [&](float v) -> u64 { return __float2ull_rz(expf((v - zmax) / temperature) * kMassOne); };

  if (small_k) {
    // ---- the gather threshold: the upper 16 bits of the k-th largest of the per-thread top-2
    //      keys (radix selection, two 8-bit digits).  At least top_k tokens have a key at or
    //      above it (a thread with fewer than two tokens holds -inf, whose key is below all others)
    uint32_t prefix = 0u, pmask = 0u;
    u64 remaining = (u64)top_k;
    for (int shift = 24; shift >= 16; shift -= 8) {
      for (int i = tid; i < 256; i += SP_THREADS) sh.hcnt[i] = 0u;
      __syncthreads();
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t key = top2_key[j];
        const bool hit = (key & pmask) == prefix;
        const unsigned hm = __ballot_sync(0xffffffffu, hit);
        if (hit) {
          const uint32_t bin = (key >> shift) & 255u;
          const unsigned peers = __match_any_sync(hm, bin);
          if (lane == __ffs(peers) - 1) atomicAdd(&sh.hcnt[bin], (unsigned)__popc(peers));
        }
      }
      __syncthreads();
      if (warp == 0) select_digit<false>(sh, remaining);
      __syncthreads();
      prefix |= sh.b32[0] << shift;
      pmask |= 0xFFu << shift;
      remaining -= sh.b64[0];
      __syncthreads();
    }
    const uint32_t tau = prefix;
    if (tid == 0) sh.ccount = 0u;
    __syncthreads();
    // ---- second pass (from L2): gather the tokens of this CTA's part whose key is at least tau
    auto gather = [&](int i, float v, bool ok) {
      const uint32_t key = order_key(v);
      const bool take = ok && key >= tau;
      const unsigned tm = __ballot_sync(0xffffffffu, take);
      if (tm) {   // warp-uniform
        unsigned slot0 = 0u;
        if (lane == 0) slot0 = atomicAdd(&sh.ccount, (unsigned)__popc(tm));
        slot0 = __shfl_sync(0xffffffffu, slot0, 0);
        if (take) {
          const unsigned slot = slot0 + __popc(tm & ((1u << lane) - 1u));
          if (slot < (unsigned)SP_CAP) {
            ckey[slot] = ((u64)key << 32) | (u64)(0xFFFFFFFFu - (uint32_t)i);
            cz[slot] = v;
          }
        }
      }
    };
    row_pass_f4<8>(z, q_lo, q_hi, [&](int q, const float4& w, bool ok) {
      if (!__any_sync(0xffffffffu, ok && order_key(max4(w)) >= tau)) return;   // most units: nothing to take
      gather(4 * q, w.x, ok); gather(4 * q + 1, w.y, ok); gather(4 * q + 2, w.z, ok); gather(4 * q + 3, w.w, ok);
    });
    row_pass4(z, V, q_hi, q_hi, tail, gather);   // the V % 4 tail
    __syncthreads();
    if (P > 1) {   // the leader appends the other CTAs' candidates to its own
      cl.sync();
      if (cr == 0) {
        unsigned total = sh.ccount;
        for (int r = 1; r < P; ++r) total += *cl.map_shared_rank(&sh.ccount, r);
        if (total <= (unsigned)SP_CAP) {
          unsigned at = sh.ccount;
          for (int r = 1; r < P; ++r) {
            const unsigned n_r = *cl.map_shared_rank(&sh.ccount, r);
            const u64* rk = cl.map_shared_rank(ckey, r);
            const float* rz = cl.map_shared_rank(cz, r);
            for (unsigned t = tid; t < n_r; t += SP_THREADS) { ckey[at + t] = rk[t]; cz[at + t] = rz[t]; }
            at += n_r;
          }
        }
        __syncthreads();
        if (tid == 0) sh.ccount = total;   // > SP_CAP: too many to rank here, the general path below
      }
      cl.sync();   // the others' shared memory stays until the leader has read it
      if (cr != 0) return;
      __syncthreads();
    }
    const unsigned gathered = sh.ccount;
    if (gathered <= (unsigned)SP_CAP && gathered >= (unsigned)top_k) {
      const int nc = (int)gathered;
      int n2 = 1;
      while (n2 < nc) n2 <<= 1;
      for (int t = nc + tid; t < n2; t += SP_THREADS) ckey[t] = 0ull;   // sorts after every candidate
      __syncthreads();
      // larger key first, then lower id (its complement is larger)
      if (nc <= SP_RANK_SORT_MAX) sort_by_rank<true>(ckey, cz, nc);
      else sort_desc(ckey, cz, n2);
      // the top-k set is the first top_k; masses in ranked order; the shortest prefix reaching
      // top_p of the top-k mass
      const int n = top_k;
      const u64 mt = tid < n ? mass(cz[tid]) : 0ull;
      u64 zk2;
      const u64 excl = block_scan_excl(mt, sh, &zk2);
      int n_p = n;
      if (top_p < 1.f) {
        u64 target = (u64)ceil((double)top_p * (double)zk2);
        target = target < 1ull ? 1ull : (target > zk2 ? zk2 : target);
        if (tid == 0) sh.bidx = n;
        __syncthreads();
        if (tid < n && excl < target && excl + mt >= target) sh.bidx = tid + 1;   // exactly one thread
        __syncthreads();
        n_p = sh.bidx;
        __syncthreads();
      }
      // the draw: kept tokens in increasing id, first whose cumulative mass exceeds u * kept mass
      const bool kept_t = tid < n_p;
      const uint32_t id_t = kept_t ? 0xFFFFFFFFu - (uint32_t)(ckey[tid] & 0xFFFFFFFFull) : 0xFFFFFFFFu;
      cmass[tid] = kept_t ? mt : 0ull;
      int m2 = 1;
      while (m2 < n_p) m2 <<= 1;
      __syncthreads();
      if (tid < m2) ckey[tid] = kept_t ? (((u64)id_t << 32) | (u64)tid) : ~0ull;   // (id, ranked slot)
      __syncthreads();
      if (n_p <= SP_RANK_SORT_MAX) { sort_by_rank<false>(ckey, nullptr, n_p); m2 = 0; }
      for (int size = 2; size <= m2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          for (int t = tid; t < m2; t += SP_THREADS) {
            const int o = t ^ stride;
            if (o > t) {
              const bool asc = (t & size) == 0;
              const u64 a = ckey[t], c = ckey[o];
              if (asc ? (a > c) : (a < c)) { ckey[t] = c; ckey[o] = a; }
            }
          }
          __syncthreads();
        }
      }
      const bool live = tid < n_p;
      const u64 m_id = live ? cmass[(uint32_t)(ckey[tid] & 0xFFFFFFFFull)] : 0ull;
      u64 zkept2;
      const u64 ex2c = block_scan_excl(m_id, sh, &zkept2);
      float uu = uniforms[row];
      uu = (uu >= 0.f) ? fminf(uu, 0.99999994f) : 0.f;
      u64 tg = (u64)floor((double)uu * (double)zkept2);
      if (tg >= zkept2) tg = zkept2 - 1;
      if (live && ex2c <= tg && tg < ex2c + m_id && in_extent(row, 1, gridDim.x / P)) tokens[row] = (int)(ckey[tid] >> 32);
      return;
    }
    // more candidates than fit: the general path below
  }

  // ---- the general path: one CTA over the whole row (with P > 1 only the leader gets here)
  if (cr != 0) return;
  // ---- top-k: the k-th largest key kk; ties at kk are kept up to id kcut
  uint32_t kk = 0u;
  int kcut = INT_MAX;
  if (top_k > 0 && top_k < V) {
    uint32_t prefix = 0u, pmask = 0u;
    u64 remaining = (u64)top_k;
    unsigned ties = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += SP_THREADS) sh.hcnt[i] = 0u;
      __syncthreads();
      // warp-aggregated: lanes that hit the same bin add once (the top bins are crowded)
      auto count = [&](int, float v, bool ok) {
        const uint32_t key = order_key(v);
        const bool hit = ok && (key & pmask) == prefix;
        const unsigned hm = __ballot_sync(0xffffffffu, hit);
        if (hit) {
          const uint32_t bin = (key >> shift) & 255u;
          const unsigned peers = __match_any_sync(hm, bin);
          if (lane == __ffs(peers) - 1) atomicAdd(&sh.hcnt[bin], (unsigned)__popc(peers));
        }
      };
      row_each(z, V, vec, count);
      __syncthreads();
      if (warp == 0) select_digit<false>(sh, remaining);
      __syncthreads();
      prefix |= sh.b32[0] << shift;
      pmask |= 0xFFu << shift;
      remaining -= sh.b64[0];
      ties = sh.b32[1];
      __syncthreads();
    }
    kk = prefix;
    if (remaining < (u64)ties) {
      const uint32_t kkey = kk;
      kcut = nth_index(z, V, (int)remaining, [kkey](int, float v) { return order_key(v) == kkey; }, sh);
    }
  }
  auto in_k = [kk, kcut](int i, uint32_t key) { return key > kk || (key == kk && i <= kcut); };

  // ---- top-p: the kept set is key > kp, or key == kp up to id pcut (the shortest prefix of the
  //      top-k ranking whose mass reaches ceil(p * top-k mass))
  uint32_t kp = kk;
  int pcut = kcut;
  if (top_p < 1.f) {
    // one pass: the top-k mass and, per bucket of d = (z_max - z) / T (1/8 wide; larger d, lower
    // rank, so a bucket's members sit together in the ranking), its mass; per-warp copies in
    // shared memory
    u64* bmass = reinterpret_cast<u64*>(dyn);
    for (int i = tid; i < SP_WARPS * SP_BUCKETS; i += SP_THREADS) bmass[i] = 0ull;
    __syncthreads();
    auto bucket_of = [&](float v) -> int {
      const float d8 = (zmax - v) / temperature * 8.f;
      return d8 < (float)SP_BUCKETS ? (int)d8 : -1;   // beyond: zero mass (or -inf)
    };
    u64 part = 0ull;
    row_each(z, V, vec, [&](int i, float v, bool ok) {
      if (!ok || !in_k(i, order_key(v))) return;
      const u64 m = mass(v);
      part += m;
      const int bk = bucket_of(v);
      if (bk >= 0 && m != 0ull) atomicAdd(&bmass[warp * SP_BUCKETS + bk], m);
    });
    __syncthreads();
    for (int bk = tid; bk < SP_BUCKETS; bk += SP_THREADS) {   // digit 255 - bk: select_digit walks down
      u64 m = 0ull;
      for (int w = 0; w < SP_WARPS; ++w) m += bmass[w * SP_BUCKETS + bk];
      sh.hmass[255 - bk] = m;
    }
    u64 zk;
    block_scan_excl(part, sh, &zk);   // synchronises
    u64 target = (u64)ceil((double)top_p * (double)zk);
    target = target < 1ull ? 1ull : (target > zk ? zk : target);
    if (warp == 0) select_digit<true>(sh, target);
    __syncthreads();
    const int bstar = 255 - (int)sh.b32[0];
    const u64 above = sh.b64[0];                 // mass of the buckets before bstar
    if (tid == 0) sh.ccount = 0u;
    __syncthreads();
    // gather bucket bstar (its zero-mass members too: they rank among it) into shared memory
    u64* ckey = reinterpret_cast<u64*>(dyn);
    float* cz = reinterpret_cast<float*>(dyn + SP_CAP * 8);
    row_each(z, V, vec, [&](int i, float v, bool ok) {
      const uint32_t key = order_key(v);
      const bool take = ok && bucket_of(v) == bstar && in_k(i, key);
      const unsigned tm = __ballot_sync(0xffffffffu, take);
      if (tm) {
        unsigned slot0 = 0u;
        if (lane == 0) slot0 = atomicAdd(&sh.ccount, (unsigned)__popc(tm));
        slot0 = __shfl_sync(0xffffffffu, slot0, 0);
        if (take) {
          const unsigned slot = slot0 + __popc(tm & ((1u << lane) - 1u));
          if (slot < (unsigned)SP_CAP) {
            ckey[slot] = ((u64)key << 32) | (u64)(0xFFFFFFFFu - (uint32_t)i);
            cz[slot] = v;
          }
        }
      }
    });
    __syncthreads();
    const unsigned bcount = sh.ccount;
    __syncthreads();
    if (bcount <= (unsigned)SP_CAP) {
      // rank bucket bstar and cut where the running mass reaches the target
      const int nc = (int)bcount;
      int n2 = 1;
      while (n2 < nc) n2 <<= 1;
      for (int t = nc + tid; t < n2; t += SP_THREADS) ckey[t] = 0ull;
      __syncthreads();
      sort_desc(ckey, cz, n2);
      // four ranked candidates per thread
      u64 m4[4], loc = 0ull;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 4 * tid + e;
        m4[e] = j < nc ? mass(cz[j]) : 0ull;
        loc += m4[e];
      }
      u64 bsum;
      u64 run = above + block_scan_excl(loc, sh, &bsum);
      if (tid == 0) sh.bidx = nc - 1;   // not reached only through rounding: keep the whole bucket
      __syncthreads();
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 4 * tid + e;
        if (j < nc && run < target && run + m4[e] >= target) sh.bidx = j;   // exactly one candidate
        run += m4[e];
      }
      __syncthreads();
      const int jc = sh.bidx;
      kp = (uint32_t)(ckey[jc] >> 32);
      pcut = (int)(0xFFFFFFFFu - (uint32_t)(ckey[jc] & 0xFFFFFFFFull));
      __syncthreads();
    } else {
      // a crowded bucket (many equal logits): radix selection on the key, by mass
      uint32_t prefix = 0u, pmask = 0u;
      u64 above_r = 0ull, bin_mass = 0ull;
      unsigned bin_cnt = 0u;
      for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += SP_THREADS) { sh.hcnt[i] = 0u; sh.hmass[i] = 0ull; }
        __syncthreads();
        row_each(z, V, vec, [&](int i, float v, bool ok) {
          const uint32_t key = order_key(v);
          if (ok && in_k(i, key) && (key & pmask) == prefix) {
            const uint32_t dg = (key >> shift) & 255u;
            atomicAdd(&sh.hmass[dg], mass(v));
            atomicAdd(&sh.hcnt[dg], 1u);
          }
        });
        __syncthreads();
        if (warp == 0) select_digit<true>(sh, target - above_r);
        __syncthreads();
        prefix |= sh.b32[0] << shift;
        pmask |= 0xFFu << shift;
        above_r += sh.b64[0];
        bin_cnt = sh.b32[1];
        bin_mass = sh.b64[1];
        __syncthreads();
      }
      kp = prefix;
      // every token at key kp has the same logit, hence the same mass
      const u64 each = bin_mass / bin_cnt;
      u64 need = (target - above_r + each - 1) / each;
      if (need > bin_cnt) need = bin_cnt;
      if (need < (u64)bin_cnt) {
        const uint32_t pkey = kp;
        pcut = nth_index(z, V, (int)need,
                         [pkey, in_k](int i, float v) { const uint32_t k = order_key(v); return k == pkey && in_k(i, k); },
                         sh);
      } else {
        pcut = kp == kk ? kcut : INT_MAX;
      }
    }
  }

  // ---- the draw: first id (increasing) whose cumulative kept mass exceeds u * (kept mass).
  //      Warp w sums the kept mass of its contiguous stretch of the row (coalesced 16-byte
  //      loads); the stretch holding the target is then scanned again by the whole block.
  auto kept = [kp, pcut](int i, uint32_t key) { return key > kp || (key == kp && i <= pcut); };
  const int nq = (V + 3) >> 2;
  const int per_warp = (nq + SP_WARPS - 1) / SP_WARPS;
  auto mass4 = [&](int q, u64 (&m)[4]) {
    const int i0 = 4 * q;
    float v[4];
    if (vec && i0 + 4 <= V) {
      const float4 w = __ldg(reinterpret_cast<const float4*>(z) + q);
      v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = i0 + e < V ? z[i0 + e] : -INFINITY;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) m[e] = (i0 + e < V && kept(i0 + e, order_key(v[e]))) ? mass(v[e]) : 0ull;
  };
  {
    u64 acc = 0ull;
    const int qa = warp * per_warp, qb = min(nq, qa + per_warp);
#pragma unroll 4
    for (int q = qa + lane; q < qb; q += 32) {
      u64 m[4];
      mass4(q, m);
      acc += m[0] + m[1] + m[2] + m[3];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) sh.wsum[warp] = acc;
  }
  __syncthreads();
  u64 zkept = 0ull;
  for (int w = 0; w < SP_WARPS; ++w) zkept += sh.wsum[w];
  float u = uniforms[row];
  u = (u >= 0.f) ? fminf(u, 0.99999994f) : 0.f;   // NaN and negatives -> 0, 1 -> largest float below 1
  u64 tgt = (u64)floor((double)u * (double)zkept);
  if (tgt >= zkept) tgt = zkept - 1;   // (double)zkept may round up
  int wstar = SP_WARPS - 1;
  u64 base = 0ull;
  for (int w = 0; w < SP_WARPS; ++w) {
    const u64 c = sh.wsum[w];
    if (tgt < base + c) { wstar = w; break; }
    base += c;
  }
  __syncthreads();
  const int qa = wstar * per_warp, qb = min(nq, qa + per_warp);
  for (int c0 = qa; c0 < qb; c0 += SP_THREADS) {   // block-uniform trip count
    const int q = c0 + tid;
    u64 m[4] = {0ull, 0ull, 0ull, 0ull};
    if (q < qb) mass4(q, m);
    const u64 sq = m[0] + m[1] + m[2] + m[3];
    u64 chunk;
    const u64 ex = block_scan_excl(sq, sh, &chunk);
    if (base + ex <= tgt && tgt < base + ex + sq) {
      u64 a = base + ex;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        a += m[e];
        if (a > tgt) {
          if (in_extent(row, 1, gridDim.x / P)) tokens[row] = 4 * q + e;
          break;
        }
      }
    }
    if (tgt < base + chunk) break;
    base += chunk;
  }
}

template <typename T, bool VEC>
__global__ void embed_kernel(const T* __restrict__ table, int64_t V, int64_t d, const int* __restrict__ tokens,
                             T* __restrict__ x, unsigned* status) {
  const int64_t row = blockIdx.x;
  const int tok = tokens[row];
  const bool ok = tok >= 0 && (int64_t)tok < V;
  if (!ok && threadIdx.x == 0) atomicOr(status, STATUS_BAD_TOKEN);
  T* dst = x + row * d;
  if (VEC) {
    const int64_t n16 = d * (int64_t)sizeof(T) / 16;
    const uint4* src = reinterpret_cast<const uint4*>(table + (ok ? (int64_t)tok : 0) * d);
    uint4* out = reinterpret_cast<uint4*>(dst);
    for (int64_t i = threadIdx.x; i < n16; i += blockDim.x)   // x: [gridDim.x rows, d]
      if (in_extent(row * n16 + i, 1, (int64_t)gridDim.x * n16)) out[i] = ok ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
  } else {
    const T* src = table + (ok ? (int64_t)tok : 0) * d;
    for (int64_t i = threadIdx.x; i < d; i += blockDim.x)
      if (in_extent(row * d + i, 1, (int64_t)gridDim.x * d)) dst[i] = ok ? src[i] : T(0);
  }
}

}  // namespace

int launch_sample(const float* logits, int64_t B, int64_t V, int64_t ld, float temperature, int64_t top_k,
                  float top_p, const float* u, int* tokens, cudaStream_t st) {
  const int k = top_k <= 0 || top_k >= V ? 0 : (int)top_k;
  int dev = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return -1;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SP_DYN_SMEM) != cudaSuccess)
      return -1;
    attr_set[dev] = true;
  }
  // CTAs per row: a power of two up to 8 such that B x P CTAs (one per SM) still fit on the GPU, each
  // taking at least 4096 logits; only for 16-byte aligned rows on the argmax and small top-k paths
  // (the general path runs on one CTA per row)
  const bool argmax = !(temperature > 0.f) || k == 1 || !(top_p > 0.f) || V == 1;
  const bool small_k = temperature > 0.f && k >= 2 && k <= SP_SMALL_K && top_p > 0.f;
  const bool aligned = (reinterpret_cast<uintptr_t>(logits) & 15) == 0 && ld % 4 == 0;
  int P = 1;
  if (aligned && (argmax || small_k))
    while (P < 8 && B * (2 * P) <= num_sms() && V / (2 * P) >= 4096) P *= 2;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)(B * P));
  cfg.blockDim = dim3(SP_THREADS);
  cfg.dynamicSmemBytes = SP_DYN_SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = P > 1 ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, sample_kernel, logits, ld, (int)V, temperature, k, top_p, u, tokens) != cudaSuccess)
    return -1;
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_embed(int dtype, const void* table, int64_t V, int64_t d, const int* tokens, int64_t n, void* x,
                 unsigned* status, cudaStream_t st) {
  const size_t es = dtype == 0 ? 4 : 2;
  const bool vec = (d * (int64_t)es) % 16 == 0 && ((uintptr_t)table % 16 == 0) && ((uintptr_t)x % 16 == 0);
  const unsigned grid = (unsigned)n;
  if (dtype == 0) {
    if (vec) embed_kernel<float, true><<<grid, 128, 0, st>>>(static_cast<const float*>(table), V, d, tokens, static_cast<float*>(x), status);
    else embed_kernel<float, false><<<grid, 128, 0, st>>>(static_cast<const float*>(table), V, d, tokens, static_cast<float*>(x), status);
  } else {
    if (vec) embed_kernel<uint16_t, true><<<grid, 128, 0, st>>>(static_cast<const uint16_t*>(table), V, d, tokens, static_cast<uint16_t*>(x), status);
    else embed_kernel<uint16_t, false><<<grid, 128, 0, st>>>(static_cast<const uint16_t*>(table), V, d, tokens, static_cast<uint16_t*>(x), status);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

LLAMA_DEFINE_BOUNDS_READER(sample)

}  // namespace llama
