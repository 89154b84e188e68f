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
// One CTA per row.  The row (up to a few hundred KB of fp32) is streamed from L2 once per pass;
// nothing is sorted.  The thresholds are found by radix selection on an order-preserving 32-bit
// key of the logit, four 8-bit digits from the top: by count for top-k, by probability mass for
// top-p.  Masses are exp((z - z_max) / T) in fp32, held as 2^-40 fixed point in 64-bit integers
// so that every sum is exact and independent of the order of the atomic adds: the same logits
// always give the same token.  Terms below 2^-40 of the largest count as zero.
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

struct SampleShared {
  u64 hmass[256];
  unsigned hcnt[256];
  u64 wsum[SP_WARPS];
  float wval[SP_WARPS];
  int widx[SP_WARPS];
  u64 b64[4];
  unsigned b32[4];
  int bidx;
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
  const int row = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* z = logits + (int64_t)row * ld;

  // ---- the largest logit and its lowest id (argmax)
  float best = -INFINITY;
  int bi = INT_MAX;
  for (int i = tid; i < V; i += SP_THREADS) {
    const float v = z[i];
    if (v > best || (v == best && i < bi)) { best = v; bi = i; }
  }
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
  const float zmax = best;
  if (!(temperature > 0.f) || top_k == 1 || !(top_p > 0.f) || !isfinite(zmax) || V == 1) {
    if (tid == 0) tokens[row] = bi == INT_MAX ? 0 : bi;
    return;
  }
  auto mass = [&](float v) -> u64 { return __float2ull_rz(expf((v - zmax) / temperature) * kMassOne); };

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
      for (int i = tid; i < V; i += SP_THREADS) {
        const uint32_t key = order_key(z[i]);
        if ((key & pmask) == prefix) atomicAdd(&sh.hcnt[(key >> shift) & 255u], 1u);
      }
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

  // ---- mass of the top-k set
  u64 part = 0;
  for (int i = tid; i < V; i += SP_THREADS) {
    const float v = z[i];
    if (in_k(i, order_key(v))) part += mass(v);
  }
  u64 zk;
  block_scan_excl(part, sh, &zk);

  // ---- top-p: the kept set is key > kp, or key == kp up to id pcut
  uint32_t kp = kk;
  int pcut = kcut;
  u64 zkept = zk;
  if (top_p < 1.f) {
    u64 target = (u64)ceil((double)top_p * (double)zk);
    target = target < 1ull ? 1ull : (target > zk ? zk : target);
    uint32_t prefix = 0u, pmask = 0u;
    u64 above = 0ull, bin_mass = 0ull;
    unsigned bin_cnt = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += SP_THREADS) { sh.hcnt[i] = 0u; sh.hmass[i] = 0ull; }
      __syncthreads();
      for (int i = tid; i < V; i += SP_THREADS) {
        const float v = z[i];
        const uint32_t key = order_key(v);
        if (in_k(i, key) && (key & pmask) == prefix) {
          const uint32_t dg = (key >> shift) & 255u;
          atomicAdd(&sh.hmass[dg], mass(v));
          atomicAdd(&sh.hcnt[dg], 1u);
        }
      }
      __syncthreads();
      if (warp == 0) select_digit<true>(sh, target - above);
      __syncthreads();
      prefix |= sh.b32[0] << shift;
      pmask |= 0xFFu << shift;
      above += sh.b64[0];
      bin_cnt = sh.b32[1];
      bin_mass = sh.b64[1];
      __syncthreads();
    }
    kp = prefix;
    // every token at key kp has the same logit, hence the same mass
    const u64 each = bin_mass / bin_cnt;
    u64 need = (target - above + each - 1) / each;
    if (need > bin_cnt) need = bin_cnt;
    if (need < (u64)bin_cnt) {
      const uint32_t pkey = kp;
      pcut = nth_index(z, V, (int)need,
                       [pkey, in_k](int i, float v) { const uint32_t k = order_key(v); return k == pkey && in_k(i, k); },
                       sh);
    } else {
      pcut = kp == kk ? kcut : INT_MAX;
    }
    zkept = above + need * each;
  }

  // ---- the draw: first id (increasing) whose cumulative kept mass exceeds u * zkept
  float u = uniforms[row];
  u = (u >= 0.f) ? fminf(u, 0.99999994f) : 0.f;   // NaN and negatives -> 0, 1 -> largest float below 1
  u64 tgt = (u64)floor((double)u * (double)zkept);
  if (tgt >= zkept) tgt = zkept - 1;   // (double)zkept may round up
  const int seg = (V + SP_THREADS - 1) / SP_THREADS;
  const int lo = min(V, tid * seg), hi = min(V, lo + seg);
  auto kept = [kp, pcut](int i, uint32_t key) { return key > kp || (key == kp && i <= pcut); };
  u64 s = 0;
  for (int i = lo; i < hi; ++i) {
    const float v = z[i];
    if (kept(i, order_key(v))) s += mass(v);
  }
  u64 total;
  const u64 before = block_scan_excl(s, sh, &total);
  if (before <= tgt && tgt < before + s) {
    u64 acc = before;
    for (int i = lo; i < hi; ++i) {
      const float v = z[i];
      if (!kept(i, order_key(v))) continue;
      acc += mass(v);
      if (acc > tgt) { tokens[row] = i; break; }
    }
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
    for (int64_t i = threadIdx.x; i < n16; i += blockDim.x) out[i] = ok ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
  } else {
    const T* src = table + (ok ? (int64_t)tok : 0) * d;
    for (int64_t i = threadIdx.x; i < d; i += blockDim.x) dst[i] = ok ? src[i] : T(0);
  }
}

}  // namespace

int launch_sample(const float* logits, int64_t B, int64_t V, int64_t ld, float temperature, int64_t top_k,
                  float top_p, const float* u, int* tokens, cudaStream_t st) {
  const int k = top_k <= 0 || top_k >= V ? 0 : (int)top_k;
  sample_kernel<<<(unsigned)B, SP_THREADS, 0, st>>>(logits, ld, (int)V, temperature, k, top_p, u, tokens);
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

}  // namespace llama
