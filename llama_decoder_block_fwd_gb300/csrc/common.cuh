// Shared device helpers for the sm_103a kernels: bf16 conversion, the RoPE angle, the device
// status word, bounded mbarrier waits, TMA (cp.async.bulk.tensor) and tcgen05 wrappers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/llama_block.h"

namespace llama {

// ---------------------------------------------------------------- status word
// Bit flags latched by kernels; read and cleared by llama_get_device_status().
enum : unsigned { STATUS_TIMEOUT = 1u, STATUS_BAD_TOKEN = 2u };

// ---------------------------------------------------------------- bounds checks (-DLLAMA_DEBUG)
// Built with -DLLAMA_DEBUG, the kernels check every global store's index range and every TMA box
// start against the extent of its tensor before issuing it.  A failed check latches this
// translation unit's bounds word (read and cleared on the host by its bounds_read_clear_* reader,
// which llama_get_device_status calls) and returns false: the caller skips the access and returns.
// Release builds compile every check to `true`.
#ifdef LLAMA_DEBUG
constexpr bool kBoundsChecks = true;
static __device__ unsigned g_bounds_fail;   // one per translation unit
#else
constexpr bool kBoundsChecks = false;
#endif

__device__ __forceinline__ bool bounds_fail() {
#ifdef LLAMA_DEBUG
  atomicOr(&g_bounds_fail, 1u);
#endif
  return false;
}
// [i, i + n) lies inside [0, extent)
__device__ __forceinline__ bool in_extent(int64_t i, int64_t n, int64_t extent) {
  if (!kBoundsChecks) return true;
  return (i >= 0 && n >= 0 && i <= extent - n) || bounds_fail();
}
// A TMA box start inside its tensor: 0 <= coordinate < extent on each dimension given.
__device__ __forceinline__ bool box_in(int64_t x, int64_t ex, int64_t y = 0, int64_t ey = 1, int64_t z = 0,
                                       int64_t ez = 1, int64_t w = 0, int64_t ew = 1) {
  if (!kBoundsChecks) return true;
  return (x >= 0 && x < ex && y >= 0 && y < ey && z >= 0 && z < ez && w >= 0 && w < ew) || bounds_fail();
}

// The host-side reader of a translation unit's bounds word (0 in release builds); each .cu file
// defines its own with LLAMA_DEFINE_BOUNDS_READER(file name).
#ifdef LLAMA_DEBUG
#define LLAMA_DEFINE_BOUNDS_READER(name)                                                  \
  unsigned bounds_read_clear_##name() {                                                  \
    unsigned v = 0;                                                                      \
    if (cudaMemcpyFromSymbol(&v, g_bounds_fail, sizeof(v)) != cudaSuccess) return 0u;    \
    if (v) {                                                                             \
      const unsigned zero = 0;                                                           \
      cudaMemcpyToSymbol(g_bounds_fail, &zero, sizeof(zero));                            \
    }                                                                                    \
    return v;                                                                            \
  }
#else
#define LLAMA_DEFINE_BOUNDS_READER(name) \
  unsigned bounds_read_clear_##name() { return 0u; }
#endif

// A bounded wait gives up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- conversions
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  return (uint32_t)f2bf(lo) | ((uint32_t)f2bf(hi) << 16);
}

template <typename T> struct Elt;
template <> struct Elt<float> {
  static __device__ __forceinline__ float ld(const float* p) { return *p; }
  static __device__ __forceinline__ void st(float* p, float v) { *p = v; }
};
template <> struct Elt<uint16_t> {
  static __device__ __forceinline__ float ld(const uint16_t* p) { return bf2f(*p); }
  static __device__ __forceinline__ void st(uint16_t* p, float v) { *p = f2bf(v); }
};

// ---------------------------------------------------------------- RoPE angle
// theta_k = theta_base^(-2k/hd) is split on the host into hi + lo floats (hi = fl(theta_k)).
// The angle m*theta_k is formed as p + e + m*lo with e the exact rounding error of p = fl(m*hi),
// and p is reduced by 2*pi with a two-part constant (Cody and Waite, "Software Manual for the
// Elementary Functions", 1980): 2*pi = 6.28125 + 1.9353071795864769e-3, the first part holding
// 8 significant bits so that n*6.28125 is exact for n < 2^16 (positions below 2^19 at theta_0=1).
struct RopeFreq { float hi, lo; };

__device__ __forceinline__ void rope_sincos(float m, RopeFreq f, float& s, float& c) {
  const float p = m * f.hi;
  const float e = fmaf(m, f.hi, -p);
  const float t = fmaf(m, f.lo, e);
  const float n = rintf(p * 0.15915494309189535f);
  float r = fmaf(-n, 6.28125f, p);
  r = fmaf(-n, 1.9353071795864769e-3f, r);
  r += t;
  sincosf(r, &s, &c);
}

// Copy the per-pair frequencies of a launch's parameters into shared memory (whole block, ends with
// a barrier).  Threads of a warp that index a kernel-parameter array with different indices are
// served one address at a time, so kernels whose lanes take different pairs read the copy instead.
__device__ __forceinline__ void stage_freq(const RopeFreq* src, int half, RopeFreq* dst) {
  for (int i = threadIdx.x + threadIdx.y * blockDim.x; i < half; i += blockDim.x * blockDim.y) dst[i] = src[i];
  __syncthreads();
}

// ---------------------------------------------------------------- shared memory / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete.  Gives up (returns false) when
// *abort is set by another role of the CTA, or after kWaitLimitNs, in which case it latches
// STATUS_TIMEOUT and sets *abort so that every role of the CTA stops.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned* status) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(a, parity)) return true;
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

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint64_t* bar, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
// Instruction descriptor, kind::f16 with bf16 A and B and an fp32 accumulator:
// bits 4-5 D type (1 = f32), 7-9 A type (1 = bf16), 10-12 B type (1 = bf16),
// 15 / 16 A / B major-ness (0 = K-major, 1 = MN-major), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major = false,
                                                  bool a_mn_major = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor with 128-byte swizzling: start address >> 4 in bits 0-13,
// leading byte offset >> 4 in bits 16-29, stride byte offset >> 4 in bits 32-45, the fixed
// value 1 in bits 46-47, base offset 0, swizzle mode 2 (128B) in bits 61-63.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 4 columns of 32-bit TMEM cells: thread t of the warp gets lane (base + t), columns
// col .. col+3 in v[0..3].
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&v)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(taddr));
}
// 32 lanes x 32 columns of 32-bit TMEM cells: thread t of the warp gets lane (base + t),
// columns col .. col+31 in v[0..31].
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
        "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
        "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
        "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T (A read from tensor memory), issued by one thread.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Programmatic dependent launch: let the next kernel of the stream begin launching, and wait until
// every earlier kernel has completed and its writes are visible (no-ops without the launch
// attribute).  A kernel reads nothing an earlier kernel wrote, and writes nothing, before pdl_wait.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace llama
