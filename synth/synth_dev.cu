// Seeded synthetic inputs, device side.
//
// Same definition as synth_host.c (SplitMix64 finaliser over a per-tensor key,
// Irwin-Hall sum of twelve 16-bit uniforms, fp64 scale and shift with separate
// roundings, round to f32, then round-to-nearest-even to bf16).  It holds no
// arithmetic of the Llama block; it only fills device buffers with the numbers
// the host side would draw, so that tensors too large to copy (a 69 GB KV cache)
// can be made where they are used and re-drawn on the host where needed.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t kG = 0x9E3779B97F4A7C15ULL;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27; z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

__host__ __device__ inline uint64_t mix64_h(uint64_t z) {
  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27; z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

__device__ __forceinline__ float draw(uint64_t key, uint64_t i, double mean, double stdv) {
  uint64_t s = 0;
#pragma unroll
  for (uint64_t j = 0; j < 3; ++j) {
    uint64_t h = mix64(key + (3 * i + j + 1) * kG);
    s += (h & 0xFFFF) + ((h >> 16) & 0xFFFF) + ((h >> 32) & 0xFFFF) + (h >> 48);
  }
  double z = (double)((int64_t)s - 393210) / 65536.0;
  double t = __dmul_rn(stdv, z);        // no contraction into an FMA
  return __double2float_rn(__dadd_rn(t, mean));
}

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0xFFFF) ? 0x40 : 0));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__global__ void fill_kernel(void* out, int dtype, int64_t n, uint64_t key, int64_t offset,
                            double mean, double stdv) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride) {
    float f = draw(key, (uint64_t)(offset + k), mean, stdv);
    if (dtype == 1) static_cast<uint16_t*>(out)[k] = f32_to_bf16_rne(f);
    else static_cast<float*>(out)[k] = f;
  }
}

}  // namespace

// Fill n elements of a device buffer with draws offset .. offset+n-1 of stream
// (seed, tid).  dtype 0 = f32, 1 = bf16.  Returns a cudaError_t code.
extern "C" int synth_fill_device(void* out, int dtype, int64_t n, uint64_t seed, uint64_t tid,
                                 int64_t offset, double mean, double stdv, void* stream) {
  if (n <= 0) return 0;
  if (!out || (dtype != 0 && dtype != 1)) return (int)cudaErrorInvalidValue;
  const uint64_t key = mix64_h(mix64_h(seed + kG) + tid * kG);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 16;
  if (blocks > cap) blocks = cap;
  fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(out, dtype, n, key, offset, mean, stdv);
  return (int)cudaGetLastError();
}
