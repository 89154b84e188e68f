// Self-test of the device-side failure path.  Every pipelined kernel of the library waits on its
// mbarriers through mbar_wait (common.cuh): a wait that has not completed after kWaitLimitNs of
// %globaltimer latches STATUS_TIMEOUT in the device status word, raises the CTA's abort flag so
// that its other roles stop too, and returns false so that the kernel winds down and exits.  This
// kernel makes two such waits run out on purpose, on phases that nothing ever completes, so that
// a test can check, without faulting or hanging the GPU, that the host reads LLAMA_ERR_TIMEOUT and
// that the context is still usable afterwards.
//
// The bounds self-test stores through the checked path (in_extent) to element 40 of a 64-element
// buffer while declaring the tensor 32 elements long: a bounds-checking build skips the store and
// latches its bounds word; a release build performs it, inside the buffer either way.
#include "kernels.h"

namespace llama {
namespace {

__global__ void wait_timeout_kernel(unsigned* status) {
  __shared__ uint64_t bar[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    // warp w waits for phase 0 of bar[w]; no thread ever arrives on either barrier.  The first
    // wait to reach its limit latches the timeout and raises the abort flag, which ends the other.
    mbar_wait(&bar[threadIdx.x >> 5], 0, &abort_flag, status);
  }
  __syncwarp();
  __syncthreads();
}

__global__ void bounds_selftest_kernel(float* scratch, int64_t declared) {
  const int64_t i = 40;
  if (threadIdx.x == 0 && in_extent(i, 1, declared)) scratch[i] = 1.0f;
}

}  // namespace

int launch_bounds_selftest(float* scratch, cudaStream_t st) {
  bounds_selftest_kernel<<<1, 32, 0, st>>>(scratch, 32);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int launch_wait_timeout_selftest(cudaStream_t st) {
  unsigned* status = status_ptr();
  if (!status) return -1;
  wait_timeout_kernel<<<1, 64, 0, st>>>(status);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

LLAMA_DEFINE_BOUNDS_READER(selftest)

}  // namespace llama

extern "C" int llama_selftest_bounded_wait(void* stream) {
  return llama::launch_wait_timeout_selftest(static_cast<cudaStream_t>(stream)) == 0 ? LLAMA_OK : LLAMA_ERR_CUDA;
}

extern "C" int llama_selftest_bounds(float* scratch, void* stream) {
  if (!scratch || (reinterpret_cast<uintptr_t>(scratch) & 15) != 0) return LLAMA_ERR_INVALID_ARG;
  return llama::launch_bounds_selftest(scratch, static_cast<cudaStream_t>(stream)) == 0 ? LLAMA_OK : LLAMA_ERR_CUDA;
}
