// Self-test of the device-side failure path.  Every pipelined kernel of the library waits on its
// mbarriers through mbar_wait (common.cuh): a wait that has not completed after kWaitLimitNs of
// %globaltimer latches STATUS_TIMEOUT in the device status word, raises the CTA's abort flag so
// that its other roles stop too, and returns false so that the kernel winds down and exits.  This
// kernel makes two such waits run out on purpose, on phases that nothing ever completes, so that
// a test can check, without faulting or hanging the GPU, that the host reads LLAMA_ERR_TIMEOUT and
// that the context is still usable afterwards.
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

}  // namespace

int launch_wait_timeout_selftest(cudaStream_t st) {
  unsigned* status = status_ptr();
  if (!status) return -1;
  wait_timeout_kernel<<<1, 64, 0, st>>>(status);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace llama

extern "C" int llama_selftest_bounded_wait(void* stream) {
  return llama::launch_wait_timeout_selftest(static_cast<cudaStream_t>(stream)) == 0 ? LLAMA_OK : LLAMA_ERR_CUDA;
}
