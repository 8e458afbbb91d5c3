// selftest.cu -- a check of the bounded-wait path that every kernel's mbarrier waits share.
//
// One warp initialises an mbarrier in shared memory that nothing ever arrives on, and one
// thread waits on it with mbar_wait (common.cuh), exactly as a producer or consumer of the
// GEMM, side-product or decode kernels waits on a stage that never fills.  After the wait
// limit the wait records kWaitSelftest in this file's device error word and the kernel
// returns; qlora_device_status then reports the code, and the device stays usable.  So a
// caller can see, on its own device, that a stuck wait ends in a status instead of a hang.
#include "common.cuh"
#include "launch.h"

namespace qlora {

__device__ int g_selftest_error = 0;

int read_and_clear_selftest_error(int* out) {
  int v = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_selftest_error, sizeof(int)) != cudaSuccess)
    return QLORA_ERR_CUDA;
  if (v && cudaMemcpyToSymbol(g_selftest_error, &zero, sizeof(int)) != cudaSuccess)
    return QLORA_ERR_CUDA;
  *out = v;
  return QLORA_OK;
}

namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel() {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    // phase 0 of `bar` never completes: no thread arrives and no copy signals it
    mbar_wait(&bar, 0, kWaitSelftest, &abort_flag, &g_selftest_error);
  }
  __syncwarp();
}

}  // namespace

int launch_wait_selftest(cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>();
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

}  // namespace qlora
