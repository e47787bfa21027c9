// fa_selftest.cu — a self-test of the library's failure reporting that needs
// no fault: one CTA of 32 threads waits on a barrier that nothing ever arrives
// on.  The wait is the bounded mbarrier wait every kernel of the library uses
// (sm103_ptx.cuh): it gives up after its time limit, raises the CTA's abort
// flag (lanes still waiting see it and stop), records its code in this file's
// device error word, and the kernel returns normally, leaving the context
// usable.  fa_get_device_error reports and clears the word like the others.
#include <cstdint>

#include <cuda_runtime.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

__device__ unsigned int g_st_error = 0;

__global__ void __launch_bounds__(32) fa_selftest_wait_kernel() {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // phase 0 of the barrier never completes: every lane's wait runs out (or
  // sees the first lane's abort flag) and returns false
  mbar_wait(&bar, 0, &abort_flag, &g_st_error, kSelftestWaitCode);
}

}  // namespace

cudaError_t launch_selftest_wait(cudaStream_t s) {
  fa_selftest_wait_kernel<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

cudaError_t st_read_clear_error(uint32_t* out, cudaStream_t s) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  uint32_t v = 0;
  e = cudaMemcpyFromSymbol(&v, g_st_error, sizeof(v));
  if (e != cudaSuccess) return e;
  if (v) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_st_error, &zero, sizeof(zero));
  }
  *out = v;
  return e;
}

}  // namespace fa
