// Self-test of the bounded wait that every staged kernel uses on its
// shared-memory barriers.  One thread waits on an mbarrier that nothing
// arrives on: the wait runs out after its limit (about one second), counts
// in a device counter of its own -- not the one rms_norm_wait_timeouts
// reads -- and the kernel returns.  No trap, no fault: the context stays
// usable, which the caller checks by running any other call afterwards.
#include <chrono>

#include "launch.h"
#include "mbar.cuh"
#include "rms_norm.h"

namespace rmsn {
namespace {

__device__ unsigned int g_selftest_timeouts;

__global__ void wait_limit_probe() {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    abort = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // one waiter, so that exactly one wait runs out; the phase never completes
  if (threadIdx.x == 0) wait_phase_counted(&bar, 0u, &abort, &g_selftest_timeouts);
}

}  // namespace
}  // namespace rmsn

extern "C" int rms_norm_selftest_wait_limit(unsigned int* timeouts, double* seconds) {
  if (!timeouts || !seconds) return RMSN_ERR_NULL;
  const unsigned int zero = 0;
  cudaError_t e = cudaMemcpyToSymbol(rmsn::g_selftest_timeouts, &zero, sizeof(zero));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return rmsn::cuda_fail(e);
  const auto t0 = std::chrono::steady_clock::now();
  rmsn::wait_limit_probe<<<1, 32>>>();
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  const auto t1 = std::chrono::steady_clock::now();
  if (e != cudaSuccess) return rmsn::cuda_fail(e);
  e = cudaMemcpyFromSymbol(timeouts, rmsn::g_selftest_timeouts, sizeof(unsigned int));
  if (e != cudaSuccess) return rmsn::cuda_fail(e);
  *seconds = std::chrono::duration<double>(t1 - t0).count();
  return RMSN_OK;
}
