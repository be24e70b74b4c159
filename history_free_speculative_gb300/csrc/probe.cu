// Probe of the bounded device waits (failure detection without a fault).
//
// Every mbarrier wait of the tensor-core kernels gives up after a time limit,
// flags DLITE_DEV_TIMEOUT in the status word and lets the kernel return; a
// kernel that starts while the flag is set skips its work. These two tiny
// kernels exercise exactly those helpers with a short, caller-chosen limit:
// the first waits on a barrier nobody arrives at (one warp through the
// warp-wide wait, one thread through the single-thread wait), the second
// makes the engines' entry check.
#include "tc_device.cuh"
#include "kernels.h"

namespace dlite {
namespace {

__global__ void __launch_bounds__(64) wait_probe_kernel(uint64_t limit_ns, int* status, int32_t* result) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = tc::su32(&bar);
  if (threadIdx.x == 0) {
    tc::mbar_init(b, 1);  // one arrival expected; none comes
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const bool got = tc::mbar_wait_warp(b, 0, status, limit_ns);
    if (threadIdx.x == 0) result[0] = got ? 0 : 1;
  } else if (threadIdx.x == 32) {
    const bool got = tc::mbar_wait(b, 0, status, limit_ns);
    result[1] = got ? 0 : 1;
  }
}

__global__ void abort_probe_kernel(int* status, int32_t* result) {
  const bool aborted = status && (*(volatile int*)status & kDevTimeout);  // as the engines check
  if (threadIdx.x == 0) result[2] = aborted ? 1 : 0;
}

}  // namespace

cudaError_t launch_wait_probe(uint64_t limit_ns, int* status, int32_t* result, cudaStream_t s) {
  wait_probe_kernel<<<1, 64, 0, s>>>(limit_ns, status, result);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  abort_probe_kernel<<<1, 32, 0, s>>>(status, result);
  return cudaGetLastError();
}

}  // namespace dlite
