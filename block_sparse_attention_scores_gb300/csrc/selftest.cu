// Failure-detection self-test: a bounded wait that is made to run out.
//
// The kernel initialises an mbarrier that expects one arrival, never arrives
// on it, and waits with a short limit; the wait gives up, writes a timeout
// into the error word and the kernel returns normally. Hosts then see
// MSA_ERR_DEVICE from msa_check_device_status(), the same path a real stall
// in any MSA kernel takes.
#include "msa_internal.h"
#include "sm100.cuh"

namespace msa {
namespace {

__global__ void wait_timeout_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, err, 901, limit_ns);  // nothing arrives: runs out after limit_ns
}

}  // namespace

cudaError_t launch_selftest_wait_timeout(int* err, long long limit_ns, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(err, (unsigned long long)limit_ns);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace msa
