// Self-test of the bounded device wait that every tensor-core kernel of the library relies on:
// one block waits on an mbarrier that nothing ever signals, through the same primitive
// (tc05::mbar_wait_limit) and the same reporting (CSA2_ETIMEOUT into the caller's status word)
// as the kernels, with a short, caller-chosen number of tries.  The wait gives up, the status
// is recorded, and the block returns: the context stays usable.
#include "../../include/csa2.h"
#include "kernels.h"
#include "tc05.cuh"

namespace csa2 {
namespace {

__global__ void wait_timeout_kernel(int32_t* dev_status, uint32_t tries) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    tc05::mbar_init(&bar, 1);  // one arrival expected; none ever comes
    tc05::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !tc05::mbar_wait_limit(&bar, 0, tries)) atomicExch(dev_status, (int)CSA2_ETIMEOUT);
}

}  // namespace
}  // namespace csa2

extern "C" csa2_status csa2_selftest_wait_timeout(int32_t* dev_status, int32_t tries, void* stream) {
  if (!dev_status || tries < 1 || tries > (1 << 20)) return CSA2_EINVAL;
  csa2::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_status, (uint32_t)tries);
  return cudaGetLastError() == cudaSuccess ? CSA2_OK : CSA2_ECUDA;
}
