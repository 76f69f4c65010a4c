// selftest.cu -- diagnostic of the bounded barrier wait (see
// treewy_selftest_wait_timeout in treewy.h): one thread waits for a phase
// of a shared-memory mbarrier that nothing completes.
#include "treewy_device.cuh"
#include "treewy_internal.h"

namespace treewy {
namespace {

__global__ void wait_selftest_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbarrier_init();
  const uint64_t t0 = globaltimer_ns();
  const bool done = mbar_wait_for(&bar, 0, limit_ns);  // no arrival ever comes
  const uint64_t waited = globaltimer_ns() - t0;
  if (!done) atomicOr(status, TREEWY_STATUS_TIMEOUT);
  status[1] = static_cast<int32_t>(waited & 0xFFFFFFFFull);
  status[2] = static_cast<int32_t>(waited >> 32);
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t* status, uint32_t limit_us, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, static_cast<uint64_t>(limit_us) * 1000ull);
  return cudaGetLastError();
}

}  // namespace treewy
