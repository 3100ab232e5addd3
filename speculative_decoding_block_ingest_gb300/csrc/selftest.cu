// selftest.cu -- exercises the bounded-wait failure path without a fault.
//
// One thread waits on a shared-memory mbarrier that nothing arrives on, for
// at most `limit_ns` of %globaltimer, exactly as every pipeline wait of the
// library does (try_wait in a loop against a deadline); when the deadline
// passes it records DERR_TIMEOUT in the handle's error word and returns.  No
// trap, no unbounded spin: the context stays usable and the host reads the
// code through dflash_device_status.
#include "kernels.cuh"
#include "ptx.cuh"

namespace dfl {

__global__ void selftest_wait_kernel(int* err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(&bar, 0)) {
    if (globaltimer() - t0 > limit_ns) {
      atomicExch(err, DERR_TIMEOUT);
      return;
    }
  }
}

void launch_selftest_wait(int* err, unsigned long long limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(err, limit_ns);
}

}  // namespace dfl
