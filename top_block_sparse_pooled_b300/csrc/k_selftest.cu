// k_selftest.cu -- self-test of the bounded-wait error path.
//
// One CTA waits on an mbarrier phase that nothing completes, with a short
// limit, exactly as the pipeline kernels wait on their copies: when the limit
// passes it records SA_ERR_TIMEOUT in the device status word and returns, so
// the host sees the failure through sa_device_status() and the context stays
// usable.  Nothing faults, traps or spins without a bound.
#pragma once

#include "sa_ptx.cuh"

namespace sa {

__global__ void selftest_wait_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);  // one arrival expected; none is ever made
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(b, 0)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      if (threadIdx.x == 0) record_error(kErrTimeout);
      break;
    }
  }
}

}  // namespace sa
