// ssd_selftest.cuh -- a kernel that exercises the library's failure path on
// purpose, without a fault: see ssd_selftest_timeout in ssd.h.
#pragma once

#include "ssd_device.cuh"

namespace ssd {

// ----------------------------------------------------------------------------
// The bounded-wait path, on its own: one warp allocates tensor memory, waits on
// an mbarrier that no thread arrives at for limit_ns, records kDevTimeout in
// the device error word as any kernel whose wait runs out does, frees the
// tensor memory and returns.  No fault, no trap: the context stays usable.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(32, 1) selftest_wait_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  tmem_alloc(&tslot, 32);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (threadIdx.x == 0) mbar_wait_limit(&bar, 0, &abort_flag, limit_ns);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  tmem_dealloc(tslot, 32);
}

}  // namespace ssd
