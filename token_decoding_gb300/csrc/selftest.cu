// selftest.cu - mars_selftest_wait_timeout: the library's own failure path,
// exercised on the device without faulting, trapping or hanging it.
//
// Every pipeline wait in the kernels of this library is an mbarrier wait with
// a poll limit (mars::mbar_wait); when the limit is reached the kernel records
// MARS_DEV_TIMEOUT in the caller's status word, stops waiting, releases what it
// holds (tensor memory) and returns, so the CUDA context stays usable.  This
// kernel runs that same helper on a barrier whose second arrival the caller
// may withhold.  Nothing asynchronous ever targets the barrier (no TMA copy, no
// tcgen05.mma commit), so a withheld arrival leaves nothing in flight.
#include "common.cuh"

namespace {

using namespace mars;

__global__ void __launch_bounds__(96, 1)
    wait_probe_kernel(int withhold, uint32_t limit, int32_t* status, unsigned long long* elapsed_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 2);  // two arrivals complete phase 0
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_slot, 32);  // held across the wait, like the real kernels' accumulators
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1 && lane == 0) mbar_arrive(&bar);
  if (warp == 2 && lane == 0 && !withhold) mbar_arrive(&bar);
  bool ok = true;
  if (warp == 0) {
    unsigned long long t0 = 0, t1 = 0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    ok = __all_sync(0xffffffffu, mbar_wait(&bar, 0, limit));
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
    if (lane == 0) {
      if (!ok) set_status(status, MARS_DEV_TIMEOUT);
      if (elapsed_ns != nullptr) *elapsed_ns = t1 - t0;
    }
  }
  // wind-down as in the kernels: every thread meets here, then the owner frees tensor memory
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_slot, 32);
  }
}

}  // namespace

extern "C" int mars_selftest_wait_timeout(int withhold_arrival, unsigned int spin_limit, int32_t* status,
                                          unsigned long long* elapsed_ns, void* stream) {
  MARS_HOST_CHECK(spin_limit >= 1 && spin_limit <= kSpinLimit, MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(status != nullptr && mars_host::aligned4(status), MARS_ERR_INVALID_ARG);
  MARS_HOST_CHECK(elapsed_ns == nullptr || (reinterpret_cast<uintptr_t>(elapsed_ns) & 7u) == 0,
                  MARS_ERR_INVALID_ARG);
  const int rc = mars_host::check_device();
  if (rc != MARS_OK) return rc;
  wait_probe_kernel<<<1, 96, 0, static_cast<cudaStream_t>(stream)>>>(withhold_arrival ? 1 : 0, spin_limit, status,
                                                                     elapsed_ns);
  return mars_host::launch_status();
}
