// Self-check of the failure path that every pipeline of this library shares:
// a bounded mbarrier wait that gives up, raises the CTA's abort flag and the
// device status bit TG_ERR_TIMEOUT, and a second waiter that leaves because
// of the abort flag.  No kernel of the hot path can be made to lose an
// arrival on purpose without breaking it, so this kernel builds the same
// situation directly: one CTA, one mbarrier that nothing ever completes.
//
//   warp 0, lane 0  waits on the barrier with the caller's short bound
//                   (mbar_wait_for), gives up, sets abort + the status bit;
//   warp 1, lane 0  waits on the same barrier with the pipelines' own bound
//                   (2 s) and must return early, as soon as it sees abort.
// Both waits sleep in try_wait with a suspend hint and check the clock, so
// the kernel ends within the caller's bound plus a few tens of microseconds.
#include "tg_device.cuh"
#include "tg_internal.h"

namespace tg {
namespace {

__global__ void __launch_bounds__(64, 1)
    bounded_wait_selftest_kernel(uint64_t timeout_ns, uint32_t* status,
                                 unsigned long long* report) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // one arrival expected; none will come
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort = &abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    const uint64_t t0 = globaltimer_ns();
    bool ok;
    if (warp == 0) {
      ok = mbar_wait_for(smem_u32(&bar), 0, abort, status, timeout_ns);
    } else {
      ok = mbar_wait(smem_u32(&bar), 0, abort, status);
    }
    const uint64_t dt = globaltimer_ns() - t0;
    if (report != nullptr) {
      report[2 * warp] = ok ? 1ull : 0ull;  // 0: the wait gave up, as it must
      report[2 * warp + 1] = dt;
    }
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(uint64_t timeout_ns, unsigned long long* report,
                                         cudaStream_t stream) {
  uint32_t* status = device_status_word();
  if (status == nullptr) return cudaErrorInvalidDevice;
  bounded_wait_selftest_kernel<<<1, 64, 0, stream>>>(timeout_ns, status, report);
  return cudaGetLastError();
}

}  // namespace tg
