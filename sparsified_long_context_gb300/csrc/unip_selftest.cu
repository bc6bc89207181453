// Self-test of the bounded device waits that every kernel of the library uses.
//
// One CTA, two roles in different warps, each waiting on its own mbarrier
// that nothing ever completes.  Role A waits with a short limit: the wait
// gives up, raises the CTA's abort flag and UNIP_DEV_TIMEOUT in the device
// status word.  Role B waits with the full one-second limit and must leave as
// soon as it sees the abort flag -- the way a kernel's other roles unwind
// after one of them timed out.  Nothing faults, traps or spins unbounded; the
// host then reads the status and can keep using the context.
#include "unip_internal.cuh"

namespace unip {
namespace {

__global__ void __launch_bounds__(64) bounded_wait_selftest_kernel(uint64_t limit_ns, int32_t *gave_up,
                                                                   uint32_t *status) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ int s_abort;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int *abort_flag = &s_abort;
  if (threadIdx.x == 0) {  // role A: short limit
    gave_up[0] = mbar_wait(smem_u32(&bars[0]), 0, abort_flag, status, limit_ns) ? 0 : 1;
  } else if (threadIdx.x == 32) {  // role B: default limit, leaves on A's abort
    const uint64_t t0 = globaltimer_ns();
    const bool done = mbar_wait(smem_u32(&bars[1]), 0, abort_flag, status);
    gave_up[1] = done ? 0 : 1;
    gave_up[2] = static_cast<int32_t>((globaltimer_ns() - t0) / 1000u);  // microseconds role B waited
  }
}

}  // namespace
}  // namespace unip

using namespace unip;

extern "C" {

UNIP_API int32_t unip_selftest_bounded_wait(uint32_t limit_us, int32_t *gave_up, void *stream) {
  if (!gave_up || limit_us == 0 || limit_us > 1000000u) return UNIP_ERR_INVALID_ARGUMENT;
  uint32_t *status = device_status_ptr();
  if (!status) return UNIP_ERR_CUDA;
  bounded_wait_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(uint64_t(limit_us) * 1000u,
                                                                               gave_up, status);
  return cudaGetLastError() == cudaSuccess ? UNIP_OK : UNIP_ERR_CUDA;
}

}  // extern "C"
