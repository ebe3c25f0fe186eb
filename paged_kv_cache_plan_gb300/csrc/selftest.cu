// Self-test of the bounded pipeline waits (decode_selftest_wait_timeout in
// include/pkvd.h): one block waits on a shared-memory barrier that nothing
// completes, through the same bounded wait the stage-1 kernels use, and
// records the outcome instead of hanging. Nothing here faults or traps.
#include <cuda_runtime.h>

#include "device.cuh"
#include "kernels.h"

namespace pkvd {
namespace {

__global__ void wait_timeout_probe(int32_t* status, unsigned long long limit_ns) {
  __shared__ alignas(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);   // one arrival completes phase 0; none comes
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long t0 = global_timer_ns();
    const bool done = mbar_wait_for(smem_addr(&bar), 0, limit_ns);
    const unsigned long long waited = global_timer_ns() - t0;
    // PKVD_ETIMEOUT when the wait gave up no earlier than its limit
    status[0] = done ? PKVD_OK : (waited >= limit_ns ? PKVD_ETIMEOUT : PKVD_ECUDA);
    status[1] = static_cast<int32_t>(waited / 1000ull);   // microseconds waited
  }
}

}  // namespace
}  // namespace pkvd

extern "C" int decode_selftest_wait_timeout(int32_t* status, int64_t limit_us,
                                            pkvd_stream_t stream) {
  if (!status || limit_us < 1 || limit_us > 10000000) return PKVD_EINVAL;
  pkvd::wait_timeout_probe<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      status, static_cast<unsigned long long>(limit_us) * 1000ull);
  return cudaGetLastError() == cudaSuccess ? PKVD_OK : PKVD_ECUDA;
}
