// Failure detection, checked without a GPU fault: every wait in the library's
// kernels is an mbarrier wait bounded by a time limit, after which the kernel
// sets bit 0 of the caller's status word and returns (bsr_last_device_error reads
// the schedule's word).  This entry point runs that same bounded wait on a barrier
// that nothing ever arrives on, so the give-up path runs for real: the wait ends
// after `limit_ns`, the bit is set, and the context stays usable for later work.
#include <cuda_runtime.h>

#include <cstdint>

#include "bsr_attn.h"
#include "bsr_internal.h"
#include "ptx.cuh"

namespace {

__global__ void __launch_bounds__(32) bounded_wait_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = bsr::ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    bsr::ptx::mbar_init(b, 1);   // one arrival expected; none is ever made
    bsr::ptx::fence_barrier_init();
  }
  __syncwarp();
  const bool done = bsr::ptx::mbar_wait_bounded(b, 0, limit_ns);
  if (!done && threadIdx.x == 0) atomicOr(status, bsr::kStatusWaitTimeout);
}

}  // namespace

extern "C" int bsr_selftest_bounded_wait(int32_t* device_status, int64_t limit_ns,
                                         void* stream) {
  if (device_status == nullptr || limit_ns <= 0 || limit_ns > 10000000000ll)
    return BSR_ERR_INVALID_ARGUMENT;
  bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(device_status,
                                                                       uint64_t(limit_ns));
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? BSR_OK : BSR_ERR_CUDA;
}
