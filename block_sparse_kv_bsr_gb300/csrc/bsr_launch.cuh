// Kernel launches with programmatic dependent launch: a kernel launched this way
// may be scheduled while the kernel before it on the stream is still finishing, so
// its CTAs' start-up (scheduling, shared-memory set-up, barrier initialisation)
// overlaps the previous kernel's tail instead of following it.  Every kernel
// launched here executes pdl_wait() -- which returns once the previous grid has
// completed and its memory operations are visible -- before its first access to
// global memory that another kernel may write (q, the pages, outputs, partial
// states, counters, the status word), so no such data is read early and none a
// previous kernel reads is overwritten early.  Only what a plan's host copy wrote
// before the launch (work lists, page table, RoPE tables) may be read before the
// wait.  Launched after a copy, or after a kernel launched the ordinary way, a
// kernel simply starts when that work is done.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace bsr {

// Let the next grid on the stream be scheduled (it still waits in pdl_wait).
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the previous grid on the stream has completed and flushed its memory.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), int grid, int threads, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(unsigned(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace bsr
