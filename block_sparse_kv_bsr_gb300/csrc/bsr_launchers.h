// Kernel launchers and the launch shape they share with the planner (device code sees
// this header; the schedule's host-side state is in bsr_schedule.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "bsr_internal.h"

namespace bsr {
// Warps per CTA (one CTA per SM) of the FP8 (E4M3) decode kernel.  Without RoPE a
// 16-key stage is half the bf16 kernel's bytes and each warp's chain of conversions
// and MMAs is latency-bound, so 12 warps (a 170-register cap; 4 stages each) keep
// more stages in flight: 88 against 97.5 us on the skewed batch (10 warps measured
// 100 us).  With RoPE (253 registers) 12 warps spill heavily, so it keeps 8.
__host__ __device__ constexpr int decode_kv8_warps(bool rope) { return rope ? kDecodeWarps : 12; }

// Kernel launchers (one translation unit per head dim).
cudaError_t launch_decode_d64(bool rope, bool r16, bool smallp, const CUtensorMap& tk,
                              const CUtensorMap& tv, const DecodeParams& p, int grid,
                              cudaStream_t stream);
cudaError_t launch_decode_d128(bool rope, bool r16, bool smallp, const CUtensorMap& tk,
                               const CUtensorMap& tv, const DecodeParams& p, int grid,
                               cudaStream_t stream);
// the grid is one CTA of decode_kv8_warps(rope) warps per p.num_warps of them
cudaError_t launch_decode_kv8(bool rope, bool r16, const CUtensorMap& tk, const CUtensorMap& tv,
                              const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_prefill(bool rope, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const PrefillParams& p, int grid,
                           cudaStream_t stream);
cudaError_t launch_prefill_merge(const PrefillMergeParams& p, cudaStream_t stream);
}  // namespace bsr
