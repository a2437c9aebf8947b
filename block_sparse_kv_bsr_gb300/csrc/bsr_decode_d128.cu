// Instantiations of the decode kernel for head_dim 128 and their launcher.
#include <atomic>
#include "bsr_decode.cuh"
#include "bsr_schedule.h"

namespace bsr {

namespace {
constexpr int kMaxDevices = 64;

template <bool ROPE, bool R16, bool SMALLP, bool WIN>
cudaError_t launch_one(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                       int grid, cudaStream_t stream) {
  auto kern = bsr_decode_kernel<128, ROPE, R16, SMALLP, WIN>;
  constexpr size_t smem = ROPE ? DecodeCfg<128>::kSmemBytesRope : DecodeCfg<128>::kSmemBytes;
  // The shared-memory opt-in is per device; set it on the first launch there so
  // that later launches (including ones under stream capture) make no extra call.
  static std::atomic<bool> opted_in[kMaxDevices];   // zero-initialized: false
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!opted_in[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    opted_in[dev].store(true, std::memory_order_release);
  }
  const cudaError_t le = launch_pdl(kern, grid, kDecodeWarps * 32, smem, stream, tk, tv, p);
  return le != cudaSuccess ? le : cudaGetLastError();
}
}  // namespace

cudaError_t launch_decode_d128(bool rope, bool r16, bool smallp, const CUtensorMap& tk,
                               const CUtensorMap& tv, const DecodeParams& p, int grid,
                               cudaStream_t stream) {
  const int key = (rope ? 4 : 0) | (r16 ? 2 : 0) | (smallp ? 1 : 0);
  if (p.window_left > 0) {
    switch (key) {
      case 0: return launch_one<false, false, false, true>(tk, tv, p, grid, stream);
      case 1: return launch_one<false, false, true, true>(tk, tv, p, grid, stream);
      case 2: return launch_one<false, true, false, true>(tk, tv, p, grid, stream);
      case 3: return launch_one<false, true, true, true>(tk, tv, p, grid, stream);
      case 4: return launch_one<true, false, false, true>(tk, tv, p, grid, stream);
      case 5: return launch_one<true, false, true, true>(tk, tv, p, grid, stream);
      case 6: return launch_one<true, true, false, true>(tk, tv, p, grid, stream);
      default: return launch_one<true, true, true, true>(tk, tv, p, grid, stream);
    }
  }
  switch (key) {
    case 0: return launch_one<false, false, false, false>(tk, tv, p, grid, stream);
    case 1: return launch_one<false, false, true, false>(tk, tv, p, grid, stream);
    case 2: return launch_one<false, true, false, false>(tk, tv, p, grid, stream);
    case 3: return launch_one<false, true, true, false>(tk, tv, p, grid, stream);
    case 4: return launch_one<true, false, false, false>(tk, tv, p, grid, stream);
    case 5: return launch_one<true, false, true, false>(tk, tv, p, grid, stream);
    case 6: return launch_one<true, true, false, false>(tk, tv, p, grid, stream);
    default: return launch_one<true, true, true, false>(tk, tv, p, grid, stream);
  }
}

}  // namespace bsr
