// bsr_merge_states and bsr_append_kv: the two small memory-bound kernels of
// the path.  Both are plain coalesced streaming kernels, grid-stride loops
// over a grid sized in multiples of the SM count, no shared memory.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "bsr_attn.h"

namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------- merge_states
// One warp per (row, head); each lane owns D / 32 consecutive columns.
// State (o, lse) is the softmax-weighted mean of its keys and their natural
// log-sum-exp; merging two states over disjoint keys reweights each mean by
// exp(lse_x - lse) ("FlashInfer: Block-Sparse KV 캐시로 …", section
// "Block-Sparse 포맷": a shared prefix composed with per-request suffixes).
template <int D, bool F32>
__global__ void __launch_bounds__(kThreads) merge_states_kernel(
    const void* __restrict__ oa, const float* __restrict__ la, const void* __restrict__ ob,
    const float* __restrict__ lb, int64_t n, void* oo, float* lo) {
  constexpr int CPL = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (kThreads / 32);
  for (int64_t w = int64_t(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5); w < n; w += warps) {
    const float a = la[w], b = lb[w];
    const float M = fmaxf(a, b);
    float wa = 0.f, wb = 0.f, l = -INFINITY;
    if (M != -INFINITY) {
      l = M + logf(expf(a - M) + expf(b - M));
      wa = expf(a - l);
      wb = expf(b - l);
    }
    const size_t off = size_t(w) * D + size_t(CPL) * lane;
    float x[CPL], y[CPL];
    if constexpr (F32) {
      const float* pa = static_cast<const float*>(oa) + off;
      const float* pb = static_cast<const float*>(ob) + off;
#pragma unroll
      for (int c = 0; c < CPL; c += 2) {
        const float2 u = *reinterpret_cast<const float2*>(pa + c);
        const float2 v = *reinterpret_cast<const float2*>(pb + c);
        x[c] = u.x; x[c + 1] = u.y; y[c] = v.x; y[c + 1] = v.y;
      }
    } else {
      const uint16_t* pa = static_cast<const uint16_t*>(oa) + off;
      const uint16_t* pb = static_cast<const uint16_t*>(ob) + off;
#pragma unroll
      for (int c = 0; c < CPL; c += 2) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(pa + c);
        const uint32_t v = *reinterpret_cast<const uint32_t*>(pb + c);
        x[c] = __uint_as_float(u << 16); x[c + 1] = __uint_as_float(u & 0xFFFF0000u);
        y[c] = __uint_as_float(v << 16); y[c + 1] = __uint_as_float(v & 0xFFFF0000u);
      }
    }
    // an empty state (weight 0) contributes exactly nothing, whatever its o holds
#pragma unroll
    for (int c = 0; c < CPL; ++c)
      x[c] = (wa != 0.f ? wa * x[c] : 0.f) + (wb != 0.f ? wb * y[c] : 0.f);
    if constexpr (F32) {
      float* po = static_cast<float*>(oo) + off;
#pragma unroll
      for (int c = 0; c < CPL; c += 2) *reinterpret_cast<float2*>(po + c) = make_float2(x[c], x[c + 1]);
    } else {
      uint16_t* po = static_cast<uint16_t*>(oo) + off;
#pragma unroll
      for (int c = 0; c < CPL; c += 2) {
        uint32_t r;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(x[c + 1]), "f"(x[c]));
        *reinterpret_cast<uint32_t*>(po + c) = r;
      }
    }
    if (lane == 0) lo[w] = l;
  }
}

// ---------------------------------------------------------------- append_kv
// One 16-byte chunk per thread: chunk c of (new token t, kv head h).  The
// request of t is found by binary search in append_indptr; its position is
// L_b - n_b + i with L_b from the (post-append) page table.
__global__ void __launch_bounds__(kThreads) append_kv_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int32_t* __restrict__ append_indptr, const int32_t* __restrict__ indptr,
    const int32_t* __restrict__ indices, const int32_t* __restrict__ last_page_len, int32_t batch,
    int64_t ntok, int32_t Hk, int32_t chunks, int32_t P, int32_t num_pages, int32_t nhd,
    uint4* k_pages, uint4* v_pages, int32_t* status) {
  const int64_t total = ntok * Hk * chunks;
  for (int64_t g = int64_t(blockIdx.x) * kThreads + threadIdx.x; g < total;
       g += int64_t(gridDim.x) * kThreads) {
    const int32_t c = int32_t(g % chunks);
    const int64_t th = g / chunks;
    const int32_t h = int32_t(th % Hk);
    const int64_t t = th / Hk;
    int32_t lo = 0, hi = batch - 1;  // last b with append_indptr[b] <= t
    while (lo < hi) {
      const int32_t mid = (lo + hi + 1) >> 1;
      if (append_indptr[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int32_t b = lo;
    const int64_t a0 = append_indptr[b], a1 = append_indptr[b + 1];
    const int64_t npg = int64_t(indptr[b + 1]) - indptr[b];
    const int32_t last = npg > 0 ? last_page_len[b] : 0;
    const int64_t L = npg > 0 ? (npg - 1) * P + last : 0;
    const int64_t n_new = a1 - a0;
    if (t < a0 || t >= a1 || npg <= 0 || last < 1 || last > P || n_new > L) {
      if (status) atomicOr(status, 1);
      continue;
    }
    const int64_t pos = L - n_new + (t - a0);
    const int32_t page = indices[indptr[b] + pos / P];
    if (page < 0 || page >= num_pages) {
      if (status) atomicOr(status, 1);
      continue;
    }
    // head-major pages [page][Hk][P][D] or token-major [page][P][Hk][D]
    const size_t dst = nhd ? ((size_t(page) * P + size_t(pos % P)) * Hk + h) * chunks + c
                           : ((size_t(page) * Hk + h) * P + size_t(pos % P)) * chunks + c;
    const size_t src = (size_t(t) * Hk + h) * chunks + c;
    k_pages[dst] = k_new[src];
    v_pages[dst] = v_new[src];
  }
}

int grid_for(int64_t work_items, int per_block) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t need = (work_items + per_block - 1) / per_block;
  const int64_t cap = int64_t(sms) * 8;  // 8 resident 256-thread blocks per SM
  return int(need < 1 ? 1 : (need < cap ? need : cap));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int bsr_merge_states(const void* o_a, const float* lse_a, const void* o_b,
                                const float* lse_b, int64_t num_rows, int32_t num_heads,
                                int32_t head_dim, int32_t dtype, void* o_out, float* lse_out,
                                void* stream_v) {
  if (num_rows < 0 || num_heads <= 0) return BSR_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128) return BSR_ERR_UNSUPPORTED;
  if (dtype != BSR_DTYPE_BF16 && dtype != BSR_DTYPE_F32) return BSR_ERR_INVALID_ARGUMENT;
  const int64_t n = num_rows * num_heads;
  if (n == 0) return BSR_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o_out || !lse_out) return BSR_ERR_INVALID_ARGUMENT;
  const uintptr_t al = dtype == BSR_DTYPE_F32 ? 8 : 4;
  if (!aligned(o_a, al) || !aligned(o_b, al) || !aligned(o_out, al)) return BSR_ERR_INVALID_ARGUMENT;
  const cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  const int grid = grid_for(n, kThreads / 32);
  if (head_dim == 128) {
    if (dtype == BSR_DTYPE_F32)
      merge_states_kernel<128, true><<<grid, kThreads, 0, stream>>>(o_a, lse_a, o_b, lse_b, n, o_out, lse_out);
    else
      merge_states_kernel<128, false><<<grid, kThreads, 0, stream>>>(o_a, lse_a, o_b, lse_b, n, o_out, lse_out);
  } else {
    if (dtype == BSR_DTYPE_F32)
      merge_states_kernel<64, true><<<grid, kThreads, 0, stream>>>(o_a, lse_a, o_b, lse_b, n, o_out, lse_out);
    else
      merge_states_kernel<64, false><<<grid, kThreads, 0, stream>>>(o_a, lse_a, o_b, lse_b, n, o_out, lse_out);
  }
  if (cudaGetLastError() != cudaSuccess) return BSR_ERR_CUDA;
  return BSR_OK;
}

extern "C" int bsr_append_kv(const void* k_new, const void* v_new, const int32_t* append_indptr,
                             const int32_t* indptr, const int32_t* indices,
                             const int32_t* last_page_len, int32_t batch, int64_t num_new_tokens,
                             int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                             int32_t num_pages_in_pool, int32_t kv_layout, void* k_pages,
                             void* v_pages, int32_t* device_status, void* stream_v) {
  if (batch < 0 || num_new_tokens < 0 || num_kv_heads <= 0 || num_pages_in_pool < 0)
    return BSR_ERR_INVALID_ARGUMENT;
  if (kv_layout != BSR_KV_HND && kv_layout != BSR_KV_NHD) return BSR_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128) return BSR_ERR_UNSUPPORTED;
  if (page_size <= 0 || page_size > 256 || (page_size & (page_size - 1))) return BSR_ERR_UNSUPPORTED;
  if (num_new_tokens == 0) return BSR_OK;
  if (batch == 0) return BSR_ERR_INVALID_ARGUMENT;
  if (!k_new || !v_new || !append_indptr || !indptr || !indices || !last_page_len || !k_pages ||
      !v_pages)
    return BSR_ERR_INVALID_ARGUMENT;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16))
    return BSR_ERR_INVALID_ARGUMENT;
  const cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  const int32_t chunks = head_dim / 8;
  const int64_t work = num_new_tokens * num_kv_heads * chunks;
  append_kv_kernel<<<grid_for(work, kThreads), kThreads, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), append_indptr, indptr,
      indices, last_page_len, batch, num_new_tokens, num_kv_heads, chunks, page_size,
      num_pages_in_pool, kv_layout == BSR_KV_NHD ? 1 : 0, static_cast<uint4*>(k_pages),
      static_cast<uint4*>(v_pages), device_status);
  if (cudaGetLastError() != cudaSuccess) return BSR_ERR_CUDA;
  return BSR_OK;
}
