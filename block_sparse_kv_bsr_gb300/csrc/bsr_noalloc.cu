// bsr_attn_decode_noalloc: split-KV decode for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc at the point where they need attention:
// an inference runtime whose memory is carved up once at start-up by its own
// allocator, code that runs where allocating would synchronize the device or
// break a fixed memory budget, or a plugin host that forbids allocation
// inside its execute callback.  This entry point serves them.  It runs the
// same decode kernel as bsr_attn_run, but the kernel's scratch memory (work
// units, per-warp ranges, merge counters, partial states) lives in one
// file-scope __device__ array of fixed size instead of a planned workspace,
// and the split of each request into key chunks is computed on the device
// from the device-resident page table.  Nothing is allocated: no cudaMalloc,
// no cudaFree, no pinned or pageable host buffer.
//
// Costs of that choice, for the user: the array (kScratchBytes, about 17 MB)
// is held on every GPU that loads this library until the process exits; all
// calls on a device share it, so two calls whose kernels overlap on the GPU
// race (serialize them on one stream); and the chunking is a fixed equal split
// per (request, kv head) rather than the host planner's balanced cut.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "bsr_attn.h"
#include "bsr_schedule.h"

namespace {

using bsr::DecodeItem;
using bsr::kDecodeWarps;
using bsr::kMaxDecodeRows;
using bsr::kStageTokens;

// Capacity of the static scratch: work units of (request, kv head, chunk).
constexpr int kMaxUnits = 2048;
// Largest number of chunks one (request, kv head) range is cut into.
constexpr int kMaxSplits = 64;
constexpr int kMaxHeadDim = 128;
constexpr int kMaxDevices = 64;

// Layout of the scratch array (byte offsets, each 256-aligned).
constexpr size_t kOffItems = 0;
constexpr size_t kOffWarpPtr = kOffItems + size_t(kMaxUnits) * sizeof(DecodeItem);
constexpr size_t kOffCounters = kOffWarpPtr + size_t(kMaxUnits + 64) * 4;
constexpr size_t kOffStatus = kOffCounters + size_t(kMaxUnits) * 4;
constexpr size_t kOffPartLse = kOffStatus + 256;
constexpr size_t kOffPartO = kOffPartLse + size_t(kMaxUnits) * kMaxDecodeRows * 4;
constexpr size_t kScratchBytes = kOffPartO + size_t(kMaxUnits) * kMaxDecodeRows * kMaxHeadDim * 4;
static_assert(kOffWarpPtr % 256 == 0 && kOffCounters % 256 == 0 && kOffStatus % 256 == 0 &&
                  kOffPartLse % 256 == 0 && kOffPartO % 256 == 0,
              "scratch regions must stay 256-byte aligned");

// The scratch itself.  In host code `g_scratch` names a host-side stand-in,
// not device memory: the host only ever passes the address returned by
// cudaGetSymbolAddress for the current device.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

// One block per request.  The block checks the request's table entries and every
// page its query reads, then writes the request's work units (one per (kv head,
// chunk)), points one warp at each, and clears their merge counters: every call
// starts from a known state whatever the previous call left behind.  A request
// whose entries are malformed (negative page count or offset, last_page_len
// outside [1, P], a length beyond 32-bit keys) or which reads a page outside the
// pool gets empty units -- all of its chunks, so its out is 0 and its lse -inf --
// and bit 1 of the status word is set.
constexpr int kFillThreads = 256;
__global__ void __launch_bounds__(kFillThreads)
    fill_units_kernel(uint8_t* scratch, const int32_t* __restrict__ indptr,
                      const int32_t* __restrict__ indices,
                      const int32_t* __restrict__ last_page_len, int32_t batch, int32_t Hk,
                      int32_t group, int32_t P, int32_t num_pages, int32_t splits,
                      int32_t window_left, int32_t* status) {
  DecodeItem* items = reinterpret_cast<DecodeItem*>(scratch + kOffItems);
  int32_t* warp_ptr = reinterpret_cast<int32_t*>(scratch + kOffWarpPtr);
  int32_t* counters = reinterpret_cast<int32_t*>(scratch + kOffCounters);
  const int32_t b = blockIdx.x;
  if (b == 0 && threadIdx.x == 0) warp_ptr[batch * Hk * splits] = batch * Hk * splits;
  const int32_t base = indptr[b];
  const int64_t n = int64_t(indptr[b + 1]) - base;
  bool bad = base < 0 || n < 0;
  int64_t L = 0;
  if (!bad && n > 0) {
    const int32_t last = last_page_len[b];
    L = (n - 1) * P + last;
    bad = last < 1 || last > P || L > INT32_MAX;
  }
  const int32_t align = P > kStageTokens ? P : kStageTokens;
  // sliding window: the range starts at the page (or 16-key stage) holding the oldest
  // key the query sees; older pages are never read (and not checked)
  int64_t kb = 0;
  if (!bad && window_left > 0 && L > window_left) kb = (L - window_left) / align * align;
  // the device table cannot be checked on the host: check the pages this query reads
  if (!bad)
    for (int64_t j = kb / P + threadIdx.x; j < (L + P - 1) / P; j += kFillThreads) {
      const int32_t page = indices[base + j];
      bad |= page < 0 || page >= num_pages;
    }
  bad = __syncthreads_or(bad) != 0;
  if (bad) {
    if (threadIdx.x == 0 && status != nullptr) atomicOr(status, 2);
    L = kb = 0;
  }
  int64_t len = (L - kb + splits - 1) / splits;
  len = (len + align - 1) / align * align;
  for (int32_t i = threadIdx.x; i < Hk * splits; i += kFillThreads) {
    const int32_t kvh = i / splits, s = i % splits;
    const int32_t bh = b * Hk + kvh;
    const int32_t u = bh * splits + s;
    int64_t t0 = kb + s * len, t1 = t0 + len < L ? t0 + len : L;
    if (t0 >= L) t0 = t1 = 0;  // an empty chunk still reports an empty state to the merge
    DecodeItem it;
    it.req = b;
    it.kvh = kvh;
    it.row0 = 0;
    it.nrows = group;
    it.tok0 = int32_t(t0);
    it.tok1 = int32_t(t1);
    it.nchunks = splits;
    it.first_slot = bh * splits;
    it.slot = splits > 1 ? u : -1;
    it.page_base = bad ? 0 : base;
    it.q_row0 = b;
    it.qpos0 = int32_t(L) - 1;
    items[u] = it;
    warp_ptr[u] = u;
    if (s == 0) counters[bh * splits] = 0;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Same stage geometry as the planned path: 16 rows x 64 columns, 128B swizzle; with
// D = 128 both 64-column blocks of a stage in one box (rows as the inner dimension).
bool encode_pool(CUtensorMap* tm, const void* base, int64_t rows, int D) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3];
  cuuint64_t strides[2];
  cuuint32_t box[3];
  cuuint32_t estr[3] = {1, 1, 1};
  cuuint32_t rank;
  if (D == 128) {
    rank = 3;
    dims[0] = 64; dims[1] = cuuint64_t(rows); dims[2] = 2;
    strides[0] = 256; strides[1] = 128;
    box[0] = 64; box[1] = kStageTokens; box[2] = 2;
  } else {
    rank = 2;
    dims[0] = 64; dims[1] = cuuint64_t(rows);
    strides[0] = 128;
    box[0] = 64; box[1] = kStageTokens;
  }
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map over an FP8 (E4M3) page pool [num_pages, Hk, P, 128] seen as rows of 128
// one-byte codes: one box of 16 rows x 128 B per 16-key stage, 128B-swizzled.
bool encode_pool_e4m3(CUtensorMap* tm, const void* base, int64_t rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {128, cuuint64_t(rows)};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, kStageTokens};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Device address of the scratch array, looked up once per device (with that
// device current) on the first call made there.
uint8_t* scratch_on(int dev) {
  static uint8_t* addr[kMaxDevices] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = static_cast<uint8_t*>(p);
  }
  return addr[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Both entry points: a bf16 cache, or (kv8) E4M3 codes with one scale per pool.
int noalloc_impl(const void* q, const void* k_pages, const void* v_pages, const int32_t* indptr,
                 const int32_t* indices, const int32_t* last_page_len, int32_t batch,
                 int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                 int32_t num_pages_in_pool, float sm_scale, bool kv8, float k_scale,
                 float v_scale, int32_t window_left, void* out, int32_t out_dtype, float* lse,
                 int32_t* device_status, void* stream_v) {
  if (window_left < 0) return BSR_ERR_INVALID_ARGUMENT;
  if (batch < 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || num_pages_in_pool < 0)
    return BSR_ERR_INVALID_ARGUMENT;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return BSR_ERR_INVALID_ARGUMENT;
  if (kv8 && (!(k_scale > 0.f) || !std::isfinite(k_scale) || !(v_scale > 0.f) ||
              !std::isfinite(v_scale)))
    return BSR_ERR_INVALID_ARGUMENT;
  // the FP8 kernel covers head_dim 128 with pages of at least one 16-key stage
  if (kv8 && (head_dim != 128 || page_size < kStageTokens)) return BSR_ERR_UNSUPPORTED;
  if (out_dtype != BSR_DTYPE_BF16 && out_dtype != BSR_DTYPE_F32) return BSR_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128) return BSR_ERR_UNSUPPORTED;
  if (page_size <= 0 || page_size > 256 || (page_size & (page_size - 1))) return BSR_ERR_UNSUPPORTED;
  if (num_qo_heads % num_kv_heads != 0 || num_qo_heads / num_kv_heads > kMaxDecodeRows)
    return BSR_ERR_UNSUPPORTED;
  if (int64_t(num_pages_in_pool) * num_kv_heads * page_size > INT32_MAX) return BSR_ERR_UNSUPPORTED;
  // The static scratch holds kMaxUnits (request, kv head, chunk) units: larger batches are
  // refused here, before anything is launched.
  if (int64_t(batch) * num_kv_heads > kMaxUnits) return BSR_ERR_UNSUPPORTED;
  if (batch == 0) return BSR_OK;
  if (!q || !k_pages || !v_pages || !indptr || !indices || !last_page_len || !out)
    return BSR_ERR_INVALID_ARGUMENT;
  if (!aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(q, 4) ||
      !aligned(out, out_dtype == BSR_DTYPE_F32 ? 8 : 4) || (lse && !aligned(lse, 4)))
    return BSR_ERR_INVALID_ARGUMENT;
  const cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return BSR_ERR_CUDA;
  }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return BSR_ERR_CUDA;
  }
  uint8_t* scratch = scratch_on(dev);
  if (scratch == nullptr) return BSR_ERR_CUDA;

  // Equal split per (request, kv head): enough units to cover every warp slot of the
  // persistent grid, never more than the scratch holds.
  const int64_t pairs = int64_t(batch) * num_kv_heads;
  // (the FP8 kernel keeps decode_kv8_warps(false) warps per SM, the bf16 one kDecodeWarps)
  const int64_t want = int64_t(sms) * (kv8 ? bsr::decode_kv8_warps(false) : kDecodeWarps);
  int64_t splits = (want + pairs - 1) / pairs;
  if (splits > kMaxSplits) splits = kMaxSplits;
  if (splits * pairs > kMaxUnits) splits = kMaxUnits / pairs;
  if (splits < 1) splits = 1;
  const int32_t units = int32_t(splits * pairs);
  const int32_t group = num_qo_heads / num_kv_heads;
  int32_t* status = device_status != nullptr
                        ? device_status
                        : reinterpret_cast<int32_t*>(scratch + kOffStatus);

  fill_units_kernel<<<batch, kFillThreads, 0, stream>>>(
      scratch, indptr, indices, last_page_len, batch, num_kv_heads, group, page_size,
      num_pages_in_pool, int32_t(splits), window_left, status);
  if (cudaGetLastError() != cudaSuccess) return BSR_ERR_CUDA;

  const bool smallp = page_size < kStageTokens;
  CUtensorMap tk{}, tv{};
  const int64_t rows = int64_t(num_pages_in_pool) * num_kv_heads * page_size;
  if (kv8) {
    if (rows <= 0 || !encode_pool_e4m3(&tk, k_pages, rows) || !encode_pool_e4m3(&tv, v_pages, rows))
      return BSR_ERR_CUDA;
  } else if (!smallp) {
    if (rows <= 0 || !encode_pool(&tk, k_pages, rows, head_dim) ||
        !encode_pool(&tv, v_pages, rows, head_dim))
      return BSR_ERR_CUDA;
  }
  bsr::DecodeParams p{};
  p.items = reinterpret_cast<const DecodeItem*>(scratch + kOffItems);
  p.warp_ptr = reinterpret_cast<const int32_t*>(scratch + kOffWarpPtr);
  p.counters = reinterpret_cast<int32_t*>(scratch + kOffCounters);
  p.part_o = reinterpret_cast<float*>(scratch + kOffPartO);
  p.part_lse = reinterpret_cast<float*>(scratch + kOffPartLse);
  p.indices = indices;
  p.rope = nullptr;
  p.q = static_cast<const uint16_t*>(q);
  p.k_pages = k_pages;
  p.v_pages = v_pages;
  p.out = out;
  p.lse = lse;
  p.error = status;
  // an FP8 cache's k_scale folds into the logit scale, v_scale into the normalisation
  p.scale_log2 = float(double(sm_scale) * (kv8 ? double(k_scale) : 1.0) * 1.4426950408889634);
  p.v_scale = kv8 ? v_scale : 1.f;
  p.Hq = num_qo_heads;
  p.Hk = num_kv_heads;
  p.group = group;
  p.P = page_size;
  p.causal = 0;
  p.out_f32 = out_dtype == BSR_DTYPE_F32;
  p.num_warps = units;
  p.window_left = window_left;
  p.rope_max_pos = 0;
  p.wait_limit_ns = 1000000000ull;
  const int grid = (units + kDecodeWarps - 1) / kDecodeWarps;
  const bool r16 = group > 8;
  const cudaError_t e =
      kv8 ? bsr::launch_decode_kv8(false, r16, tk, tv, p, stream)
          : head_dim == 128 ? bsr::launch_decode_d128(false, r16, smallp, tk, tv, p, grid, stream)
                            : bsr::launch_decode_d64(false, r16, smallp, tk, tv, p, grid, stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return BSR_ERR_CUDA;
  }
  return BSR_OK;
}

}  // namespace

extern "C" int bsr_attn_decode_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                       const int32_t* indptr, const int32_t* indices,
                                       const int32_t* last_page_len, int32_t batch,
                                       int32_t num_qo_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t page_size,
                                       int32_t num_pages_in_pool, float sm_scale, void* out,
                                       int32_t out_dtype, float* lse, int32_t* device_status,
                                       void* stream) {
  return noalloc_impl(q, k_pages, v_pages, indptr, indices, last_page_len, batch, num_qo_heads,
                      num_kv_heads, head_dim, page_size, num_pages_in_pool, sm_scale, false, 1.f,
                      1.f, 0, out, out_dtype, lse, device_status, stream);
}

extern "C" int bsr_attn_decode_noalloc_kv8(const void* q, const void* k_pages,
                                           const void* v_pages, const int32_t* indptr,
                                           const int32_t* indices, const int32_t* last_page_len,
                                           int32_t batch, int32_t num_qo_heads,
                                           int32_t num_kv_heads, int32_t head_dim,
                                           int32_t page_size, int32_t num_pages_in_pool,
                                           float sm_scale, float k_scale, float v_scale,
                                           void* out, int32_t out_dtype, float* lse,
                                           int32_t* device_status, void* stream) {
  return noalloc_impl(q, k_pages, v_pages, indptr, indices, last_page_len, batch, num_qo_heads,
                      num_kv_heads, head_dim, page_size, num_pages_in_pool, sm_scale, true,
                      k_scale, v_scale, 0, out, out_dtype, lse, device_status, stream);
}

extern "C" int bsr_attn_decode_noalloc_ex(const void* q, const void* k_pages, const void* v_pages,
                                          const int32_t* indptr, const int32_t* indices,
                                          const int32_t* last_page_len, int32_t batch,
                                          int32_t num_qo_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t page_size,
                                          int32_t num_pages_in_pool, float sm_scale,
                                          int32_t kv_dtype, float k_scale, float v_scale,
                                          int32_t window_left, void* out, int32_t out_dtype,
                                          float* lse, int32_t* device_status, void* stream) {
  if (kv_dtype != BSR_KV_DTYPE_BF16 && kv_dtype != BSR_KV_DTYPE_E4M3) return BSR_ERR_INVALID_ARGUMENT;
  const bool kv8 = kv_dtype == BSR_KV_DTYPE_E4M3;
  return noalloc_impl(q, k_pages, v_pages, indptr, indices, last_page_len, batch, num_qo_heads,
                      num_kv_heads, head_dim, page_size, num_pages_in_pool, sm_scale, kv8,
                      kv8 ? k_scale : 1.f, kv8 ? v_scale : 1.f, window_left, out, out_dtype, lse,
                      device_status, stream);
}
