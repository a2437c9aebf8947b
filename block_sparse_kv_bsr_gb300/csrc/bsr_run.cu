// bsr_attn_run: executes a planned schedule on the GPU.
//
// Host work here is argument checking, encoding the TMA tensor maps of the
// caller's K/V page pools (cached per pool pointer), and one kernel launch.
// Nothing is allocated and the host is never synchronized, so the call can
// be captured in a CUDA graph.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "bsr_attn.h"
#include "bsr_schedule.h"

namespace {

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

// Tensor map over a page pool [num_pages, Hk, P, D] bf16 seen as rows of D
// elements, loaded 16 rows x 64 columns at a time into 128B-swizzled tiles.
// D = 128: rank 3 {64 cols, 2 column blocks, rows} so one box is one column
// block of 16 rows; D = 64: rank 2 {64 cols, rows}.
// Page pools are [pages, Hk, P, D] (HND: a (page, head) block of P rows is
// contiguous; rows = pages * Hk * P, row (page * Hk + h) * P + t) or
// [pages, P, Hk, D] (NHD: token-major; token rows = pages * P, row page * P + t,
// the head an outer map dimension of stride D elements).  Every map below lands
// the same shared-memory layout in both cases; only the coordinates differ.
struct PoolGeom {
  int64_t rows;     // HND rows (pages * Hk * P)
  int32_t Hk;
  bool nhd;
  int64_t tok_rows() const { return rows / Hk; }
};

bool encode(CUtensorMap* tm, CUtensorMapDataType dt, cuuint32_t rank, const void* base,
            const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(tm, dt, rank, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map over a page pool for the decode kernel's 16-key stages.  D = 128: the two 64-column blocks are
// an outer dimension (stride 128 B), so one box {64, rows, 2} lands the tile as
// [column block][rows][128 B], 128B-swizzled: one copy where two would do (a TMA
// copy's cost is mostly per box: ~26 B/clk per SM with 4 KB boxes against ~20
// with 2 KB ones).  D = 64: one box of [rows][128 B].
bool encode_pool_stage(CUtensorMap* tm, const void* base, const PoolGeom& g, int D,
                       int box_rows = bsr::kStageTokens) {
  constexpr auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint64_t hs = cuuint64_t(D) * 2;   // bytes of one head row
  if (D == 128) {
    if (!g.nhd) {
      const cuuint64_t dims[3] = {64, cuuint64_t(g.rows), 2};
      const cuuint64_t strides[2] = {hs, 128};
      const cuuint32_t box[3] = {64, cuuint32_t(box_rows), 2};
      return encode(tm, BF, 3, base, dims, strides, box);
    }
    const cuuint64_t dims[4] = {64, cuuint64_t(g.tok_rows()), 2, cuuint64_t(g.Hk)};
    const cuuint64_t strides[3] = {cuuint64_t(g.Hk) * hs, 128, hs};
    const cuuint32_t box[4] = {64, cuuint32_t(box_rows), 2, 1};
    return encode(tm, BF, 4, base, dims, strides, box);
  }
  if (!g.nhd) {
    const cuuint64_t dims[2] = {64, cuuint64_t(g.rows)};
    const cuuint64_t strides[1] = {hs};
    const cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
    return encode(tm, BF, 2, base, dims, strides, box);
  }
  const cuuint64_t dims[3] = {64, cuuint64_t(g.tok_rows()), cuuint64_t(g.Hk)};
  const cuuint64_t strides[2] = {cuuint64_t(g.Hk) * hs, hs};
  const cuuint32_t box[3] = {64, cuuint32_t(box_rows), 1};
  return encode(tm, BF, 3, base, dims, strides, box);
}

// Tensor map over an FP8 (E4M3, one byte per element) page pool with D = 128: one
// box is a 16-key stage, [16 rows][128 B], 128B-swizzled (a row is a whole head).
bool encode_pool_e4m3(CUtensorMap* tm, const void* base, const PoolGeom& g) {
  constexpr auto U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  if (!g.nhd) {
    const cuuint64_t dims[2] = {128, cuuint64_t(g.rows)};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, bsr::kStageTokens};
    return encode(tm, U8, 2, base, dims, strides, box);
  }
  const cuuint64_t dims[3] = {128, cuuint64_t(g.tok_rows()), cuuint64_t(g.Hk)};
  const cuuint64_t strides[2] = {cuuint64_t(g.Hk) * 128, 128};
  const cuuint32_t box[3] = {128, bsr::kStageTokens, 1};
  return encode(tm, U8, 3, base, dims, strides, box);
}

// Tensor map over a D = 64 or 128 page pool for the prefill kernel's K and V tiles: a
// box {64 cols, 8 rows, 2 column blocks, box_rows / 8 row groups} lands as [row group]
// [column block][8 rows][128 B], 128B-swizzled, so the boxes of a 128-key tile
// stack into one uniform layout (8-row groups 2 KB apart, the column blocks of a
// group 1 KB apart) whatever the page size: one box per page-sized piece.
// Rows (token rows with NHD) must be a multiple of 8.  A D = 64 pool has one column
// block: the box still spans two and the second lands as zeros, so a D = 64 head runs
// the 128-wide tile program with its upper 64 dimensions zero.
bool encode_pool_groups(CUtensorMap* tm, const void* base, const PoolGeom& g, int box_rows,
                        int D) {
  constexpr auto BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (box_rows % 8 != 0 || (D != 64 && D != 128)) return false;
  const cuuint64_t hs = cuuint64_t(D) * 2;   // bytes of one head row
  const cuuint64_t blocks = cuuint64_t(D / 64);
  if (!g.nhd) {
    if (g.rows % 8 != 0) return false;
    const cuuint64_t dims[4] = {64, 8, blocks, cuuint64_t(g.rows / 8)};
    const cuuint64_t strides[3] = {hs, 128, 8 * hs};
    const cuuint32_t box[4] = {64, 8, 2, cuuint32_t(box_rows / 8)};
    return encode(tm, BF, 4, base, dims, strides, box);
  }
  if (g.tok_rows() % 8 != 0) return false;
  const cuuint64_t rs = cuuint64_t(g.Hk) * hs;   // token row stride
  const cuuint64_t dims[5] = {64, 8, blocks, cuuint64_t(g.tok_rows() / 8), cuuint64_t(g.Hk)};
  const cuuint64_t strides[4] = {rs, 128, 8 * rs, hs};
  const cuuint32_t box[5] = {64, 8, 2, cuuint32_t(box_rows / 8), 1};
  return encode(tm, BF, 5, base, dims, strides, box);
}

// Tensor map over q [rows, Hq, D] (bf16, D = 64 or 128) for the prefill kernel's
// query tiles: rank 4 {64 cols, D / 64 column blocks, Hq heads, rows}; one box is one
// 64-column block of `group` heads x 128 / group queries -- the 128 packed rows of a
// query tile, 128B-swizzled.  The kernel loads two column blocks; with D = 64 the
// second starts past the tensor and lands as zeros.
bool encode_q(CUtensorMap* tm, const void* base, int64_t rows, int Hq, int group, int D) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t hs = cuuint64_t(D) * 2;   // bytes of one head row
  cuuint64_t dims[4] = {64, cuuint64_t(D / 64), cuuint64_t(Hq), cuuint64_t(rows)};
  cuuint64_t strides[3] = {128, hs, cuuint64_t(Hq) * hs};
  cuuint32_t box[4] = {64, 1, cuuint32_t(group), cuuint32_t(bsr::kPrefillKeyTile / group)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int bsr_attn_run(bsr_schedule_t s, const void* q, const void* k_pages,
                            const void* v_pages, float sm_scale, float rope_theta, int32_t causal,
                            void* out, int32_t out_dtype, float* lse, void* stream_v) {
  if (s == nullptr || s->d_ws == nullptr) return BSR_ERR_INVALID_ARGUMENT;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return BSR_ERR_INVALID_ARGUMENT;
  if (out_dtype != BSR_DTYPE_BF16 && out_dtype != BSR_DTYPE_F32) return BSR_ERR_INVALID_ARGUMENT;
  if (rope_theta != s->rope_theta || causal != s->causal) return BSR_ERR_SCHEDULE_MISMATCH;
  if (s->kv_dtype != BSR_KV_DTYPE_BF16) return BSR_ERR_SCHEDULE_MISMATCH;   // planned for FP8
  if (s->n_items == 0 && s->n_pitems == 0) return BSR_OK;
  if (q == nullptr || out == nullptr || k_pages == nullptr || v_pages == nullptr)
    return BSR_ERR_INVALID_ARGUMENT;
  if (!aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(q, 16) || !aligned(out, 16) ||
      (lse && !aligned(lse, 4)))
    return BSR_ERR_INVALID_ARGUMENT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != s->device) return BSR_ERR_SCHEDULE_MISMATCH;
  const cudaStream_t stream = static_cast<cudaStream_t>(stream_v);

  const bool smallp = s->P < bsr::kStageTokens;
  const int64_t rows = int64_t(s->num_pages) * s->Hk * s->P;
  if (!smallp && (s->tm_k_ptr != k_pages || s->tm_v_ptr != v_pages)) {
    const PoolGeom geom{rows, s->Hk, s->kv_layout == BSR_KV_NHD};
    if (rows <= 0 || !encode_pool_stage(&s->tm_k, k_pages, geom, s->D) ||
        !encode_pool_stage(&s->tm_v, v_pages, geom, s->D)) {
      s->tm_k_ptr = s->tm_v_ptr = nullptr;
      return BSR_ERR_CUDA;
    }
    s->tm_k_ptr = k_pages;
    s->tm_v_ptr = v_pages;
  }

  // optional stage timing: events around each launch, in the next slot of the ring
  int t_slot = -1;
  if (s->t_max > 0) {
    t_slot = int(s->t_count % s->t_max);
    ++s->t_count;
    for (int st = 0; st < bsr_schedule::kStages; ++st) s->t_ran[t_slot * bsr_schedule::kStages + st] = 0;
  }
  auto t_mark = [&](int stage, int edge) {
    if (t_slot < 0) return;
    cudaEventRecord(s->t_ev[(t_slot * bsr_schedule::kStages + stage) * 2 + edge], stream);
    if (edge == 1) s->t_ran[t_slot * bsr_schedule::kStages + stage] = 1;
  };

  const bool rope = s->rope_rows > 0;
  const float scale_log2 = float(double(sm_scale) * 1.4426950408889634);
  const uint64_t wait_limit_ns = 1000000000ull;  // 1 s: orders of magnitude above any healthy wait
  CUtensorMap dummy{};
  const CUtensorMap& tk = smallp ? dummy : s->tm_k;
  const CUtensorMap& tv = smallp ? dummy : s->tm_v;

  if (s->n_items > 0) {
    bsr::DecodeParams p{};
    p.items = s->dev<const bsr::DecodeItem>(s->off_items);
    p.warp_ptr = s->dev<const int32_t>(s->off_warp_ptr);
    p.counters = s->dev<int32_t>(s->off_counters);
    p.part_o = s->dev<float>(s->off_part_o);
    p.part_lse = s->dev<float>(s->off_part_lse);
    p.indices = s->dev<const int32_t>(s->off_indices);
    p.rope = rope ? reinterpret_cast<const float2*>(s->d_rope) : nullptr;
    p.page_pos = s->has_page_pos ? s->dev<const int32_t>(s->off_page_pos) : nullptr;
    p.qshift = s->has_page_pos ? s->dev<const int32_t>(s->off_qshift) : nullptr;
    p.q = static_cast<const uint16_t*>(q);
    p.k_pages = k_pages;
    p.v_pages = v_pages;
    p.out = out;
    p.lse = lse;
    p.error = s->dev<int32_t>(s->off_error);
    p.scale_log2 = scale_log2;
    p.v_scale = 1.f;
    p.Hq = s->Hq;
    p.Hk = s->Hk;
    p.group = s->group;
    p.P = s->P;
    p.causal = s->causal;
    p.out_f32 = out_dtype == BSR_DTYPE_F32;
    p.num_warps = s->dec_warps;
    p.rope_max_pos = rope ? s->rope_rows - 1 : 0;
    p.window_left = s->window_left;
    p.nhd = s->kv_layout == BSR_KV_NHD;
    p.plan_uploaded = 1;   // the work list and page table came with the plan's copy
    p.n_dyn = smallp ? 0 : s->n_dyn;
    p.dyn_begin = s->dyn_begin;
    p.dyn_ctr = s->dev<int32_t>(s->off_dyn_ctr);
    p.wait_limit_ns = wait_limit_ns;
    const bool r16 = s->max_rows > 8;
    t_mark(0, 0);
    const cudaError_t e =
        s->D == 128 ? bsr::launch_decode_d128(rope, r16, smallp, tk, tv, p, s->dec_ctas, stream)
                    : bsr::launch_decode_d64(rope, r16, smallp, tk, tv, p, s->dec_ctas, stream);
    t_mark(0, 1);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return BSR_ERR_CUDA;
    }
  }
  if (s->n_pitems > 0) {
    // query tiles come straight from q (with RoPE the kernel rotates them in shared memory)
    if (s->tm_q_ptr != q) {
      if (!encode_q(&s->tm_q, q, s->sum_qo, s->Hq, s->group, s->D)) {
        s->tm_q_ptr = nullptr;
        return BSR_ERR_CUDA;
      }
      s->tm_q_ptr = q;
    }
    // K/V boxes of min(P, 128) rows (the prefill class has P >= 16)
    const int box_rows = s->P < bsr::kPrefillKeyTile ? s->P : bsr::kPrefillKeyTile;
    if (s->tm_pk_ptr != k_pages || s->tm_pv_ptr != v_pages) {
      const PoolGeom pgeom{rows, s->Hk, s->kv_layout == BSR_KV_NHD};
      // K and V alike: one box per page-sized piece of a tile (row-group layout)
      if (rows <= 0 || !encode_pool_groups(&s->tm_pk, k_pages, pgeom, box_rows, s->D) ||
          !encode_pool_groups(&s->tm_pv, v_pages, pgeom, box_rows, s->D)) {
        s->tm_pk_ptr = s->tm_pv_ptr = nullptr;
        return BSR_ERR_CUDA;
      }
      s->tm_pk_ptr = k_pages;
      s->tm_pv_ptr = v_pages;
    }
    bsr::PrefillParams p{};
    p.box_rows = box_rows;
    p.rope = rope ? reinterpret_cast<const float4*>(s->d_rope + s->rope_bytes) : nullptr;
    p.page_pos = rope && s->has_page_pos ? s->dev<const int32_t>(s->off_page_pos) : nullptr;
    p.qshift = rope && s->has_page_pos ? s->dev<const int32_t>(s->off_qshift) : nullptr;
    p.rope_max_pos = rope ? s->rope_rows - 1 : 0;
    p.items = s->dev<const bsr::DecodeItem>(s->off_pitems);
    p.cta_ptr = s->dev<const int32_t>(s->off_cta_ptr);
    p.part_o = s->dev<float>(s->off_ppart_o);
    p.part_lse = s->dev<float>(s->off_ppart_lse);
    p.indices = s->dev<const int32_t>(s->off_indices);
    p.out = out;
    p.lse = lse;
    p.error = s->dev<int32_t>(s->off_error);
    p.scale_log2 = scale_log2;
    p.Hq = s->Hq;
    p.Hk = s->Hk;
    p.group = s->group;
    p.P = s->P;
    p.causal = s->causal;
    p.out_f32 = out_dtype == BSR_DTYPE_F32;
    p.out_v8 = aligned(out, 32);
    p.num_ctas = s->pre_ctas;
    p.window_left = s->window_left;
    p.nhd = s->kv_layout == BSR_KV_NHD;
    p.head_dim = s->D;
    p.wait_limit_ns = wait_limit_ns;
    t_mark(1, 0);
    cudaError_t e =
        bsr::launch_prefill(rope, s->tm_q, s->tm_pk, s->tm_pv, p, s->pre_ctas, stream);
    t_mark(1, 1);
    if (e == cudaSuccess && s->n_pmerge > 0) {
      bsr::PrefillMergeParams m{};
      m.units = s->dev<const bsr::DecodeItem>(s->off_pmerge);
      m.part_o = p.part_o;
      m.part_lse = p.part_lse;
      m.out = out;
      m.lse = lse;
      m.n_units = s->n_pmerge;
      m.Hq = s->Hq;
      m.group = s->group;
      m.out_f32 = p.out_f32;
      m.head_dim = s->D;
      t_mark(2, 0);
      e = bsr::launch_prefill_merge(m, stream);
      t_mark(2, 1);
    }
    if (e != cudaSuccess) {
      cudaGetLastError();
      return BSR_ERR_CUDA;
    }
  }
  return BSR_OK;
}

extern "C" int bsr_attn_run_host(bsr_schedule_t s, const void* q_host, const void* k_pages,
                                 const void* v_pages, float k_scale, float v_scale,
                                 float sm_scale, float rope_theta, int32_t causal, void* out_host,
                                 int32_t out_dtype, float* lse_host, void* stream_v) {
  if (s == nullptr || s->d_ws == nullptr) return BSR_ERR_INVALID_ARGUMENT;
  if (out_dtype != BSR_DTYPE_BF16 && out_dtype != BSR_DTYPE_F32) return BSR_ERR_INVALID_ARGUMENT;
  const cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  const size_t n = size_t(s->sum_qo) * size_t(s->Hq) * size_t(s->D);   // q / out elements
  if (n == 0) return s->kv_dtype == BSR_KV_DTYPE_E4M3
                         ? bsr_attn_run_kv8(s, nullptr, k_pages, v_pages, k_scale, v_scale, sm_scale,
                                            rope_theta, causal, nullptr, out_dtype, nullptr, stream_v)
                         : bsr_attn_run(s, nullptr, k_pages, v_pages, sm_scale, rope_theta, causal,
                                        nullptr, out_dtype, nullptr, stream_v);
  if (q_host == nullptr || out_host == nullptr) return BSR_ERR_INVALID_ARGUMENT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != s->device) return BSR_ERR_SCHEDULE_MISMATCH;
  // staging: q (bf16), out (room for fp32), lse, each 256-byte aligned
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = size_t(s->sum_qo) * size_t(s->Hq);
  const size_t q_bytes = n * 2, out_bytes = n * (out_dtype == BSR_DTYPE_F32 ? 4 : 2);
  const size_t need = up(q_bytes) + up(n * 4) + up(rows * 4);
  if (s->io_cap < need) {
    if (s->d_io != nullptr) {
      if (cudaFree(s->d_io) != cudaSuccess) {   // synchronizes: no copy can still use it
        cudaGetLastError();
        return BSR_ERR_CUDA;
      }
      s->d_io = nullptr;
      s->io_cap = 0;
    }
    if (cudaMalloc(reinterpret_cast<void**>(&s->d_io), need) != cudaSuccess) {
      cudaGetLastError();
      return BSR_ERR_OUT_OF_MEMORY;
    }
    s->io_cap = need;
  }
  uint8_t* dq = s->d_io;
  uint8_t* dout = dq + up(q_bytes);
  float* dlse = reinterpret_cast<float*>(dout + up(n * 4));
  if (cudaMemcpyAsync(dq, q_host, q_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess) {
    cudaGetLastError();
    return BSR_ERR_CUDA;
  }
  const int rc = s->kv_dtype == BSR_KV_DTYPE_E4M3
                     ? bsr_attn_run_kv8(s, dq, k_pages, v_pages, k_scale, v_scale, sm_scale,
                                        rope_theta, causal, dout, out_dtype,
                                        lse_host != nullptr ? dlse : nullptr, stream_v)
                     : bsr_attn_run(s, dq, k_pages, v_pages, sm_scale, rope_theta, causal, dout,
                                    out_dtype, lse_host != nullptr ? dlse : nullptr, stream_v);
  if (rc != BSR_OK) return rc;
  if (cudaMemcpyAsync(out_host, dout, out_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      (lse_host != nullptr &&
       cudaMemcpyAsync(lse_host, dlse, rows * 4, cudaMemcpyDeviceToHost, stream) != cudaSuccess)) {
    cudaGetLastError();
    return BSR_ERR_CUDA;
  }
  return BSR_OK;
}

extern "C" int bsr_schedule_set_stage_timing(bsr_schedule_t s, int32_t max_calls) {
  if (s == nullptr || max_calls < 0 || max_calls > (1 << 16)) return BSR_ERR_INVALID_ARGUMENT;
  if (s->device >= 0 && cudaSetDevice(s->device) != cudaSuccess) return BSR_ERR_CUDA;
  for (cudaEvent_t e : s->t_ev) cudaEventDestroy(e);
  s->t_ev.clear();
  s->t_ran.clear();
  s->t_max = 0;
  s->t_count = 0;
  if (max_calls == 0) return BSR_OK;
  const size_t n = size_t(max_calls) * bsr_schedule::kStages * 2;
  s->t_ev.reserve(n);
  for (size_t i = 0; i < n; ++i) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) {
      cudaGetLastError();
      for (cudaEvent_t x : s->t_ev) cudaEventDestroy(x);
      s->t_ev.clear();
      return BSR_ERR_CUDA;
    }
    s->t_ev.push_back(e);
  }
  s->t_ran.assign(size_t(max_calls) * bsr_schedule::kStages, 0);
  s->t_max = max_calls;
  return BSR_OK;
}

extern "C" int bsr_schedule_stage_times(bsr_schedule_t s, int32_t call, float* ms) {
  if (s == nullptr || ms == nullptr || s->t_max == 0) return BSR_ERR_INVALID_ARGUMENT;
  const int64_t kept = s->t_count < s->t_max ? s->t_count : s->t_max;
  if (call < 0 || call >= kept) return BSR_ERR_INVALID_ARGUMENT;
  const int slot = int((s->t_count - kept + call) % s->t_max);
  for (int st = 0; st < bsr_schedule::kStages; ++st) {
    ms[st] = -1.f;
    if (!s->t_ran[size_t(slot) * bsr_schedule::kStages + st]) continue;
    cudaEvent_t b = s->t_ev[(size_t(slot) * bsr_schedule::kStages + st) * 2];
    cudaEvent_t e = s->t_ev[(size_t(slot) * bsr_schedule::kStages + st) * 2 + 1];
    if (cudaEventSynchronize(e) != cudaSuccess || cudaEventElapsedTime(&ms[st], b, e) != cudaSuccess) {
      cudaGetLastError();
      return BSR_ERR_CUDA;
    }
  }
  return int(kept);
}

extern "C" int bsr_attn_run_kv8(bsr_schedule_t s, const void* q, const void* k_pages,
                                const void* v_pages, float k_scale, float v_scale, float sm_scale,
                                float rope_theta, int32_t causal, void* out, int32_t out_dtype,
                                float* lse, void* stream_v) {
  if (s == nullptr || s->d_ws == nullptr) return BSR_ERR_INVALID_ARGUMENT;
  if (!(sm_scale > 0.f) || !std::isfinite(sm_scale)) return BSR_ERR_INVALID_ARGUMENT;
  if (!(k_scale > 0.f) || !std::isfinite(k_scale) || !(v_scale > 0.f) || !std::isfinite(v_scale))
    return BSR_ERR_INVALID_ARGUMENT;
  if (out_dtype != BSR_DTYPE_BF16 && out_dtype != BSR_DTYPE_F32) return BSR_ERR_INVALID_ARGUMENT;
  if (rope_theta != s->rope_theta || causal != s->causal) return BSR_ERR_SCHEDULE_MISMATCH;
  if (s->kv_dtype != BSR_KV_DTYPE_E4M3) return BSR_ERR_SCHEDULE_MISMATCH;   // planned for bf16
  // the FP8 path covers the decode kernel's work: D = 128, pages of at least 16
  // keys, every request on the decode kernel (RoPE included)
  if (s->D != 128 || s->P < bsr::kStageTokens || s->n_pitems > 0) return BSR_ERR_UNSUPPORTED;
  if (s->n_items == 0) return BSR_OK;
  if (q == nullptr || out == nullptr || k_pages == nullptr || v_pages == nullptr)
    return BSR_ERR_INVALID_ARGUMENT;
  if (!aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(q, 16) || !aligned(out, 16) ||
      (lse && !aligned(lse, 4)))
    return BSR_ERR_INVALID_ARGUMENT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != s->device) return BSR_ERR_SCHEDULE_MISMATCH;
  const cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  const int64_t rows = int64_t(s->num_pages) * s->Hk * s->P;
  if (s->tm_k8_ptr != k_pages || s->tm_v8_ptr != v_pages) {
    const PoolGeom geom{rows, s->Hk, s->kv_layout == BSR_KV_NHD};
    if (rows <= 0 || !encode_pool_e4m3(&s->tm_k8, k_pages, geom) ||
        !encode_pool_e4m3(&s->tm_v8, v_pages, geom)) {
      s->tm_k8_ptr = s->tm_v8_ptr = nullptr;
      return BSR_ERR_CUDA;
    }
    s->tm_k8_ptr = k_pages;
    s->tm_v8_ptr = v_pages;
  }
  int t_slot = -1;
  if (s->t_max > 0) {
    t_slot = int(s->t_count % s->t_max);
    ++s->t_count;
    for (int st = 0; st < bsr_schedule::kStages; ++st) s->t_ran[t_slot * bsr_schedule::kStages + st] = 0;
  }
  auto t_mark = [&](int stage, int edge) {
    if (t_slot < 0) return;
    cudaEventRecord(s->t_ev[(t_slot * bsr_schedule::kStages + stage) * 2 + edge], stream);
    if (edge == 1) s->t_ran[t_slot * bsr_schedule::kStages + stage] = 1;
  };
  bsr::DecodeParams p{};
  p.items = s->dev<const bsr::DecodeItem>(s->off_items);
  p.warp_ptr = s->dev<const int32_t>(s->off_warp_ptr);
  p.counters = s->dev<int32_t>(s->off_counters);
  p.part_o = s->dev<float>(s->off_part_o);
  p.part_lse = s->dev<float>(s->off_part_lse);
  p.indices = s->dev<const int32_t>(s->off_indices);
  // the FP8 kernel reads the cos/sin table in pair order
  const bool rope = s->rope_rows > 0;
  p.rope = rope ? reinterpret_cast<const float2*>(s->d_rope + s->rope_bytes) : nullptr;
  p.page_pos = rope && s->has_page_pos ? s->dev<const int32_t>(s->off_page_pos) : nullptr;
  p.qshift = rope && s->has_page_pos ? s->dev<const int32_t>(s->off_qshift) : nullptr;
  p.q = static_cast<const uint16_t*>(q);
  p.k_pages = k_pages;
  p.v_pages = v_pages;
  p.out = out;
  p.lse = lse;
  p.error = s->dev<int32_t>(s->off_error);
  p.scale_log2 = float(double(sm_scale) * double(k_scale) * 1.4426950408889634);
  p.v_scale = v_scale;
  p.Hq = s->Hq;
  p.Hk = s->Hk;
  p.group = s->group;
  p.P = s->P;
  p.causal = s->causal;
  p.out_f32 = out_dtype == BSR_DTYPE_F32;
  p.num_warps = s->dec_warps;
  p.rope_max_pos = rope ? s->rope_rows - 1 : 0;
  p.window_left = s->window_left;
  p.nhd = s->kv_layout == BSR_KV_NHD;
  p.plan_uploaded = 1;   // the work list and page table came with the plan's copy
  p.wait_limit_ns = 1000000000ull;
  t_mark(0, 0);
  const cudaError_t e = bsr::launch_decode_kv8(rope, s->max_rows > 8, s->tm_k8, s->tm_v8, p, stream);
  t_mark(0, 1);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return BSR_ERR_CUDA;
  }
  return BSR_OK;
}
