// Host-side state of one schedule (opaque to C callers as bsr_schedule_t).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <vector>

#include "bsr_internal.h"
#include "bsr_launchers.h"

struct bsr_schedule {
  int device = -1;
  int num_sms = 0;
  int32_t sm_budget = 0;       // plans spread their work over at most this many SMs (0: all)

  // problem the schedule was planned for
  int32_t batch = 0, Hq = 0, Hk = 0, D = 0, P = 0, group = 0, causal = 0;
  float rope_theta = 0.f;
  int32_t num_pages = 0;
  int64_t sum_qo = 0, active_tokens = 0;
  int32_t rope_rows = 0;       // rows of the cos/sin table (0 without RoPE)
  int32_t window_left = 0;     // sliding window (0: none)
  int32_t kv_layout = 0;       // BSR_KV_HND or BSR_KV_NHD
  int32_t kv_dtype = 0;        // BSR_KV_DTYPE_BF16 or BSR_KV_DTYPE_E4M3 (sets the decode warps)
  // per-page logical positions for RoPE (uploaded with the image when given)
  bool has_page_pos = false;
  size_t off_page_pos = 0, off_qshift = 0;
  int32_t max_rows = 0;        // largest packed-row count of one decode unit

  // decode plan
  int32_t n_items = 0, n_partials = 0, n_split = 0, dec_warps = 0, dec_ctas = 0;
  int32_t n_dyn = 0, dyn_begin = 0;   // run-time units (decode): count, first item
  size_t off_dyn_ctr = 0;             // their queue counters in the workspace
  int32_t dec_warps_per_cta = 0;   // warps one decode CTA runs (one CTA per SM)
  double dec_imbalance = 0.0;
  // prefill plan (tensor-core kernel)
  int32_t n_pitems = 0, n_ppartials = 0, n_psplit = 0, pre_ctas = 0;
  double pre_imbalance = 1.0;
  size_t rope_bytes = 0;     // one of the two device cos/sin tables (fragment, then frequency order)

  // one device allocation holding everything the kernels read or own
  uint8_t* d_ws = nullptr;
  size_t ws_cap = 0, ws_used = 0, upload_bytes = 0;
  size_t off_indices = 0, off_items = 0, off_warp_ptr = 0, off_counters = 0, off_error = 0,
         off_part_o = 0, off_part_lse = 0;
  size_t off_pitems = 0, off_cta_ptr = 0, off_pmerge = 0, off_ppart_o = 0, off_ppart_lse = 0;
  int32_t n_pmerge = 0;      // prefill units whose key range was split (merged by a second kernel)
  // prefill K/V tiles: boxes of min(P, 128) rows over the caller's pools
  CUtensorMap tm_pk;
  CUtensorMap tm_pv;
  const void* tm_pk_ptr = nullptr;
  const void* tm_pv_ptr = nullptr;
  // prefill query tiles over q
  CUtensorMap tm_q;
  const void* tm_q_ptr = nullptr;

  // device staging of bsr_attn_run_host (q in, out and lse back), allocated on its
  // first call and when a larger batch needs more, kept until destroy
  uint8_t* d_io = nullptr;
  size_t io_cap = 0;

  // pinned staging buffer for the single host-to-device upload
  uint8_t* h_stage = nullptr;
  size_t stage_cap = 0;
  cudaEvent_t upload_done = nullptr;
  bool upload_pending = false;

  // cos/sin tables: built on the host and uploaded to their own device buffer only
  // when theta or head_dim change or the longest request outgrows them (rows grow
  // in powers of two), so re-planning a decode step uploads no table
  float rope_cache_theta = 0.f;
  int32_t rope_cache_D = 0, rope_cache_rows = 0;
  uint8_t* h_rope = nullptr;   // [fragment order | frequency order] (malloc)
  uint8_t* d_rope = nullptr;   // device copy of h_rope
  size_t d_rope_cap = 0;
  bool d_rope_valid = false;

  // tensor maps of the last k/v pools seen by run (re-encoded when they change)
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  const void* tm_k_ptr = nullptr;
  const void* tm_v_ptr = nullptr;
  // the same for FP8 (E4M3) pools
  CUtensorMap tm_k8;
  CUtensorMap tm_v8;
  const void* tm_k8_ptr = nullptr;
  const void* tm_v8_ptr = nullptr;

  // optional per-stage timing of runs: events [run slot][stage][begin, end]
  static constexpr int kStages = 3;   // decode, prefill, prefill merge
  std::vector<cudaEvent_t> t_ev;
  std::vector<uint8_t> t_ran;         // [run slot][stage]
  int32_t t_max = 0;
  int64_t t_count = 0;

  template <typename T>
  T* dev(size_t off) const { return reinterpret_cast<T*>(d_ws + off); }
};
