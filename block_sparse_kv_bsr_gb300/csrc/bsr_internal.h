// Internal data layout shared by the host planner and the CUDA kernels.
// The planner (bsr_plan.cpp) writes these records into one device workspace
// with a single host-to-device copy; the kernels only read them (plus the
// merge counters and partial states, which they own at run time).
#pragma once

#include <cstddef>
#include <cstdint>

#include "bsr_attn.h"

namespace bsr {

// Keys per pipeline stage of the decode kernel: one m16n8k16 K-step of the
// P.V product and two n-tiles of the Q.K^T product.
constexpr int kStageTokens = 16;
// Packed (query, head) rows per decode work unit: the M of one mma tile.
constexpr int kMaxDecodeRows = 16;
// Warps per decode CTA (each warp is an independent workgroup) and pipeline
// stages per warp; one CTA per SM, so warps x stages x stage bytes must fit
// the 227 KB of shared memory.  Overridable at build time for tuning sweeps.
#ifndef BSR_DECODE_WARPS
#define BSR_DECODE_WARPS 8
#endif
#ifndef BSR_DECODE_STAGES_D128
#define BSR_DECODE_STAGES_D128 3
#endif
#ifndef BSR_DECODE_STAGES_D64
#define BSR_DECODE_STAGES_D64 6
#endif
constexpr int kDecodeWarps = BSR_DECODE_WARPS;

// One decode work unit: rows [row0, row0 + nrows) of the packed rows of
// (request req, kv head kvh) against keys [tok0, tok1).  Packed row R is
// query R / group of the request, qo head kvh * group + R % group.  Every
// field the kernel needs is stored here so that no pointer is chased.
struct alignas(16) DecodeItem {
  int32_t req;
  int32_t kvh;
  int32_t row0;
  int32_t nrows;
  int32_t tok0;        // first key; a multiple of max(page_size, kStageTokens)
  int32_t tok1;        // one past the last key
  int32_t slot;        // -1: the unit covers all keys and writes out/lse; else partial slot
  int32_t first_slot;  // first partial slot (and merge counter) of a split range
  int32_t page_base;   // indptr[req]
  int32_t q_row0;      // qo_indptr[req]
  int32_t qpos0;       // position of the request's first query: kv_len - qo_len
  int32_t nchunks;     // units the range was cut into (1 when unsplit)
};

struct DecodeParams {
  const DecodeItem* items;
  const int32_t* warp_ptr;        // [num_warps + 1] item ranges per warp
  int32_t* counters;              // [num_partials] arrivals per split range (at first_slot)
  float* part_o;                  // [num_partials, kMaxDecodeRows, D] normalized partial outputs
  float* part_lse;                // [num_partials, kMaxDecodeRows] partial LSE (log2 domain)
  const int32_t* indices;         // [nnz] page ids
  const float2* rope;             // RoPE cos/sin table, or null: the bf16 kernel's fragment order
                                  // [rows, 4, D / 8] (cos, sin); the FP8 kernel's pair order
                                  // [rows, D / 4] float4 (cos f, cos f+1, sin f, sin f+1)
  const int32_t* page_pos;        // RoPE: logical position of each page entry's first key, or null
  const int32_t* qshift;          // RoPE with page_pos: logical minus cached end per request
  const uint16_t* q;              // bf16 [sum_qo, Hq, D]
  const void* k_pages;            // bf16 [num_pages, Hk, P, D] (read directly when P < 16)
  const void* v_pages;
  void* out;                      // bf16 or fp32 [sum_qo, Hq, D]
  float* lse;                     // fp32 [sum_qo, Hq] or null
  int32_t* error;                 // device status word
  float scale_log2;               // sm_scale * log2(e) (times k_scale for an FP8 cache)
  float v_scale;                  // FP8 cache: value of one V code unit (1 otherwise)
  int32_t Hq, Hk, group, P;
  int32_t causal, out_f32, num_warps;
  int32_t rope_max_pos;           // last row of the cos/sin table
  int32_t window_left;            // sliding window: keys >= position - window_left + 1 (0: none)
  int32_t nhd;                    // page pools token-major [pages, P, Hk, D] (else [pages, Hk, P, D])
  int32_t plan_uploaded;          // 1: items, warp_ptr, indices, page_pos and rope were written
                                  // by a host copy before the launch, so the kernel may read
                                  // them before the previous grid on the stream completes
  // Units taken at run time: items [dyn_begin, dyn_begin + n_dyn) (whole short ranges,
  // longest first) go to whichever warp has finished its own list, one at a time, so
  // that warps which ran slow take fewer.  dyn_ctr[0] is the next one to take,
  // dyn_ctr[1] the warps that found the queue empty; both are 0 between launches (the
  // plan uploads zeros, the last warp of a launch resets them).  n_dyn = 0: none.
  int32_t n_dyn, dyn_begin;
  int32_t* dyn_ctr;
  uint64_t wait_limit_ns;         // bound on every barrier wait
};

// Work units of the tensor-core prefill kernel use the same record with up to
// kPrefillRows packed rows (two 128-row query tiles that share every key
// tile); partial states are [slot][kPrefillRows][D].  Key ranges are cut at
// multiples of kPrefillKeyTile keys.  The head group divides 128, so a query
// tile is whole queries and is one TMA box of q.
constexpr int kPrefillRows = 256;
constexpr int kPrefillKeyTile = 128;
// Rotated (RoPE) q and k enter the products as fp16 scaled by 2^-4 (an exact
// power of two), so rotated values up to 2^20 in magnitude fit.
constexpr float kRopeOperandScale = 0.0625f;
constexpr float kRopeOperandMax = 65504.f;
// Device status bits (the status word of a schedule).  Bit 1: an fp16 operand of
// the products was out of range -- a rotated q or k of magnitude 2^20 or more, or
// on the tensor-core prefill path a V value beyond 65504 -- so the scores or
// outputs involving it are not finite.
constexpr int32_t kStatusWaitTimeout = 1;
constexpr int32_t kStatusOperandRange = 2;

struct PrefillParams {
  const DecodeItem* items;
  const int32_t* cta_ptr;         // [num_ctas + 1] unit ranges per CTA
  float* part_o;                  // [num_partials, kPrefillRows, D] fp32
  float* part_lse;                // [num_partials, kPrefillRows] (log2 domain)
  const int32_t* indices;
  const float4* rope;             // RoPE: [rope rows, D / 4] (cos f, cos f+1, sin f, sin f+1), f even; or null
  const int32_t* page_pos;        // RoPE: logical position of each page entry's first key, or null
  const int32_t* qshift;          // RoPE with page_pos: logical minus cached end per request
  int32_t rope_max_pos;           // last row of the cos/sin table
  void* out;
  float* lse;
  int32_t* error;
  float scale_log2;
  int32_t Hq, Hk, group, P;
  int32_t causal, out_f32, out_v8, num_ctas;
  int32_t window_left;            // sliding window (0: none)
  int32_t nhd;                    // page pools token-major (else head-major)
  int32_t box_rows;               // rows per K/V box of the prefill tensor maps: min(P, 128)
  int32_t head_dim;               // 64 or 128 (a D = 64 head runs the 128-wide tile program
                                  // with its upper 64 dimensions zero)
  uint64_t wait_limit_ns;
};

// Second pass for split prefill units: one warp per packed row combines the
// unit's partial states (in key order) into out / lse.
struct PrefillMergeParams {
  const DecodeItem* units;        // [n_units] the first piece of each split unit
  const float* part_o;
  const float* part_lse;
  void* out;
  float* lse;
  int32_t n_units, Hq, group, out_f32;
  int32_t head_dim;               // 64 or 128
};

}  // namespace bsr
