/*
 * bsr_attn.h — C ABI of a GB300 (sm_103a) attention engine for batched
 * attention over a KV cache stored in Block-Sparse-Row (paged) form.
 *
 * What it computes follows "FlashInfer: Block-Sparse KV 캐시로 어텐션 병목을
 * 해소하다 (MLSys 2025 Best Paper)" (visionhong.com):
 *   - section "FlashInfer는 KV 캐시를 어떻게 통합하는가?: Block-Sparse 포맷":
 *     the KV cache is a block-sparse tensor whose blocks are runs of
 *     consecutive tokens and whose sparse metadata lists the active blocks;
 *     paged and contiguous caches are instances of it; inactive blocks are
 *     skipped; a shared prefix is stored once (at its own block size) and
 *     composed with per-request suffixes;
 *   - section "어텐션 연산에서 진짜 병목은 어디인가?": decode is bound by
 *     memory bandwidth (the whole KV history is read per generated token),
 *     prefill by compute;
 *   - section "JIT 컴파일은 어텐션을 어떻게 빠르게 만드는가?": RoPE is fused
 *     into the attention kernel instead of running as its own pass;
 *   - section "벤치마크: FlashInfer는 얼마나 빠른가?": a load-balanced scheduler
 *     cuts long sequences into smaller work units and interleaves them with
 *     short ones so that no workgroup idles on a skewed batch.
 * The pages give no signatures; these calls state that problem directly.
 *
 * Conventions for every call
 *   - All tensors are dense, row-major, and live in device memory unless a
 *     parameter says "host".  bf16 is IEEE bfloat16 (uint16 storage).
 *   - q, out      : [sum_qo, Hq, D]        (sum_qo = qo_indptr[batch])
 *   - k/v pages   : [num_pages, Hk, P, D]  (HND: one (page, kv head) block of
 *                   P*D elements is contiguous)
 *   - lse         : [sum_qo, Hq] fp32, natural-log log-sum-exp of the scaled
 *                   logits of the row; -inf (and out = 0) for a row that
 *                   attends to no key.
 *   - Page table (indptr, indices, last_page_len) for request b: its pages
 *     are indices[indptr[b] .. indptr[b+1]); every page is full except the
 *     last, which holds last_page_len[b] tokens (1..P); a request with no
 *     page has length 0.  Key j of b is slot j mod P of page j / P of that
 *     list; dropped (inactive) blocks are simply absent from the list.
 *   - Query i of request b (qo_indptr[b] <= row < qo_indptr[b+1]) sits at
 *     position L_b - qo_len_b + i; with causal masking it sees keys at
 *     positions <= its own.  qo head h reads kv head h / (Hq / Hk).
 *   - RoPE (rope_theta > 0): rotate-half form, frequency theta^(-2i/D) for
 *     pair (i, i + D/2); keys are stored un-rotated and rotated on load at
 *     their position in the request's page list; queries at their position.
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - Every call returns BSR_OK (0) or a negative BSR_ERR_* code.  No call
 *     aborts the process and no kernel traps.
 *   - Supported: head_dim 64 or 128; page_size a power of two in [1, 256];
 *     Hq a multiple of Hk with Hq / Hk <= 16.
 */
#ifndef BSR_ATTN_H_
#define BSR_ATTN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  BSR_OK = 0,
  BSR_ERR_INVALID_ARGUMENT = -1, /* null pointer, bad size, bad scale */
  BSR_ERR_UNSUPPORTED = -2,      /* head_dim / page_size / group size outside the set */
  BSR_ERR_PAGE_TABLE = -3,       /* malformed indptr / indices / last_page_len / qo_indptr */
  BSR_ERR_OUT_OF_MEMORY = -4,    /* device or pinned host allocation failed */
  BSR_ERR_CUDA = -5,             /* a CUDA runtime/driver call or launch failed */
  BSR_ERR_DEVICE_TIMEOUT = -6,   /* a kernel gave up on a bounded wait (see bsr_last_device_error) */
  BSR_ERR_SCHEDULE_MISMATCH = -7 /* run arguments disagree with what the schedule was planned for */
};

enum { BSR_DTYPE_BF16 = 0, BSR_DTYPE_F32 = 1 };
/* page pool layouts: head-major [pages, Hk, P, D] or token-major [pages, P, Hk, D] */
enum { BSR_KV_HND = 0, BSR_KV_NHD = 1 };
/* element type of a KV cache (bsr_attn_plan, bsr_attn_decode_noalloc_ex) */
enum { BSR_KV_DTYPE_BF16 = 0, BSR_KV_DTYPE_E4M3 = 1 };

typedef struct bsr_schedule* bsr_schedule_t;

/*
 * bsr_attn_plan — build the load-balanced work schedule for one batch.
 * (Scheduler: "벤치마크: FlashInfer는 얼마나 빠른가?"; block table:
 * "Block-Sparse 포맷".)
 *
 * indptr [batch+1], indices [indptr[batch]], last_page_len [batch] and
 * qo_indptr [batch+1] are HOST arrays; the caller keeps ownership and may
 * free them on return.  qo_indptr may be NULL, meaning one query per request.
 * The planner validates the table (indptr and qo_indptr start at 0 and never
 * decrease, page ids in [0, num_pages_in_pool), 1 <= last_page_len <=
 * page_size for non-empty requests, qo_len <= kv_len when causal or RoPE),
 * cuts every (request, kv head) key range into page-aligned chunks, spreads
 * the chunks over persistent warps at equal cost (long sequences cut and
 * interleaved with short ones), and uploads the page table, the work lists and
 * zeroed merge counters with ONE asynchronous host-to-device copy on `stream`;
 * with rope_theta > 0 an fp32 cos/sin table built in fp64 goes to its own
 * device buffer, uploaded only when theta or head_dim change or the longest
 * request outgrows it.
 * The planner's host working arrays are kept per calling thread and reused by
 * that thread's later plans (in a serving loop that re-plans every step the
 * large per-plan arrays are not allocated again), and its budget search starts from
 * the last plan's; the resulting schedule depends only on the arguments.
 *
 * window_left >= 0: 0 attends every key; W > 0 is the sliding-window variant
 * ("JIT 컴파일은 …": Sliding Window among the fused variants) -- a query at
 * position p sees keys p - W + 1 .. p (and causal still bounds it above).  The
 * planner starts each work unit at the oldest key any of its rows sees, so
 * pages wholly older than every window are never read.  The window is part of
 * the schedule (reported in bsr_schedule_info_t.window_left).
 *
 * page_pos (HOST int32 [indptr[batch]], may be NULL): the logical position of
 * each page-table entry's first token, for RoPE over a cache whose inactive
 * blocks were dropped ("Block-Sparse 포맷": discarded blocks are skipped; the
 * kept tokens keep their positions).  Key j of request b is rotated at
 * page_pos[indptr[b] + j / P] + j % P and its queries at the positions after
 * the last cached token, page_pos[last entry] + last_page_len - qo_len + i.
 * NULL: positions are the cached order j.  Causal and window masks use the
 * cached order.  Entries must be in [0, 2^29); with RoPE, page_size must be at
 * least 16 (else BSR_ERR_UNSUPPORTED).  Without RoPE the array is not used.
 *
 * kv_layout: BSR_KV_HND, pages [num_pages_in_pool, Hk, P, D] (one head's P
 * tokens contiguous), or BSR_KV_NHD, pages [num_pages_in_pool, P, Hk, D] (one
 * token's heads contiguous, the token-major layout some serving engines keep).
 * Every run of the schedule reads k_pages / v_pages in that layout.
 *
 * kv_dtype: BSR_KV_DTYPE_BF16 (the schedule runs with bsr_attn_run) or
 * BSR_KV_DTYPE_E4M3 (with bsr_attn_run_kv8).  The decode work is balanced over
 * the warps the cache's decode kernel keeps per SM -- 12 for an FP8 cache without
 * RoPE (its stages are half the bytes, so more warps hide the latency), 8
 * otherwise; a run of the other type returns BSR_ERR_SCHEDULE_MISMATCH.
 *
 * *schedule must be NULL (a new schedule is created) or a schedule returned
 * by an earlier plan or by bsr_schedule_create, which is then (re-)planned in
 * place: its device workspace is reused when large enough.  Re-planning is ordered on `stream` after work
 * already queued there; work on other streams that still reads the old
 * schedule is the caller's to finish first.
 * The schedule binds the current CUDA device.
 */
int bsr_attn_plan(const int32_t* indptr, const int32_t* indices, const int32_t* last_page_len,
                  int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t page_size, const int32_t* qo_indptr, int32_t num_pages_in_pool,
                  int32_t causal, int32_t window_left, const int32_t* page_pos,
                  int32_t kv_layout, int32_t kv_dtype, float rope_theta, void* stream,
                  bsr_schedule_t* schedule);

/*
 * bsr_schedule_create — an empty schedule, bound to the current CUDA device,
 * whose plans spread their work over at most sm_budget SMs (0: all of the
 * device's SMs); plan into it with bsr_attn_plan.  A budget lets two schedules
 * run at the same time on disjoint parts of the GPU, each launched on its own
 * stream -- the composable levels of a cascade ("Block-Sparse 포맷": a shared
 * prefix stored once, composed with per-request suffixes), whose prefix level
 * keeps the tensor cores busy while the suffix level streams its pages from
 * HBM.  sm_budget >= 0 (else BSR_ERR_INVALID_ARGUMENT).  Free with
 * bsr_schedule_destroy.
 */
int bsr_schedule_create(int32_t sm_budget, bsr_schedule_t* schedule);

/*
 * bsr_attn_run — execute a schedule: out = softmax(sm_scale * q k^T) v and
 * lse per (query row, qo head).  ("어텐션 연산에서 진짜 병목은 어디인가?",
 * "Block-Sparse 포맷", "JIT 컴파일은 …" for the fused RoPE.)
 *
 * q (bf16), k_pages, v_pages (bf16, num_pages_in_pool pages as planned) are
 * read; out (out_dtype: BSR_DTYPE_BF16 or BSR_DTYPE_F32) and lse (fp32, may
 * be NULL) are written.  All are caller-owned device buffers; no buffer may
 * alias another.  sm_scale must be finite and > 0.  rope_theta and causal
 * must equal the values given to plan, which was for BSR_KV_DTYPE_BF16 (else
 * BSR_ERR_SCHEDULE_MISMATCH).
 * q, k_pages, v_pages and out must be 16-byte aligned (else
 * BSR_ERR_INVALID_ARGUMENT).
 * The call allocates nothing, never synchronizes the host, and is
 * stream-ordered; it may be captured in a CUDA graph.  Two runs of one
 * schedule must not overlap in time (they share its merge workspace).
 */
int bsr_attn_run(bsr_schedule_t schedule, const void* q, const void* k_pages, const void* v_pages,
                 float sm_scale, float rope_theta, int32_t causal, void* out, int32_t out_dtype,
                 float* lse, void* stream);

/*
 * bsr_attn_run_kv8 — bsr_attn_run over an FP8 KV cache (the quantisation /
 * dequant variant of the attention operator, "JIT 컴파일은 …"): k_pages and
 * v_pages hold OCP FP8 E4M3 codes, one byte per element, in the same
 * [num_pages_in_pool, Hk, P, D] layout; the cached keys and values are
 * k_scale * code and v_scale * code (per-pool scales, finite and > 0; codes
 * S.1111.111 are NaN).  Dequantisation is fused into the page gather: the
 * codes are converted to fp16 in registers (exact) right before the MMAs.
 * With rope_theta > 0 (planned so) the keys are rotated in registers after
 * that conversion, RoPE and dequantisation fused into one kernel ("JIT 컴파일은
 * …" names both): the rotated q and k enter Q K^T as fp16 x 2^-4, as on the
 * bf16 path, at the positions the plan gives (page_pos included).
 * The schedule must be planned with kv_dtype BSR_KV_DTYPE_E4M3 (else
 * BSR_ERR_SCHEDULE_MISMATCH).  Everything else (q bf16, out, lse, alignment,
 * ownership, stream semantics) is as for bsr_attn_run.  Covered: head_dim 128, page_size >= 16, every
 * request on the decode kernel (info.num_prefill_items == 0); other schedules
 * return BSR_ERR_UNSUPPORTED.
 */
int bsr_attn_run_kv8(bsr_schedule_t schedule, const void* q, const void* k_pages,
                     const void* v_pages, float k_scale, float v_scale, float sm_scale,
                     float rope_theta, int32_t causal, void* out, int32_t out_dtype, float* lse,
                     void* stream);

/*
 * bsr_attn_run_host — one decode or prefill step with HOST buffers: q_host (bf16
 * [sum_qo, Hq, D]) is copied to the device, the schedule runs (bsr_attn_run, or
 * bsr_attn_run_kv8 with k_scale / v_scale for a schedule planned for
 * BSR_KV_DTYPE_E4M3; the scales are not used otherwise), and out (out_dtype) and lse
 * (fp32, may be NULL) are copied back into out_host / lse_host -- all ordered on
 * `stream`, so the host buffers hold the result once the stream has completed (the
 * call itself does not wait).  With pinned host memory the copies are asynchronous;
 * pageable memory works, but then the copies hold the host.  The device staging for
 * q, out and lse belongs to the schedule: allocated by the first call (or when a
 * larger plan needs more; the old one is freed, which waits for the device) and kept
 * until bsr_schedule_destroy -- the only allocation on a run path, so a caller that
 * must not allocate later makes one call while warming up.  The page pools are device
 * buffers, as for bsr_attn_run; the other rules and error codes are the same.
 */
int bsr_attn_run_host(bsr_schedule_t schedule, const void* q_host, const void* k_pages,
                      const void* v_pages, float k_scale, float v_scale, float sm_scale,
                      float rope_theta, int32_t causal, void* out_host, int32_t out_dtype,
                      float* lse_host, void* stream);

/*
 * bsr_merge_states — combine two attention states over disjoint key sets
 * (split chunks, or the shared-prefix and suffix levels of a cascade;
 * "Block-Sparse 포맷", composition of a stored-once prefix with suffixes):
 *   lse = M + ln(exp(lse_a - M) + exp(lse_b - M)),  M = max(lse_a, lse_b)
 *   o   = exp(lse_a - lse) o_a + exp(lse_b - lse) o_b
 * A row whose two states are both empty (lse = -inf) gets o = 0, lse = -inf.
 * o_a, o_b, o_out: [num_rows, num_heads, head_dim] of `dtype`; lse_*:
 * [num_rows, num_heads] fp32.  o_out may equal o_a and lse_out may equal
 * lse_a (in-place); no other aliasing.  Device buffers, caller-owned.
 */
int bsr_merge_states(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b,
                     int64_t num_rows, int32_t num_heads, int32_t head_dim, int32_t dtype,
                     void* o_out, float* lse_out, void* stream);

/*
 * bsr_append_kv — write new tokens' (un-rotated) k and v into their pages
 * (the append step of chunked prefill / decode).
 *
 * All arrays are DEVICE arrays.  The page table (indptr, indices,
 * last_page_len; batch requests) describes the cache AFTER the append:
 * request b appends n_b = append_indptr[b+1] - append_indptr[b] tokens, which
 * take positions L_b - n_b .. L_b - 1.  k_new, v_new: bf16
 * [num_new_tokens, Hk, D]; k_pages, v_pages: bf16 [num_pages_in_pool, Hk, P, D],
 * written in place (kv_layout: BSR_KV_HND or BSR_KV_NHD, as for plan); every
 * other slot keeps its bits.  The device-resident
 * table cannot be checked on the host: a token whose page id falls outside
 * [0, num_pages_in_pool) or whose request cannot hold it is skipped, and bit
 * 1 is OR-ed into *device_status (a device int32, may be NULL) for the caller
 * to read after synchronizing.
 */
int bsr_append_kv(const void* k_new, const void* v_new, const int32_t* append_indptr,
                  const int32_t* indptr, const int32_t* indices, const int32_t* last_page_len,
                  int32_t batch, int64_t num_new_tokens, int32_t num_kv_heads, int32_t head_dim,
                  int32_t page_size, int32_t num_pages_in_pool, int32_t kv_layout,
                  void* k_pages, void* v_pages, int32_t* device_status, void* stream);

/* Free a schedule's device workspace and host buffers after synchronizing
 * the device.  NULL is ignored. */
void bsr_schedule_destroy(bsr_schedule_t schedule);

/* What a plan produced (sizes are per schedule). */
typedef struct bsr_schedule_info {
  int32_t batch, num_qo_heads, num_kv_heads, head_dim, page_size, causal;
  float rope_theta;
  int64_t sum_qo;
  int64_t active_tokens;      /* sum of attended key counts over requests */
  int32_t num_decode_items;   /* work units of the split-KV decode kernel */
  int32_t num_prefill_items;  /* work units of the tensor-core prefill kernel */
  int32_t num_split_streams;  /* (request, kv head, row group) ranges cut into >1 chunk */
  int32_t num_partials;       /* partial states written before merging */
  int32_t decode_ctas, decode_warps_per_cta;  /* one decode CTA per SM; its warps follow kv_dtype */
  int32_t prefill_ctas;
  int32_t num_sms;
  int64_t workspace_bytes;    /* device workspace of the schedule */
  int64_t upload_bytes;       /* bytes of the one host-to-device copy a plan makes */
  double decode_imbalance;    /* max planned cost of a decode warp / mean decode cost per
                                 warp (run-time units counted in the mean only) */
  double prefill_imbalance;   /* max / mean planned cost over prefill CTAs */
  int32_t kernels_per_run;    /* kernels one bsr_attn_run launches (decode, prefill,
                                 split-range merge; 0 when there is no work) */
  int32_t window_left;        /* sliding window given to plan (0: none) */
  int32_t kv_layout;          /* BSR_KV_HND or BSR_KV_NHD */
  int32_t kv_dtype;           /* BSR_KV_DTYPE_BF16 or BSR_KV_DTYPE_E4M3 (as planned) */
} bsr_schedule_info_t;

int bsr_schedule_get_info(bsr_schedule_t schedule, bsr_schedule_info_t* info);

/*
 * Optional per-stage timing of bsr_attn_run (a measurement hook; the pages
 * have no counterpart).  Off by default.
 *
 * bsr_schedule_set_stage_timing: with max_calls > 0 every later run records
 * CUDA events on its stream around each kernel it launches -- stage 0 decode,
 * 1 prefill, 2 split-range merge of the prefill -- and the schedule keeps
 * the last max_calls runs; 0 turns timing off and frees the events.  Returns
 * BSR_OK or a negative BSR_ERR_* code.
 *
 * bsr_schedule_stage_times: waits for the events of kept run `call` (0 = the
 * oldest kept) and writes its three stage durations in milliseconds to ms[3]
 * (-1 for a stage that did not run).  Returns the number of runs kept, or a
 * negative BSR_ERR_* code (BSR_ERR_INVALID_ARGUMENT for a call not kept).
 */
int bsr_schedule_set_stage_timing(bsr_schedule_t schedule, int32_t max_calls);
int bsr_schedule_stage_times(bsr_schedule_t schedule, int32_t call, float* ms);

/*
 * bsr_attn_plan_host — the host half of bsr_attn_plan, for a given SM count,
 * touching no GPU: validates the table exactly like bsr_attn_plan (kv_dtype
 * included, which sets the decode warps per SM) and returns the number of work
 * units, decode and prefill (or a negative BSR_ERR_* code).  If `info` is non-NULL
 * it is filled as bsr_schedule_get_info would (without the workspace size); if
 * `units` is non-NULL (capacity max_units rows) each unit is written as
 * int32[8]: request, kv head, first packed row, packed rows, first key, end key,
 * partial slot (-1 = unsplit), then the decode warp that runs it, or -1 - CTA for
 * a unit of the tensor-core prefill kernel, or -- for a whole range the plan leaves to
 * run time (skewed bf16 batches without RoPE: warps that have finished their own lists
 * take these from a queue, longest first) -- the number of decode warps plus its place
 * in the queue.  Packed row R of
 * (request, kv head) is query R / (Hq/Hk), qo head kv_head * (Hq/Hk) +
 * R % (Hq/Hk).  All arrays are host arrays owned by the caller.  Use it to
 * inspect or test a schedule (coverage of every key, balance) without a device.
 */
int bsr_attn_plan_host(const int32_t* indptr, const int32_t* indices,
                       const int32_t* last_page_len, int32_t batch, int32_t num_qo_heads,
                       int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                       const int32_t* qo_indptr, int32_t num_pages_in_pool, int32_t causal,
                       int32_t window_left, const int32_t* page_pos, int32_t kv_layout,
                       int32_t kv_dtype, float rope_theta, int32_t num_sms,
                       bsr_schedule_info_t* info, int32_t* units, int64_t max_units);

/*
 * bsr_attn_decode_noalloc — decode attention that allocates nothing.
 * The paper has no counterpart; this is a service to callers that cannot call
 * cudaMalloc where they need attention (a runtime that carves all device
 * memory once at start-up with its own allocator, or a host that forbids
 * allocation inside its execute step).
 *
 * Computes what bsr_attn_plan + bsr_attn_run compute for one query per
 * request, non-causal, without RoPE: q [batch, Hq, D] bf16; k_pages/v_pages
 * [num_pages_in_pool, Hk, P, D] bf16; indptr [batch+1], indices, last_page_len
 * [batch] are DEVICE arrays; out [batch, Hq, D] (out_dtype) and lse
 * [batch, Hq] fp32 (may be NULL) are written.  All buffers are the caller's.
 * Each (request, kv head) key range is cut into equal chunks on the device.
 * The kernel's scratch lives in one static device array of about 17 MB that
 * every GPU loading this library holds until the process exits; it holds at
 * most 2048 (request, kv head, chunk) units, so batch * num_kv_heads above
 * 2048 is refused with BSR_ERR_UNSUPPORTED before anything runs.  The first
 * call on a device looks up the array's device address (make that call before
 * any stream capture).  All calls on a device share the array and every call
 * rewrites it: calls whose kernels overlap on the GPU race, so keep them on
 * one stream.  The device table is checked on the device, request by request:
 * a request whose entries are malformed (indptr[b] < 0, a negative page count,
 * last_page_len outside [1, page_size], a length beyond 2^31 - 1 keys) or any
 * page of which that its query reads lies outside [0, num_pages_in_pool) is
 * treated as empty as a whole -- its out rows are 0 and its lse -inf -- and bit
 * 1 is OR-ed into *device_status (device int32, may be NULL); the other
 * requests are unaffected.  indptr[b + 1] must not exceed the length of
 * `indices` (the library is not told that length).  Bit 0 means a bounded
 * wait gave up.
 */
int bsr_attn_decode_noalloc(const void* q, const void* k_pages, const void* v_pages,
                            const int32_t* indptr, const int32_t* indices,
                            const int32_t* last_page_len, int32_t batch, int32_t num_qo_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                            int32_t num_pages_in_pool, float sm_scale, void* out,
                            int32_t out_dtype, float* lse, int32_t* device_status, void* stream);

/* bsr_attn_decode_noalloc over an FP8 (E4M3) KV cache: k_pages / v_pages hold one-byte
 * codes in the same layout, the cached values k_scale * code and v_scale * code (as
 * bsr_attn_run_kv8).  head_dim 128 and page_size >= 16 only (else
 * BSR_ERR_UNSUPPORTED); k_scale and v_scale finite and > 0.  Allocation, scratch,
 * status and ordering as bsr_attn_decode_noalloc. */
int bsr_attn_decode_noalloc_kv8(const void* q, const void* k_pages, const void* v_pages,
                                const int32_t* indptr, const int32_t* indices,
                                const int32_t* last_page_len, int32_t batch,
                                int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t page_size, int32_t num_pages_in_pool, float sm_scale,
                                float k_scale, float v_scale, void* out, int32_t out_dtype,
                                float* lse, int32_t* device_status, void* stream);

/* The general no-allocation decode: kv_dtype BSR_KV_DTYPE_BF16 (k_scale / v_scale
 * ignored) or BSR_KV_DTYPE_E4M3 (as bsr_attn_decode_noalloc_kv8), and window_left >= 0
 * (0: every key; W > 0: the query at position L - 1 sees keys L - W .. L - 1, and each
 * (request, kv head) range starts at the page holding key L - W, so older pages are
 * never read). */
int bsr_attn_decode_noalloc_ex(const void* q, const void* k_pages, const void* v_pages,
                               const int32_t* indptr, const int32_t* indices,
                               const int32_t* last_page_len, int32_t batch,
                               int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t page_size, int32_t num_pages_in_pool, float sm_scale,
                               int32_t kv_dtype, float k_scale, float v_scale,
                               int32_t window_left, void* out, int32_t out_dtype, float* lse,
                               int32_t* device_status, void* stream);

/* Self-test of failure detection (no GPU fault involved): runs, on `stream`, the
 * bounded mbarrier wait the library's kernels use, on a barrier that nothing ever
 * arrives on; after `limit_ns` (1 ns .. 10 s) the wait gives up and bit 0 of the
 * int32 at `device_status` (device memory) is set, as a kernel whose wait ran out
 * sets its schedule's status word.  BSR_OK once launched. */
int bsr_selftest_bounded_wait(int32_t* device_status, int64_t limit_ns, void* stream);

/* Device-side status word of a schedule (0 = fine; bit 0: a kernel gave up on
 * a bounded wait; bit 1: a value was beyond the range of its fp16 operand, so
 * the scores or outputs involving it are not finite -- with RoPE a rotated q or
 * k of magnitude 2^20 or more (the rotated operands are fp16 x 2^-4), or, for
 * requests on the tensor-core prefill path, a V value beyond 65504 (P and V
 * enter P.V as fp16)).  Bits stay set until the schedule is planned again.
 * Synchronizes the schedule's device; returns the word, or a negative BSR_ERR_*
 * code. */
int bsr_last_device_error(bsr_schedule_t schedule);

/* Static, human-readable text for a status code. */
const char* bsr_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* BSR_ATTN_H_ */
