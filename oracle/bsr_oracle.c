/*
 * Oracle for batched attention over a Block-Sparse-Row (paged) KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain fp64 CPU statement
 * of what the GPU path computes.  Only the tests, the package smoke check and
 * the bench's CPU-baseline leg may load it; the product library never does.
 * It shares no code, header, table or constant with the CUDA sources.
 *
 * Source: "FlashInfer: Block-Sparse KV 캐시로 어텐션 병목을 해소하다 (MLSys 2025
 * Best Paper)" (visionhong.com), sections
 *   - "FlashInfer는 KV 캐시를 어떻게 통합하는가?: Block-Sparse 포맷": the KV cache
 *     is a block-sparse tensor; a block is a run of consecutive tokens; sparse
 *     metadata names the active blocks; paged and contiguous caches are both
 *     instances; inactive blocks are skipped; a shared prefix is stored once
 *     and composed with per-request suffixes.
 *   - "어텐션 연산에서 진짜 병목은 어디인가?": decode reads the whole KV history
 *     for each generated token; prefill handles many query tokens at once.
 *   - "JIT 컴파일은 어텐션을 어떻게 빠르게 만드는가?": RoPE is one of the
 *     operations fused into attention.
 * The pages give no formulas for these, so every function below is the plain
 * definition, and each reading of an open point is named where it is used.
 *
 * Parity pins (tests/test_oracle.py): brute-force dense attention through
 * torch CPU fp64 library routines, closed forms, page-size and page-permutation
 * invariance, block dropping == masking, split+merge == unsplit,
 * cascade == flat, RoPE against the complex-exponential form.
 *
 * Storage conventions (the inputs the GPU path also reads):
 *   q        bf16 bits [sum_qo, Hq, D]
 *   k_pages  bf16 bits [num_pages, Hk, P, D]   (one (page, head) is P*D contiguous)
 *   v_pages  same as k_pages
 *   FP8 KV cache: k_pages / v_pages as E4M3 codes (one byte each, same
 *   layout) with one float scale per pool (oracle_attention_kv8)
 *   indptr [B+1], indices [indptr[B]], last_page_len [B], qo_indptr [B+1]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32; widening to double is exact. */
static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point E4M3 (the FP8 KV-cache format): 1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits.  Exponent field 0 holds the
 * subnormals m/8 * 2^-6; there are no infinities, S.1111.111 is NaN and the
 * largest finite magnitude is 1.75 * 2^8 = 448.  Every code is exact in fp64. */
static double e4m3_to_double(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  const double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

double oracle_e4m3(uint8_t code) { return e4m3_to_double(code); }

/* One K or V element of the page pools: bf16 bits (kv_fp8 = 0) or an E4M3 code
 * times the pool's per-tensor scale (kv_fp8 = 1; the FP8 KV cache stores
 * value / scale, "quantisation/dequant" fused into attention). */
static double kv_elem(const void* pool, int32_t kv_fp8, double scale, int64_t idx) {
  if (kv_fp8) return scale * e4m3_to_double(((const uint8_t*)pool)[idx]);
  return bf16_bits_to_double(((const uint16_t*)pool)[idx]);
}

/* Element offset of (page, kv head h, slot t) in a page pool: HND pages hold
 * [Hk][P][D] (one head's P tokens contiguous), NHD pages [P][Hk][D] (one token's
 * heads contiguous, the token-major layout some serving engines keep). */
static int64_t kv_off(int64_t page, int32_t h, int64_t t, int32_t Hk, int32_t P, int32_t D,
                      int32_t nhd) {
  if (nhd) return ((page * P + t) * Hk + h) * (int64_t)D;
  return ((page * Hk + h) * P + t) * (int64_t)D;
}

/* Attended KV length of request b: all of its pages are full except the last,
 * which holds last_page_len tokens (reading: 1 <= last_page_len <= P whenever
 * the request has a page; a request with no page has length 0). Returns -1 on
 * a malformed table. */
static int64_t kv_len_of(const int32_t* indptr, const int32_t* last_page_len,
                         int32_t b, int32_t page_size) {
  int64_t n = (int64_t)indptr[b + 1] - indptr[b];
  if (n < 0) return -1;
  if (n == 0) return 0;
  if (last_page_len[b] < 1 || last_page_len[b] > page_size) return -1;
  return (n - 1) * page_size + last_page_len[b];
}

int oracle_kv_len(const int32_t* indptr, const int32_t* last_page_len,
                  int32_t batch, int32_t page_size, int64_t* kv_len_out) {
  for (int32_t b = 0; b < batch; ++b) {
    int64_t L = kv_len_of(indptr, last_page_len, b, page_size);
    if (L < 0) return -1;
    kv_len_out[b] = L;
  }
  return 0;
}

/* Rotate-half RoPE at position pos (reading: non-interleaved halves, omega_i =
 * theta^(-2i/D), no frequency scaling).  x has D entries; rotated in place. */
static void rope_rotate(double* x, int32_t D, double pos, double theta) {
  int32_t half = D / 2;
  for (int32_t i = 0; i < half; ++i) {
    double omega = pow(theta, -2.0 * (double)i / (double)D);
    double c = cos(pos * omega), s = sin(pos * omega);
    double a = x[i], b = x[i + half];
    x[i] = a * c - b * s;
    x[i + half] = b * c + a * s;
  }
}

void oracle_rope(const double* x_in, double* x_out, int32_t D, double pos, double theta) {
  memcpy(x_out, x_in, sizeof(double) * (size_t)D);
  rope_rotate(x_out, D, pos, theta);
}

/* Find the request owning query row t: qo_indptr[b] <= t < qo_indptr[b+1]. */
static int32_t owner_of(const int32_t* qo_indptr, int32_t batch, int64_t t) {
  int32_t lo = 0, hi = batch - 1;
  while (lo < hi) {
    int32_t mid = (lo + hi + 1) / 2;
    if (qo_indptr[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

/*
 * Attention for selected (query row, qo head) pairs, or for all of them when
 * sel_rows == NULL.  For request b with L keys and qo_len queries, query i
 * sits at position L - qo_len + i (bottom-right alignment; for decode this is
 * L - 1).  Key j of b is token (j mod P) of page indices[indptr[b] + j / P].
 * qo head h reads kv head h / (Hq / Hk).  With causal != 0 key j is kept only
 * when j <= the query position.  Scores s_j = sm_scale * <q, k_j> (after RoPE
 * when rope_theta > 0); lse = ln sum_j exp(s_j); out = sum_j exp(s_j - lse) v_j.
 * No kept key: out = 0, lse = -inf.
 *
 * Output: out [rows, D] and lse [rows] in fp64, where rows are either
 * (sum_qo * Hq) in [t][h] order or num_sel in selection order.
 * Returns 0, or -1 for a malformed input (bad page id, last_page_len, heads).
 */
static int attention_impl(const uint16_t* q, const void* k_pages, const void* v_pages,
                          int32_t kv_fp8, double k_scale, double v_scale,
                          const int32_t* indptr, const int32_t* indices,
                          const int32_t* last_page_len, const int32_t* qo_indptr,
                          int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t page_size, int64_t num_pages,
                          double sm_scale, double rope_theta, int32_t causal,
                          int32_t window_left, const int32_t* page_pos, int32_t nhd,
                          const int64_t* sel_rows, const int32_t* sel_heads, int64_t num_sel,
                          double* out, double* lse, int32_t num_threads) {
  const int32_t D = head_dim, P = page_size, Hq = num_qo_heads, Hk = num_kv_heads;
  if (nhd != 0 && nhd != 1) return -1;
  if (window_left < 0) return -1;
  if (batch < 0 || Hq <= 0 || Hk <= 0 || Hq % Hk != 0 || D <= 0 || D % 2 != 0 || P <= 0)
    return -1;
  const int32_t group = Hq / Hk;
  /* validate the whole table once */
  for (int32_t b = 0; b < batch; ++b) {
    if (kv_len_of(indptr, last_page_len, b, P) < 0) return -1;
    if (qo_indptr[b + 1] < qo_indptr[b]) return -1;
    for (int32_t e = indptr[b]; e < indptr[b + 1]; ++e)
      if (indices[e] < 0 || (int64_t)indices[e] >= num_pages) return -1;
  }
  const int64_t total_rows = (int64_t)qo_indptr[batch];
  const int64_t n_work = sel_rows ? num_sel : total_rows * Hq;
  int bad = 0;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel
#endif
  {
    double* scores = NULL;
    int64_t scores_cap = 0;
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    double* kv = (double*)malloc(sizeof(double) * (size_t)D);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t w = 0; w < n_work; ++w) {
      int64_t t;
      int32_t h;
      if (sel_rows) { t = sel_rows[w]; h = sel_heads[w]; }
      else { t = w / Hq; h = (int32_t)(w % Hq); }
      double* o = out + w * D;
      if (t < 0 || t >= total_rows || h < 0 || h >= Hq) { bad = 1; continue; }
      const int32_t b = owner_of(qo_indptr, batch, t);
      const int64_t L = kv_len_of(indptr, last_page_len, b, P);
      const int64_t qo_len = (int64_t)qo_indptr[b + 1] - qo_indptr[b];
      const int64_t qpos = L - qo_len + (t - qo_indptr[b]);
      const int32_t kvh = h / group;
      /* RoPE positions: the key index j, or with page_pos (per-page logical
       * position of its first token, for caches whose dropped blocks leave gaps)
       * page_pos[page entry] + j mod P; the queries follow the last cached token,
       * at page_pos[last] + last_page_len - qo_len + i.  Causal and window masks
       * use the cached order (the two agree while page positions increase). */
      const int64_t qlog = (page_pos && L > 0)
                               ? (int64_t)page_pos[indptr[b + 1] - 1] + last_page_len[b] - qo_len +
                                     (t - qo_indptr[b])
                               : qpos;
      for (int32_t d = 0; d < D; ++d)
        qv[d] = bf16_bits_to_double(q[(t * Hq + h) * (int64_t)D + d]);
      if (rope_theta > 0.0) rope_rotate(qv, D, (double)qlog, rope_theta);
      if (L > scores_cap) {
        free(scores);
        scores_cap = L;
        scores = (double*)malloc(sizeof(double) * (size_t)scores_cap);
      }
      int64_t kept = 0;
      double m = -INFINITY;
      for (int64_t j = 0; j < L; ++j) {
        if (causal && j > qpos) { scores[j] = -INFINITY; continue; }
        /* sliding window: only the window_left most recent positions up to the
         * query's own (reading of the JIT section's "Sliding Window" variant) */
        if (window_left > 0 && j < qpos - window_left + 1) { scores[j] = -INFINITY; continue; }
        const int64_t page = indices[indptr[b] + j / P];
        const int64_t off = kv_off(page, kvh, j % P, Hk, P, D, nhd);
        for (int32_t d = 0; d < D; ++d) kv[d] = kv_elem(k_pages, kv_fp8, k_scale, off + d);
        if (rope_theta > 0.0) {
          const int64_t kpos = page_pos ? (int64_t)page_pos[indptr[b] + j / P] + j % P : j;
          rope_rotate(kv, D, (double)kpos, rope_theta);
        }
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += qv[d] * kv[d];
        scores[j] = sm_scale * dot;
        if (scores[j] > m) m = scores[j];
        ++kept;
      }
      for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
      if (kept == 0) { lse[w] = -INFINITY; continue; }
      double sum = 0.0;
      for (int64_t j = 0; j < L; ++j)
        if (scores[j] != -INFINITY) sum += exp(scores[j] - m);
      const double l = m + log(sum);
      lse[w] = l;
      for (int64_t j = 0; j < L; ++j) {
        if (scores[j] == -INFINITY) continue;
        const double p = exp(scores[j] - l);
        const int64_t page = indices[indptr[b] + j / P];
        const int64_t off = kv_off(page, kvh, j % P, Hk, P, D, nhd);
        for (int32_t d = 0; d < D; ++d) o[d] += p * kv_elem(v_pages, kv_fp8, v_scale, off + d);
      }
    }
    free(scores);
    free(qv);
    free(kv);
  }
  return bad ? -1 : 0;
}

int oracle_attention(const uint16_t* q, const uint16_t* k_pages, const uint16_t* v_pages,
                     const int32_t* indptr, const int32_t* indices,
                     const int32_t* last_page_len, const int32_t* qo_indptr,
                     int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
                     int32_t head_dim, int32_t page_size, int64_t num_pages,
                     double sm_scale, double rope_theta, int32_t causal, int32_t window_left,
                     const int32_t* page_pos, int32_t kv_layout, const int64_t* sel_rows, const int32_t* sel_heads, int64_t num_sel,
                     double* out, double* lse, int32_t num_threads) {
  return attention_impl(q, k_pages, v_pages, 0, 1.0, 1.0, indptr, indices, last_page_len,
                        qo_indptr, batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                        num_pages, sm_scale, rope_theta, causal, window_left, page_pos,
                        kv_layout, sel_rows, sel_heads, num_sel, out, lse, num_threads);
}

/* The same attention over an FP8 (E4M3) KV cache: K = k_scale * code,
 * V = v_scale * code, everything else as above. */
int oracle_attention_kv8(const uint16_t* q, const uint8_t* k_pages, const uint8_t* v_pages,
                         double k_scale, double v_scale,
                         const int32_t* indptr, const int32_t* indices,
                         const int32_t* last_page_len, const int32_t* qo_indptr,
                         int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t page_size, int64_t num_pages,
                         double sm_scale, double rope_theta, int32_t causal,
                         int32_t window_left, const int32_t* page_pos, int32_t kv_layout,
                         const int64_t* sel_rows, const int32_t* sel_heads, int64_t num_sel,
                         double* out, double* lse, int32_t num_threads) {
  return attention_impl(q, k_pages, v_pages, 1, k_scale, v_scale, indptr, indices,
                        last_page_len, qo_indptr, batch, num_qo_heads, num_kv_heads, head_dim,
                        page_size, num_pages, sm_scale, rope_theta, causal, window_left,
                        page_pos, kv_layout, sel_rows, sel_heads, num_sel, out, lse,
                        num_threads);
}

/*
 * Merge two attention states over disjoint key sets (what a split chunk or a
 * prefix/suffix cascade level produces).  Each state is (o, lse) with o the
 * softmax-weighted mean over its keys.  With M = max(lse_a, lse_b):
 *   lse = M + ln(exp(lse_a - M) + exp(lse_b - M))
 *   o   = exp(lse_a - lse) o_a + exp(lse_b - lse) o_b
 * Both states empty (lse = -inf): o = 0, lse = -inf.
 * o_* are [n, D], lse_* are [n].
 */
void oracle_merge_states(const double* o_a, const double* lse_a, const double* o_b,
                         const double* lse_b, int64_t n, int32_t D, double* o_out,
                         double* lse_out) {
  for (int64_t r = 0; r < n; ++r) {
    const double a = lse_a[r], b = lse_b[r];
    const double M = a > b ? a : b;
    if (M == -INFINITY) {
      lse_out[r] = -INFINITY;
      for (int32_t d = 0; d < D; ++d) o_out[r * D + d] = 0.0;
      continue;
    }
    const double l = M + log(exp(a - M) + exp(b - M));
    const double wa = exp(a - l), wb = exp(b - l);
    lse_out[r] = l;
    for (int32_t d = 0; d < D; ++d) o_out[r * D + d] = wa * o_a[r * D + d] + wb * o_b[r * D + d];
  }
}

/*
 * Append new tokens into their pages.  The page table describes the cache
 * AFTER the append: request b appends n_b = append_indptr[b+1]-append_indptr[b]
 * tokens, which take KV positions L_b - n_b ... L_b - 1.  Token i of b is
 * written to slot (pos mod P) of page indices[indptr[b] + pos / P], for every
 * kv head.  k_new/v_new are bf16 bits [sum_n, Hk, D]; pages are modified in
 * place.  Returns 0, or -1 for a malformed input.
 */
int oracle_append_kv(const uint16_t* k_new, const uint16_t* v_new,
                     const int32_t* append_indptr, const int32_t* indptr,
                     const int32_t* indices, const int32_t* last_page_len, int32_t batch,
                     int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                     int64_t num_pages, int32_t kv_layout, uint16_t* k_pages,
                     uint16_t* v_pages) {
  const int32_t D = head_dim, P = page_size, Hk = num_kv_heads, nhd = kv_layout;
  if (nhd != 0 && nhd != 1) return -1;
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t L = kv_len_of(indptr, last_page_len, b, P);
    const int64_t n_new = (int64_t)append_indptr[b + 1] - append_indptr[b];
    if (L < 0 || n_new < 0 || n_new > L) return -1;
    for (int64_t i = 0; i < n_new; ++i) {
      const int64_t pos = L - n_new + i;
      const int64_t page = indices[indptr[b] + pos / P];
      if (page < 0 || page >= num_pages) return -1;
      const int64_t src_tok = append_indptr[b] + i;
      for (int32_t h = 0; h < Hk; ++h) {
        const int64_t dst = kv_off(page, h, pos % P, Hk, P, D, nhd);
        const int64_t src = (src_tok * Hk + h) * (int64_t)D;
        memcpy(k_pages + dst, k_new + src, sizeof(uint16_t) * (size_t)D);
        memcpy(v_pages + dst, v_new + src, sizeof(uint16_t) * (size_t)D);
      }
    }
  }
  return 0;
}
