// Split-KV decode attention over an FP8 (E4M3) paged KV cache, sm_103a.
//
// The "quantisation / dequant" variant of the attention operator ("FlashInfer:
// Block-Sparse KV 캐시로 어텐션 병목을 해소하다", section "JIT 컴파일은 …"):
// the cache holds K and V as one-byte E4M3 codes with one float scale per pool
// (K = k_scale * code, V = v_scale * code), which halves the bytes a decode
// step streams from HBM.  The dequantisation is fused into the page gather:
// TMA copies the codes (one 2 KB box per 16-key stage for K and for V: a
// 128-byte row is a whole D = 128 head), and each warp converts them to fp16
// in registers right before its MMAs.  Every E4M3 code is exact in fp16, so
// QK^T and PV see the cached values unchanged; k_scale folds into the logit
// scale and v_scale into the output normalisation.
//
// Structure and scheduling are the bf16 decode kernel's (persistent warps,
// private TMA rings, planned work units, in-kernel merge of split ranges).
// What differs is how fragments are formed from one-byte elements:
//  * S = Q K^T: ldmatrix on the code tile gives a thread 4 consecutive codes
//    (dims 4t..4t+3 of a 16-dim block) of one key.  The head dimension is
//    taken in that order for q as well (q . k is a sum over dims, so the same
//    permutation on both sides leaves it unchanged): a0 = q dims 4t, 4t+1,
//    a2 = dims 4t+2, 4t+3.
//  * O += P V: ldmatrix.trans on byte pairs gives a thread dims (2g, 2g+1) of
//    keys 2t and 2t+1; a byte permute splits them into the even-dim and the
//    odd-dim n-tile of the block, so each thread's accumulators hold dims
//    4t..4t+3 of every 16-dim block (stored contiguously).
//  * P enters PV as fp16 (11 significant bits).
//  * A step consumes two ring stages (32 keys) while two remain: their Q K^T
//    products interleave and the max, its shuffles and the O rescale run once
//    per 32 keys (the conversions make a stage about three times the bf16
//    kernel's instructions per byte, so per-step latency matters here).
// Every barrier wait is bounded; on timeout the warp sets bit 0 of the status
// word, drains its own copies (bounded) and exits.
#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <type_traits>

#include "bsr_decode.cuh"
#include "bsr_launchers.h"

#ifndef BSR_DECODE_STAGES_KV8
#define BSR_DECODE_STAGES_KV8 4
#endif

namespace bsr {
namespace {

constexpr int kD8 = 128;                                      // head dim (bytes per row)
constexpr int kTile8 = kStageTokens * kD8;                    // one K (or V) stage: 2 KB
constexpr int kStage8 = 2 * kTile8;
constexpr int kStages8 = BSR_DECODE_STAGES_KV8;
// RoPE: one table row per stage (the angles of the stage's first key, pair order:
// D / 4 float4 (cos f, cos f+1, sin f, sin f+1)) beside the ring, and the CTA's 16
// offset rows t < 16 (times the operand scale)
constexpr int kRowBytes8 = kD8 / 4 * 16;
// dynamic shared memory of a CTA: the warps' rings and barriers (+ RoPE rows)
constexpr size_t smem8(bool rope) {
  const size_t w = size_t(decode_kv8_warps(rope));
  return w * kStages8 * kStage8 + w * kStages8 * 8 + 1024 +
         (rope ? w * kStages8 * kRowBytes8 + size_t(kStageTokens) * kRowBytes8 : 0);
}
static_assert(smem8(false) <= 232448 && smem8(true) <= 232448,
              "FP8 decode stages exceed the shared memory of one SM");

// Byte offset of (token t, 16-byte chunk c of 8) in a [16 rows][128 B] tile with
// the TMA 128-byte swizzle.
__device__ __forceinline__ uint32_t tile8_off(int t, int c) {
  return uint32_t((t << 7) + ((c ^ (t & 7)) << 4));
}

// Two E4M3 codes (the low 16 bits, low byte first) as an fp16 pair (low half
// first): the PTX conversion instruction, exact (every E4M3 value is an fp16).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t d;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(d) : "r"(two));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  return ptx::pack_f16(ptx::bf16_lo(v), ptx::bf16_hi(v));
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t v) {
  float2 r;
  asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}" : "=f"(r.x), "=f"(r.y) : "r"(v));
  return r;
}

// RoPE on a pair of frequencies (f, f + 1): x are dims f, f + 1, y their rotate-half
// partners; (c, s) the angles' cosines and sines.  x <- x c - y s, y <- y c + x s.
__device__ __forceinline__ void rotate2(float2& x, float2& y, float2 c, float2 s) {
  const float2 u = ptx::fsub2(ptx::fmul2(x, c), ptx::fmul2(y, s));
  y = ptx::ffma2(y, c, ptx::fmul2(x, s));
  x = u;
}

template <bool R16, bool WIN, bool ROPE>
__global__ void __launch_bounds__(decode_kv8_warps(ROPE) * 32, 1)
    bsr_decode_kv8_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  constexpr int D = kD8;
  constexpr int NR = R16 ? 4 : 2;       // accumulator registers per n-tile that carry rows
  constexpr int KB = D / 16;            // 16-dim blocks
  constexpr int NT = D / 8;             // n-tiles of the output
  extern __shared__ uint8_t smem_raw[];
  // launched as a programmatic dependent (see bsr_launch.cuh); a plan's work list, page
  // table and tables are read before the wait, as in bsr_decode_kernel
  pdl_trigger();
  const bool early = p.plan_uploaded != 0;
  if (!early) pdl_wait();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - ptx::smem_u32(smem_raw));
  // RoPE: this warp's per-stage table rows, then the CTA's offset rows
  constexpr int W = decode_kv8_warps(ROPE);   // warps of this CTA
  const uint32_t grows = base + uint32_t(W * kStages8 * (kStage8 + 8) +
                                         warp * kStages8 * kRowBytes8);
  const uint8_t* const grows_ptr = base_ptr + (grows - base);
  uint8_t* const frows_ptr =
      base_ptr + W * kStages8 * (kStage8 + 8) + W * kStages8 * kRowBytes8;
  if constexpr (ROPE) {
    const float4* src = reinterpret_cast<const float4*>(p.rope);
    for (int i = threadIdx.x; i < kStageTokens * (kD8 / 4); i += W * 32) {
      const float4 v = __ldg(src + i);
      reinterpret_cast<float4*>(frows_ptr)[i] =
          make_float4(v.x * kRopeOperandScale, v.y * kRopeOperandScale, v.z * kRopeOperandScale,
                      v.w * kRopeOperandScale);
    }
    __syncthreads();
  }
  const int gw = blockIdx.x * W + warp;
  if (gw >= p.num_warps) return;
  const int it_begin = __ldg(p.warp_ptr + gw), it_end = __ldg(p.warp_ptr + gw + 1);
  if (it_begin >= it_end) return;

  const uint32_t ring = base + uint32_t(warp * kStages8 * kStage8);
  const uint32_t bars = base + uint32_t(W * kStages8 * kStage8 + warp * kStages8 * 8);
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kStages8; ++s) ptx::mbar_init(bars + 8 * s, 1);
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tm_k);
    ptx::prefetch_tensormap(&tm_v);
  }
  __syncwarp();
  const uint64_t pol = ptx::policy_evict_first();
  const int g4 = lane >> 2, t4 = lane & 3;
  const int log2P = 31 - __clz(p.P);

  // ------------------------------------------------------------------ producer
  // Up to kStages8 stages ahead of the consumer; page ids of the next 32 stages
  // of the current unit sit one per lane in `win`.
  int p_it = it_begin, p_st = 0, p_nst = 0, win = 0, win_next = 0, win_base = 0;
  int wpos = 0, wpos_next = 0;   // RoPE with page positions: the stages' first-key positions
  uint32_t p_seq = 0;
  DecodeItem pi;
  const uint64_t pol_rope = ptx::policy_evict_normal();
  auto load_window = [&](const DecodeItem& it, int ws) -> int {
    const int s = ws + lane;
    if (s < stages_of(it))
      return __ldg(p.indices + it.page_base + ((it.tok0 + kStageTokens * s) >> log2P));
    return 0;
  };
  auto load_pos_window = [&](const DecodeItem& it, int ws) -> int {
    const int s = ws + lane;
    if (!ROPE || p.page_pos == nullptr || s >= stages_of(it)) return 0;
    const int tok = it.tok0 + kStageTokens * s;
    return __ldg(p.page_pos + it.page_base + (tok >> log2P)) + (tok & (p.P - 1));
  };
  auto producer_seek = [&]() {
    while (p_it < it_end) {
      pi = load_item(p.items, p_it);
      p_nst = stages_of(pi);
      if (p_nst > 0) break;
      ++p_it;
    }
    if (p_it < it_end) {
      win_base = 0;
      win = load_window(pi, 0);
      win_next = load_window(pi, 32);
      if constexpr (ROPE) {
        wpos = load_pos_window(pi, 0);
        wpos_next = load_pos_window(pi, 32);
      }
    }
  };
  auto producer_issue = [&]() {
    if (p_it >= it_end) return;
    const int slot = int(p_seq % kStages8);
    const int page = __shfl_sync(0xffffffffu, win, p_st - win_base);
    const int spos = ROPE ? __shfl_sync(0xffffffffu, wpos, p_st - win_base) : 0;
    if (lane == 0) {
      const uint32_t bar = bars + 8 * slot;
      const uint32_t dk = ring + uint32_t(slot * kStage8), dv = dk + kTile8;
      const int tok = pi.tok0 + kStageTokens * p_st;
      const int row = (page * p.Hk + pi.kvh) * p.P + (tok & (p.P - 1));
      ptx::mbar_arrive_expect_tx(bar, kStage8 + (ROPE ? kRowBytes8 : 0));
      if constexpr (ROPE) {
        // the table row of the stage's first key: its index, or its logical position
        const int rpos = min(p.page_pos ? spos : tok, p.rope_max_pos);
        ptx::bulk_load(grows + uint32_t(slot * kRowBytes8),
                       reinterpret_cast<const float4*>(p.rope) + size_t(rpos) * (kD8 / 4),
                       kRowBytes8, bar, pol_rope);
      }
      if (p.nhd) {   // token row page * P + slot, the head as the map's outer coordinate
        const int trow = page * p.P + (tok & (p.P - 1));
        ptx::tma_load_3d(dk, &tm_k, bar, 0, trow, pi.kvh, pol);
        ptx::tma_load_3d(dv, &tm_v, bar, 0, trow, pi.kvh, pol);
      } else {
        ptx::tma_load_2d(dk, &tm_k, bar, 0, row, pol);
        ptx::tma_load_2d(dv, &tm_v, bar, 0, row, pol);
      }
    }
    ++p_seq;
    ++p_st;
    if (p_st == p_nst) {
      ++p_it;
      p_st = 0;
      producer_seek();
    } else if (p_st - win_base == 32) {
      win_base += 32;
      win = win_next;
      win_next = load_window(pi, win_base + 32);
      if constexpr (ROPE) {
        wpos = wpos_next;
        wpos_next = load_pos_window(pi, win_base + 32);
      }
    }
  };
  producer_seek();
  if (early) pdl_wait();
#pragma unroll 1
  for (int i = 0; i < kStages8; ++i) producer_issue();

  // ------------------------------------------------------------------ consumer
  // ldmatrix lane addressing (matrix mi = lane / 8, row lane % 8):
  //  K (x4): mi covers keys (mi / 2) * 8.., 16-byte chunk 2 * pair + mi % 2
  //  V (x4, trans): mi covers keys (mi % 2) * 8.., chunk 2 * pair + mi / 2
  const int mi = lane >> 3;
  const int k_tok = ((mi >> 1) << 3) + (lane & 7), k_cb = mi & 1;
  const int v_tok = ((mi & 1) << 3) + (lane & 7), v_cb = mi >> 1;
  constexpr float kLn2 = 0.69314718055994530942f;

  uint32_t c_seq = 0;
  bool failed = false;
  float rmag = 0.f;   // RoPE: largest rotated q / k magnitude of a valid row or key
#pragma unroll 1
  for (int c_it = it_begin; c_it < it_end; ++c_it) {
    const DecodeItem ci = load_item(p.items, c_it);
    const int nst = stages_of(ci);
    const int group = p.group;
    const int rA = ci.row0 + g4, rB = ci.row0 + g4 + 8;
    const bool vA = g4 < ci.nrows, vB = R16 && (g4 + 8 < ci.nrows);
    const int qposA = ci.qpos0 + rA / group, qposB = ci.qpos0 + rB / group;
    const int qpos_min = ci.qpos0 + ci.row0 / group;
    // sliding window: row r sees keys >= its position - window_left + 1; the last
    // row's bound is the highest, so a stage at or above it is unmasked for all rows
    // (compiled in only for WIN: the predicates cost a few percent in the hot loop)
    const int wlo_A = WIN ? qposA - p.window_left + 1 : 0;
    const int wlo_B = WIN ? qposB - p.window_left + 1 : 0;
    const int wlo_max = WIN ? ci.qpos0 + (ci.row0 + ci.nrows - 1) / group - p.window_left + 1 : 0;

    // q fragments in fp16, head dims of block kb in the order 4t..4t+3:
    // [kb][0] = row g4 dims 4t, 4t+1; [kb][NR/2] = row g4 dims 4t+2, 4t+3;
    // with R16 [kb][1] / [kb][3] the same for row g4 + 8.
    uint32_t qh[KB][NR];
    if constexpr (ROPE) {
      // rotate q at its (logical) position in fp32, then fp16 x 2^-4; dims 4t..4t+3 of
      // block kb (< KB / 2) pair with the same dims of block kb + KB / 2
      const int qsh = p.qshift != nullptr ? __ldg(p.qshift + ci.req) : 0;
#pragma unroll
      for (int rr = 0; rr < (R16 ? 2 : 1); ++rr) {
        const int R = rr == 0 ? rA : rB;
        const bool valid = rr == 0 ? vA : vB;
        const uint16_t* qr =
            p.q + (size_t(ci.q_row0 + R / group) * p.Hq + ci.kvh * group + R % group) * D;
        const int pos = min(max(ci.qpos0 + R / group + qsh, 0), p.rope_max_pos);
        const float4* tab = reinterpret_cast<const float4*>(p.rope) + size_t(pos) * (D / 4) + 2 * t4;
        const int lo = rr == 0 ? 0 : 1, hi = rr == 0 ? NR / 2 : 3;
#pragma unroll
        for (int kb = 0; kb < KB / 2; ++kb) {
          const int d0 = 16 * kb + 4 * t4;
          const uint2 a = valid ? __ldg(reinterpret_cast<const uint2*>(qr + d0)) : make_uint2(0u, 0u);
          const uint2 b = valid ? __ldg(reinterpret_cast<const uint2*>(qr + d0 + D / 2))
                                : make_uint2(0u, 0u);
          const float4 t01 = __ldg(tab + 8 * kb), t23 = __ldg(tab + 8 * kb + 1);
          float2 x01 = make_float2(ptx::bf16_lo(a.x), ptx::bf16_hi(a.x));
          float2 x23 = make_float2(ptx::bf16_lo(a.y), ptx::bf16_hi(a.y));
          float2 y01 = make_float2(ptx::bf16_lo(b.x), ptx::bf16_hi(b.x));
          float2 y23 = make_float2(ptx::bf16_lo(b.y), ptx::bf16_hi(b.y));
          const float2 sc = make_float2(kRopeOperandScale, kRopeOperandScale);
          rotate2(x01, y01, ptx::fmul2(make_float2(t01.x, t01.y), sc), ptx::fmul2(make_float2(t01.z, t01.w), sc));
          rotate2(x23, y23, ptx::fmul2(make_float2(t23.x, t23.y), sc), ptx::fmul2(make_float2(t23.z, t23.w), sc));
          rmag = ptx::fmax3(rmag, fmaxf(fabsf(x01.x), fabsf(x01.y)), fmaxf(fabsf(x23.x), fabsf(x23.y)));
          rmag = ptx::fmax3(rmag, fmaxf(fabsf(y01.x), fabsf(y01.y)), fmaxf(fabsf(y23.x), fabsf(y23.y)));
          qh[kb][lo] = ptx::pack_f16(x01.x, x01.y);
          qh[kb][hi] = ptx::pack_f16(x23.x, x23.y);
          qh[kb + KB / 2][lo] = ptx::pack_f16(y01.x, y01.y);
          qh[kb + KB / 2][hi] = ptx::pack_f16(y23.x, y23.y);
        }
      }
    } else {
      const uint16_t* qa =
          p.q + (size_t(ci.q_row0 + rA / group) * p.Hq + ci.kvh * group + rA % group) * D;
      const uint16_t* qb =
          p.q + (size_t(ci.q_row0 + rB / group) * p.Hq + ci.kvh * group + rB % group) * D;
#pragma unroll
      for (int kb = 0; kb < KB; ++kb) {
        const int d0 = 16 * kb + 4 * t4;
        const uint2 a = vA ? __ldg(reinterpret_cast<const uint2*>(qa + d0)) : make_uint2(0u, 0u);
        qh[kb][0] = bf16x2_to_f16x2(a.x);
        qh[kb][NR / 2] = bf16x2_to_f16x2(a.y);
        if constexpr (R16) {
          const uint2 b = vB ? __ldg(reinterpret_cast<const uint2*>(qb + d0)) : make_uint2(0u, 0u);
          qh[kb][1] = bf16x2_to_f16x2(b.x);
          qh[kb][3] = bf16x2_to_f16x2(b.y);
        }
      }
    }

    float o[NT][NR];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int r = 0; r < NR; ++r) o[n][r] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

    // One step consumes NS ring stages (16 keys each): two while at least two
    // remain, so that the Q K^T products of both interleave (four independent
    // accumulator chains) and the max, its shuffles and the O rescale run once
    // per 32 keys; a last odd stage goes alone.
    auto step = [&](auto ns_c, int st) -> bool {
      constexpr int NS = decltype(ns_c)::value;
      uint32_t kt[NS], vt[NS];
      int tok[NS], nvalid[NS];
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        const uint32_t sq = c_seq + uint32_t(s);
        const int slot = int(sq % kStages8);
        kt[s] = ring + uint32_t(slot * kStage8);
        vt[s] = kt[s] + kTile8;
        tok[s] = ci.tok0 + kStageTokens * (st + s);
        nvalid[s] = min(kStageTokens, ci.tok1 - tok[s]);
        if (!ptx::mbar_wait_bounded(bars + 8 * slot, (sq / kStages8) & 1u, p.wait_limit_ns))
          return false;
      }
      bool zeroed = false;
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        if (nvalid[s] < kStageTokens) {
          // Rows past the valid keys may hold another page's tail (NaN codes
          // included): zero their V codes so that P = 0 contributes exactly 0.
          zeroed = true;
#pragma unroll 1
          for (int idx = lane; idx < (kStageTokens - nvalid[s]) * 8; idx += 32) {
            const int t = nvalid[s] + idx / 8, c = idx % 8;
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vt[s] + tile8_off(t, c)),
                         "r"(0u)
                         : "memory");
          }
        }
      }
      __syncwarp();

      // ---------------- S = Q K^T  (per stage two n-tiles of 8 keys), 32 dims per ldmatrix
      float sacc[NS][2][4];
#pragma unroll
      for (int s = 0; s < NS; ++s)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int r = 0; r < 4; ++r) sacc[s][n][r] = 0.f;
      if constexpr (ROPE) {
        // keys are rotated in registers: codes -> fp16 -> fp32, angle of key tok + t =
        // angle of tok (the stage's table row) (+) angle of t (offset row), then fp16 x
        // 2^-4.  A thread holds keys g4 (n-tile 0) and 8 + g4 (n-tile 1), dims 4 t4 ..
        // 4 t4 + 3 of each block: block kb pairs with block kb + KB / 2.
        const float4* fo[2] = {reinterpret_cast<const float4*>(frows_ptr + g4 * kRowBytes8) + 2 * t4,
                               reinterpret_cast<const float4*>(frows_ptr + (g4 + 8) * kRowBytes8) + 2 * t4};
#pragma unroll
        for (int pr = 0; pr < KB / 4; ++pr) {
          uint32_t kl[NS][4], kh[NS][4];
#pragma unroll
          for (int s = 0; s < NS; ++s) {
            ptx::ldsm_x4(kl[s], kt[s] + tile8_off(k_tok, 2 * pr + k_cb));
            ptx::ldsm_x4(kh[s], kt[s] + tile8_off(k_tok, 2 * pr + KB / 2 + k_cb));
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int kb = 2 * pr + h;
            const uint32_t a0 = qh[kb][0], a2 = qh[kb][NR / 2];
            const uint32_t a1 = R16 ? qh[kb][1] : 0u, a3 = R16 ? qh[kb][NR - 1] : 0u;
            const int kb2 = kb + KB / 2;
            const uint32_t b0 = qh[kb2][0], b2 = qh[kb2][NR / 2];
            const uint32_t b1 = R16 ? qh[kb2][1] : 0u, b3 = R16 ? qh[kb2][NR - 1] : 0u;
#pragma unroll
            for (int s = 0; s < NS; ++s) {
              const float4* gr = reinterpret_cast<const float4*>(
                                     grows_ptr + int((c_seq + uint32_t(s)) % kStages8) * kRowBytes8) +
                                 2 * t4;
              const float4 g01 = gr[8 * kb], g23 = gr[8 * kb + 1];
#pragma unroll
              for (int n = 0; n < 2; ++n) {
                const float4 o01 = fo[n][8 * kb], o23 = fo[n][8 * kb + 1];
                // cos / sin of (tok + t) omega for the four frequencies, times 2^-4
                const float2 cg01 = make_float2(g01.x, g01.y), sg01 = make_float2(g01.z, g01.w);
                const float2 cg23 = make_float2(g23.x, g23.y), sg23 = make_float2(g23.z, g23.w);
                const float2 co01 = make_float2(o01.x, o01.y), so01 = make_float2(o01.z, o01.w);
                const float2 co23 = make_float2(o23.x, o23.y), so23 = make_float2(o23.z, o23.w);
                const float2 c01 = ptx::fsub2(ptx::fmul2(cg01, co01), ptx::fmul2(sg01, so01));
                const float2 s01 = ptx::ffma2(sg01, co01, ptx::fmul2(cg01, so01));
                const float2 c23 = ptx::fsub2(ptx::fmul2(cg23, co23), ptx::fmul2(sg23, so23));
                const float2 s23 = ptx::ffma2(sg23, co23, ptx::fmul2(cg23, so23));
                const uint32_t lo = kl[s][2 * n + h], hi = kh[s][2 * n + h];
                float2 x01 = f16x2_to_f32x2(e4m3x2_to_f16x2(lo)), x23 = f16x2_to_f32x2(e4m3x2_to_f16x2(lo >> 16));
                float2 y01 = f16x2_to_f32x2(e4m3x2_to_f16x2(hi)), y23 = f16x2_to_f32x2(e4m3x2_to_f16x2(hi >> 16));
                rotate2(x01, y01, c01, s01);
                rotate2(x23, y23, c23, s23);
                if (8 * n + g4 < nvalid[s]) {
                  rmag = ptx::fmax3(rmag, fmaxf(fabsf(x01.x), fabsf(x01.y)), fmaxf(fabsf(x23.x), fabsf(x23.y)));
                  rmag = ptx::fmax3(rmag, fmaxf(fabsf(y01.x), fabsf(y01.y)), fmaxf(fabsf(y23.x), fabsf(y23.y)));
                }
                float* acc = sacc[s][n];
                ptx::mma_f16(acc[0], acc[1], acc[2], acc[3], a0, a1, a2, a3, ptx::pack_f16(x01.x, x01.y),
                             ptx::pack_f16(x23.x, x23.y));
                ptx::mma_f16(acc[0], acc[1], acc[2], acc[3], b0, b1, b2, b3, ptx::pack_f16(y01.x, y01.y),
                             ptx::pack_f16(y23.x, y23.y));
              }
            }
          }
        }
      } else {
#pragma unroll
      for (int pr = 0; pr < KB / 2; ++pr) {
        uint32_t kr[NS][4];
#pragma unroll
        for (int s = 0; s < NS; ++s) ptx::ldsm_x4(kr[s], kt[s] + tile8_off(k_tok, 2 * pr + k_cb));
        // kr[s][h]: keys g4 (n-tile 0), block 2 pr + h; kr[s][2 + h]: keys 8 + g4 (n-tile 1)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int kb = 2 * pr + h;
          const uint32_t a0 = qh[kb][0], a2 = qh[kb][NR / 2];
          const uint32_t a1 = R16 ? qh[kb][1] : 0u, a3 = R16 ? qh[kb][NR - 1] : 0u;
#pragma unroll
          for (int s = 0; s < NS; ++s) {
            float* s0 = sacc[s][0];
            float* s1 = sacc[s][1];
            ptx::mma_f16(s0[0], s0[1], s0[2], s0[3], a0, a1, a2, a3, e4m3x2_to_f16x2(kr[s][h]),
                         e4m3x2_to_f16x2(kr[s][h] >> 16));
            ptx::mma_f16(s1[0], s1[1], s1[2], s1[3], a0, a1, a2, a3, e4m3x2_to_f16x2(kr[s][2 + h]),
                         e4m3x2_to_f16x2(kr[s][2 + h] >> 16));
          }
        }
      }
      }

      // ---------------- mask + online softmax (log2 domain; k_scale is in scale_log2)
      float xa[NS][4], xb[NS][4];
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        const bool full = (nvalid[s] == kStageTokens) &&
                          (!p.causal || tok[s] + kStageTokens - 1 <= qpos_min) &&
                          (!WIN || tok[s] >= wlo_max);
        // with RoPE q and k are both scaled by 2^-4
        const float sc = ROPE ? p.scale_log2 * (1.f / (kRopeOperandScale * kRopeOperandScale))
                              : p.scale_log2;
        const int k0 = tok[s] + 2 * t4;
        const int kidx[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
        const float sa[4] = {sacc[s][0][0], sacc[s][0][1], sacc[s][1][0], sacc[s][1][1]};
        const float sb[4] = {sacc[s][0][2], sacc[s][0][3], sacc[s][1][2], sacc[s][1][3]};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool inr = full || (kidx[j] < ci.tok1);
          const bool okA =
              full || (inr && (!p.causal || kidx[j] <= qposA) && (!WIN || kidx[j] >= wlo_A));
          const bool okB =
              full || (inr && (!p.causal || kidx[j] <= qposB) && (!WIN || kidx[j] >= wlo_B));
          xa[s][j] = okA ? sa[j] * sc : -INFINITY;
          xb[s][j] = okB ? sb[j] * sc : -INFINITY;
        }
      }
      float mxA = -INFINITY;
#pragma unroll
      for (int s = 0; s < NS; ++s)
        mxA = fmaxf(mxA, fmaxf(fmaxf(xa[s][0], xa[s][1]), fmaxf(xa[s][2], xa[s][3])));
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
      const float mnA = fmaxf(mA, mxA);
      const float muA = mnA == -INFINITY ? 0.f : mnA;
      const float alA = ptx::ex2(mA - muA);
      mA = mnA;
      float pa[NS][4];
      float sumA = 0.f;
#pragma unroll
      for (int s = 0; s < NS; ++s) {
#pragma unroll
        for (int j = 0; j < 4; ++j) pa[s][j] = ptx::ex2(xa[s][j] - muA);
        sumA += (pa[s][0] + pa[s][1]) + (pa[s][2] + pa[s][3]);
      }
      lA = lA * alA + sumA;
      float alB = 1.f;
      float pb[NS][4];
#pragma unroll
      for (int s = 0; s < NS; ++s)
#pragma unroll
        for (int j = 0; j < 4; ++j) pb[s][j] = 0.f;
      if constexpr (R16) {
        float mxB = -INFINITY;
#pragma unroll
        for (int s = 0; s < NS; ++s)
          mxB = fmaxf(mxB, fmaxf(fmaxf(xb[s][0], xb[s][1]), fmaxf(xb[s][2], xb[s][3])));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
        const float mnB = fmaxf(mB, mxB);
        const float muB = mnB == -INFINITY ? 0.f : mnB;
        alB = ptx::ex2(mB - muB);
        mB = mnB;
        float sumB = 0.f;
#pragma unroll
        for (int s = 0; s < NS; ++s) {
#pragma unroll
          for (int j = 0; j < 4; ++j) pb[s][j] = ptx::ex2(xb[s][j] - muB);
          sumB += (pb[s][0] + pb[s][1]) + (pb[s][2] + pb[s][3]);
        }
        lB = lB * alB + sumB;
      }
      if (__any_sync(0xffffffffu, alA != 1.f || alB != 1.f)) {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          o[n][0] *= alA;
          o[n][1] *= alA;
          if constexpr (R16) {
            o[n][NR - 2] *= alB;
            o[n][NR - 1] *= alB;
          }
        }
      }

      // ---------------- O += P V  (P in fp16), 32 dims per ldmatrix; stage by stage,
      // so that the two products into one accumulator are 16 MMAs apart
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        const uint32_t ph0 = ptx::pack_f16(pa[s][0], pa[s][1]), ph2 = ptx::pack_f16(pa[s][2], pa[s][3]);
        [[maybe_unused]] const uint32_t ph1 = R16 ? ptx::pack_f16(pb[s][0], pb[s][1]) : 0u;
        [[maybe_unused]] const uint32_t ph3 = R16 ? ptx::pack_f16(pb[s][2], pb[s][3]) : 0u;
#pragma unroll
        for (int pr = 0; pr < KB / 2; ++pr) {
          uint32_t vr[4];
          ptx::ldsm_x4_trans(vr, vt[s] + tile8_off(v_tok, 2 * pr + v_cb));
          // vr[2h]: keys 2t, 2t+1 of the first 8 keys, dims (2 g4, 2 g4 + 1) of block
          // 2 pr + h; vr[2h + 1]: the same for keys 8 + 2t, 8 + 2t + 1
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int cb = 2 * pr + h;
            const uint32_t lo = vr[2 * h], hi = vr[2 * h + 1];
            // even dims of the block (2 g4), then odd dims (2 g4 + 1)
            const uint32_t be0 = e4m3x2_to_f16x2(__byte_perm(lo, 0u, 0x0020));
            const uint32_t be1 = e4m3x2_to_f16x2(__byte_perm(hi, 0u, 0x0020));
            const uint32_t bo0 = e4m3x2_to_f16x2(__byte_perm(lo, 0u, 0x0031));
            const uint32_t bo1 = e4m3x2_to_f16x2(__byte_perm(hi, 0u, 0x0031));
            float* e = o[2 * cb];
            float* f = o[2 * cb + 1];
            if constexpr (R16) {
              ptx::mma_f16(e[0], e[1], e[NR - 2], e[NR - 1], ph0, ph1, ph2, ph3, be0, be1);
              ptx::mma_f16(f[0], f[1], f[NR - 2], f[NR - 1], ph0, ph1, ph2, ph3, bo0, bo1);
            } else {
              // rows g4 + 8 are padding: their accumulators are dead scratch
              float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;
              ptx::mma_f16(e[0], e[1], z0, z1, ph0, 0u, ph2, 0u, be0, be1);
              ptx::mma_f16(f[0], f[1], z2, z3, ph0, 0u, ph2, 0u, bo0, bo1);
            }
          }
        }
      }
      __syncwarp();
      // generic writes (the zero fill) must be ordered before the TMA that reuses the slot
      if (zeroed) ptx::fence_proxy_async_smem();
      __syncwarp();
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        ++c_seq;
        producer_issue();
      }
      return true;
    };
    {
      int st = 0;
#pragma unroll 1
      for (; st + 2 <= nst; st += 2)
        if (!step(std::integral_constant<int, 2>{}, st)) {
          failed = true;
          break;
        }
      if (!failed && st < nst && !step(std::integral_constant<int, 1>{}, st)) failed = true;
    }
    if (failed) break;

    // ---------------- epilogue: dims 16 c + 4 t .. + 3 of every block c are
    // o[2c][c0], o[2c+1][c0], o[2c][c0+1], o[2c+1][c0+1]
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    if constexpr (R16) {
      lB += __shfl_xor_sync(0xffffffffu, lB, 1);
      lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    }
    const float lseA = lA > 0.f ? mA + ptx::lg2(lA) : -INFINITY;
    const float lseB = lB > 0.f ? mB + ptx::lg2(lB) : -INFINITY;
    const float invA = lA > 0.f ? p.v_scale / lA : 0.f;
    const float invB = lB > 0.f ? p.v_scale / lB : 0.f;
    if (ci.slot < 0) {
#pragma unroll
      for (int rr = 0; rr < (R16 ? 2 : 1); ++rr) {
        const bool ok = rr == 0 ? vA : vB;
        if (!ok) continue;
        const int R = rr == 0 ? rA : rB;
        const float inv = rr == 0 ? invA : invB;
        const int c0 = rr == 0 ? 0 : NR - 2;
        const size_t orow = size_t(ci.q_row0 + R / group) * p.Hq + ci.kvh * group + R % group;
        if (p.out_f32) {
          float* dst = static_cast<float*>(p.out) + orow * D + 4 * t4;
#pragma unroll
          for (int cb = 0; cb < KB; ++cb)
            *reinterpret_cast<float4*>(dst + 16 * cb) =
                make_float4(o[2 * cb][c0] * inv, o[2 * cb + 1][c0] * inv,
                            o[2 * cb][c0 + 1] * inv, o[2 * cb + 1][c0 + 1] * inv);
        } else {
          uint16_t* dst = static_cast<uint16_t*>(p.out) + orow * D + 4 * t4;
#pragma unroll
          for (int cb = 0; cb < KB; ++cb)
            *reinterpret_cast<uint2*>(dst + 16 * cb) =
                make_uint2(ptx::pack_bf16(o[2 * cb][c0] * inv, o[2 * cb + 1][c0] * inv),
                           ptx::pack_bf16(o[2 * cb][c0 + 1] * inv, o[2 * cb + 1][c0 + 1] * inv));
        }
        if (p.lse != nullptr && t4 == 0) p.lse[orow] = (rr == 0 ? lseA : lseB) * kLn2;
      }
    } else {
#pragma unroll
      for (int rr = 0; rr < (R16 ? 2 : 1); ++rr) {
        const int r = g4 + 8 * rr;
        const float inv = rr == 0 ? invA : invB;
        const int c0 = rr == 0 ? 0 : NR - 2;
        float* dst = p.part_o + (size_t(ci.slot) * kMaxDecodeRows + r) * D + 4 * t4;
#pragma unroll
        for (int cb = 0; cb < KB; ++cb)
          __stcg(reinterpret_cast<float4*>(dst + 16 * cb),
                 make_float4(o[2 * cb][c0] * inv, o[2 * cb + 1][c0] * inv,
                             o[2 * cb][c0 + 1] * inv, o[2 * cb + 1][c0 + 1] * inv));
        if (t4 == 0)
          __stcg(p.part_lse + size_t(ci.slot) * kMaxDecodeRows + r, rr == 0 ? lseA : lseB);
      }
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) last = atomicAdd(p.counters + ci.first_slot, 1) == ci.nchunks - 1;
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence();
        merge_range<D>(p, ci, lane);
        if (lane == 0) atomicExch(p.counters + ci.first_slot, 0);
      }
    }
  }

  if (ROPE && __any_sync(0xffffffffu, rmag > kRopeOperandMax) && lane == 0)
    atomicOr(p.error, kStatusOperandRange);
  if (failed) {
    if (lane == 0) atomicOr(p.error, 1);
    // let the copies this warp still has in flight land before the CTA exits
#pragma unroll 1
    for (uint32_t s = c_seq; s < p_seq; ++s)
      ptx::mbar_wait_bounded(bars + 8 * (s % kStages8), (s / kStages8) & 1u, 50000000ull);
  }
}

constexpr int kMaxDevices = 64;

template <bool R16, bool WIN, bool ROPE>
cudaError_t launch_one(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                       cudaStream_t stream) {
  auto kern = bsr_decode_kv8_kernel<R16, WIN, ROPE>;
  constexpr int W = decode_kv8_warps(ROPE);
  constexpr size_t smem = smem8(ROPE);
  const int grid = (p.num_warps + W - 1) / W;
  if (grid <= 0) return cudaSuccess;
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
  const cudaError_t le = launch_pdl(kern, grid, W * 32, smem, stream, tk, tv, p);
  return le != cudaSuccess ? le : cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_kv8(bool rope, bool r16, const CUtensorMap& tk, const CUtensorMap& tv,
                              const DecodeParams& p, cudaStream_t stream) {
  const bool win = p.window_left > 0;
  if (rope) {
    if (r16) return win ? launch_one<true, true, true>(tk, tv, p, stream)
                        : launch_one<true, false, true>(tk, tv, p, stream);
    return win ? launch_one<false, true, true>(tk, tv, p, stream)
               : launch_one<false, false, true>(tk, tv, p, stream);
  }
  if (r16) return win ? launch_one<true, true, false>(tk, tv, p, stream)
                      : launch_one<true, false, false>(tk, tv, p, stream);
  return win ? launch_one<false, true, false>(tk, tv, p, stream)
             : launch_one<false, false, false>(tk, tv, p, stream);
}

}  // namespace bsr
