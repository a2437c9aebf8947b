// Split-KV decode attention over a paged (BSR) KV cache, sm_103a.
//
// Decode is bound by HBM bandwidth: every generated token re-reads its whole
// KV history ("FlashInfer: Block-Sparse KV 캐시로 어텐션 병목을 해소하다",
// section "어텐션 연산에서 진짜 병목은 어디인가?").  The kernel is therefore
// built around keeping enough bytes in flight:
//
//  * Persistent CTAs of kDecodeWarps warps.  Every warp is an independent
//    workgroup that walks its own planned list of work units (request,
//    kv head, packed-row group, page-aligned key chunk) — the load-balanced
//    split of long sequences into pieces interleaved with short ones
//    (section "벤치마크: FlashInfer는 얼마나 빠른가?").  For skewed batches the
//    plan leaves the shortest whole ranges out of those lists: a warp that has
//    finished its own list takes them one at a time from a shared queue (an
//    atomic counter; the last warp of a launch resets it), so the warps that
//    stream faster take more and the kernel does not wait for the slowest list.
//  * Each warp feeds itself through a private ring of shared-memory stages:
//    one elected lane issues TMA (cp.async.bulk.tensor) loads of the next
//    16-token K and V tiles of the unit's pages, straight from the page ids
//    in `indices` (dropped blocks are absent there and never read), into
//    128B-swizzled tiles completing on an mbarrier -- one box per tile (with
//    D = 128 the map takes the two 64-column blocks as its outer dimension,
//    so one 4 KB copy lands both: the copy engine's cost is mostly per box,
//    and two 2 KB boxes per tile held a CTA to ~20 B/clk).  Only active blocks are
//    gathered ("Block-Sparse 포맷").
//  * The (query, head) rows of one GQA group are packed into the M dimension
//    of warp-level m16n8k16 bf16 MMAs: S = Q K^T for 16 keys, online softmax
//    in registers (exp2 domain), O += P V with P split into bf16 hi + lo so
//    the probabilities keep ~16 bits.  K is rotated on load when RoPE is on
//    (section "JIT 컴파일은 …": RoPE fused into attention); rotated q and k
//    are fp16 operands scaled by 2^-4.  The angle of key p0 + t (p0 the
//    stage's first key) is composed from the table row of p0, copied into
//    the stage with its K and V, and the row of t < 16, kept in shared memory
//    for the whole CTA, so no table load waits on L2 inside the stage.
//  * A unit that covers all keys of its range writes out (bf16 / fp32) and the
//    natural-log LSE; a split unit writes a normalized fp32 partial state and
//    the last arriving unit of the range merges all partials in chunk order
//    (deterministic) and resets the range's counter for the next launch.
//
// Every barrier wait is bounded; on timeout the warp sets bit 0 of the
// schedule's status word, drains its outstanding copies (bounded) and exits.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "bsr_internal.h"
#include "bsr_launch.cuh"
#include "ptx.cuh"

namespace bsr {

template <int D>
struct DecodeCfg {
  static constexpr int kHalves = D / 64;                        // 128-byte column blocks per row
  static constexpr int kStageKBytes = kStageTokens * D * 2;      // one K (or V) tile
  static constexpr int kStageBytes = 2 * kStageKBytes;           // K + V
  static constexpr int kStages = (D == 128) ? BSR_DECODE_STAGES_D128 : BSR_DECODE_STAGES_D64;
  static constexpr int kKSteps = D / 16;
  static constexpr int kNTiles = D / 8;
  // cos/sin table: one position is D/2 (cos, sin) fp32 pairs = D/4 float4s,
  // float4 (i, quad t) at i * 4 + t holding frequencies 16(i/2) + 8(i%2) + 2t + {0, 1}
  static constexpr int kRopeRowF4 = D / 4;
  static constexpr int kRopeRowBytes = 16 * kRopeRowF4;
  // offset rows t < 16 in shared memory, padded so that rows t and t + 1 fall
  // on different bank halves (conflict-free 16-byte loads)
  static constexpr int kRopeOffStride = kRopeRowBytes + 64;
  static constexpr size_t kRingBytes = size_t(kDecodeWarps) * kStages * kStageBytes;
  static constexpr size_t kBarBytes = size_t(kDecodeWarps) * kStages * 8;
  // per warp: the item ids of the run-time units it has taken, by position (a ring: the
  // producer runs at most kStages stages, so at most kStages units, ahead)
  static constexpr int kTakenRing = 8;
  static constexpr size_t kTakenBytes = size_t(kDecodeWarps) * kTakenRing * 4;
  static constexpr size_t kSmemBytes = kRingBytes + kBarBytes + kTakenBytes + 1024;
  static constexpr size_t kSmemBytesRope = kSmemBytes +
                                           size_t(kDecodeWarps) * kStages * kRopeRowBytes +
                                           size_t(kStageTokens) * kRopeOffStride;
  static_assert((kBarBytes + kTakenBytes) % 16 == 0,
                "stage-row copies need 16-byte aligned destinations");
  static_assert(kTakenRing > kStages && (kTakenRing & (kTakenRing - 1)) == 0, "taken-unit ring");
  static_assert(kSmemBytesRope <= 232448, "decode stages exceed the shared memory of one SM");
};

// Byte offset of (token t, column d) in a 16-token tile stored as
// [column block][16 tokens][128 bytes] with the TMA 128-byte swizzle
// (16-byte chunk index XOR row index mod 8).  d must be a multiple of 8.
__device__ __forceinline__ uint32_t tile_off(int t, int d) {
  const int h = d >> 6, c = (d & 63) >> 3;
  return uint32_t(((h * kStageTokens + t) << 7) + ((c ^ (t & 7)) << 4));
}

__device__ __forceinline__ DecodeItem load_item(const DecodeItem* items, int i) {
  const int4* src = reinterpret_cast<const int4*>(items + i);
  const int4 a = __ldg(src), b = __ldg(src + 1), c = __ldg(src + 2);
  DecodeItem it;
  it.req = a.x; it.kvh = a.y; it.row0 = a.z; it.nrows = a.w;
  it.tok0 = b.x; it.tok1 = b.y; it.slot = b.z; it.first_slot = b.w;
  it.page_base = c.x; it.q_row0 = c.y; it.qpos0 = c.z; it.nchunks = c.w;
  return it;
}

__device__ __forceinline__ int stages_of(const DecodeItem& it) {
  return it.tok1 > it.tok0 ? (it.tok1 - it.tok0 + kStageTokens - 1) / kStageTokens : 0;
}

// Rotate the pairs (x, y) = (dims d, d + D/2) of two bf16x2 registers by the
// (cos, sin) pairs cs0 (element 0) and cs1 (element 1); returns fp32 values.
__device__ __forceinline__ void rope_pair(uint32_t xlo, uint32_t xhi, float2 cs0, float2 cs1,
                                          float (&x)[2], float (&y)[2]) {
  const float a0 = ptx::bf16_lo(xlo), a1 = ptx::bf16_hi(xlo);
  const float b0 = ptx::bf16_lo(xhi), b1 = ptx::bf16_hi(xhi);
  x[0] = a0 * cs0.x - b0 * cs0.y;
  y[0] = b0 * cs0.x + a0 * cs0.y;
  x[1] = a1 * cs1.x - b1 * cs1.y;
  y[1] = b1 * cs1.x + a1 * cs1.y;
}

// (cos, sin) of a + b from those of a and b, for the two frequencies of a table float4.
__device__ __forceinline__ float4 rot_compose(float4 a, float4 b) {
  return make_float4(a.x * b.x - a.y * b.y, a.y * b.x + a.x * b.y,
                     a.z * b.z - a.w * b.w, a.w * b.z + a.z * b.w);
}

// Merge the partial states of one split range (the last-arriving warp calls
// this).  Rows are taken four at a time; the chunk maxima and sums are
// computed lane-parallel over chunks, and the weighted sum of partial outputs
// (each lane owns D/32 columns) is accumulated in chunk order, so the result
// does not depend on which warp merges.  The merge sits on the kernel's tail, so
// its loads are issued as early as possible: the chunk LSEs and the first four
// chunks' partial rows in one go, then four chunks at a time.
template <int D>
__device__ __forceinline__ void merge_range(const DecodeParams& p, const DecodeItem& ci, int lane) {
  constexpr int CPL = D / 32;
  constexpr float kLn2 = 0.69314718055994530942f;
  const int nck = ci.nchunks, group = p.group;
  const float* lse_base = p.part_lse + size_t(ci.first_slot) * kMaxDecodeRows;
  const float* o_base = p.part_o + size_t(ci.first_slot) * kMaxDecodeRows * D;
  // lane's CPL columns of the partial row of chunk k, row r (0 where `on` is false)
  auto load_o = [&](int k, int r, bool on, float (&v)[CPL]) {
    const size_t sl = size_t(k) * kMaxDecodeRows + r;
    if constexpr (CPL == 4) {
      const float4 t = on ? __ldcg(reinterpret_cast<const float4*>(o_base + sl * D) + lane)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
      v[0] = t.x; v[1 % CPL] = t.y; v[2 % CPL] = t.z; v[3 % CPL] = t.w;
    } else {
      const float2 t = on ? __ldcg(reinterpret_cast<const float2*>(o_base + sl * D) + lane)
                          : make_float2(0.f, 0.f);
      v[0] = t.x; v[1 % CPL] = t.y;
    }
  };
#pragma unroll 1
  for (int r0 = 0; r0 < ci.nrows; r0 += 4) {
    const int nr = min(4, ci.nrows - r0);
    // The chunk LSEs (lane k holds chunk k) and the first four chunks' partial rows are
    // requested together: for ranges of up to four chunks the merge waits on memory once.
    float v0[4][4][CPL];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) load_o(kk, r0 + rr, kk < nck && rr < nr, v0[kk][rr]);
    float lk[4], M[4], S[4], L2[4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      lk[rr] = lane < nck && rr < nr ? __ldcg(lse_base + size_t(lane) * kMaxDecodeRows + r0 + rr)
                                     : -INFINITY;
      M[rr] = lk[rr];
    }
    // chunks 32, 33, ... (long ranges only) are read again where they are needed
#pragma unroll 1
    for (int k = lane + 32; k < nck; k += 32) {
#pragma unroll
      for (int rr = 0; rr < 4; ++rr)
        if (rr < nr) M[rr] = fmaxf(M[rr], __ldcg(lse_base + size_t(k) * kMaxDecodeRows + r0 + rr));
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M[rr] = fmaxf(M[rr], __shfl_xor_sync(0xffffffffu, M[rr], o));
      S[rr] = M[rr] != -INFINITY && lk[rr] != -INFINITY ? ptx::ex2(lk[rr] - M[rr]) : 0.f;
    }
#pragma unroll 1
    for (int k = lane + 32; k < nck; k += 32) {
#pragma unroll
      for (int rr = 0; rr < 4; ++rr)
        if (rr < nr && M[rr] != -INFINITY)
          S[rr] += ptx::ex2(__ldcg(lse_base + size_t(k) * kMaxDecodeRows + r0 + rr) - M[rr]);
    }
    float wk[4];   // this lane's chunk weight exp2(lse_k - L)
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) S[rr] += __shfl_xor_sync(0xffffffffu, S[rr], o);
      L2[rr] = M[rr] == -INFINITY ? -INFINITY : M[rr] + ptx::lg2(S[rr]);
      wk[rr] = L2[rr] == -INFINITY || lk[rr] == -INFINITY ? 0.f : ptx::ex2(lk[rr] - L2[rr]);
    }
    // weight of chunk k, row rr: from lane k for the first 32 chunks, else from memory
    auto weight = [&](int k, int rr) {
      if (k < 32) return __shfl_sync(0xffffffffu, wk[rr], k);
      if (rr >= nr || L2[rr] == -INFINITY) return 0.f;
      const float l = __ldcg(lse_base + size_t(k) * kMaxDecodeRows + r0 + rr);
      return l == -INFINITY ? 0.f : ptx::ex2(l - L2[rr]);
    };
    float acc[4][CPL];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[rr][c] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float wt = weight(kk, rr);
        if (wt != 0.f) {   // an empty chunk's row (weight 0) is not read into the sum
#pragma unroll
          for (int c = 0; c < CPL; ++c) acc[rr][c] += wt * v0[kk][rr][c];
        }
      }
    }
#pragma unroll 1
    for (int k0 = 4; k0 < nck; k0 += 4) {
      float v[4][4][CPL];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) load_o(k0 + kk, r0 + rr, k0 + kk < nck && rr < nr, v[kk][rr]);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          const float wt = k0 + kk < nck ? weight(k0 + kk, rr) : 0.f;
          if (wt != 0.f) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[rr][c] += wt * v[kk][rr][c];
          }
        }
    }
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      if (rr >= nr) break;
      const int R = ci.row0 + r0 + rr;
      const size_t orow = size_t(ci.q_row0 + R / group) * p.Hq + ci.kvh * group + R % group;
      if (p.out_f32) {
        float* dst = static_cast<float*>(p.out) + orow * D + CPL * lane;
#pragma unroll
        for (int c = 0; c < CPL; ++c) dst[c] = acc[rr][c];
      } else {
        uint16_t* dst = static_cast<uint16_t*>(p.out) + orow * D + CPL * lane;
#pragma unroll
        for (int c = 0; c < CPL; c += 2)
          *reinterpret_cast<uint32_t*>(dst + c) = ptx::pack_bf16(acc[rr][c], acc[rr][c + 1]);
      }
      if (p.lse != nullptr && lane == 0) p.lse[orow] = L2[rr] * kLn2;
    }
  }
}

template <int D, bool ROPE, bool R16, bool SMALLP, bool WIN>
__global__ void __launch_bounds__(kDecodeWarps * 32, 1)
    bsr_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  using C = DecodeCfg<D>;
  constexpr int NR = R16 ? 4 : 2;       // accumulator registers per n-tile that carry rows
  constexpr int KS = C::kKSteps;
  constexpr int NT = C::kNTiles;
  constexpr int KH = KS / 2;            // k-steps in the first half of the head dim
  extern __shared__ uint8_t smem_raw[];
  // launched as a programmatic dependent: let the next grid start its set-up.  q, the
  // pages and every output may be another grid's, so they wait until the previous grid
  // has completed; a plan's work list, page table and tables came with its host copy
  // and are read before that wait (the set-up below overlaps the previous grid's tail)
  pdl_trigger();
  const bool early = p.plan_uploaded != 0;
  if (!early) pdl_wait();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - ptx::smem_u32(smem_raw));
  const uint32_t ring = base + uint32_t(warp * C::kStages * C::kStageBytes);
  const uint32_t bars = base + uint32_t(C::kRingBytes + warp * C::kStages * 8);
  // this warp's taken run-time units, then with RoPE its per-stage table rows, then the
  // CTA's offset rows t < 16
  volatile int* const taken =
      reinterpret_cast<volatile int*>(base_ptr + C::kRingBytes + C::kBarBytes) + warp * C::kTakenRing;
  const size_t rope_off = C::kRingBytes + C::kBarBytes + C::kTakenBytes;
  const uint32_t grows = base + uint32_t(rope_off + warp * C::kStages * C::kRopeRowBytes);
  uint8_t* const goff_ptr = base_ptr + (grows - base);
  uint8_t* const frows_ptr =
      base_ptr + rope_off + size_t(kDecodeWarps) * C::kStages * C::kRopeRowBytes;
  if constexpr (ROPE) {
    const float4* src = reinterpret_cast<const float4*>(p.rope);
    for (int i = threadIdx.x; i < kStageTokens * C::kRopeRowF4; i += kDecodeWarps * 32) {
      const int t = i / C::kRopeRowF4, c = i % C::kRopeRowF4;
      *reinterpret_cast<float4*>(frows_ptr + t * C::kRopeOffStride + 16 * c) = __ldg(src + i);
    }
    __syncthreads();
  }

  const int gw = blockIdx.x * kDecodeWarps + warp;
  if (gw >= p.num_warps) return;
  const int it_begin = __ldg(p.warp_ptr + gw), it_end = __ldg(p.warp_ptr + gw + 1);
  // positions 0 .. nstat - 1 of this warp's sequence are its planned items; after them
  // come run-time units taken from the shared queue until it is empty (dyn)
  const bool dyn = !SMALLP && p.n_dyn > 0;
  const int nstat = it_end - it_begin;
  if (nstat <= 0 && !dyn) return;
  if (dyn && lane < C::kTakenRing) taken[lane] = p.dyn_begin;   // always a valid item id
  __syncwarp();
  if (!SMALLP) {
    if (lane == 0) {
#pragma unroll
      for (int s = 0; s < C::kStages; ++s) ptx::mbar_init(bars + 8 * s, 1);
      ptx::fence_barrier_init();
      ptx::prefetch_tensormap(&tm_k);
      ptx::prefetch_tensormap(&tm_v);
    }
    __syncwarp();
  }
  const uint64_t pol = ptx::policy_evict_first();
  const uint64_t pol_rope = ptx::policy_evict_normal();   // table rows are shared by all units
  const int g4 = lane >> 2, t4 = lane & 3;
  const int log2P = 31 - __clz(p.P);

  // ------------------------------------------------------------------ producer
  // The producer runs up to kStages stages ahead of the consumer.  Page ids of
  // the next 32 stages of the current unit sit one per lane in `win`; the next
  // window is requested before it is needed.
  // p_end: the first position with no item (known for a warp without run-time units;
  // otherwise found when the queue is empty); p_have: pi is the unit at position p_q
  int p_q = 0, p_end = dyn ? INT_MAX : nstat, p_st = 0, p_nst = 0;
  int win = 0, win_next = 0, win_base = 0;
  bool p_have = false, may_take = !early, took_last = false;
  // with RoPE and per-page positions: each stage's logical position, same windows
  int wpos = 0, wpos_next = 0;
  uint32_t p_seq = 0;
  DecodeItem pi;
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
  // item id at position q (a run-time unit's was recorded when the producer took it)
  auto item_at = [&](int q) { return q < nstat ? it_begin + q : taken[q & (C::kTakenRing - 1)]; };
  // this warp has found the queue empty: the last planned warp to do so empties the
  // counters for the next launch (every taker of this launch has finished taking)
  auto done_taking = [&]() {
    took_last = true;
    if (lane == 0 && atomicAdd(p.dyn_ctr + 1, 1) == p.num_warps - 1) {
      atomicExch(p.dyn_ctr, 0);
      atomicExch(p.dyn_ctr + 1, 0);
    }
  };
  // take the next run-time unit for position q; false when the queue is empty
  auto take = [&](int q) -> bool {
    int d = 0;
    if (lane == 0) d = atomicAdd(p.dyn_ctr, 1);
    d = __shfl_sync(0xffffffffu, d, 0);
    if (d >= p.n_dyn) {
      done_taking();
      return false;
    }
    if (lane == 0) taken[q & (C::kTakenRing - 1)] = p.dyn_begin + d;
    __syncwarp();
    return true;
  };
  auto producer_seek = [&]() {
    p_have = false;
    while (p_q < p_end) {
      if (p_q >= nstat) {
        if (!may_take) return;   // run-time units wait for the grid-dependency wait
        if (!take(p_q)) {
          p_end = p_q;
          return;
        }
      }
      pi = load_item(p.items, item_at(p_q));
      p_nst = stages_of(pi);
      if (p_nst > 0) {
        p_have = true;
        break;
      }
      ++p_q;
    }
    if (p_have) {
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
    if (!p_have) return;
    const int slot = int(p_seq % C::kStages);
    const int page = __shfl_sync(0xffffffffu, win, p_st - win_base);
    const int spos = ROPE ? __shfl_sync(0xffffffffu, wpos, p_st - win_base) : 0;
    if (lane == 0) {
      const uint32_t bar = bars + 8 * slot;
      const uint32_t dk = ring + uint32_t(slot * C::kStageBytes), dv = dk + C::kStageKBytes;
      const int tok = pi.tok0 + kStageTokens * p_st;
      const int row = (page * p.Hk + pi.kvh) * p.P + (tok & (p.P - 1));
      ptx::mbar_arrive_expect_tx(bar, C::kStageBytes + (ROPE ? C::kRopeRowBytes : 0));
      if constexpr (ROPE) {
        // the table row of the stage's first key: its index, or its logical position
        const int rpos = p.page_pos ? spos : tok;
        ptx::bulk_load(grows + slot * C::kRopeRowBytes,
                       reinterpret_cast<const float4*>(p.rope) + size_t(rpos) * C::kRopeRowF4,
                       C::kRopeRowBytes, bar, pol_rope);
      }
      // HND pools: row (page * Hk + head) * P + slot; NHD: token row page * P + slot
      // and the head as the map's outer coordinate
      const int trow = page * p.P + (tok & (p.P - 1));
      if constexpr (D == 128) {
        // one box per tile: both 64-column blocks, [block][16 rows][128 B]
        if (p.nhd) {
          ptx::tma_load_4d(dk, &tm_k, bar, 0, trow, 0, pi.kvh, pol);
          ptx::tma_load_4d(dv, &tm_v, bar, 0, trow, 0, pi.kvh, pol);
        } else {
          ptx::tma_load_3d(dk, &tm_k, bar, 0, row, 0, pol);
          ptx::tma_load_3d(dv, &tm_v, bar, 0, row, 0, pol);
        }
      } else {
        if (p.nhd) {
          ptx::tma_load_3d(dk, &tm_k, bar, 0, trow, pi.kvh, pol);
          ptx::tma_load_3d(dv, &tm_v, bar, 0, trow, pi.kvh, pol);
        } else {
          ptx::tma_load_2d(dk, &tm_k, bar, 0, row, pol);
          ptx::tma_load_2d(dv, &tm_v, bar, 0, row, pol);
        }
      }
    }
    ++p_seq;
    ++p_st;
    if (p_st == p_nst) {
      ++p_q;
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

  if (!SMALLP) producer_seek();
  if (early) pdl_wait();
  if (!may_take) {
    may_take = true;
    if (!SMALLP && !p_have) producer_seek();
  }
  if (!SMALLP) {
#pragma unroll 1
    for (int i = 0; i < C::kStages; ++i) producer_issue();
  }

  // ------------------------------------------------------------------ consumer
  // Per-lane smem addressing for ldmatrix (see tile_off):
  //  K (x4, non-trans): matrix mi = lane/8 covers tokens (mi/2)*8.., columns +(mi%2)*8
  //  V (x4, trans):     matrix mi covers tokens (mi%2)*8.., columns +(mi/2)*8
  const int k_tok = ((lane >> 4) << 3) + (lane & 7), k_hb = (lane >> 3) & 1;
  const int v_tok = (((lane >> 3) & 1) << 3) + (lane & 7), v_hb = lane >> 4;
  constexpr float kLn2 = 0.69314718055994530942f;

  uint32_t c_seq = 0;
  bool failed = false;
#pragma unroll 1
  for (int c_q = 0; c_q < p_end; ++c_q) {
    // the producer has placed position c_q (or found the end) before the consumer
    // gets here: it moves past a unit as soon as it has issued its last stage
    const DecodeItem ci = load_item(p.items, item_at(c_q));
    const int nst = stages_of(ci);
    const int group = p.group;
    const int rA = ci.row0 + g4, rB = ci.row0 + g4 + 8;
    const bool vA = g4 < ci.nrows, vB = R16 && (g4 + 8 < ci.nrows);
    const int qposA = ci.qpos0 + rA / group, qposB = ci.qpos0 + rB / group;
    const int qpos_min = ci.qpos0 + ci.row0 / group;
    // RoPE with per-page positions: queries sit after the request's last logical key
    const int qsh = (ROPE && p.qshift != nullptr) ? __ldg(p.qshift + ci.req) : 0;
    // sliding window: row r sees keys >= its position - window_left + 1; the last
    // row's bound is the highest, so a stage at or above it is unmasked for all rows
    // (compiled in only for WIN: the predicates cost a few percent in the hot loop)
    const int wlo_A = WIN ? qposA - p.window_left + 1 : 0;
    const int wlo_B = WIN ? qposB - p.window_left + 1 : 0;
    const int wlo_max = WIN ? ci.qpos0 + (ci.row0 + ci.nrows - 1) / group - p.window_left + 1 : 0;
    const int wlo_min = WIN ? qpos_min - p.window_left + 1 : 0;

    // q fragments (A operand): regs [0] and [NR/2] hold row g4 (columns 2t4.. and
    // 8+2t4..); with R16 regs [1] and [3] hold row g4 + 8.
    // With RoPE the rotated q and k are fp16 operands scaled by 2^-4 (11
    // significant bits; the scale keeps values up to 2^20 in range).
    uint32_t qh[KS][NR];
    {
      const uint16_t* qa =
          p.q + (size_t(ci.q_row0 + rA / group) * p.Hq + ci.kvh * group + rA % group) * D;
      const uint16_t* qb =
          p.q + (size_t(ci.q_row0 + rB / group) * p.Hq + ci.kvh * group + rB % group) * D;
      uint32_t raw[KS][NR];
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int d0 = 16 * ks + 2 * t4;
        raw[ks][0] = vA ? __ldg(reinterpret_cast<const uint32_t*>(qa + d0)) : 0u;
        raw[ks][NR / 2] = vA ? __ldg(reinterpret_cast<const uint32_t*>(qa + d0 + 8)) : 0u;
        if constexpr (R16) {
          raw[ks][1] = vB ? __ldg(reinterpret_cast<const uint32_t*>(qb + d0)) : 0u;
          raw[ks][3] = vB ? __ldg(reinterpret_cast<const uint32_t*>(qb + d0 + 8)) : 0u;
        }
      }
      if constexpr (!ROPE) {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
          for (int r = 0; r < NR; ++r) qh[ks][r] = raw[ks][r];
      } else {
        // rotate the (ks, ks + KH) pairs at the query positions of rows g4 / g4 + 8
#pragma unroll
        for (int rr = 0; rr < (R16 ? 2 : 1); ++rr) {
          const int pos = (rr == 0 ? qposA : qposB) + qsh;
          const bool ok = rr == 0 ? vA : vB;
          const int tpos = ok ? min(max(pos, 0), p.rope_max_pos) : 0;
          const float4* tab =
              reinterpret_cast<const float4*>(p.rope) + size_t(tpos) * C::kRopeRowF4 + t4;
          const int r0 = rr == 0 ? 0 : 1, r1 = rr == 0 ? NR / 2 : 3;
#pragma unroll
          for (int ks = 0; ks < KH; ++ks) {
            const float4 c01 = __ldg(tab + 8 * ks), c23 = __ldg(tab + 8 * ks + 4);
            float x[2], y[2];
            rope_pair(raw[ks][r0], raw[ks + KH][r0], make_float2(c01.x, c01.y),
                      make_float2(c01.z, c01.w), x, y);
            qh[ks][r0] = ptx::pack_f16(x[0] * kRopeOperandScale, x[1] * kRopeOperandScale);
            qh[ks + KH][r0] = ptx::pack_f16(y[0] * kRopeOperandScale, y[1] * kRopeOperandScale);
            rope_pair(raw[ks][r1], raw[ks + KH][r1], make_float2(c23.x, c23.y),
                      make_float2(c23.z, c23.w), x, y);
            qh[ks][r1] = ptx::pack_f16(x[0] * kRopeOperandScale, x[1] * kRopeOperandScale);
            qh[ks + KH][r1] = ptx::pack_f16(y[0] * kRopeOperandScale, y[1] * kRopeOperandScale);
          }
        }
      }
    }

    float o[NT][NR];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int r = 0; r < NR; ++r) o[n][r] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

#pragma unroll 1
    for (int st = 0; st < nst; ++st) {
      const int slot = SMALLP ? 0 : int(c_seq % C::kStages);
      const uint32_t kt = ring + uint32_t(slot * C::kStageBytes), vt = kt + C::kStageKBytes;
      const int tok = ci.tok0 + kStageTokens * st;
      const int nvalid = min(kStageTokens, ci.tok1 - tok);
      if constexpr (SMALLP) {
        // Page size below the stage: gather the stage's tokens with plain 16-byte loads.
        const uint16_t* kp = static_cast<const uint16_t*>(p.k_pages);
        const uint16_t* vp = static_cast<const uint16_t*>(p.v_pages);
#pragma unroll 1
        for (int idx = lane; idx < nvalid * (D / 8); idx += 32) {
          const int t = idx / (D / 8), c = idx % (D / 8);
          const int key = tok + t;
          uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
          // keys older than every row's window: their page may be recycled, not read
          if (!WIN || key >= wlo_min) {
            const int page = __ldg(p.indices + ci.page_base + (key >> log2P));
            const size_t off =
                (p.nhd ? size_t(page * p.P + (key & (p.P - 1))) * p.Hk + ci.kvh
                       : size_t(page * p.Hk + ci.kvh) * p.P + (key & (p.P - 1))) * D + c * 8;
            kv = __ldg(reinterpret_cast<const uint4*>(kp + off));
            vv = __ldg(reinterpret_cast<const uint4*>(vp + off));
          }
          const uint32_t to = tile_off(t, c * 8);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(kt + to), "r"(kv.x),
                       "r"(kv.y), "r"(kv.z), "r"(kv.w)
                       : "memory");
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(vt + to), "r"(vv.x),
                       "r"(vv.y), "r"(vv.z), "r"(vv.w)
                       : "memory");
        }
        if constexpr (ROPE) {
          if (lane < C::kRopeRowF4)
            reinterpret_cast<float4*>(goff_ptr)[lane] =
                __ldg(reinterpret_cast<const float4*>(p.rope) + size_t(tok) * C::kRopeRowF4 + lane);
        }
      } else {
        if (!ptx::mbar_wait_bounded(bars + 8 * slot, (c_seq / C::kStages) & 1u, p.wait_limit_ns)) {
          failed = true;
          break;
        }
      }
      if (nvalid < kStageTokens) {
        // Rows past the valid keys may hold another page's tail or stale bits
        // (NaN included): zero V there so that P = 0 contributes exactly 0.
#pragma unroll 1
        for (int idx = lane; idx < (kStageTokens - nvalid) * (D / 8); idx += 32) {
          const int t = nvalid + idx / (D / 8), c = idx % (D / 8);
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vt + tile_off(t, c * 8)),
                       "r"(0u)
                       : "memory");
        }
      }
      __syncwarp();

      // ---------------- S = Q K^T  (two n-tiles of 8 keys)
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (!ROPE) {
        float u0[4] = {0.f, 0.f, 0.f, 0.f}, u1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t kb[4];
          ptx::ldsm_x4(kb, kt + tile_off(k_tok, 16 * ks + 8 * k_hb));
          const uint32_t a0 = qh[ks][0], a2 = qh[ks][NR / 2];
          const uint32_t a1 = R16 ? qh[ks][1] : 0u, a3 = R16 ? qh[ks][NR - 1] : 0u;
          if (ks & 1) {
            ptx::mma_bf16(u0[0], u0[1], u0[2], u0[3], a0, a1, a2, a3, kb[0], kb[1]);
            ptx::mma_bf16(u1[0], u1[1], u1[2], u1[3], a0, a1, a2, a3, kb[2], kb[3]);
          } else {
            ptx::mma_bf16(s0[0], s0[1], s0[2], s0[3], a0, a1, a2, a3, kb[0], kb[1]);
            ptx::mma_bf16(s1[0], s1[1], s1[2], s1[3], a0, a1, a2, a3, kb[2], kb[3]);
          }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          s0[r] += u0[r];
          s1[r] += u1[r];
        }
      } else {
        // angle of key tok + t = angle of tok (this stage's table row) + angle of t
        const float4* g = reinterpret_cast<const float4*>(goff_ptr + slot * C::kRopeRowBytes) + t4;
        const float4* fa = reinterpret_cast<const float4*>(frows_ptr + g4 * C::kRopeOffStride) + t4;
        const float4* fb =
            reinterpret_cast<const float4*>(frows_ptr + (g4 + 8) * C::kRopeOffStride) + t4;
#pragma unroll
        for (int ks = 0; ks < KH; ++ks) {
          uint32_t kl[4], kh[4];
          ptx::ldsm_x4(kl, kt + tile_off(k_tok, 16 * ks + 8 * k_hb));
          ptx::ldsm_x4(kh, kt + tile_off(k_tok, 16 * (ks + KH) + 8 * k_hb));
          const float4 g01 = g[8 * ks], g23 = g[8 * ks + 4];
          uint32_t lh[4], hh[4];
          // kl[0], kl[1]: key g4 (n-tile 0); kl[2], kl[3]: key 8 + g4 (n-tile 1)
          const float4 cs01[4] = {rot_compose(g01, fa[8 * ks]), rot_compose(g23, fa[8 * ks + 4]),
                                  rot_compose(g01, fb[8 * ks]), rot_compose(g23, fb[8 * ks + 4])};
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            float x[2], y[2];
            rope_pair(kl[r], kh[r], make_float2(cs01[r].x, cs01[r].y),
                      make_float2(cs01[r].z, cs01[r].w), x, y);
            lh[r] = ptx::pack_f16(x[0] * kRopeOperandScale, x[1] * kRopeOperandScale);
            hh[r] = ptx::pack_f16(y[0] * kRopeOperandScale, y[1] * kRopeOperandScale);
          }
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int kk = half == 0 ? ks : ks + KH;
            const uint32_t* bh = half == 0 ? lh : hh;
            const uint32_t h0 = qh[kk][0], h2 = qh[kk][NR / 2];
            const uint32_t h1 = R16 ? qh[kk][1] : 0u, h3 = R16 ? qh[kk][NR - 1] : 0u;
            ptx::mma_f16(s0[0], s0[1], s0[2], s0[3], h0, h1, h2, h3, bh[0], bh[1]);
            ptx::mma_f16(s1[0], s1[1], s1[2], s1[3], h0, h1, h2, h3, bh[2], bh[3]);
          }
        }
      }

      // ---------------- mask + online softmax (log2 domain)
      // s*[0..1]: row g4, keys tok + {0,8} + 2t4 + {0,1};  s*[2..3]: row g4 + 8
      const bool full = (nvalid == kStageTokens) &&
                        (!p.causal || tok + kStageTokens - 1 <= qpos_min) &&
                        (!WIN || tok >= wlo_max);
      float xa[4], xb[4];
      {
        // with RoPE both operands carry 2^-4
        const float sc = ROPE ? p.scale_log2 * (1.f / (kRopeOperandScale * kRopeOperandScale))
                              : p.scale_log2;
        const int k0 = tok + 2 * t4;
        const int kidx[4] = {k0, k0 + 1, k0 + 8, k0 + 9};
        const float sa[4] = {s0[0], s0[1], s1[0], s1[1]};
        const float sb[4] = {s0[2], s0[3], s1[2], s1[3]};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool inr = full || (kidx[j] < ci.tok1);
          const bool okA =
              full || (inr && (!p.causal || kidx[j] <= qposA) && (!WIN || kidx[j] >= wlo_A));
          const bool okB =
              full || (inr && (!p.causal || kidx[j] <= qposB) && (!WIN || kidx[j] >= wlo_B));
          xa[j] = okA ? sa[j] * sc : -INFINITY;
          xb[j] = okB ? sb[j] * sc : -INFINITY;
        }
      }
      float mxA = fmaxf(fmaxf(xa[0], xa[1]), fmaxf(xa[2], xa[3]));
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
      mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
      const float mnA = fmaxf(mA, mxA);
      const float muA = mnA == -INFINITY ? 0.f : mnA;
      const float alA = ptx::ex2(mA - muA);
      mA = mnA;
      float pa[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) pa[j] = ptx::ex2(xa[j] - muA);
      lA = lA * alA + ((pa[0] + pa[1]) + (pa[2] + pa[3]));
      float alB = 1.f;
      float pb[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (R16) {
        float mxB = fmaxf(fmaxf(xb[0], xb[1]), fmaxf(xb[2], xb[3]));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
        mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
        const float mnB = fmaxf(mB, mxB);
        const float muB = mnB == -INFINITY ? 0.f : mnB;
        alB = ptx::ex2(mB - muB);
        mB = mnB;
#pragma unroll
        for (int j = 0; j < 4; ++j) pb[j] = ptx::ex2(xb[j] - muB);
        lB = lB * alB + ((pb[0] + pb[1]) + (pb[2] + pb[3]));
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

      // ---------------- O += P V  (P = hi + lo, both bf16)
      uint32_t ph[4], pl[4];
      ptx::split_bf16(pa[0], pa[1], ph[0], pl[0]);
      ptx::split_bf16(pa[2], pa[3], ph[2], pl[2]);
      if constexpr (R16) {
        ptx::split_bf16(pb[0], pb[1], ph[1], pl[1]);
        ptx::split_bf16(pb[2], pb[3], ph[3], pl[3]);
      } else {
        ph[1] = ph[3] = pl[1] = pl[3] = 0u;
      }
#pragma unroll
      for (int np = 0; np < D / 16; ++np) {
        uint32_t vb[4];
        ptx::ldsm_x4_trans(vb, vt + tile_off(v_tok, 16 * np + 8 * v_hb));
        if constexpr (R16) {
          float* e = o[2 * np];
          float* f = o[2 * np + 1];
          ptx::mma_bf16(e[0], e[1], e[NR - 2], e[NR - 1], ph[0], ph[1], ph[2], ph[3], vb[0], vb[1]);
          ptx::mma_bf16(e[0], e[1], e[NR - 2], e[NR - 1], pl[0], pl[1], pl[2], pl[3], vb[0], vb[1]);
          ptx::mma_bf16(f[0], f[1], f[NR - 2], f[NR - 1], ph[0], ph[1], ph[2], ph[3], vb[2], vb[3]);
          ptx::mma_bf16(f[0], f[1], f[NR - 2], f[NR - 1], pl[0], pl[1], pl[2], pl[3], vb[2], vb[3]);
        } else {
          // rows g4 + 8 are padding: their accumulators are dead scratch
          float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;
          ptx::mma_bf16(o[2 * np][0], o[2 * np][1], z0, z1, ph[0], 0u, ph[2], 0u, vb[0], vb[1]);
          ptx::mma_bf16(o[2 * np][0], o[2 * np][1], z0, z1, pl[0], 0u, pl[2], 0u, vb[0], vb[1]);
          ptx::mma_bf16(o[2 * np + 1][0], o[2 * np + 1][1], z2, z3, ph[0], 0u, ph[2], 0u, vb[2], vb[3]);
          ptx::mma_bf16(o[2 * np + 1][0], o[2 * np + 1][1], z2, z3, pl[0], 0u, pl[2], 0u, vb[2], vb[3]);
        }
      }
      __syncwarp();
      if constexpr (!SMALLP) {
        // generic writes (the zero fill) must be ordered before the TMA that reuses the slot
        if (nvalid < kStageTokens) ptx::fence_proxy_async_smem();
        __syncwarp();
        ++c_seq;
        producer_issue();
      }
    }
    if (failed) break;

    // ---------------- epilogue
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    if constexpr (R16) {
      lB += __shfl_xor_sync(0xffffffffu, lB, 1);
      lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    }
    if constexpr (ROPE) {
      // a rotated q or k beyond the fp16 operand range shows as a non-finite row sum
      const bool bad = (vA && !isfinite(lA)) || (vB && !isfinite(lB));
      if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.error, kStatusOperandRange);
    }
    const float lseA = lA > 0.f ? mA + ptx::lg2(lA) : -INFINITY;
    const float lseB = lB > 0.f ? mB + ptx::lg2(lB) : -INFINITY;
    const float invA = lA > 0.f ? 1.f / lA : 0.f;
    const float invB = lB > 0.f ? 1.f / lB : 0.f;
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
          float* dst = static_cast<float*>(p.out) + orow * D + 2 * t4;
#pragma unroll
          for (int n = 0; n < NT; ++n)
            *reinterpret_cast<float2*>(dst + 8 * n) =
                make_float2(o[n][c0] * inv, o[n][c0 + 1] * inv);
        } else {
          uint16_t* dst = static_cast<uint16_t*>(p.out) + orow * D + 2 * t4;
#pragma unroll
          for (int n = 0; n < NT; ++n)
            *reinterpret_cast<uint32_t*>(dst + 8 * n) =
                ptx::pack_bf16(o[n][c0] * inv, o[n][c0 + 1] * inv);
        }
        if (p.lse != nullptr && t4 == 0) p.lse[orow] = (rr == 0 ? lseA : lseB) * kLn2;
      }
    } else {
#pragma unroll
      for (int rr = 0; rr < (R16 ? 2 : 1); ++rr) {
        const int r = g4 + 8 * rr;
        const float inv = rr == 0 ? invA : invB;
        const int c0 = rr == 0 ? 0 : NR - 2;
        float* dst = p.part_o + (size_t(ci.slot) * kMaxDecodeRows + r) * D + 2 * t4;
#pragma unroll
        for (int n = 0; n < NT; ++n)
          __stcg(reinterpret_cast<float2*>(dst + 8 * n),
                 make_float2(o[n][c0] * inv, o[n][c0 + 1] * inv));
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

  if (failed) {
    if (lane == 0) atomicOr(p.error, 1);
    if (dyn && !took_last) done_taking();   // the queue's count of finished warps stays exact
    // let the copies this warp still has in flight land before the CTA exits
#pragma unroll 1
    for (uint32_t s = c_seq; s < p_seq; ++s)
      ptx::mbar_wait_bounded(bars + 8 * (s % C::kStages), (s / C::kStages) & 1u, 50000000ull);
  }
}

}  // namespace bsr
