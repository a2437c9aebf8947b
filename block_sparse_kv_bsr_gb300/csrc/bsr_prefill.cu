// Prefill / multi-query attention over a paged (BSR) KV cache on the sm_103a
// tensor cores (tcgen05 + TMEM), head_dim 128.
//
// Prefill is compute-bound ("FlashInfer: Block-Sparse KV 캐시로 어텐션 병목을
// 해소하다", section "어텐션 연산에서 진짜 병목은 어디인가?"): many query rows
// share every key, so the work is a real dense contraction.  One work unit is
// up to 256 packed (query, head) rows of one (request, kv head) -- two 128-row
// query tiles -- against a page-aligned key range; a CTA walks its planned
// list of units.  Both query tiles consume the same key tiles, so each K/V
// tile is staged once for 256 rows, and while the softmax of one query tile
// runs, the tensor cores work on the other's products.
//
// Roles (576 threads; 704 with RoPE):
//   warps 0-15 softmax, two threads per row: warp w works on query tile w / 8,
//              key/column half (w / 4) % 2 and row quarter w % 4 (the TMEM lanes
//              it may access).  Each half reads its 64 scores of a row from TMEM,
//              the halves swap their partial max (and at the end their partial
//              sum) through shared memory and an mbarrier, then each writes its
//              half of P (fp16) over S columns it has already read, rescales its
//              64 O columns in TMEM when the running max grows by more than 2^8,
//              and writes out / lse (or the fp32 partial state of a split key
//              range, combined afterwards by bsr_prefill_merge_kernel).  Between
//              handing over P of key tile j and waiting for the scores of tile
//              j + 1 -- time they would otherwise spend idle -- they turn V of tile
//              j + 1 into fp16 in place: P enters P V as fp16 (11 significant bits),
//              because rows that see only a few keys, such as the first rows of a
//              causal prompt, cannot average out the rounding of a bf16 P.  Rows past
//              the last key of a ragged tile are zeroed there (they may hold another
//              page's tail, NaN included, and P = 0 must contribute exactly 0).
//   warp 16    TMA producer, the whole warp: each unit's query tiles (one box per
//              64 columns: whole queries of the kv head's group, straight from q)
//              as soon as the previous unit's last Q K^T has read them, and a FIFO
//              ring of 32 KB stages with the K and V tiles of every key tile in
//              turn (K(j), V(j), K(j+1), ...), gathered box by box from `indices`
//              (inactive blocks are absent, "Block-Sparse 포맷") into one row-group
//              layout, 128B-swizzled: one box per page-sized piece with both column
//              blocks (a 4 KB box for 16-token pages where per-block boxes would be
//              2 KB: the copy engine's cost is mostly per box).  Lane b fetches box
//              b's page id two key tiles ahead.
//   warp 17    allocates TMEM and issues the MMAs: S_i = Q_i K^T (M 128, N 128,
//              K-major operands from shared memory) and O_i += P_i V (P from
//              TMEM, V MN-major from shared memory), i = 0, 1.
//   warps 18-21 (RoPE) rotate every query tile and every K tile in shared memory
//              once its copy has landed and before the MMA reads it -- RoPE fused
//              into the attention kernel, so rotated keys never go back to global
//              memory ("JIT 컴파일은 어텐션을 어떻게 빠르게 만드는가?") -- and write
//              them in place as fp16 scaled by 2^-4, the operand type of the RoPE
//              Q K^T.
// TMEM columns: S_0 | S_1 | O_0 | O_1, 128 fp32 columns each; P_i (fp16 pairs)
// overwrites columns 0-31 and 64-95 of S_i.  MMAs run in issue order, so the
// Q K^T of the next key tile may be queued right behind the P V that reads P_i.
// Every mbarrier wait is bounded and warp-agreed.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <type_traits>

#include "bsr_internal.h"
#include "bsr_launch.cuh"
#include "bsr_schedule.h"
#include "ptx.cuh"
#include "umma.cuh"

namespace bsr {
namespace {

constexpr int D = 128;                      // width of the tile program (head_dim 64 runs it with zeros above)
constexpr int kTileM = 128;                 // rows per query tile (TMEM lanes)
constexpr int kUnitRows = kPrefillRows;     // two query tiles
constexpr int kTileN = kPrefillKeyTile;     // keys per key tile
constexpr int kHalfBytes = kTileN * 128;    // one 64-column block of a 128-row tile: 16 KB
constexpr int kTileBytes = 2 * kHalfBytes;
constexpr int kStages = 4;                  // K/V ring depth (32 KB stages)
constexpr uint32_t kTmemCols = 512;
constexpr int kSoftmaxWarps = 16;           // two per row quarter and query tile
constexpr int kProducerWarp = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + 1;
// RoPE warps (the RoPE variant only) rotate the query and K tiles.
constexpr int kRotWarp0 = kSoftmaxWarps + 2, kRotWarps = 4;
constexpr int kRotThreads = 32 * kRotWarps;
template <bool ROPE>
constexpr int threads_of() { return 32 * (kSoftmaxWarps + 2 + (ROPE ? kRotWarps : 0)); }
static_assert(kUnitRows == 2 * kTileM, "a unit is two query tiles");
// A rotating thread takes one 16-byte chunk (8 frequencies) of 8 consecutive rows of a
// tile: 16 row blocks x 8 chunks = 128 threads, a row block inside one 16-key group.
static_assert(kRotThreads == (kTileN / 8) * 8 && kTileM == kTileN, "RoPE thread map");
constexpr int kVChunks = kTileBytes / 16;    // 16-byte chunks of a V stage
// Largest magnitude of an fp16 tensor-core operand.
constexpr float kF16Max = 65504.f;

struct Smem {
  static constexpr int kQ = 0;                               // Q_0, Q_1
  static constexpr int kRing = 2 * kTileBytes;
  // row-half exchange: [parity][query tile][half][row] fp32
  static constexpr int kXchData = kRing + kStages * kTileBytes;
  // RoPE: cos / sin of t * omega_f for t < 16, times the operand scale, as
  // [t][frequency pair within the chunk][chunk] float4 (cos_f, sin_f, cos_f+1, sin_f+1)
  static constexpr int kRopeT = kXchData + 2 * 2 * 2 * kTileM * 4;
  static constexpr int kBars = kRopeT + 16 * (D / 2) * 8;
  // full[kStages], empty[kStages], s_full[2], p_full[2], o_full[2], q_full[2], q_empty[2],
  // drain, xch[2][4] (query tile, row quarter), ready[kStages] (the operand warps are
  // done with a stage: every V stage, and with RoPE every K stage), q_rot[2] (RoPE)
  static constexpr int kFull = 0, kEmpty = kStages, kSFull = 2 * kStages, kPFull = kSFull + 2,
                       kOFull = kPFull + 2, kQFull = kOFull + 2, kQEmpty = kQFull + 2,
                       kDrain = kQEmpty + 2, kXch = kDrain + 1, kReady = kXch + 8,
                       kQRot = kReady + kStages;
  static constexpr int kNumBars = kQRot + 2;
  static constexpr int kTmemSlot = kBars + 8 * kNumBars;
  static constexpr int kFlags = kTmemSlot + 16;   // abort flag
  static constexpr int kTotal = kFlags + 16;
  static constexpr size_t kDynBytes = size_t(kTotal) + 1024;
  static_assert(kDynBytes <= 232448, "prefill tiles exceed the shared memory of one SM");
};

struct Waiter {
  uint32_t abort_flag;  // smem address of the shared abort word
  uint64_t limit;
  int32_t* error;
  // Wait for a barrier phase; false when this CTA is aborting (timeout here or elsewhere).
  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
#pragma unroll 1
      for (int i = 0; i < 16; ++i)
        if (ptx::mbar_try_wait(bar, parity)) return true;
      uint32_t ab;
      asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(ab) : "r"(abort_flag));
      if (ab) return false;
      if (ptx::globaltimer_ns() - t0 > limit) {
        asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(abort_flag), "r"(1u));
        atomicOr(error, kStatusWaitTimeout);
        return false;
      }
    }
  }
  // All lanes wait; the warp proceeds only if every lane saw the phase complete.
  __device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) const {
    return __all_sync(0xffffffffu, wait(bar, parity));
  }
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ int ntiles_of(const DecodeItem& it) {
  return it.tok1 > it.tok0 ? (it.tok1 - it.tok0 + kTileN - 1) / kTileN : 0;
}

// Row of `out` (and `lse`) of packed row R of a unit: query R / group of the
// request, head kvh * group + R % group.
__device__ __forceinline__ size_t out_row(const DecodeItem& it, int R, int group, int Hq) {
  return size_t(it.q_row0 + R / group) * Hq + it.kvh * group + R % group;
}

// Write 32 columns (chunk c) of one output row as bf16 or fp32; 32-byte stores
// (one full sector per thread) when `out` allows them.
__device__ __forceinline__ void store_row_chunk(const PrefillParams& p, size_t orow, int c,
                                                const float (&v)[32]) {
  if (p.out_f32) {
    float* dst = static_cast<float*>(p.out) + orow * size_t(p.head_dim) + 32 * c;
    if (p.out_v8) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        ptx::st_global_v8(dst + 8 * i, __float_as_uint(v[8 * i]), __float_as_uint(v[8 * i + 1]),
                          __float_as_uint(v[8 * i + 2]), __float_as_uint(v[8 * i + 3]),
                          __float_as_uint(v[8 * i + 4]), __float_as_uint(v[8 * i + 5]),
                          __float_as_uint(v[8 * i + 6]), __float_as_uint(v[8 * i + 7]));
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        reinterpret_cast<float4*>(dst)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  } else {
    uint16_t* dst = static_cast<uint16_t*>(p.out) + orow * size_t(p.head_dim) + 32 * c;
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = ptx::pack_bf16(v[2 * i], v[2 * i + 1]);
    if (p.out_v8) {
#pragma unroll
      for (int i = 0; i < 2; ++i)
        ptx::st_global_v8(dst + 16 * i, w[8 * i], w[8 * i + 1], w[8 * i + 2], w[8 * i + 3],
                          w[8 * i + 4], w[8 * i + 5], w[8 * i + 6], w[8 * i + 7]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        reinterpret_cast<uint4*>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
  }
}

// (cos, sin) of the frequency pairs (8 ch + 2 e, 8 ch + 2 e + 1), e < 4, of one chunk.
struct Angles {
  float2 c[4], s[4];
};

// Angles of chunk ch at table row `pos` (four float4 of the pair-order table, whose
// rows hold head_dim / 4 float4).
__device__ __forceinline__ Angles load_angles(const float4* rope, int pos, int ch, int row_f4) {
  const float4* row = rope + size_t(pos) * row_f4 + 4 * ch;
  Angles an;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float4 v = __ldg(row + e);
    an.c[e] = make_float2(v.x, v.y);
    an.s[e] = make_float2(v.z, v.w);
  }
  return an;
}

// Rotate dimensions 8 ch .. 8 ch + 7 of row r of a 128B-swizzled bf16 tile together
// with their rotate-half partners, two frequencies per packed instruction, and write
// both back in place as fp16.  With head_dim 128 the partners are 64 further (the same
// bytes of the other column block); with 64 (D64, ch < 4) they are 32 further, chunk
// ch + 4 of the same 128-byte row.  A query tile is [2 column blocks][128 rows][128 B];
// a key tile (GROUPED) is [16 row groups][2 column blocks][8 rows][128 B].  The angles
// are already times the operand scale.  Returns the largest magnitude written.
template <bool GROUPED, bool D64>
__device__ __forceinline__ float rotate_row_chunk(uint32_t tile, int r, int ch, const Angles& an) {
  const uint32_t rowb = GROUPED ? tile + uint32_t(r >> 3) * 2048u + uint32_t(r & 7) * 128u
                                : tile + uint32_t(r) * 128u;
  const uint32_t lo = rowb + (uint32_t(ch ^ (r & 7)) << 4);
  const uint32_t hi = D64 ? rowb + (uint32_t((ch + 4) ^ (r & 7)) << 4)
                          : lo + (GROUPED ? 1024u : uint32_t(kHalfBytes));
  uint32_t a[4], b[4];
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]) : "r"(lo));
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]) : "r"(hi));
  float m = 0.f;
  uint32_t xo[4], yo[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = make_float2(ptx::bf16_lo(a[e]), ptx::bf16_hi(a[e]));
    const float2 y = make_float2(ptx::bf16_lo(b[e]), ptx::bf16_hi(b[e]));
    const float2 u = ptx::fsub2(ptx::fmul2(x, an.c[e]), ptx::fmul2(y, an.s[e]));
    const float2 v = ptx::ffma2(y, an.c[e], ptx::fmul2(x, an.s[e]));
    m = ptx::fmax3(m, fabsf(u.x), fabsf(u.y));
    m = ptx::fmax3(m, fabsf(v.x), fabsf(v.y));
    xo[e] = ptx::pack_f16(u.x, u.y);
    yo[e] = ptx::pack_f16(v.x, v.y);
  }
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
               ::"r"(lo), "r"(xo[0]), "r"(xo[1]), "r"(xo[2]), "r"(xo[3]) : "memory");
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
               ::"r"(hi), "r"(yo[0]), "r"(yo[1]), "r"(yo[2]), "r"(yo[3]) : "memory");
  return m;
}

// One CTA per SM.  Each of the 4 SM sub-partitions holds a quarter of the register
// file (16K registers) and up to 6 of the 22 warps of the RoPE variant, so 80
// registers per thread is its ceiling (96 for the 18 warps without RoPE).
// D64: head_dim 64 with RoPE (its rotation pairs lie 32 apart); head_dim 64 without
// RoPE needs nothing of its own beyond the run-time output width.
template <bool ROPE, bool WIN, bool D64>
__global__ void __launch_bounds__(threads_of<ROPE>()) __maxnreg__(ROPE ? 80 : 96)
    bsr_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using L = Smem;
  extern __shared__ uint8_t smem_raw[];
  // launched as a programmatic dependent (see bsr_launch.cuh): the set-up below --
  // barriers, TMEM, the plan's CTA ranges (written by the plan's host copy) -- overlaps
  // the previous grid's tail; everything after it waits for that grid
  pdl_trigger();
  const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar0 = base + L::kBars;
  auto BAR = [&](int i) { return bar0 + 8u * uint32_t(i); };
  auto FULL = [&](uint32_t c) { return BAR(L::kFull + int(c % kStages)); };
  auto EMPTY = [&](uint32_t c) { return BAR(L::kEmpty + int(c % kStages)); };
  auto STAGE = [&](uint32_t c) { return base + L::kRing + (c % kStages) * uint32_t(kTileBytes); };
  auto PHASE = [&](uint32_t c) { return (c / kStages) & 1u; };
  const uint32_t abort_addr = base + L::kFlags;
  Waiter wt{abort_addr, p.wait_limit_ns, p.error};

  const int u_begin = __ldg(p.cta_ptr + blockIdx.x), u_end = __ldg(p.cta_ptr + blockIdx.x + 1);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      ptx::mbar_init(BAR(L::kFull + i), 1);
      ptx::mbar_init(BAR(L::kEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(BAR(L::kSFull + i), 1);
      ptx::mbar_init(BAR(L::kPFull + i), kSoftmaxWarps / 2);   // one arrival per warp of the tile
      ptx::mbar_init(BAR(L::kOFull + i), 1);
      ptx::mbar_init(BAR(L::kQFull + i), 1);
      ptx::mbar_init(BAR(L::kQEmpty + i), 1);
    }
    ptx::mbar_init(BAR(L::kDrain), 1);
    for (int i = 0; i < 8; ++i) ptx::mbar_init(BAR(L::kXch + i), 2);   // the two halves of a row quarter
    // ready: K stages sit at even ring positions (one arrival per RoPE warp), V stages
    // at odd ones (arrivals of the softmax warps: 16 in all per use)
    for (int i = 0; i < kStages; ++i)
      ptx::mbar_init(BAR(L::kReady + i), (i & 1) ? kSoftmaxWarps : kRotWarps);
    for (int i = 0; i < 2; ++i) ptx::mbar_init(BAR(L::kQRot + i), kRotWarps);
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(abort_addr), "r"(0u));
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tm_q);
    ptx::prefetch_tensormap(&tm_k);
    ptx::prefetch_tensormap(&tm_v);
  }
  if (warp == kMmaWarp) {
    umma::tmem_alloc(base + L::kTmemSlot, kTmemCols);
    umma::tmem_relinquish();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  pdl_wait();
  uint32_t tmem;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(base + L::kTmemSlot));
  auto S_T = [&](int i) { return tmem + 128u * uint32_t(i); };
  auto O_T = [&](int i) { return tmem + 256u + 128u * uint32_t(i); };
  auto Q_S = [&](int i) { return base + L::kQ + uint32_t(i) * kTileBytes; };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop: lane 0 waits on the ring and posts the byte
    // counts, lane b gathers box b of a paged key tile, and each lane fetches its
    // box's page id two tiles ahead, so no page-table load is on the issue path.
    // K/V tiles are re-read by the other row units of the same (request, kv head),
    // which run concurrently on other SMs: keep them in L2 at normal priority.
    // Query tiles are read once.
    const uint64_t pol = ptx::policy_evict_normal();
    const uint64_t pol_q = ptx::policy_evict_first();
    uint32_t c = 0, nq0 = 0, nq1 = 0;
    bool ok = true;
    // lane 0 waits; the warp goes on only if the wait succeeded
    auto ring_wait = [&](uint32_t bar, uint32_t parity) -> bool {
      bool r = true;
      if (lane == 0) r = wt.wait(bar, parity);
      return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
    };
    // query tile i of a unit, once the previous unit's last Q K^T has read the buffer
    auto load_q = [&](int i, uint32_t& nq, const DecodeItem& it) -> bool {
      if (nq > 0 && !ring_wait(BAR(L::kQEmpty + i), (nq - 1) & 1u)) return false;
      ++nq;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(BAR(L::kQFull + i), uint32_t(kTileBytes));
        const int q0 = it.q_row0 + (it.row0 + kTileM * i) / p.group;
        for (int h = 0; h < 2; ++h)
          ptx::tma_load_4d(Q_S(i) + h * kHalfBytes, &tm_q, BAR(L::kQFull + i), 0, h,
                           it.kvh * p.group, q0, pol_q);
      }
      return true;
    };
    // K/V come in boxes of R = min(P, 128) rows (R and P powers of two): one page
    // holds a whole box, and a key tile (its start a multiple of max(P, 128)) is
    // 128 / R boxes
    const int lr = 31 - __clz(p.box_rows), lp = 31 - __clz(p.P);
    const uint32_t box_bytes = 128u << lr;
    auto boxes_of = [&](const DecodeItem& it, int j) {
      return (min(kTileN, it.tok1 - it.tok0 - kTileN * j) + p.box_rows - 1) >> lr;
    };
    auto page_of = [&](const DecodeItem& it, int j, int nsub) {
      return lane < nsub ? __ldg(p.indices + it.page_base + ((it.tok0 + kTileN * j + (lane << lr)) >> lp))
                         : 0;
    };
    // gather the paged boxes of key tile j into the stage of ring position cc (lane b:
    // box b).  K and V tiles alike land in the row-group layout, one copy per box.
    int last_pos[kStages];
#pragma unroll
    for (int sl = 0; sl < kStages; ++sl) last_pos[sl] = -1;
    auto issue_paged = [&](uint32_t cc, const CUtensorMap* tm, const DecodeItem& it, int j,
                           int nsub, int page) {
      if (lane == 0) ptx::mbar_arrive_expect_tx(FULL(cc), uint32_t(nsub) * 2u * box_bytes);
      __syncwarp();
      if (lane < nsub) {
        const int key = it.tok0 + kTileN * j + (lane << lr);
        // HND pools: row (page * Hk + head) * P + slot; NHD: token row page * P + slot
        // with the head as the map's outer coordinate
        const int row = p.nhd ? page * p.P + (key & (p.P - 1))
                              : (page * p.Hk + it.kvh) * p.P + (key & (p.P - 1));
        const uint32_t dst = STAGE(cc) + uint32_t(lane) * 2u * box_bytes;
        if (p.nhd) ptx::tma_load_5d(dst, tm, FULL(cc), 0, 0, 0, row >> 3, it.kvh, pol);
        else ptx::tma_load_4d(dst, tm, FULL(cc), 0, 0, 0, row >> 3, pol);
      }
      last_pos[cc % kStages] = int(cc);
    };
    // K(j) sits at ring position base + 2 j and V(j) at base + 2 j + 1, issued in
    // that order (issuing K(j + 1) ahead of V(j) measured slower)
    auto issue = [&](uint32_t cc, const CUtensorMap* tm, const DecodeItem& it, int j, int nsub,
                     int page) {
      if (cc >= kStages && !ring_wait(EMPTY(cc), PHASE(cc) ^ 1u)) return false;
      issue_paged(cc, tm, it, j, nsub, page);
      return true;
    };
    for (int u = u_begin; u < u_end && ok; ++u) {
      const DecodeItem it = p.items[u];
      const int nt = ntiles_of(it);
      if (nt == 0) continue;
      const uint32_t c0 = c;
      int nsub0 = boxes_of(it, 0), page0 = page_of(it, 0, nsub0);
      int nsub1 = nt > 1 ? boxes_of(it, 1) : 0, page1 = nt > 1 ? page_of(it, 1, nsub1) : 0;
      if (!issue(c0, &tm_k, it, 0, nsub0, page0) || !load_q(0, nq0, it) ||
          (it.nrows > kTileM && !load_q(1, nq1, it))) { ok = false; break; }
      for (int j = 0; j < nt; ++j) {
        int nsub2 = 0, page2 = 0;
        if (j + 2 < nt) {
          nsub2 = boxes_of(it, j + 2);
          page2 = page_of(it, j + 2, nsub2);
        }
        if (j > 0 && !issue(c0 + 2u * uint32_t(j), &tm_k, it, j, nsub0, page0)) {
          ok = false;
          break;
        }
        if (!issue(c0 + 2u * uint32_t(j) + 1u, &tm_v, it, j, nsub0, page0)) { ok = false; break; }
        nsub0 = nsub1, page0 = page1, nsub1 = nsub2, page1 = page2;
      }
      c = c0 + 2u * uint32_t(nt);
    }
    // on abort, let the copies still in flight land before shared memory is released:
    // a slot's earlier positions completed before the slot was reissued, so its latest
    // issued position is the only one that can be outstanding
    if (!ok && lane == 0) {
      for (int sl = 0; sl < kStages; ++sl)
        if (last_pos[sl] >= 0)
          ptx::mbar_wait_bounded(FULL(uint32_t(last_pos[sl])), PHASE(uint32_t(last_pos[sl])),
                                 50000000ull);
      if (nq0 > 0) ptx::mbar_wait_bounded(BAR(L::kQFull), (nq0 - 1) & 1u, 50000000ull);
      if (nq1 > 0) ptx::mbar_wait_bounded(BAR(L::kQFull + 1), (nq1 - 1) & 1u, 50000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = ROPE ? umma::idesc_f16_f32(kTileM, kTileN, 0, 0)
                                         : umma::idesc_bf16_f32(kTileM, kTileN, 0, 0);
      constexpr uint32_t idesc_pv = umma::idesc_f16_f32(kTileM, D, 0, 1);
      uint32_t c = 0;
      uint32_t nq[2] = {0, 0}, np[2] = {0, 0};
      bool ok = true;
      // Shared-memory descriptors are built once; per MMA only a constant offset is
      // added to the address field (bits 0-13, address / 16: shared memory ends below
      // 256 KB, so the field never carries).
      const uint64_t dq0 = umma::sdesc_sw128(Q_S(0), 16, 1024);
      const uint64_t dq1 = umma::sdesc_sw128(Q_S(1), 16, 1024);
      // K (K-major) by row groups like V: 8-key groups 2 KB apart (SBO), the second
      // 64-column block of a group 1 KB in
      const uint64_t dk = umma::sdesc_sw128(STAGE(0), 16, 2048);
      // V (MN-major) by row groups: column blocks 1 KB apart (LBO), 8-key groups 2 KB
      // apart (SBO), a 16-key step 4 KB
      const uint64_t dv = umma::sdesc_sw128(STAGE(0), 1024, 2048);
      auto stage_field = [&](uint32_t c) { return uint64_t((c % kStages) * uint32_t(kTileBytes / 16)); };
      // S_i = Q_i K^T from the K stage at ring position kc
      auto qk = [&](int i, uint32_t kc) {
        const uint64_t kd = dk + stage_field(kc), qd = i == 0 ? dq0 : dq1;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t qoff = uint64_t(((k >> 2) * kHalfBytes + (k & 3) * 32) >> 4);
          const uint64_t koff = uint64_t(((k >> 2) * 1024 + (k & 3) * 32) >> 4);
          umma::mma_f16_ss(S_T(i), qd + qoff, kd + koff, idesc_qk, k > 0);
        }
        umma::commit(BAR(L::kSFull + i));
      };
      // O_i (+)= P_i V from the V stage at ring position vc
      auto pv = [&](int i, uint32_t vc, int nk16, bool acc) {
        const uint64_t vd = dv + stage_field(vc);
#pragma unroll
        for (int k = 0; k < kTileN / 16; ++k)
          if (k < nk16)
            umma::mma_f16_ts(O_T(i), S_T(i) + 8u * uint32_t(k) + (k >= 4 ? 32u : 0u), vd + uint64_t((k * 4096) >> 4),
                             idesc_pv, (acc || k > 0) ? 1u : 0u);
      };
      auto wait_p = [&](int i) {
        const bool r = wt.wait(BAR(L::kPFull + i), np[i] & 1u);
        ++np[i];
        return r;
      };
      // V stages (and with RoPE the query tiles and K stages) are read once the operand
      // warps are done with them; their barriers complete once per use, like full / q_full
      const int q_ready = ROPE ? L::kQRot : L::kQFull;
      auto ready = [&](uint32_t c) { return BAR(L::kReady + int(c % kStages)); };
      auto k_ready = [&](uint32_t c) { return ROPE ? ready(c) : FULL(c); };
      for (int u = u_begin; u < u_end && ok; ++u) {
        const DecodeItem it = p.items[u];
        const int nt = ntiles_of(it);
        if (nt == 0) continue;
        const bool two = it.nrows > kTileM;
        if (!wt.wait(BAR(q_ready), nq[0]++ & 1u)) break;
        if (two && !wt.wait(BAR(q_ready + 1), nq[1]++ & 1u)) break;
        if (!wt.wait(k_ready(c), PHASE(c))) break;
        umma::fence_after_sync();
        qk(0, c);
        if (two) qk(1, c);
        umma::commit(EMPTY(c));
        if (nt == 1) {   // the query tiles are free once these products complete
          umma::commit(BAR(L::kQEmpty));
          if (two) umma::commit(BAR(L::kQEmpty + 1));
        }
        ++c;
        for (int j = 0; j < nt; ++j) {
          const bool last = j + 1 == nt;
          const int nkeys = min(kTileN, it.tok1 - it.tok0 - kTileN * j);
          const int nk16 = (nkeys + 15) >> 4;
          const uint32_t vc = c, kc = c + 1;
          if (!wt.wait(ready(vc), PHASE(vc))) { ok = false; break; }
          if (!wait_p(0)) { ok = false; break; }
          umma::fence_after_sync();
          pv(0, vc, nk16, j > 0);
          if (last) umma::commit(BAR(L::kOFull));
          if (!last) {
            if (!wt.wait(k_ready(kc), PHASE(kc))) { ok = false; break; }
            umma::fence_after_sync();
            qk(0, kc);
            if (j + 2 == nt) umma::commit(BAR(L::kQEmpty));
          }
          if (two) {
            if (!wait_p(1)) { ok = false; break; }
            umma::fence_after_sync();
            pv(1, vc, nk16, j > 0);
            if (last) umma::commit(BAR(L::kOFull + 1));
          }
          umma::commit(EMPTY(vc));
          if (!last) {
            if (two) {
              qk(1, kc);
              if (j + 2 == nt) umma::commit(BAR(L::kQEmpty + 1));
            }
            umma::commit(EMPTY(kc));
          }
          c += last ? 1 : 2;
        }
      }
      // every MMA issued so far completes before TMEM is released
      umma::commit(BAR(L::kDrain));
      ptx::mbar_wait_bounded(BAR(L::kDrain), 0, 50000000ull);
    }
  } else if (ROPE && warp >= kRotWarp0) {
    // ------------------------------------------------------------ RoPE warps
    // Thread rt rotates chunk ch (frequencies 8 ch .. 8 ch + 7 and their partners 64
    // further) of rows 8 blk .. 8 blk + 7 of each query and K tile.  A row's angles come
    // from two table rows by angle addition: a base position (a key row: the first key
    // of its 16-key group, from `indices` order or the page's logical position; a query
    // row: the position of the thread's first row) and an offset below 16, whose (cos,
    // sin) sit in shared memory.  Base rows are fetched a tile ahead.  A quarter warp
    // covers one row's eight chunks, so its shared-memory accesses hit distinct banks.
    const int rt = tid - 32 * kRotWarp0;
    const int ch = rt & 7, blk = rt >> 3;
    // head_dim 64: 32 rotation pairs per row, chunks 0-3 with 4-7 (threads of chunks
    // 4-7 have nothing to rotate and load no angles)
    const bool rot_on = !D64 || ch < 4;
    constexpr int row_f4 = D64 ? 16 : D / 4;
    const uint32_t ttab = base + L::kRopeT;
    for (int i = rt; i < 16 * row_f4; i += kRotThreads) {
      const int t = i / row_f4, fp = i % row_f4;   // offset, frequency pair
      const float4 v = __ldg(p.rope + size_t(t) * row_f4 + fp);
      const uint32_t dst = ttab + uint32_t(((t * 4 + (fp & 3)) * 8 + (fp >> 2)) * 16);
      asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst),
                   "f"(v.x * kRopeOperandScale), "f"(v.y * kRopeOperandScale),
                   "f"(v.z * kRopeOperandScale), "f"(v.w * kRopeOperandScale) : "memory");
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kRotThreads) : "memory");
    const int lp = 31 - __clz(p.P);
    const int g = blk >> 1;                  // 16-key group of this thread's key rows
    const int t0 = (blk & 1) * 8;            // offset of its first row within the group
    uint32_t c = 0, nq[2] = {0, 0};
    float mag = 0.f;                         // largest rotated magnitude of a valid row
    bool ok = true;
    // base angles of this thread's key rows in tile j (nothing to rotate past the end)
    auto key_base = [&](const DecodeItem& it, int j) {
      Angles b{};
      const int nkeys = min(kTileN, it.tok1 - it.tok0 - kTileN * j);
      if (rot_on && j < ntiles_of(it) && 16 * g < nkeys) {
        const int kg = it.tok0 + kTileN * j + 16 * g;
        const int bpos = p.page_pos != nullptr
                             ? __ldg(p.page_pos + it.page_base + (kg >> lp)) + (kg & (p.P - 1))
                             : kg;
        b = load_angles(p.rope, min(bpos, p.rope_max_pos), ch, row_f4);
      }
      return b;
    };
    // rows 8 blk + t of a tile at `tile`: compose base (+) offset off(t), rotate in place
    auto rotate_rows = [&](auto grouped, uint32_t tile, const Angles& b, int first_off,
                           int step_div, int valid_rows) {
      if (!rot_on) return;
#pragma unroll 1
      for (int t = 0; t < 8; ++t) {
        const int r = 8 * blk + t;
        const int off = step_div == 1 ? first_off + t : (first_off + t) / step_div;
        const uint32_t trow = ttab + uint32_t((off * 32 + ch) * 16);
        Angles an;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float2 ct, st;
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(ct.x), "=f"(ct.y), "=f"(st.x), "=f"(st.y) : "r"(trow + e * 128));
          an.c[e] = ptx::fsub2(ptx::fmul2(b.c[e], ct), ptx::fmul2(b.s[e], st));
          an.s[e] = ptx::ffma2(b.s[e], ct, ptx::fmul2(b.c[e], st));
        }
        const float m = rotate_row_chunk<decltype(grouped)::value, D64>(tile, r, ch, an);
        if (r < valid_rows) mag = fmaxf(mag, m);
      }
    };
    // query tile i: row R of the unit is query R / group at position qpos0 + R / group
    // (plus the logical shift of a cache with dropped blocks); this thread's rows start
    // at R0 = row0 + 128 i + 8 blk, and row R0 + t sits (R0 % group + t) / group after it
    auto q_base = [&](const DecodeItem& it, int i) {
      const int qsh = p.qshift != nullptr ? __ldg(p.qshift + it.req) : 0;
      const int R0 = it.row0 + kTileM * i + 8 * blk;
      const int pos = min(max(it.qpos0 + R0 / p.group + qsh, 0), p.rope_max_pos);
      return rot_on ? load_angles(p.rope, pos, ch, row_f4) : Angles{};
    };
    auto rotate_q = [&](const DecodeItem& it, int i, const Angles& b) -> bool {
      if (!wt.warp_wait(BAR(L::kQFull + i), nq[i] & 1u)) return false;
      ++nq[i];
      const int R0 = it.row0 + kTileM * i + 8 * blk;
      rotate_rows(std::false_type{}, Q_S(i), b, R0 % p.group, p.group, it.nrows - kTileM * i);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(L::kQRot + i));
      return true;
    };
    for (int u = u_begin; u < u_end && ok; ++u) {
      const DecodeItem it = p.items[u];
      const int nt = ntiles_of(it);
      if (nt == 0) continue;
      const bool two = it.nrows > kTileM;
      Angles bk = key_base(it, 0);
      // K(0) lands first (the producer issues it before the query tiles), then the
      // query tiles, then K(1), ... (every key tile's K at an even ring position)
      for (int j = 0; j < nt && ok; ++j) {
        const uint32_t kc = c + 2 * uint32_t(j);
        const int nkeys = min(kTileN, it.tok1 - it.tok0 - kTileN * j);
        if (!wt.warp_wait(FULL(kc), PHASE(kc))) { ok = false; break; }
        const Angles bnext = key_base(it, j + 1);
        rotate_rows(std::true_type{}, STAGE(kc), bk, t0, 1, nkeys);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(L::kReady + int(kc % kStages)));
        bk = bnext;
        if (j == 0) {
          ok = rotate_q(it, 0, q_base(it, 0));
          if (ok && two) ok = rotate_q(it, 1, q_base(it, 1));
        }
      }
      c += 2 * uint32_t(nt);
    }
    if (mag > kF16Max) atomicOr(p.error, kStatusOperandRange);
  } else {
    // ------------------------------------------------------------ softmax warps
    // Two threads per row: warp w works on query tile w / 8, key/column half
    // (w / 4) % 2 and row quarter w % 4 (the TMEM lanes it may access); thread t of
    // the quarter owns row t.  The halves of a row exchange their partial max (and
    // at the end their partial sum) through shared memory and an mbarrier.
    const int qt = warp >> 3;
    const int half = (warp >> 2) & 1;
    const int quad = warp & 3;
    const int t = quad * 32 + lane;        // row within the tile == TMEM lane
    const uint32_t lane_off = uint32_t(quad * 32) << 16;
    // this half's 64 S columns (keys 64 half ..), later its 32 columns of P; its O columns
    const uint32_t s_t = S_T(qt) + lane_off + 64u * half, o_t = O_T(qt) + lane_off + 64u * half;
    const uint32_t xbar = BAR(L::kXch + qt * 4 + quad);
    auto xslot = [&](uint32_t par, int h) {
      return base + L::kXchData + uint32_t((((par * 2 + qt) * 2 + h) * kTileM + t) * 4);
    };
    const float sl2 = ROPE ? p.scale_log2 * (1.f / (kRopeOperandScale * kRopeOperandScale))
                           : p.scale_log2;
    uint32_t ns = 0, no = 0, nx = 0;
    bool ok = true;
    // Swap a value with the other half of the row; false when this CTA is aborting.
    auto exchange = [&](float mine, float& other) -> bool {
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(xslot(nx & 1u, half)), "f"(mine) : "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar);
      if (!wt.warp_wait(xbar, nx & 1u)) return false;
      asm volatile("ld.shared.f32 %0, [%1];" : "=f"(other) : "r"(xslot(nx & 1u, half ^ 1)) : "memory");
      ++nx;
      return true;
    };
    // V of key tile j of a unit (ring position cring + 2 j + 1) to fp16 in place, rows
    // past the last key zeroed.  Every softmax warp takes 1 / 16 of the 16-byte chunks
    // of every V tile (q = 32 warp + lane + 512 k: a quarter warp covers 128 contiguous
    // bytes), in ring order, even for a unit where its query tile has no rows: a barrier
    // wait more than one use ahead of a stage would be satisfied by an older phase of
    // the same parity.  In the row-group layout chunk q holds row 8 (q / 128) + (q / 8) % 8.
    uint32_t cring = 0;
    float vmag = 0.f;                      // largest V magnitude of a valid row
    auto convert_v = [&](const DecodeItem& it, int j) -> bool {
      const uint32_t vc = cring + 2 * uint32_t(j) + 1;
      if (!wt.warp_wait(FULL(vc), PHASE(vc))) return false;
      const int nkeys = min(kTileN, it.tok1 - it.tok0 - kTileN * j);
      const uint32_t vs = STAGE(vc);
#pragma unroll 2
      for (int q = 32 * warp + lane; q < kVChunks; q += 32 * kSoftmaxWarps) {
        const int r = 8 * (q >> 7) + ((q >> 3) & 7);
        const uint32_t addr = vs + uint32_t(q) * 16u;
        uint32_t o[4] = {0u, 0u, 0u, 0u};
        if (r < nkeys) {
          uint32_t a[4];
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]) : "r"(addr));
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = ptx::bf16_lo(a[e]), x1 = ptx::bf16_hi(a[e]);
            vmag = ptx::fmax3(vmag, fabsf(x0), fabsf(x1));
            o[e] = ptx::pack_f16(x0, x1);
          }
        }
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                     ::"r"(addr), "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3]) : "memory");
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(L::kReady + int(vc % kStages)));
      return true;
    };
    for (int u = u_begin; u < u_end && ok; ++u) {
      const DecodeItem it = p.items[u];
      const int nt = ntiles_of(it);
      const int rows_here = it.nrows - kTileM * qt;
      if (rows_here <= 0) {
        // second query tile of a short unit: only its share of the unit's V tiles
        for (int j = 0; j < nt && ok; ++j) ok = convert_v(it, j);
        cring += 2 * uint32_t(nt);
        continue;
      }
      const int group = p.group;
      const int prow = kTileM * qt + t;    // row within the unit
      const int R = it.row0 + prow;
      const bool vrow = t < rows_here;
      const int qpos = it.qpos0 + R / group;
      float m_used = -INFINITY, l = 0.f;   // l: this half's partial sum
      if (nt > 0) {
        if (!convert_v(it, 0)) { ok = false; break; }
        for (int j = 0; j < nt; ++j) {
          const int key0 = it.tok0 + kTileN * j + 64 * half;
          const int nkeys = min(64, it.tok1 - key0);                          // may be <= 0
          const int klim = p.causal ? min(nkeys, qpos - key0 + 1) : nkeys;
          // sliding window: keys [klo, klim) of this half are visible
          // (compiled in only for WIN)
          const int klo = WIN ? qpos - p.window_left + 1 - key0 : 0;

          // ---- online softmax (log2 domain, lazy rescale) over this half's 64 scores,
          // read in 32-column quarters: max pass, exchange, exp2 / pack / store pass
          if (!wt.warp_wait(BAR(L::kSFull + qt), ns & 1u)) { ok = false; break; }
          ++ns;
          umma::fence_after_sync();
          const bool masked = __any_sync(0xffffffffu, klim < 64 || (WIN && klo > 0));
          auto load_quarter = [&](int qq, float (&sv)[32]) {
            umma::tmem_ld32(s_t + 32 * qq, sv);
            if (masked) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                sv[i] = (32 * qq + i < klim && (!WIN || 32 * qq + i >= klo)) ? sv[i] : -INFINITY;
            }
          };
          float mpart = -INFINITY;
#pragma unroll
          for (int qq = 0; qq < 2; ++qq) {
            float sv[32];
            load_quarter(qq, sv);
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < 32; i += 8)
#pragma unroll
              for (int k = 0; k < 4; ++k) m4[k] = ptx::fmax3(m4[k], sv[i + 2 * k], sv[i + 2 * k + 1]);
            mpart = ptx::fmax3(mpart, ptx::fmax3(m4[0], m4[1], m4[2]), m4[3]);
          }
          float mother;
          if (!exchange(mpart, mother)) { ok = false; break; }
          float mx = fmaxf(mpart, mother);
          mx = mx == -INFINITY ? mx : mx * sl2;
          float alpha = 1.f;
          if (mx > m_used + 8.f) {          // also true the first time a row sees a key
            alpha = m_used == -INFINITY ? 0.f : ptx::ex2(m_used - mx);
            m_used = mx;
          }
          const float mu = m_used == -INFINITY ? 0.f : m_used;
          // O_i is stable here: this S was committed after the previous P V
          if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
            for (int c2 = 0; c2 < 2; ++c2) {
              float v[32];
              umma::tmem_ld32(o_t + 32 * c2, v);
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] *= alpha;
              umma::tmem_st32(o_t + 32 * c2, v);
            }
          }
          const float2 sc2 = make_float2(sl2, sl2), nmu2 = make_float2(-mu, -mu);
          float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                           make_float2(0.f, 0.f)};
#pragma unroll
          for (int qq = 0; qq < 2; ++qq) {
            float sv[32];
            load_quarter(qq, sv);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 x = ptx::ffma2(make_float2(sv[i], sv[i + 1]), sc2, nmu2);
              const float2 e = make_float2(ptx::ex2(x.x), ptx::ex2(x.y));
              rs2[(i >> 1) & 3] = ptx::fadd2(rs2[(i >> 1) & 3], e);
              pk[i / 2] = ptx::pack_f16(e.x, e.y);
            }
            // P (fp16 pairs, at most 2^8 with the lazy rescale) over this half's S
            // columns already read
            umma::tmem_st16u(s_t + 16 * qq, pk);
          }
          const float2 r01 = ptx::fadd2(rs2[0], rs2[1]), r23 = ptx::fadd2(rs2[2], rs2[3]);
          const float2 r = ptx::fadd2(r01, r23);
          l = l * alpha + (r.x + r.y);
          umma::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(L::kPFull + qt));
          // while the tensor cores take P V and the next Q K^T: V of the next key tile
          if (j + 1 < nt && !convert_v(it, j + 1)) { ok = false; break; }
        }
        if (!ok) break;
        cring += 2 * uint32_t(nt);
        if (!wt.warp_wait(BAR(L::kOFull + qt), no & 1u)) { ok = false; break; }
        ++no;
        umma::fence_after_sync();
        float lother;
        if (!exchange(l, lother)) { ok = false; break; }
        l += lother;
      }
      // ---- epilogue: this half's 64 columns of O row t / l (an empty unit writes 0 /
      // -inf); a split range writes its fp32 partial state instead.  With head_dim 64
      // only the first half's columns are real (the second half's are zero padding).
      const size_t orow = out_row(it, R, group, p.Hq);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse2 = l > 0.f ? m_used + ptx::lg2(l) : -INFINITY;
      constexpr float kLn2 = 0.69314718055994530942f;
      float* part_row =
          p.part_o + (size_t(it.slot < 0 ? 0 : it.slot) * kUnitRows + prow) * size_t(p.head_dim);
#pragma unroll 1
      for (int c2 = 0; c2 < 2; ++c2) {
        const int c4 = 2 * half + c2;      // 32-column chunk of the row
        if (32 * c4 >= p.head_dim) break;
        float v[32];
        if (nt > 0) {
          umma::tmem_ld32(o_t + 32 * c2, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= inv;
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        if (it.slot >= 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            ptx::st_global_v8(part_row + 32 * c4 + 8 * i, __float_as_uint(v[8 * i]),
                              __float_as_uint(v[8 * i + 1]), __float_as_uint(v[8 * i + 2]),
                              __float_as_uint(v[8 * i + 3]), __float_as_uint(v[8 * i + 4]),
                              __float_as_uint(v[8 * i + 5]), __float_as_uint(v[8 * i + 6]),
                              __float_as_uint(v[8 * i + 7]));
        } else if (vrow) {
          store_row_chunk(p, orow, c4, v);
        }
      }
      umma::fence_before_sync();
      if (half == 0) {
        if (it.slot < 0) {
          if (vrow && p.lse != nullptr) p.lse[orow] = lse2 * kLn2;
        } else {
          p.part_lse[size_t(it.slot) * kUnitRows + prow] = lse2;
        }
      }
    }
    if (vmag > kF16Max) atomicOr(p.error, kStatusOperandRange);
  }

  // ------------------------------------------------------------ teardown
  umma::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- split-range merge
// One thread per 16-byte column chunk (4 columns) of a packed row of a split unit.
// The partial states (fp32, log2-domain lse) are combined in key order:
//   lse = M + log2(sum_k 2^(lse_k - M)),  o = sum_k 2^(lse_k - M) o_k / sum_k 2^(lse_k - M).
// Every thread of a row reads the row's few chunk lse values itself (one broadcast load
// per warp) and the partial columns of the first kMergeAhead chunks before the weights
// are known, so a split of up to that many chunks waits on memory once; no shuffles.
constexpr int kMergeThreads = 256;
constexpr int kMergeAhead = 4;
__global__ void __launch_bounds__(kMergeThreads) bsr_prefill_merge_kernel(const PrefillMergeParams p) {
  // launched as a programmatic dependent of the prefill kernel, whose partial states it reads
  pdl_trigger();
  pdl_wait();
  const int cpr = p.head_dim / 4;                       // 16-byte chunks per row
  const int64_t gid = int64_t(blockIdx.x) * kMergeThreads + threadIdx.x;
  const int64_t grow = gid / cpr;                       // unit * kUnitRows + packed row
  const int ch = int(gid - grow * cpr);
  const int unit = int(grow / kUnitRows), prow = int(grow % kUnitRows);
  if (unit >= p.n_units) return;
  const DecodeItem it = p.units[unit];
  if (prow >= it.nrows) return;
  const int n = it.nchunks;
  const size_t hd = size_t(p.head_dim);
  const float* lse_k = p.part_lse + size_t(it.first_slot) * kUnitRows + prow;
  const float* po = p.part_o + (size_t(it.first_slot) * kUnitRows + prow) * hd + 4 * ch;
  const size_t slot_stride = size_t(kUnitRows) * hd;
  float lk[kMergeAhead];
  float4 x[kMergeAhead];
#pragma unroll
  for (int k = 0; k < kMergeAhead; ++k) {
    lk[k] = k < n ? __ldg(lse_k + size_t(k) * kUnitRows) : -INFINITY;
    x[k] = k < n ? __ldcg(reinterpret_cast<const float4*>(po + size_t(k) * slot_stride))
                 : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < kMergeAhead; ++k) M = fmaxf(M, lk[k]);
  for (int k = kMergeAhead; k < n; ++k) M = fmaxf(M, __ldg(lse_k + size_t(k) * kUnitRows));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lt = -INFINITY;
  if (M != -INFINITY) {
    float sum = 0.f;
    auto add = [&](float l, const float4& v) {
      const float wk = l == -INFINITY ? 0.f : ptx::ex2(l - M);
      sum += wk;
      acc.x += wk * v.x; acc.y += wk * v.y; acc.z += wk * v.z; acc.w += wk * v.w;
    };
#pragma unroll
    for (int k = 0; k < kMergeAhead; ++k)
      if (k < n) add(lk[k], x[k]);
    for (int k = kMergeAhead; k < n; ++k)
      add(__ldg(lse_k + size_t(k) * kUnitRows),
          __ldcg(reinterpret_cast<const float4*>(po + size_t(k) * slot_stride)));
    const float inv = 1.f / sum;
    acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
    lt = M + ptx::lg2(sum);
  }
  const size_t orow = out_row(it, it.row0 + prow, p.group, p.Hq);
  if (p.out_f32) {
    reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * hd)[ch] = acc;
  } else {
    reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + orow * hd)[ch] =
        make_uint2(ptx::pack_bf16(acc.x, acc.y), ptx::pack_bf16(acc.z, acc.w));
  }
  if (ch == 0 && p.lse != nullptr) p.lse[orow] = lt * 0.69314718055994530942f;
}

template <bool ROPE, bool WIN, bool D64>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const PrefillParams& p, int grid, cudaStream_t stream) {
  auto kern = bsr_prefill_kernel<ROPE, WIN, D64>;
  constexpr size_t smem = Smem::kDynBytes;
  static std::atomic<bool> opted_in[64];   // zero-initialized: false
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!opted_in[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    opted_in[dev].store(true, std::memory_order_release);
  }
  const cudaError_t le = launch_pdl(kern, grid, threads_of<ROPE>(), smem, stream, tq, tk, tv, p);
  return le != cudaSuccess ? le : cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(bool rope, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const PrefillParams& p, int grid,
                           cudaStream_t stream) {
  const bool d64 = p.head_dim == 64;
  if (p.window_left > 0) {
    if (!rope) return launch_one<false, true, false>(tq, tk, tv, p, grid, stream);
    return d64 ? launch_one<true, true, true>(tq, tk, tv, p, grid, stream)
               : launch_one<true, true, false>(tq, tk, tv, p, grid, stream);
  }
  if (!rope) return launch_one<false, false, false>(tq, tk, tv, p, grid, stream);
  return d64 ? launch_one<true, false, true>(tq, tk, tv, p, grid, stream)
             : launch_one<true, false, false>(tq, tk, tv, p, grid, stream);
}

cudaError_t launch_prefill_merge(const PrefillMergeParams& p, cudaStream_t stream) {
  const int64_t threads = int64_t(p.n_units) * kUnitRows * (p.head_dim / 4);
  const int64_t grid = (threads + kMergeThreads - 1) / kMergeThreads;
  if (grid <= 0) return cudaSuccess;
  const cudaError_t le = launch_pdl(bsr_prefill_merge_kernel, int(grid), kMergeThreads, 0, stream, p);
  return le != cudaSuccess ? le : cudaGetLastError();
}

}  // namespace bsr
