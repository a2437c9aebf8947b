// Prefill / multi-query attention over a paged (BSR) KV cache on the sm_103a
// tensor cores (tcgen05 + TMEM), head_dim 128.
//
// Prefill is compute-bound ("FlashInfer: Block-Sparse KV 캐시로 어텐션 병목을
// 해소하다", section "어텐션 연산에서 진짜 병목은 어디인가?"): many query rows
// share every key, so the work is a real dense contraction.  One work unit is
// a tile of 128 packed (query, head) rows of one (request, kv head) against a
// page-aligned key range; a CTA walks its planned list of units.
//
// Roles:
//   warps 0-3  row owners: thread t owns packed row t of the tile and TMEM lane
//              t.  They load Q (RoPE-rotated and split into bf16 hi + lo, so
//              QK^T takes two passes), run the online softmax on S
//              rows read from TMEM (two passes: row max, then exp2 / P), write
//              P (bf16) to shared memory, rescale O in TMEM when the running
//              max grows by more than 2^8, and write out / lse.
//   warp 4     TMA producer: gathers 128-key K and V tiles page by page from
//              `indices` (inactive blocks are absent, "Block-Sparse 포맷") into a
//              two-stage ring of 128B-swizzled tiles.
//   warp 5     allocates TMEM and issues the MMAs: S = Q K^T (M 128, N 128,
//              8 x K16, K-major operands) into one of two TMEM S buffers, and
//              O += P V (P K-major from shared memory, V MN-major) into a TMEM
//              O buffer.  S is double-buffered so that QK^T of the next tile
//              runs on the tensor cores while the row owners work on this one.
//   warps 6-7  (RoPE only) rotate each landed K tile in place, ahead of the MMA
//              ("JIT 컴파일은 …": RoPE fused into attention, k stored un-rotated).
// A unit whose key range was split writes an fp32 partial state; for each
// 32-row quarter the last arriving warp merges the partials in key order.
// Every mbarrier wait is bounded and warp-agreed.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bsr_internal.h"
#include "bsr_schedule.h"
#include "ptx.cuh"
#include "umma.cuh"

namespace bsr {
namespace {

constexpr int D = 128;
constexpr int kTileM = 128;              // packed rows per unit
constexpr int kTileN = 128;              // keys per KV tile
constexpr int kHalfBytes = kTileN * 128; // one 64-column block of a 128-row tile: 16 KB
constexpr int kTileBytes = 2 * kHalfBytes;
constexpr uint32_t kTmemCols = 512;      // S0 | S1 | O | (unused)

template <bool ROPE>
struct PrefillSmem {
  static constexpr int kThreads = ROPE ? 256 : 192;
  static constexpr int kQ = 0;
  static constexpr int kQlo = kQ + kTileBytes;                     // RoPE: low half of the split q
  static constexpr int kStage0 = ROPE ? kQlo + kTileBytes : kQlo;  // K then V per stage
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kP = kStage0 + 2 * kStageBytes;
  static constexpr int kBars = kP + kTileBytes;
  // barriers: kv_full[2], kv_ready[2], kv_empty[2], s_full[2], p_full, pv_done, q_full
  static constexpr int kNumBars = 11;
  static constexpr int kTmemSlot = kBars + 8 * kNumBars;
  static constexpr int kFlags = kTmemSlot + 16;   // abort flag
  static constexpr int kTotal = kFlags + 16;
  static constexpr size_t kDynBytes = size_t(kTotal) + 1024;
  static_assert(kDynBytes <= 232448, "prefill tiles exceed the shared memory of one SM");
};

// Offset of (row r, 16-byte chunk c of 16) in a [2 blocks][128 rows][128 B]
// 128B-swizzled tile.
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return uint32_t((c >> 3) * kHalfBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

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
        atomicOr(error, 1);
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

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// Rotate one 128-column row of a swizzled tile in place at position `pos`
// (rotate-half pairs (d, d + 64), cos/sin from the frequency-ordered table).
__device__ __forceinline__ void rope_row_inplace(uint32_t tile, int r, const float2* rope_nat,
                                                 int pos) {
  const float4* tab = reinterpret_cast<const float4*>(rope_nat + size_t(pos) * (D / 2));
#pragma unroll 2
  for (int c = 0; c < 8; ++c) {
    float4 cs[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) cs[e] = __ldg(tab + 4 * c + e);   // frequencies 8c + 2e, 8c + 2e + 1
    uint4 av, bv;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(av.x), "=r"(av.y), "=r"(av.z), "=r"(av.w) : "r"(tile + sw_off(r, c)));
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(bv.x), "=r"(bv.y), "=r"(bv.z), "=r"(bv.w) : "r"(tile + sw_off(r, c + 8)));
    const uint32_t* a = reinterpret_cast<const uint32_t*>(&av);
    const uint32_t* b = reinterpret_cast<const uint32_t*>(&bv);
    uint32_t xo[4], yo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a0 = ptx::bf16_lo(a[e]), a1 = ptx::bf16_hi(a[e]);
      const float b0 = ptx::bf16_lo(b[e]), b1 = ptx::bf16_hi(b[e]);
      xo[e] = ptx::pack_bf16(a0 * cs[e].x - b0 * cs[e].y, a1 * cs[e].z - b1 * cs[e].w);
      yo[e] = ptx::pack_bf16(b0 * cs[e].x + a0 * cs[e].y, b1 * cs[e].z + a1 * cs[e].w);
    }
    sts128(tile + sw_off(r, c), xo[0], xo[1], xo[2], xo[3]);
    sts128(tile + sw_off(r, c + 8), yo[0], yo[1], yo[2], yo[3]);
  }
}

// Write 32 columns (chunk c) of one output row as bf16 or fp32.
__device__ __forceinline__ void store_row_chunk(const PrefillParams& p, size_t orow, int c,
                                                const float (&v)[32]) {
  if (p.out_f32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * D + 32 * c);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow * D + 32 * c);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      dst[i] = make_uint4(ptx::pack_bf16(v[8 * i], v[8 * i + 1]), ptx::pack_bf16(v[8 * i + 2], v[8 * i + 3]),
                          ptx::pack_bf16(v[8 * i + 4], v[8 * i + 5]), ptx::pack_bf16(v[8 * i + 6], v[8 * i + 7]));
  }
}

template <bool ROPE>
__global__ void __launch_bounds__(PrefillSmem<ROPE>::kThreads, 1)
    bsr_prefill_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using L = PrefillSmem<ROPE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar0 = base + L::kBars;
  auto BAR = [&](int i) { return bar0 + 8u * uint32_t(i); };
  enum { KV_FULL = 0, KV_READY = 2, KV_EMPTY = 4, S_FULL = 6, P_FULL = 8, PV_DONE = 9, Q_FULL = 10 };
  const uint32_t abort_addr = base + L::kFlags;
  Waiter wt{abort_addr, p.wait_limit_ns, p.error};

  const int u_begin = __ldg(p.cta_ptr + blockIdx.x), u_end = __ldg(p.cta_ptr + blockIdx.x + 1);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(BAR(KV_FULL + i), 1);
      ptx::mbar_init(BAR(KV_READY + i), 64);
      ptx::mbar_init(BAR(KV_EMPTY + i), 1);
      ptx::mbar_init(BAR(S_FULL + i), 1);
    }
    ptx::mbar_init(BAR(P_FULL), 128);
    ptx::mbar_init(BAR(PV_DONE), 1);
    ptx::mbar_init(BAR(Q_FULL), 128);
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(abort_addr), "r"(0u));
    ptx::fence_barrier_init();
  }
  if (warp == 5) {
    umma::tmem_alloc(base + L::kTmemSlot, kTmemCols);
    umma::tmem_relinquish();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  uint32_t tmem;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(tmem) : "r"(base + L::kTmemSlot));
  const uint32_t O_T = tmem + 256;
  auto S_T = [&](uint32_t g) { return tmem + 128u * (g & 1u); };
  auto stage_k = [&](uint32_t g) { return base + L::kStage0 + (g & 1u) * L::kStageBytes; };

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // K/V tiles are re-read by the other row tiles of the same (request, kv head),
      // which run concurrently on other SMs: keep them in L2 at normal priority.
      const uint64_t pol = ptx::policy_evict_normal();
      uint32_t gt = 0;
      bool ok = true;
      for (int u = u_begin; u < u_end && ok; ++u) {
        const DecodeItem it = p.items[u];
        const int nt = ntiles_of(it);
        for (int j = 0; j < nt; ++j, ++gt) {
          const int stage = gt & 1;
          const uint32_t n = gt >> 1;
          if (gt >= 2 && !wt.wait(BAR(KV_EMPTY + stage), (n - 1) & 1)) { ok = false; break; }
          const int key0 = it.tok0 + kTileN * j;
          const int nkeys = min(kTileN, it.tok1 - key0);
          const int nsub = (nkeys + 15) >> 4;
          const uint32_t ks = stage_k(gt), vs = ks + kTileBytes;
          ptx::mbar_arrive_expect_tx(BAR(KV_FULL + stage), uint32_t(nsub) * 4u * 2048u);
          for (int sb = 0; sb < nsub; ++sb) {
            const int key = key0 + 16 * sb;
            const int page = __ldg(p.indices + it.page_base + key / p.P);
            const int row = (page * p.Hk + it.kvh) * p.P + (key % p.P);
            for (int h = 0; h < 2; ++h) {
              ptx::tma_load_3d(ks + h * kHalfBytes + sb * 2048, &tm_k, BAR(KV_FULL + stage), 0, h, row, pol);
              ptx::tma_load_3d(vs + h * kHalfBytes + sb * 2048, &tm_v, BAR(KV_FULL + stage), 0, h, row, pol);
            }
          }
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma::idesc_bf16_f32(kTileM, kTileN, 0, 0);
      constexpr uint32_t idesc_pv = umma::idesc_bf16_f32(kTileM, D, 0, 1);
      uint32_t gt = 0, qc = 0;   // tiles and non-empty units seen so far
      bool ok = true;
      // S(g) = Q K(g)^T into S buffer g % 2, once tile g's K is in shared memory
      auto issue_qk = [&](uint32_t g) -> bool {
        if (!wt.wait(BAR((ROPE ? KV_READY : KV_FULL) + (g & 1)), (g >> 1) & 1)) return false;
        umma::fence_after_sync();
        const uint32_t ks = stage_k(g);
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
          umma::mma_f16_ss(S_T(g), umma::sdesc_sw128(base + L::kQ + off, 16, 1024),
                           umma::sdesc_sw128(ks + off, 16, 1024), idesc_qk, k > 0);
        }
        if constexpr (ROPE) {
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
            umma::mma_f16_ss(S_T(g), umma::sdesc_sw128(base + L::kQlo + off, 16, 1024),
                             umma::sdesc_sw128(ks + off, 16, 1024), idesc_qk, 1);
          }
        }
        umma::commit(BAR(S_FULL + (g & 1)));
        return true;
      };
      for (int u = u_begin; u < u_end && ok; ++u) {
        const DecodeItem it = p.items[u];
        const int nt = ntiles_of(it);
        if (nt == 0) continue;
        if (!wt.wait(BAR(Q_FULL), qc & 1)) break;
        ++qc;
        umma::fence_after_sync();
        if (!issue_qk(gt)) break;
        if (nt > 1 && !issue_qk(gt + 1)) break;
        for (int j = 0; j < nt; ++j, ++gt) {
          if (!wt.wait(BAR(P_FULL), gt & 1)) { ok = false; break; }
          umma::fence_after_sync();
          const uint32_t vs = stage_k(gt) + kTileBytes;
          const int key0 = it.tok0 + kTileN * j;
          const int nk16 = (min(kTileN, it.tok1 - key0) + 15) >> 4;
          for (int k = 0; k < nk16; ++k) {
            const uint32_t aoff = (k >> 2) * kHalfBytes + (k & 3) * 32;
            umma::mma_f16_ss(O_T, umma::sdesc_sw128(base + L::kP + aoff, 16, 1024),
                             umma::sdesc_sw128(vs + k * 2048, kHalfBytes, 1024), idesc_pv,
                             (j > 0 || k > 0) ? 1u : 0u);
          }
          umma::commit(BAR(KV_EMPTY + (gt & 1)));
          umma::commit(BAR(PV_DONE));
          // S buffer gt % 2 was read by the row owners before P_FULL: refill it with tile j + 2
          if (j + 2 < nt && !issue_qk(gt + 2)) { ok = false; break; }
        }
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ RoPE on K (ROPE only)
    const int t = tid - 192;           // this thread rotates key rows t and t + 64 of the tile
    uint32_t gt = 0;
    bool ok = true;
    for (int u = u_begin; u < u_end && ok; ++u) {
      const DecodeItem it = p.items[u];
      const int nt = ntiles_of(it);
      for (int j = 0; j < nt; ++j, ++gt) {
        if (!wt.warp_wait(BAR(KV_FULL + (gt & 1)), (gt >> 1) & 1)) { ok = false; break; }
        const int key0 = it.tok0 + kTileN * j;
        const int nkeys = min(kTileN, it.tok1 - key0);
#pragma unroll 1
        for (int r = t; r < nkeys; r += 64)
          rope_row_inplace(stage_k(gt), r, p.rope_nat, min(key0 + r, p.rope_max_pos));
        ptx::fence_proxy_async_smem();
        mbar_arrive(BAR(KV_READY + (gt & 1)));
      }
    }
  } else {
    // ------------------------------------------------------------ row owners
    const int t = tid;                     // packed row within the tile == TMEM lane
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    uint32_t gt = 0;
    bool ok = true;
    for (int u = u_begin; u < u_end && ok; ++u) {
      const DecodeItem it = p.items[u];
      const int nt = ntiles_of(it);
      const int group = p.group;
      const int R = it.row0 + t;
      const bool vrow = t < it.nrows;
      const int qpos = it.qpos0 + R / group;
      const size_t orow = size_t(it.q_row0 + R / group) * p.Hq + it.kvh * group + R % group;
      float m_used = -INFINITY, l = 0.f;
      if (nt > 0) {
        // ---- Q row t (RoPE-rotated at its position when RoPE is on)
        uint4 qraw[16];
        const uint4* src = reinterpret_cast<const uint4*>(p.q + orow * D);
#pragma unroll
        for (int c = 0; c < 16; ++c) qraw[c] = vrow ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        if constexpr (!ROPE) {
#pragma unroll
          for (int c = 0; c < 16; ++c)
            sts128(base + L::kQ + sw_off(t, c), qraw[c].x, qraw[c].y, qraw[c].z, qraw[c].w);
        } else {
          // The rotated query is split into bf16 hi + lo (two QK^T passes): its rounding
          // error would not average out over keys the way the keys' does.
          const float4* tab = reinterpret_cast<const float4*>(
              p.rope_nat + size_t(vrow ? min(max(qpos, 0), p.rope_max_pos) : 0) * (D / 2));
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t* a = reinterpret_cast<const uint32_t*>(&qraw[c]);
            const uint32_t* b = reinterpret_cast<const uint32_t*>(&qraw[c + 8]);
            uint32_t xh[4], xl[4], yh[4], yl[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float4 cs = __ldg(tab + 4 * c + e);   // frequencies 8c + 2e, 8c + 2e + 1
              const float a0 = ptx::bf16_lo(a[e]), a1 = ptx::bf16_hi(a[e]);
              const float b0 = ptx::bf16_lo(b[e]), b1 = ptx::bf16_hi(b[e]);
              ptx::split_bf16(a0 * cs.x - b0 * cs.y, a1 * cs.z - b1 * cs.w, xh[e], xl[e]);
              ptx::split_bf16(b0 * cs.x + a0 * cs.y, b1 * cs.z + a1 * cs.w, yh[e], yl[e]);
            }
            sts128(base + L::kQ + sw_off(t, c), xh[0], xh[1], xh[2], xh[3]);
            sts128(base + L::kQ + sw_off(t, c + 8), yh[0], yh[1], yh[2], yh[3]);
            sts128(base + L::kQlo + sw_off(t, c), xl[0], xl[1], xl[2], xl[3]);
            sts128(base + L::kQlo + sw_off(t, c + 8), yl[0], yl[1], yl[2], yl[3]);
          }
        }
        ptx::fence_proxy_async_smem();
        mbar_arrive(BAR(Q_FULL));

        for (int j = 0; j < nt; ++j, ++gt) {
          const int key0 = it.tok0 + kTileN * j;
          const int nkeys = min(kTileN, it.tok1 - key0);
          const uint32_t vs = stage_k(gt) + kTileBytes;
          const int klim = p.causal ? min(nkeys, qpos - key0 + 1) : nkeys;   // keys [0, klim) visible

          // ---- S row t: one 128-column TMEM load; mask, online softmax (log2, lazy rescale)
          if (!wt.warp_wait(BAR(S_FULL + (gt & 1)), (gt >> 1) & 1)) { ok = false; break; }
          umma::fence_after_sync();
          float sv[kTileN];
          umma::tmem_ld128(S_T(gt) + lane_off, sv);
          float mx = -INFINITY;
#pragma unroll
          for (int i = 0; i < kTileN; ++i)
            if (i < klim) mx = fmaxf(mx, sv[i]);
          mx = mx == -INFINITY ? mx : mx * p.scale_log2;
          float alpha = 1.f;
          if (mx > m_used + 8.f) {          // also true the first time a row sees a key
            alpha = m_used == -INFINITY ? 0.f : ptx::ex2(m_used - mx);
            m_used = mx;
          }
          const float mu = m_used == -INFINITY ? 0.f : m_used;
          float rs = 0.f;
          uint32_t pk[kTileN / 2];
#pragma unroll
          for (int i = 0; i < kTileN; i += 2) {
            const float p0 = i < klim ? ptx::ex2(sv[i] * p.scale_log2 - mu) : 0.f;
            const float p1 = i + 1 < klim ? ptx::ex2(sv[i + 1] * p.scale_log2 - mu) : 0.f;
            rs += p0 + p1;
            pk[i / 2] = ptx::pack_bf16(p0, p1);
          }

          // P buffer and O are free once the previous P.V has completed
          if (j > 0) {
            if (!wt.warp_wait(BAR(PV_DONE), (gt - 1) & 1)) { ok = false; break; }
            umma::fence_after_sync();
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                float v[32];
                umma::tmem_ld32(O_T + lane_off + 32 * c, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] *= alpha;
                umma::tmem_st32(O_T + lane_off + 32 * c, v);
              }
            }
          }
#pragma unroll
          for (int c = 0; c < 16; ++c)
            sts128(base + L::kP + sw_off(t, c), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          l = l * alpha + rs;
          // V rows past the last valid key of the final 16-key group may hold
          // another page's tail: zero them so that P = 0 contributes exactly 0.
          if (t >= nkeys && t < ((nkeys + 15) & ~15)) {
#pragma unroll
            for (int c = 0; c < 16; ++c) sts128(vs + sw_off(t, c), 0u, 0u, 0u, 0u);
          }
          ptx::fence_proxy_async_smem();
          umma::fence_before_sync();
          mbar_arrive(BAR(P_FULL));
        }
        if (!ok) break;
        if (!wt.warp_wait(BAR(PV_DONE), (gt - 1) & 1)) { ok = false; break; }
        umma::fence_after_sync();
      }
      // ---- epilogue: O row t / l  (an empty unit writes 0 / -inf), 32 columns at a time
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse2 = l > 0.f ? m_used + ptx::lg2(l) : -INFINITY;
      constexpr float kLn2 = 0.69314718055994530942f;
      float* part_row = p.part_o + (size_t(it.slot < 0 ? 0 : it.slot) * kTileM + t) * D;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float v[32];
        if (nt > 0) {
          umma::tmem_ld32(O_T + lane_off + 32 * c, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= inv;
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        if (it.slot >= 0) {
          float4* dst = reinterpret_cast<float4*>(part_row + 32 * c);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            __stcg(dst + i, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
        } else if (vrow) {
          store_row_chunk(p, orow, c, v);
        }
      }
      umma::fence_before_sync();
      if (it.slot < 0) {
        if (vrow && p.lse != nullptr) p.lse[orow] = lse2 * kLn2;
      } else {
        __stcg(p.part_lse + size_t(it.slot) * kTileM + t, lse2);
        __threadfence();
        __syncwarp();
        // each warp owns 32 rows of the tile and its own arrival counter, so the
        // merge needs no CTA-wide synchronization
        int last = 0;
        if (lane == 0) last = atomicAdd(p.counters + it.first_slot * 4 + warp, 1) == it.nchunks - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          __threadfence();
          if (vrow) {
            const float* lse_k = p.part_lse + size_t(it.first_slot) * kTileM + t;
            float M = -INFINITY;
            for (int k = 0; k < it.nchunks; ++k) M = fmaxf(M, __ldcg(lse_k + size_t(k) * kTileM));
            float lt = -INFINITY;
            if (M != -INFINITY) {
              float sum = 0.f;
              for (int k = 0; k < it.nchunks; ++k) sum += ptx::ex2(__ldcg(lse_k + size_t(k) * kTileM) - M);
              lt = M + ptx::lg2(sum);
            }
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
              float acc[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[i] = 0.f;
              if (M != -INFINITY) {
                for (int k = 0; k < it.nchunks; ++k) {
                  const size_t sl = size_t(it.first_slot + k) * kTileM + t;
                  const float w = ptx::ex2(__ldcg(p.part_lse + sl) - lt);
                  const float4* srcp = reinterpret_cast<const float4*>(p.part_o + sl * D + 32 * c);
#pragma unroll
                  for (int i = 0; i < 8; ++i) {
                    const float4 x = __ldcg(srcp + i);
                    acc[4 * i] += w * x.x;
                    acc[4 * i + 1] += w * x.y;
                    acc[4 * i + 2] += w * x.z;
                    acc[4 * i + 3] += w * x.w;
                  }
                }
              }
              store_row_chunk(p, orow, c, acc);
            }
            if (p.lse != nullptr) p.lse[orow] = lt * kLn2;
          }
          if (lane == 0) atomicExch(p.counters + it.first_slot * 4 + warp, 0);
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 4 && lane == 0) {
    uint32_t ab;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(ab) : "r"(abort_addr));
    if (ab) {   // let this CTA's copies land before its shared memory is released
      for (int i = 0; i < 2; ++i) {
        ptx::mbar_wait_bounded(BAR(KV_FULL + i), 0, 50000000ull);
        ptx::mbar_wait_bounded(BAR(KV_FULL + i), 1, 50000000ull);
      }
    }
  }
  if (warp == 5) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}

template <bool ROPE>
cudaError_t launch_one(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                       int grid, cudaStream_t stream) {
  auto kern = bsr_prefill_kernel<ROPE>;
  constexpr size_t smem = PrefillSmem<ROPE>::kDynBytes;
  static bool opted_in[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!opted_in[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    opted_in[dev] = true;
  }
  kern<<<grid, PrefillSmem<ROPE>::kThreads, smem, stream>>>(tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(bool rope, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int grid, cudaStream_t stream) {
  return rope ? launch_one<true>(tk, tv, p, grid, stream)
              : launch_one<false>(tk, tv, p, grid, stream);
}

}  // namespace bsr
