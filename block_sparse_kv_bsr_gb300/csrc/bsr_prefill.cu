// Prefill / multi-query attention over a paged (BSR) KV cache on the sm_103a
// tensor cores (tcgen05 + TMEM), head_dim 128.
//
// Prefill is compute-bound ("FlashInfer: Block-Sparse KV 캐시로 어텐션 병목을
// 해소하다", section "어텐션 연산에서 진짜 병목은 어디인가?"): many query rows
// share every key, so the work is a real dense contraction.  One work unit is
// a tile of 128 packed (query, head) rows of one (request, kv head) against a
// page-aligned key range; a CTA walks its planned list of units.
//
// Roles (192 threads):
//   warps 0-3  row owners: thread t owns packed row t of the tile and TMEM lane
//              t.  They load Q (RoPE-rotated and split into bf16 hi + lo, so
//              QK^T takes two passes), run the online softmax on S rows read
//              from TMEM (one 128-column load per tile), write P (bf16) to
//              shared memory, rescale O in TMEM when the running max grows by
//              more than 2^8, and write out / lse.
//   warp 4     TMA producer: gathers 128-key K and V tiles page by page from
//              `indices` (inactive blocks are absent, "Block-Sparse 포맷") into
//              two-stage K and V rings of 128B-swizzled tiles.  A K stage is
//              released as soon as Q K^T has read it, so K runs ahead of V.
//              With RoPE, K comes already rotated from a dense buffer that a
//              pre-pass fills once per run (every key is read by many row
//              tiles, so rotating it once is cheaper than once per tile).
//   warp 5     allocates TMEM and issues the MMAs: S = Q K^T (M 128, N 128,
//              8 x K16, K-major operands) into one of two TMEM S buffers, and
//              O += P V (P K-major from shared memory, V MN-major) into a TMEM
//              O buffer.  S is double-buffered so that Q K^T of a tile runs on
//              the tensor cores while the row owners work on the previous one.
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
  static constexpr int kThreads = 192;
  static constexpr int kQ = 0;
  static constexpr int kQlo = kQ + kTileBytes;                     // RoPE: low half of the split q
  static constexpr int kK0 = ROPE ? kQlo + kTileBytes : kQlo;      // K ring: 2 tiles
  static constexpr int kV0 = kK0 + 2 * kTileBytes;                 // V ring: 2 tiles
  static constexpr int kP = kV0 + 2 * kTileBytes;
  static constexpr int kBars = kP + kTileBytes;
  // barriers: k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full, pv_done, q_full
  static constexpr int kNumBars = 13;
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
  enum { K_FULL = 0, K_EMPTY = 2, V_FULL = 4, V_EMPTY = 6, S_FULL = 8, P_FULL = 10, PV_DONE = 11,
         Q_FULL = 12 };
  const uint32_t abort_addr = base + L::kFlags;
  Waiter wt{abort_addr, p.wait_limit_ns, p.error};

  const int u_begin = __ldg(p.cta_ptr + blockIdx.x), u_end = __ldg(p.cta_ptr + blockIdx.x + 1);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(BAR(K_FULL + i), 1);
      ptx::mbar_init(BAR(K_EMPTY + i), 1);
      ptx::mbar_init(BAR(V_FULL + i), 1);
      ptx::mbar_init(BAR(V_EMPTY + i), 1);
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
  auto stage_k = [&](uint32_t g) { return base + L::kK0 + (g & 1u) * kTileBytes; };
  auto stage_v = [&](uint32_t g) { return base + L::kV0 + (g & 1u) * kTileBytes; };

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      // K/V tiles are re-read by the other row tiles of the same (request, kv head),
      // which run concurrently on other SMs: keep them in L2 at normal priority.
      const uint64_t pol = ptx::policy_evict_normal();
      // Tiles are issued in order; the V of tile g - 1 goes out after the K of tile g,
      // so K (released early, after Q K^T) runs ahead of V (released after P V).
      struct Tile {
        int pages[kTileN / 16];   // page id of each 16-key block
        int kvh, nsub, key0, krow;
      };
      Tile cur{}, prev{};
      bool have_prev = false;
      uint32_t gt = 0;
      bool ok = true;
      auto issue_v = [&](const Tile& tl, uint32_t g) -> bool {
        const int st = g & 1;
        if (g >= 2 && !wt.wait(BAR(V_EMPTY + st), ((g >> 1) - 1) & 1)) return false;
        ptx::mbar_arrive_expect_tx(BAR(V_FULL + st), uint32_t(tl.nsub) * 2u * 2048u);
        const uint32_t vs = stage_v(g);
        for (int sb = 0; sb < tl.nsub; ++sb) {
          const int row = (tl.pages[sb] * p.Hk + tl.kvh) * p.P + ((tl.key0 + 16 * sb) % p.P);
          for (int h = 0; h < 2; ++h)
            ptx::tma_load_3d(vs + h * kHalfBytes + sb * 2048, &tm_v, BAR(V_FULL + st), 0, h, row, pol);
        }
        return true;
      };
      for (int u = u_begin; u < u_end && ok; ++u) {
        const DecodeItem it = p.items[u];
        const int nt = ntiles_of(it);
        const int koff = ROPE ? __ldg(p.rk_off + it.req) : 0;
        for (int j = 0; j < nt; ++j, ++gt) {
          cur.kvh = it.kvh;
          cur.key0 = it.tok0 + kTileN * j;
          cur.nsub = (min(kTileN, it.tok1 - cur.key0) + 15) >> 4;
          // all page ids of the tile first (independent loads), then the copies
#pragma unroll
          for (int sb = 0; sb < kTileN / 16; ++sb)
            cur.pages[sb] = sb < cur.nsub ? __ldg(p.indices + it.page_base + (cur.key0 + 16 * sb) / p.P) : 0;
          const int st = gt & 1;
          if (gt >= 2 && !wt.wait(BAR(K_EMPTY + st), ((gt >> 1) - 1) & 1)) { ok = false; break; }
          const uint32_t ks = stage_k(gt);
          if (ROPE) {
            // rotated keys are dense per (kv head, request): one box per 64-column block
            ptx::mbar_arrive_expect_tx(BAR(K_FULL + st), 2u * uint32_t(kHalfBytes));
            const int row = it.kvh * p.rk_total + koff + cur.key0;
            for (int h = 0; h < 2; ++h)
              ptx::tma_load_3d(ks + h * kHalfBytes, &tm_k, BAR(K_FULL + st), 0, h, row, pol);
          } else {
            ptx::mbar_arrive_expect_tx(BAR(K_FULL + st), uint32_t(cur.nsub) * 2u * 2048u);
            for (int sb = 0; sb < cur.nsub; ++sb) {
              const int row = (cur.pages[sb] * p.Hk + it.kvh) * p.P + ((cur.key0 + 16 * sb) % p.P);
              for (int h = 0; h < 2; ++h)
                ptx::tma_load_3d(ks + h * kHalfBytes + sb * 2048, &tm_k, BAR(K_FULL + st), 0, h, row, pol);
            }
          }
          if (have_prev && !issue_v(prev, gt - 1)) { ok = false; break; }
          prev = cur;
          have_prev = true;
        }
      }
      if (ok && have_prev) issue_v(prev, gt - 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma::idesc_bf16_f32(kTileM, kTileN, 0, 0);
      constexpr uint32_t idesc_pv = umma::idesc_bf16_f32(kTileM, D, 0, 1);
      uint32_t gt = 0, qc = 0;   // tiles and non-empty units seen so far
      bool ok = true;
      // S(g) = Q K(g)^T into S buffer g % 2, once tile g's K is in shared memory;
      // the K stage is handed back to the producer as soon as these MMAs complete.
      auto issue_qk = [&](uint32_t g) -> bool {
        if (!wt.wait(BAR(K_FULL + (g & 1)), (g >> 1) & 1)) return false;
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
        umma::commit(BAR(K_EMPTY + (g & 1)));
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
          if (!wt.wait(BAR(V_FULL + (gt & 1)), (gt >> 1) & 1)) { ok = false; break; }
          umma::fence_after_sync();
          const uint32_t vs = stage_v(gt);
          const int key0 = it.tok0 + kTileN * j;
          const int nk16 = (min(kTileN, it.tok1 - key0) + 15) >> 4;
          for (int k = 0; k < nk16; ++k) {
            const uint32_t aoff = (k >> 2) * kHalfBytes + (k & 3) * 32;
            umma::mma_f16_ss(O_T, umma::sdesc_sw128(base + L::kP + aoff, 16, 1024),
                             umma::sdesc_sw128(vs + k * 2048, kHalfBytes, 1024), idesc_pv,
                             (j > 0 || k > 0) ? 1u : 0u);
          }
          umma::commit(BAR(V_EMPTY + (gt & 1)));
          umma::commit(BAR(PV_DONE));
          // S buffer gt % 2 was read by the row owners before P_FULL: refill it with tile j + 2
          if (j + 2 < nt && !issue_qk(gt + 2)) { ok = false; break; }
        }
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
          // another page's tail: zero them (once the copy has landed) so that
          // P = 0 contributes exactly 0.
          if (nkeys & 15) {
            const bool mine = t >= nkeys && t < ((nkeys + 15) & ~15);
            if (__any_sync(0xffffffffu, mine)) {
              if (!wt.warp_wait(BAR(V_FULL + (gt & 1)), (gt >> 1) & 1)) { ok = false; break; }
              if (mine) {
#pragma unroll
                for (int c = 0; c < 16; ++c) sts128(stage_v(gt) + sw_off(t, c), 0u, 0u, 0u, 0u);
              }
            }
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
        for (int b = 0; b < 2; ++b) {
          ptx::mbar_wait_bounded(BAR(K_FULL + i), b, 50000000ull);
          ptx::mbar_wait_bounded(BAR(V_FULL + i), b, 50000000ull);
        }
      }
    }
  }
  if (warp == 5) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}


// ---------------------------------------------------------------- RoPE pre-pass
// One thread per (kv head, key row, 16-byte column chunk of the first half):
// rotates the pair of chunks (d, d + 64) of one key at its position in the
// request's page list and writes it to the dense rotated-K buffer.  Threads
// walk rows fastest, so reads follow the pages and writes are contiguous.
__global__ void __launch_bounds__(256) rope_k_prepass_kernel(const RopeKParams p) {
  const int64_t total = int64_t(p.Hk) * p.rk_total * 8;
  for (int64_t g = int64_t(blockIdx.x) * 256 + threadIdx.x; g < total; g += int64_t(gridDim.x) * 256) {
    const int c = int(g & 7);
    const int64_t hr = g >> 3;
    const int kvh = int(hr / p.rk_total);
    const int r = int(hr % p.rk_total);
    int lo = 0, hi = p.n - 1;   // request i with rk_start[i] <= r < rk_start[i + 1]
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.rk_start + mid) <= r) lo = mid; else hi = mid - 1;
    }
    const int j = r - __ldg(p.rk_start + lo);
    const int page = __ldg(p.indices + __ldg(p.rk_req_pbase + lo) + j / p.P);
    const uint16_t* src = p.k_pages + ((size_t(page) * p.Hk + kvh) * p.P + (j % p.P)) * D;
    const uint4 av = __ldg(reinterpret_cast<const uint4*>(src) + c);
    const uint4 bv = __ldg(reinterpret_cast<const uint4*>(src) + 8 + c);
    const float4* tab = reinterpret_cast<const float4*>(p.rope_nat + size_t(min(j, p.rope_max_pos)) * (D / 2));
    const uint32_t* a = reinterpret_cast<const uint32_t*>(&av);
    const uint32_t* b = reinterpret_cast<const uint32_t*>(&bv);
    uint32_t xo[4], yo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float4 cs = __ldg(tab + 4 * c + e);   // frequencies 8c + 2e, 8c + 2e + 1
      const float a0 = ptx::bf16_lo(a[e]), a1 = ptx::bf16_hi(a[e]);
      const float b0 = ptx::bf16_lo(b[e]), b1 = ptx::bf16_hi(b[e]);
      xo[e] = ptx::pack_bf16(a0 * cs.x - b0 * cs.y, a1 * cs.z - b1 * cs.w);
      yo[e] = ptx::pack_bf16(b0 * cs.x + a0 * cs.y, b1 * cs.z + a1 * cs.w);
    }
    uint4* dst = reinterpret_cast<uint4*>(p.rotk + (size_t(kvh) * p.rk_total + r) * D);
    dst[c] = make_uint4(xo[0], xo[1], xo[2], xo[3]);
    dst[8 + c] = make_uint4(yo[0], yo[1], yo[2], yo[3]);
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

cudaError_t launch_rope_k_prepass(const RopeKParams& p, int num_sms, cudaStream_t stream) {
  const int64_t work = int64_t(p.Hk) * p.rk_total * 8;
  int64_t grid = (work + 255) / 256;
  if (grid > int64_t(num_sms) * 8) grid = int64_t(num_sms) * 8;
  if (grid < 1) grid = 1;
  rope_k_prepass_kernel<<<int(grid), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prefill(bool rope, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int grid, cudaStream_t stream) {
  return rope ? launch_one<true>(tk, tv, p, grid, stream)
              : launch_one<false>(tk, tv, p, grid, stream);
}

}  // namespace bsr
