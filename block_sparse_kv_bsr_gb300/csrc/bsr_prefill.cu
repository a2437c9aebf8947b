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
//              t.  They load (and RoPE-rotate) Q, rotate each K tile in place
//              when RoPE is on, run the online softmax on S rows read from
//              TMEM, write P (bf16) to shared memory, rescale O in TMEM when the
//              running max grows by more than 2^8, and write out / lse.
//   warp 4     TMA producer: gathers 128-key K and V tiles page by page from
//              `indices` (inactive blocks are absent, "Block-Sparse 포맷") into a
//              two-stage ring of 128B-swizzled tiles.
//   warp 5     allocates TMEM and issues the MMAs: S = Q K^T (M 128, N 128,
//              8 x K16, K-major operands) into TMEM columns [0, 128) and
//              O += P V (P K-major from shared memory, V MN-major) into columns
//              [128, 256); completion is signalled with tcgen05.commit.
// With RoPE the rotated q is split into bf16 hi + lo (two QK passes) so the
// fused rotation costs no accuracy on the query side.  A unit whose key range
// was split writes an fp32 partial state; the last arriving CTA merges the
// partials in key order.  Every mbarrier wait is bounded.
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
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;

template <bool ROPE>
struct PrefillSmem {
  static constexpr int kQ = 0;
  static constexpr int kQlo = kQ + kTileBytes;
  static constexpr int kStage0 = ROPE ? kQlo + kTileBytes : kQlo;   // K then V per stage
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kP = kStage0 + 2 * kStageBytes;
  static constexpr int kBars = kP + kTileBytes;
  // barriers: kv_full[2], kv_ready[2], kv_empty[2], s_full, p_full, pv_done, q_full
  static constexpr int kNumBars = 10;
  static constexpr int kTmemSlot = kBars + 8 * kNumBars;
  static constexpr int kFlags = kTmemSlot + 16;   // abort flag, last-arriver flag
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
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ int ntiles_of(const DecodeItem& it) {
  return it.tok1 > it.tok0 ? (it.tok1 - it.tok0 + kTileN - 1) / kTileN : 0;
}

template <bool ROPE>
__global__ void __launch_bounds__(kThreads, 1)
    bsr_prefill_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  using L = PrefillSmem<ROPE>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = (ptx::smem_u32(smem_raw) + 1023u) & ~1023u;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar0 = base + L::kBars;
  auto BAR = [&](int i) { return bar0 + 8u * uint32_t(i); };
  enum { KV_FULL = 0, KV_READY = 2, KV_EMPTY = 4, S_FULL = 6, P_FULL = 7, PV_DONE = 8, Q_FULL = 9 };
  const uint32_t abort_addr = base + L::kFlags;
  Waiter wt{abort_addr, p.wait_limit_ns, p.error};

  const int u_begin = __ldg(p.cta_ptr + blockIdx.x), u_end = __ldg(p.cta_ptr + blockIdx.x + 1);

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(BAR(KV_FULL + i), 1);
      ptx::mbar_init(BAR(KV_READY + i), 128);
      ptx::mbar_init(BAR(KV_EMPTY + i), 1);
    }
    ptx::mbar_init(BAR(S_FULL), 1);
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
  const uint32_t S_T = tmem, O_T = tmem + 128;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_first();
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
          const uint32_t ks = base + L::kStage0 + stage * L::kStageBytes, vs = ks + kTileBytes;
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
      for (int u = u_begin; u < u_end && ok; ++u) {
        const DecodeItem it = p.items[u];
        const int nt = ntiles_of(it);
        if (nt == 0) continue;
        if (!wt.wait(BAR(Q_FULL), qc & 1)) break;
        ++qc;
        umma::fence_after_sync();
        for (int j = 0; j < nt; ++j, ++gt) {
          const int stage = gt & 1;
          const uint32_t n = gt >> 1;
          if (!wt.wait(BAR((ROPE ? KV_READY : KV_FULL) + stage), n & 1)) { ok = false; break; }
          umma::fence_after_sync();
          const uint32_t ks = base + L::kStage0 + stage * L::kStageBytes, vs = ks + kTileBytes;
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
            umma::mma_f16_ss(S_T, umma::sdesc_sw128(base + L::kQ + off, 16, 1024),
                             umma::sdesc_sw128(ks + off, 16, 1024), idesc_qk, k > 0);
          }
          if (ROPE) {
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
              umma::mma_f16_ss(S_T, umma::sdesc_sw128(base + L::kQlo + off, 16, 1024),
                               umma::sdesc_sw128(ks + off, 16, 1024), idesc_qk, 1);
            }
          }
          umma::commit(BAR(S_FULL));
          if (!wt.wait(BAR(P_FULL), gt & 1)) { ok = false; break; }
          umma::fence_after_sync();
          const int key0 = it.tok0 + kTileN * j;
          const int nk16 = (min(kTileN, it.tok1 - key0) + 15) >> 4;
          for (int k = 0; k < nk16; ++k) {
            const uint32_t aoff = (k >> 2) * kHalfBytes + (k & 3) * 32;
            umma::mma_f16_ss(O_T, umma::sdesc_sw128(base + L::kP + aoff, 16, 1024),
                             umma::sdesc_sw128(vs + k * 2048, kHalfBytes, 1024), idesc_pv,
                             (j > 0 || k > 0) ? 1u : 0u);
          }
          umma::commit(BAR(KV_EMPTY + stage));
          umma::commit(BAR(PV_DONE));
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
        // ---- Q row t (RoPE-rotated, split hi/lo when RoPE is on)
        uint4 qraw[16];
        const uint4* src = reinterpret_cast<const uint4*>(p.q + orow * D);
#pragma unroll
        for (int c = 0; c < 16; ++c) qraw[c] = vrow ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        if (!ROPE) {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + L::kQ + sw_off(t, c)),
                         "r"(qraw[c].x), "r"(qraw[c].y), "r"(qraw[c].z), "r"(qraw[c].w) : "memory");
          }
        } else {
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
              const float x0 = a0 * cs.x - b0 * cs.y, y0 = b0 * cs.x + a0 * cs.y;
              const float x1 = a1 * cs.z - b1 * cs.w, y1 = b1 * cs.z + a1 * cs.w;
              ptx::split_bf16(x0, x1, xh[e], xl[e]);
              ptx::split_bf16(y0, y1, yh[e], yl[e]);
            }
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + L::kQ + sw_off(t, c)),
                         "r"(xh[0]), "r"(xh[1]), "r"(xh[2]), "r"(xh[3]) : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + L::kQ + sw_off(t, c + 8)),
                         "r"(yh[0]), "r"(yh[1]), "r"(yh[2]), "r"(yh[3]) : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + L::kQlo + sw_off(t, c)),
                         "r"(xl[0]), "r"(xl[1]), "r"(xl[2]), "r"(xl[3]) : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + L::kQlo + sw_off(t, c + 8)),
                         "r"(yl[0]), "r"(yl[1]), "r"(yl[2]), "r"(yl[3]) : "memory");
          }
        }
        ptx::fence_proxy_async_smem();
        mbar_arrive(BAR(Q_FULL));

        for (int j = 0; j < nt; ++j, ++gt) {
          const int stage = gt & 1;
          const uint32_t n = gt >> 1;
          const int key0 = it.tok0 + kTileN * j;
          const int nkeys = min(kTileN, it.tok1 - key0);
          const uint32_t ks = base + L::kStage0 + stage * L::kStageBytes, vs = ks + kTileBytes;
          if (ROPE) {
            // rotate key row t of the tile in place (both 64-column blocks)
            if (!__all_sync(0xffffffffu, wt.wait(BAR(KV_FULL + stage), n & 1))) { ok = false; break; }
            if (t < nkeys) {
              const float4* tab = reinterpret_cast<const float4*>(
                  p.rope_nat + size_t(min(key0 + t, p.rope_max_pos)) * (D / 2));
#pragma unroll 2
              for (int c = 0; c < 8; ++c) {
                uint4 av, bv;
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(av.x), "=r"(av.y), "=r"(av.z), "=r"(av.w) : "r"(ks + sw_off(t, c)));
                asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(bv.x), "=r"(bv.y), "=r"(bv.z), "=r"(bv.w) : "r"(ks + sw_off(t, c + 8)));
                const uint32_t* a = reinterpret_cast<const uint32_t*>(&av);
                const uint32_t* b = reinterpret_cast<const uint32_t*>(&bv);
                uint32_t xo[4], yo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const float4 cs = __ldg(tab + 4 * c + e);
                  const float a0 = ptx::bf16_lo(a[e]), a1 = ptx::bf16_hi(a[e]);
                  const float b0 = ptx::bf16_lo(b[e]), b1 = ptx::bf16_hi(b[e]);
                  xo[e] = ptx::pack_bf16(a0 * cs.x - b0 * cs.y, a1 * cs.z - b1 * cs.w);
                  yo[e] = ptx::pack_bf16(b0 * cs.x + a0 * cs.y, b1 * cs.z + a1 * cs.w);
                }
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(ks + sw_off(t, c)),
                             "r"(xo[0]), "r"(xo[1]), "r"(xo[2]), "r"(xo[3]) : "memory");
                asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(ks + sw_off(t, c + 8)),
                             "r"(yo[0]), "r"(yo[1]), "r"(yo[2]), "r"(yo[3]) : "memory");
              }
            }
            ptx::fence_proxy_async_smem();
            mbar_arrive(BAR(KV_READY + stage));
          }

          // ---- S row t from TMEM; mask, online softmax (log2 domain, lazy rescale)
          if (!__all_sync(0xffffffffu, wt.wait(BAR(S_FULL), gt & 1))) { ok = false; break; }
          umma::fence_after_sync();
          float s[kTileN];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float v[32];
            umma::tmem_ld32(S_T + lane_off + 32 * c, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) s[32 * c + i] = v[i];
          }
          const int klim = p.causal ? min(nkeys, qpos - key0 + 1) : nkeys;   // keys [0, klim) visible
          float mx = -INFINITY;
#pragma unroll
          for (int c = 0; c < kTileN; ++c) {
            s[c] = c < klim ? s[c] * p.scale_log2 : -INFINITY;
            mx = fmaxf(mx, s[c]);
          }
          float alpha = 1.f;
          if (mx > m_used + 8.f) {          // also true the first time a row sees a key
            alpha = m_used == -INFINITY ? 0.f : ptx::ex2(m_used - mx);
            m_used = mx;
          }
          const float mu = m_used == -INFINITY ? 0.f : m_used;
          float rs = 0.f;
          uint32_t pk[kTileN / 2];
#pragma unroll
          for (int c = 0; c < kTileN; c += 2) {
            const float p0 = ptx::ex2(s[c] - mu), p1 = ptx::ex2(s[c + 1] - mu);
            rs += p0 + p1;
            pk[c / 2] = ptx::pack_bf16(p0, p1);
          }
          l = l * alpha + rs;

          // P buffer and O are free once the previous P.V has completed
          if (j > 0) {
            if (!__all_sync(0xffffffffu, wt.wait(BAR(PV_DONE), (gt - 1) & 1))) { ok = false; break; }
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
          // V rows past the last valid key of the final 16-key group may hold
          // another page's tail: zero them so that P = 0 contributes exactly 0.
          if (t >= nkeys && t < ((nkeys + 15) & ~15)) {
#pragma unroll
            for (int c = 0; c < 16; ++c)
              asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vs + sw_off(t, c)), "r"(0u)
                           : "memory");
          }
#pragma unroll
          for (int c = 0; c < 16; ++c)
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(base + L::kP + sw_off(t, c)),
                         "r"(pk[4 * c]), "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                         : "memory");
          ptx::fence_proxy_async_smem();
          umma::fence_before_sync();
          mbar_arrive(BAR(P_FULL));
        }
        if (!ok) break;
        if (!__all_sync(0xffffffffu, wt.wait(BAR(PV_DONE), (gt - 1) & 1))) { ok = false; break; }
        umma::fence_after_sync();
      }

      // ---- epilogue: O row t / l  (an empty unit writes 0 / -inf)
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse2 = l > 0.f ? m_used + ptx::lg2(l) : -INFINITY;
      constexpr float kLn2 = 0.69314718055994530942f;
      float o[kTileN];
      if (nt > 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[32];
          umma::tmem_ld32(O_T + lane_off + 32 * c, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[32 * c + i] = v[i] * inv;
        }
      } else {
#pragma unroll
        for (int i = 0; i < D; ++i) o[i] = 0.f;
      }
      umma::fence_before_sync();
      if (it.slot < 0) {
        if (vrow) {
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * D);
#pragma unroll
            for (int c = 0; c < D / 4; ++c)
              dst[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow * D);
#pragma unroll
            for (int c = 0; c < D / 8; ++c)
              dst[c] = make_uint4(ptx::pack_bf16(o[8 * c], o[8 * c + 1]),
                                  ptx::pack_bf16(o[8 * c + 2], o[8 * c + 3]),
                                  ptx::pack_bf16(o[8 * c + 4], o[8 * c + 5]),
                                  ptx::pack_bf16(o[8 * c + 6], o[8 * c + 7]));
          }
          if (p.lse != nullptr) p.lse[orow] = lse2 * kLn2;
        }
      } else {
        float4* dst = reinterpret_cast<float4*>(p.part_o + (size_t(it.slot) * kTileM + t) * D);
#pragma unroll
        for (int c = 0; c < D / 4; ++c)
          __stcg(dst + c, make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]));
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
            float M = -INFINITY;
            for (int k = 0; k < it.nchunks; ++k)
              M = fmaxf(M, __ldcg(p.part_lse + size_t(it.first_slot + k) * kTileM + t));
            float acc[D];
#pragma unroll
            for (int i = 0; i < D; ++i) acc[i] = 0.f;
            float lt = -INFINITY;
            if (M != -INFINITY) {
              float sum = 0.f;
              for (int k = 0; k < it.nchunks; ++k)
                sum += ptx::ex2(__ldcg(p.part_lse + size_t(it.first_slot + k) * kTileM + t) - M);
              lt = M + ptx::lg2(sum);
              for (int k = 0; k < it.nchunks; ++k) {
                const size_t sl = size_t(it.first_slot + k) * kTileM + t;
                const float w = ptx::ex2(__ldcg(p.part_lse + sl) - lt);
                const float4* srcp = reinterpret_cast<const float4*>(p.part_o + sl * D);
#pragma unroll
                for (int c = 0; c < D / 4; ++c) {
                  const float4 v = __ldcg(srcp + c);
                  acc[4 * c] += w * v.x;
                  acc[4 * c + 1] += w * v.y;
                  acc[4 * c + 2] += w * v.z;
                  acc[4 * c + 3] += w * v.w;
                }
              }
            }
            if (p.out_f32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * D);
#pragma unroll
              for (int c = 0; c < D / 4; ++c)
                dst[c] = make_float4(acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + orow * D);
#pragma unroll
              for (int c = 0; c < D / 8; ++c)
                dst[c] = make_uint4(ptx::pack_bf16(acc[8 * c], acc[8 * c + 1]),
                                    ptx::pack_bf16(acc[8 * c + 2], acc[8 * c + 3]),
                                    ptx::pack_bf16(acc[8 * c + 4], acc[8 * c + 5]),
                                    ptx::pack_bf16(acc[8 * c + 6], acc[8 * c + 7]));
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
  kern<<<grid, kThreads, smem, stream>>>(tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(bool rope, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int grid, cudaStream_t stream) {
  return rope ? launch_one<true>(tk, tv, p, grid, stream)
              : launch_one<false>(tk, tv, p, grid, stream);
}

}  // namespace bsr
