// Host planner for BSR (paged) attention: validates the block table, cuts each
// (request, kv head, packed-row group) key range into page-aligned work units,
// spreads the units over persistent warps at equal cost, and uploads
// everything the kernels read in one asynchronous copy.
//
// The scheduling idea follows "FlashInfer: Block-Sparse KV 캐시로 어텐션
// 병목을 해소하다" (visionhong.com), section "벤치마크: FlashInfer는 얼마나
// 빠른가?": long sequences are split into smaller work units and interleaved
// with short ones so that every workgroup stays busy on a skewed batch.  The
// block table follows section "FlashInfer는 KV 캐시를 어떻게 통합하는가?:
// Block-Sparse 포맷" (active blocks listed per request, inactive ones absent).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <numeric>
#include <vector>

#include "bsr_attn.h"
#include "bsr_schedule.h"

namespace {

using bsr::DecodeItem;
using bsr::kDecodeWarps;
using bsr::kMaxDecodeRows;
using bsr::kStageTokens;

constexpr size_t kAlign = 256;
// Cost of one decode work unit beyond its keys (q load, epilogue), in key-equivalents,
// and the extra cost of each piece of a split range (its partial write, arrival and
// its share of the merge); used only to weigh units against each other.  A fit of the
// decode kernel's per-warp busy times (clock stamps of every warp of the skewed
// 128-request batch over 16 launches, against the keys, pieces and split pieces each
// warp was given) put them at ~33 and ~69 key-equivalents.  The split surcharge stays
// at 16: at the fitted value a uniform batch (512 equal ranges over 1216 warps) is cut
// into fewer pieces than it has warps, 3-4 % slower; at 16 its cut is unchanged.
constexpr int64_t kUnitOverhead = 32;
constexpr int64_t kSplitOverhead = 16;
// Shortest piece a key range is cut into (keys): below this the partial
// write and merge cost more than the balance gains.
constexpr int64_t kMinPiece = 64;
// The same for a batch too small to give every warp of the GPU kMinWarpWork.
// Such a batch is latency-bound: its longest range's chain of dependent stages
// sets the time, and a warp takes ~0.6 us per 16-key stage even with the data
// landed, against ~4 us for a split range's partial write, arrival and merge.
// Cutting a 255-key range into four pieces instead of two took a 4-request
// decode from ~10 to ~7.5 us; applied to full batches the shorter pieces only
// add merges (1.3 % on the skewed 128-request decode), so they stay at kMinPiece.
constexpr int64_t kMinPieceSmall = 32;
// Least work (key-equivalents) worth a warp of its own: small batches use
// fewer warps instead of many tiny pieces.
constexpr int64_t kMinWarpWork = 64;
// Run-time units: the shortest whole ranges, up to this share of a decode batch's cost,
// each at most a quarter of a warp's mean share, are left out of the static cut and taken at
// run time by warps that have finished their own lists (longest first), so the spread
// of finishing times that a static cut cannot foresee (SMs that stream slower, units
// that cost more than planned) is filled instead of waited for.  Only for skewed
// batches (some range is at least kDynSkew warps' mean share: the long ranges are cut
// over many warps anyway and the short ones are the natural fill) with enough work to
// keep every warp busy, pages of 16 keys or more, a bf16 cache and no RoPE.  Measured
// on GB300: the skewed 128-request decode 3.5 % faster (NHD pages 4 %); with RoPE at
// logical positions 9 % slower and on a cascade's suffix level (no range longer than a
// warp's share) 3.4 % slower, hence the conditions.
constexpr double kDynShare = 0.15;
constexpr int64_t kDynMinWarpWork = 256;
constexpr int64_t kDynSkew = 4;
// Prefill: packed rows from which a request takes the tensor-core kernel, the
// per-unit overhead (Q load, pipeline fill, epilogue) in keys, the shortest
// key piece and the least work per CTA.
constexpr int32_t kPrefillMinRows = 64;
constexpr int64_t kPrefillOverhead = 256;
constexpr int64_t kPrefillMinPiece = 512;
constexpr int64_t kPrefillMinCtaWork = 1024;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
// warps per SM that the decode kernel of a cache type keeps
int decode_warps_per_sm(int32_t kv_dtype, bool rope) {
  return kv_dtype == BSR_KV_DTYPE_E4M3 ? bsr::decode_kv8_warps(rope) : kDecodeWarps;
}
bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

// A (request, kv head, row group) range of keys before chunking.
struct Unit {
  int32_t req, kvh, row0, nrows, kend;
  int32_t page_base, q_row0, qpos0;
  int32_t kbegin;   // first key any of the rows may see (aligned down to the cut alignment)
};

// cos/sin of every (position, frequency), angles in fp64 rounded once to fp32, in two
// orders.  frag: the order the decode kernel's fragments consume them, per position
// D/4 groups of two (cos, sin) pairs, group i * 4 + t (quad t < 4, i < D/16) holding
// frequencies 16 * (i / 2) + 8 * (i % 2) + 2t + {0, 1}.  pairs: frequency order by
// pairs, per position D/4 float4 (cos f, cos f+1, sin f, sin f+1) for f = 0, 2, ...
// (the tensor-core prefill kernel, which rotates its tiles in shared memory two
// frequencies per packed instruction).
void build_rope_tables(float* frag, float* pairs, int32_t rows, int32_t D, double theta) {
  std::vector<double> omega(D / 2);
  for (int f = 0; f < D / 2; ++f) omega[f] = std::pow(theta, -2.0 * double(f) / double(D));
  for (int32_t pos = 0; pos < rows; ++pos)
    for (int f = 0; f < D / 2; ++f) {
      const double a = double(pos) * omega[f];
      const float c = float(std::cos(a)), sn = float(std::sin(a));
      const int i = 2 * (f / 16) + (f % 16) / 8, t = (f % 8) / 2, e = f % 2;
      float* fr = frag + ((size_t(pos) * (D / 4) + i * 4 + t) * 2 + e) * 2;
      float* pr = pairs + (size_t(pos) * (D / 4) + f / 2) * 4 + e;
      fr[0] = pr[0] = c;
      fr[1] = pr[2] = sn;
    }
}

int fail_cuda(cudaError_t e) {
  cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? BSR_ERR_OUT_OF_MEMORY : BSR_ERR_CUDA;
}

// One kernel's work list: items grouped by worker (a decode warp or a prefill CTA).
struct WorkList {
  std::vector<DecodeItem> items;
  std::vector<int32_t> ptr;          // [workers + 1]
  int32_t n_partials = 0, n_split = 0, workers = 0;
  double imbalance = 1.0;
  // decode only: items [dyn_begin, dyn_begin + n_dyn), after every worker's list, are
  // taken at run time by whichever worker is free (longest first)
  int32_t n_dyn = 0, dyn_begin = 0;
};

// The ranges to cut, longest first, and the limits of the cut.
struct CutInput {
  const int64_t* kb;   // first key of each range, in cut order
  const int64_t* ke;   // one past its last key
  size_t n;
  int64_t overhead, align_mask, min_piece, max_workers;   // align_mask: ~(align - 1)
  int workers;
  int64_t split_overhead;   // extra cost of every piece of a range that is cut
};

// Cut with budget T: ranges are laid end to end and each worker takes pieces until
// the next one would pass T; a range that does not fit is cut at an `align`-key
// boundary (no piece shorter than `min_piece`) and continues on the next worker.
// `align` is a power of two, so rounding down is a mask (a negative length rounds
// to a negative take, which places no piece, as a truncating division would).
// Calls emit(range, tok0, tok1, worker) for every piece in order and returns the
// number of workers the cut needs (anything above `workers` means "does not fit").
template <class Emit>
int64_t cut_ranges(const CutInput& in, int64_t T, Emit&& emit) {
  int64_t w = 0, room = T;
  for (size_t oi = 0; oi < in.n; ++oi) {
    const int64_t kend = in.ke[oi];
    int64_t pos = in.kb[oi];
    for (;;) {   // until the piece ending at kend is placed (an empty range still needs one)
      const int64_t rest = kend - pos;
      const int64_t last_cost = rest + in.overhead + (pos != in.kb[oi] ? in.split_overhead : 0);
      if (last_cost <= room) {
        emit(oi, pos, kend, w);
        room -= last_cost;
        break;
      }
      int64_t take = (room - in.overhead - in.split_overhead) & in.align_mask;
      if (rest - take < in.min_piece) take = (rest - in.min_piece) & in.align_mask;
      if (take >= in.min_piece) {
        emit(oi, pos, pos + take, w);
        pos += take;
      } else if (room == T) {
        return in.max_workers + 2;  // budget below one piece: cannot make progress
      }
      ++w;
      room = T;
      if (w >= in.workers) return w + 1;
    }
  }
  return w + 1;
}

// Cut key ranges into pieces and spread them over at most `max_workers`
// workers at equal cost.  Ranges are laid end to end, longest first, and the
// sequence is cut into consecutive per-worker segments of (almost) equal
// cost: a range that does not fit the current worker's budget is cut at an
// `align`-key boundary and its remainder continues on the next worker.  Long
// ranges therefore spread over many workers while short ones fill the rest
// (the interleaving of long and short work).  The budget is the smallest one
// for which the cut fits the workers, found by bisection, so the busiest
// worker carries about one piece-alignment more than the mean.  The result
// is a pure function of its inputs.  `align` is a power of two (a page or a
// key tile).
void balance(const std::vector<Unit>& units, int64_t max_workers, int64_t align, int64_t overhead,
             int64_t min_piece, int64_t min_worker_work, WorkList* out, int64_t* k_hint = nullptr,
             int64_t min_piece_small = 0, int64_t split_overhead = 0) {
  // Working arrays live across calls (per thread), so a plan per decode step reuses
  // their memory instead of faulting in fresh pages.
  struct Scratch {
    std::vector<uint32_t> key, key_tmp;
    std::vector<int32_t> order, order_tmp, pieces_of_unit, first_slot, next_slot;
    std::vector<int64_t> kb, ke, load;
  };
  thread_local Scratch sc;
  const size_t n = units.size();
  // Longest first, ties in unit order: a stable radix sort (8-bit digits, least
  // significant first) on INT32_MAX - length, skipping digits all ranges share.
  sc.key.resize(n);
  sc.key_tmp.resize(n);
  sc.order.resize(n);
  sc.order_tmp.resize(n);
  uint32_t hist[4][256] = {};
  for (size_t i = 0; i < n; ++i) {
    const uint32_t d = uint32_t(INT32_MAX - (units[i].kend - units[i].kbegin));
    sc.key[i] = d;
    sc.order[i] = int32_t(i);
    for (int b = 0; b < 4; ++b) ++hist[b][(d >> (8 * b)) & 255u];
  }
  for (int b = 0; b < 4 && n > 0; ++b) {
    const int sh = 8 * b;
    if (hist[b][(sc.key[0] >> sh) & 255u] == n) continue;
    uint32_t off[256], run = 0;
    for (int v = 0; v < 256; ++v) {
      off[v] = run;
      run += hist[b][v];
    }
    for (size_t i = 0; i < n; ++i) {
      const uint32_t dst = off[(sc.key[i] >> sh) & 255u]++;
      sc.key_tmp[dst] = sc.key[i];
      sc.order_tmp[dst] = sc.order[i];
    }
    sc.key.swap(sc.key_tmp);
    sc.order.swap(sc.order_tmp);
  }
  const std::vector<int32_t>& order = sc.order;
  // key ranges in that order, contiguous for the cut passes
  std::vector<int64_t>& kb = sc.kb;
  std::vector<int64_t>& ke = sc.ke;
  kb.resize(n);
  ke.resize(n);
  for (size_t i = 0; i < n; ++i) {
    kb[i] = units[order[i]].kbegin;
    ke[i] = units[order[i]].kend;
  }
  int64_t total = 0;
  for (const Unit& u : units) total += u.kend - u.kbegin + overhead;
  const int workers =
      units.empty() ? 0
                    : int(std::max<int64_t>(1, std::min<int64_t>(max_workers, (total + min_worker_work - 1) / min_worker_work)));
  // a batch that leaves workers idle may be cut finer (min_piece_small, when given)
  if (min_piece_small > 0 && workers < max_workers) min_piece = min_piece_small;
  const CutInput in{kb.data(), ke.data(), n, overhead, ~(align - 1), min_piece, max_workers, workers,
                    split_overhead};
  std::vector<int32_t>& pieces_of_unit = sc.pieces_of_unit;
  pieces_of_unit.assign(n, 0);
  int64_t T = 0;
  if (!units.empty()) {
    int64_t lo = std::max<int64_t>((total + workers - 1) / workers, 2 * min_piece + overhead + align);
    // The budget is the smallest T = lo + k (k >= 0) for which the cut fits (the cut
    // needs fewer workers as T grows).  A caller that re-plans similar batches passes
    // the last k as a hint: two cuts confirm it (it fits, k - 1 does not); otherwise
    // a doubling search from one alignment step, then halving.  Either way the same k.
    auto fits = [&](int64_t k) {
      return cut_ranges(in, lo + k, [](size_t, int64_t, int64_t, int64_t) {}) <= workers;
    };
    auto count = [&](size_t oi, int64_t, int64_t, int64_t) { ++pieces_of_unit[order[oi]]; };
    int64_t k = -1;
    // pieces_of_unit is valid only while `counted` is true: the hinted cut below fills it
    // as a side effect, and every path that leaves `counted` false (the hint does not fit,
    // is not the smallest, or the cut stops early) is followed by a reset and a fresh
    // counting cut at the final budget.  Never set `counted` on any other path.
    bool counted = false;
    if (k_hint != nullptr && *k_hint >= 0 && cut_ranges(in, lo + *k_hint, count) <= workers &&
        (*k_hint == 0 || !fits(*k_hint - 1))) {
      k = *k_hint;
      counted = true;
    }
    if (k < 0) {
      if (fits(0)) {
        k = 0;
      } else {
        int64_t bad = 0, good = align;
        while (!fits(good)) {
          bad = good;
          good *= 2;
        }
        while (good - bad > 1) {
          const int64_t mid = bad + (good - bad) / 2;
          if (fits(mid)) good = mid; else bad = mid;
        }
        k = good;
      }
    }
    if (k_hint != nullptr) *k_hint = k;
    T = lo + k;
    if (!counted) {
      pieces_of_unit.assign(n, 0);
      cut_ranges(in, T, count);
    }
  }

  std::vector<int32_t>& first_slot = sc.first_slot;
  std::vector<int32_t>& next_slot = sc.next_slot;
  first_slot.assign(n, -1);
  next_slot.assign(n, 0);
  out->n_partials = 0;
  out->n_split = 0;
  int64_t n_pieces = 0;
  for (size_t u = 0; u < n; ++u) {
    n_pieces += pieces_of_unit[u];
    if (pieces_of_unit[u] > 1) {
      first_slot[u] = out->n_partials;
      out->n_partials += pieces_of_unit[u];
      ++out->n_split;
    }
  }
  // the cut emits pieces worker by worker, so item order is grouped by worker
  out->items.resize(size_t(n_pieces));
  out->ptr.assign(workers + 1, 0);
  std::vector<int64_t>& load = sc.load;
  load.assign(workers, 0);
  if (!units.empty()) {
    int64_t cur = 0;
    int32_t idx = 0;
    cut_ranges(in, T, [&](size_t oi, int64_t tok0, int64_t tok1, int64_t w) {
      while (cur < w) out->ptr[++cur] = idx;
      const int32_t ui = order[oi];
      const Unit& u = units[ui];
      DecodeItem& it = out->items[idx++];
      it.req = u.req;
      it.kvh = u.kvh;
      it.row0 = u.row0;
      it.nrows = u.nrows;
      it.tok0 = int32_t(tok0);
      it.tok1 = int32_t(tok1);
      it.nchunks = pieces_of_unit[ui];
      it.first_slot = first_slot[ui];
      // pieces of a range are cut in key order, so slot order is key order
      it.slot = it.nchunks > 1 ? first_slot[ui] + next_slot[ui]++ : -1;
      it.page_base = u.page_base;
      it.q_row0 = u.q_row0;
      it.qpos0 = u.qpos0;
      load[w] += tok1 - tok0 + overhead + (it.nchunks > 1 ? split_overhead : 0);
    });
    while (cur < workers) out->ptr[++cur] = idx;
  }
  out->workers = workers;
  out->imbalance = 1.0;
  if (workers > 0) {
    const int64_t mx = *std::max_element(load.begin(), load.end());
    const double mean = double(std::accumulate(load.begin(), load.end(), int64_t(0))) / workers;
    out->imbalance = mean > 0 ? double(mx) / mean : 1.0;
  }
}

// Prefill units of one (request, kv head) read the same K/V tiles.  They are planned in
// gangs of up to kMaxGang row units: the gangs are cut and balanced over groups of G
// CTAs (G = the largest gang; balance() with a gang's longest member as its key
// range), and every piece of a gang goes to all its members at once, member r of the
// k-th piece of a group to CTA G * group + (r + k) mod G.  The members of a gang thus
// read each K/V tile within a short window, all but the first from L2, where a cut of
// single units would run them on neighbouring CTAs at drifting times (K/V then come
// from DRAM once per member); the rotation spreads the longer causal members over the
// group.  Gangs too uneven to fill their groups (cost-weighted fill below 90 %) fall
// back to the cut of single units.
void balance_gangs(const std::vector<Unit>& units, int64_t num_ctas, int64_t align,
                   int64_t overhead, int64_t min_piece, int64_t min_cta_work, WorkList* out) {
  constexpr int kMaxGang = 8;
  // gangs: runs of consecutive units of the same (request, kv head), at most kMaxGang long
  std::vector<int32_t> gstart;
  for (size_t i = 0; i < units.size(); ++i) {
    const bool fresh = gstart.empty() || units[i].req != units[gstart.back()].req ||
                       units[i].kvh != units[gstart.back()].kvh ||
                       int32_t(i) - gstart.back() == kMaxGang;
    if (fresh) gstart.push_back(int32_t(i));
  }
  const int ngang = int(gstart.size());
  gstart.push_back(int32_t(units.size()));
  int kGang = 1;
  double filled = 0.0, offered = 0.0;
  for (int g = 0; g < ngang; ++g) kGang = std::max(kGang, int(gstart[g + 1] - gstart[g]));
  for (int g = 0; g < ngang; ++g) {
    int64_t kend = 0, kbegin = INT64_MAX, sum = 0;
    for (int32_t i = gstart[g]; i < gstart[g + 1]; ++i) {
      kend = std::max<int64_t>(kend, units[i].kend);
      kbegin = std::min<int64_t>(kbegin, units[i].kbegin);
      sum += units[i].kend - units[i].kbegin + overhead;
    }
    filled += double(sum);
    offered += double(kGang) * double(kend - kbegin + overhead);
  }
  if (kGang == 1 || num_ctas < kGang || filled < 0.9 * offered) {
    balance(units, num_ctas, align, overhead, min_piece, min_cta_work, out);
    return;
  }
  std::vector<Unit> gunits(ngang);
  for (int g = 0; g < ngang; ++g) {
    Unit u = units[gstart[g]];
    for (int32_t i = gstart[g]; i < gstart[g + 1]; ++i) {
      u.kend = std::max(u.kend, units[i].kend);
      u.kbegin = std::min(u.kbegin, units[i].kbegin);
    }
    u.row0 = g;   // carried through balance() to name the gang
    gunits[g] = u;
  }
  WorkList gw;
  balance(gunits, std::max<int64_t>(1, num_ctas / kGang), align, overhead, min_piece,
          min_cta_work, &gw);

  // a member takes the part of a piece inside its own key range (at least one, possibly
  // empty, piece when it has no key at all)
  auto takes = [&](const DecodeItem& gp, const Unit& u) {
    const int32_t lo = std::max(gp.tok0, u.kbegin), hi = std::min(gp.tok1, u.kend);
    return hi > lo || (u.kend == u.kbegin && gp.tok0 <= u.kbegin && u.kbegin <= gp.tok1);
  };
  std::vector<int32_t> npieces(units.size(), 0);
  for (const DecodeItem& gp : gw.items)
    for (int32_t i = gstart[gp.row0]; i < gstart[gp.row0 + 1]; ++i)
      if (takes(gp, units[i])) ++npieces[i];
  std::vector<int32_t> first_slot(units.size(), -1), next_slot(units.size(), 0);
  out->n_partials = 0;
  out->n_split = 0;
  for (size_t i = 0; i < units.size(); ++i)
    if (npieces[i] > 1) {
      first_slot[i] = out->n_partials;
      out->n_partials += npieces[i];
      ++out->n_split;
    }
  const int workers = gw.workers * kGang;
  std::vector<std::vector<DecodeItem>> per(workers);
  std::vector<int64_t> load(workers, 0);
  // balance() emits a gang's pieces in key order over consecutive groups, so each
  // member meets its pieces in key order: slot order is key order
  for (int w = 0; w < gw.workers; ++w)
    for (int32_t idx = gw.ptr[w], k = 0; idx < gw.ptr[w + 1]; ++idx, ++k) {
      const DecodeItem& gp = gw.items[idx];
      for (int32_t i = gstart[gp.row0]; i < gstart[gp.row0 + 1]; ++i) {
        const Unit& u = units[i];
        if (!takes(gp, u)) continue;
        DecodeItem it{};
        it.req = u.req;
        it.kvh = u.kvh;
        it.row0 = u.row0;
        it.nrows = u.nrows;
        it.tok0 = std::max(gp.tok0, u.kbegin);
        it.tok1 = std::max(it.tok0, std::min(gp.tok1, u.kend));
        it.nchunks = npieces[i];
        it.first_slot = first_slot[i];
        it.slot = it.nchunks > 1 ? first_slot[i] + next_slot[i]++ : -1;
        it.page_base = u.page_base;
        it.q_row0 = u.q_row0;
        it.qpos0 = u.qpos0;
        const int cta = w * kGang + int((i - gstart[gp.row0] + k) % kGang);
        per[cta].push_back(it);
        load[cta] += int64_t(it.tok1 - it.tok0) + overhead;
      }
    }
  out->items.clear();
  out->ptr.assign(workers + 1, 0);
  for (int w = 0; w < workers; ++w) {
    out->items.insert(out->items.end(), per[w].begin(), per[w].end());
    out->ptr[w + 1] = int32_t(out->items.size());
  }
  out->workers = workers;
  out->imbalance = 1.0;
  if (workers > 0) {
    const int64_t mx = *std::max_element(load.begin(), load.end());
    const double mean = double(std::accumulate(load.begin(), load.end(), int64_t(0))) / workers;
    out->imbalance = mean > 0 ? double(mx) / mean : 1.0;
  }
}

// Everything the planner decides without a GPU: validation, units, cuts,
// per-warp item lists.
struct HostPlan {
  int32_t group = 0;
  int64_t sum_qo = 0, active = 0;
  int32_t max_len = 0, max_rows = 0;
  WorkList dec;   // split-KV decode kernel, workers = warps
  int32_t dec_warps_per_cta = 0;   // warps of one decode CTA (one CTA per SM)
  WorkList pre;   // tensor-core prefill kernel, workers = CTAs
  std::vector<DecodeItem> pmerge;   // one entry per prefill unit whose key range was split
  // per-page positions: logical minus cached end of each request, and one past the
  // largest position a stage may touch (sizes the cos/sin table)
  std::vector<int32_t> qshift;
  int64_t max_pos_end = 0;
  // working arrays, kept with the plan so that re-planning reuses their memory
  std::vector<int32_t> kv_len, qo_len, q_row0;
  std::vector<Unit> dunits, punits, dyn_units, dyn_sorted;
  std::vector<int32_t> dyn_idx;
  std::vector<uint8_t> dyn_mark;
};

int make_host_plan(const int32_t* indptr, const int32_t* indices, const int32_t* last_page_len,
                   int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                   int32_t page_size, const int32_t* qo_indptr, int32_t num_pages_in_pool,
                   int32_t causal, int32_t window_left, const int32_t* page_pos,
                   float rope_theta, int num_sms, int dec_warps_per_sm, bool allow_dyn,
                   HostPlan* hp) {
  if (indptr == nullptr || batch < 0 || num_pages_in_pool < 0 || num_sms <= 0)
    return BSR_ERR_INVALID_ARGUMENT;
  if (batch > 0 && last_page_len == nullptr) return BSR_ERR_INVALID_ARGUMENT;
  if (num_qo_heads <= 0 || num_kv_heads <= 0) return BSR_ERR_INVALID_ARGUMENT;
  if (!(rope_theta >= 0.f) || !std::isfinite(rope_theta)) return BSR_ERR_INVALID_ARGUMENT;
  if (causal != 0 && causal != 1) return BSR_ERR_INVALID_ARGUMENT;
  if (window_left < 0) return BSR_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128) return BSR_ERR_UNSUPPORTED;
  if (!is_pow2(page_size) || page_size > 256) return BSR_ERR_UNSUPPORTED;
  if (num_qo_heads % num_kv_heads != 0) return BSR_ERR_UNSUPPORTED;
  const int32_t group = num_qo_heads / num_kv_heads;
  if (group > kMaxDecodeRows) return BSR_ERR_UNSUPPORTED;
  if (int64_t(num_pages_in_pool) * num_kv_heads * page_size > INT32_MAX) return BSR_ERR_UNSUPPORTED;
  const bool rope = rope_theta > 0.f;

  // ---------------------------------------------------------------- table validation
  if (indptr[0] != 0) return BSR_ERR_PAGE_TABLE;
  if (qo_indptr != nullptr && qo_indptr[0] != 0) return BSR_ERR_PAGE_TABLE;
  std::vector<int32_t>& kv_len = hp->kv_len;
  std::vector<int32_t>& qo_len = hp->qo_len;
  std::vector<int32_t>& q_row0 = hp->q_row0;
  kv_len.resize(batch);
  qo_len.resize(batch);
  q_row0.resize(batch);
  int64_t sum_qo = 0, active = 0;
  int32_t max_len = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t n = int64_t(indptr[b + 1]) - indptr[b];
    if (n < 0) return BSR_ERR_PAGE_TABLE;
    int64_t L = 0;
    if (n > 0) {
      if (last_page_len[b] < 1 || last_page_len[b] > page_size) return BSR_ERR_PAGE_TABLE;
      L = (n - 1) * page_size + last_page_len[b];
    }
    if (L > INT32_MAX / 2) return BSR_ERR_UNSUPPORTED;
    const int64_t nq = qo_indptr ? int64_t(qo_indptr[b + 1]) - qo_indptr[b] : 1;
    if (nq < 0) return BSR_ERR_PAGE_TABLE;
    if ((causal || rope) && L > 0 && nq > L) return BSR_ERR_PAGE_TABLE;
    kv_len[b] = int32_t(L);
    qo_len[b] = int32_t(nq);
    q_row0[b] = int32_t(sum_qo);
    sum_qo += nq;
    // keys some row attends: all of them, or the union of the rows' windows
    active += window_left > 0 ? L - std::max<int64_t>(0, L - nq - window_left + 1) : L;
    max_len = std::max<int32_t>(max_len, int32_t(L));
  }
  if (sum_qo > INT32_MAX / num_qo_heads) return BSR_ERR_UNSUPPORTED;
  const int64_t nnz = indptr[batch];
  if (nnz > 0 && indices == nullptr) return BSR_ERR_INVALID_ARGUMENT;
  // range checks as min/max reductions (no early exit, so the loops vectorize)
  auto min_max = [](const int32_t* v, int64_t n, int32_t* mn, int32_t* mx) {
    int32_t a = INT32_MAX, b = INT32_MIN;
    for (int64_t e = 0; e < n; ++e) {
      a = std::min(a, v[e]);
      b = std::max(b, v[e]);
    }
    *mn = a;
    *mx = b;
  };
  if (nnz > 0) {
    int32_t mn, mx;
    min_max(indices, nnz, &mn, &mx);
    if (mn < 0 || mx >= num_pages_in_pool) return BSR_ERR_PAGE_TABLE;
  }
  // per-page logical positions (RoPE over caches with dropped blocks): a 16-key stage
  // must lie inside one page, so pages of fewer than 16 keys are refused with RoPE
  hp->qshift.assign(page_pos ? batch : 0, 0);
  hp->max_pos_end = 0;
  if (page_pos != nullptr) {
    if (rope && page_size < kStageTokens) return BSR_ERR_UNSUPPORTED;
    if (nnz > 0) {
      int32_t mn, mx;
      min_max(page_pos, nnz, &mn, &mx);
      if (mn < 0 || mx > INT32_MAX / 4) return BSR_ERR_PAGE_TABLE;
      hp->max_pos_end = int64_t(mx) + page_size;
    }
    for (int32_t b = 0; b < batch; ++b)
      if (indptr[b + 1] > indptr[b])
        hp->qshift[b] = int32_t(int64_t(page_pos[indptr[b + 1] - 1]) + last_page_len[b] -
                                kv_len[b]);
  }

  // ---------------------------------------------------------------- units
  // A request goes to the tensor-core prefill kernel when its packed rows fill
  // at least half of a 128-row query tile and the layout suits it (pages of at
  // least 16 keys, a head group that divides the 128-row tile, so that a tile is
  // whole queries; head_dim 64 runs the 128-wide tile program with its upper 64
  // dimensions zero); the others use the decode kernel's 16-row groups.  Prefill
  // units hold up to two query tiles (256 rows).
  std::vector<Unit>& dunits = hp->dunits;
  std::vector<Unit>& punits = hp->punits;
  dunits.clear();
  punits.clear();
  int32_t max_rows = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const int32_t rows = qo_len[b] * group;
    const int32_t qpos0 = kv_len[b] - qo_len[b];
    const bool prefill = page_size >= kStageTokens && rows >= kPrefillMinRows &&
                         bsr::kPrefillKeyTile % group == 0;
    const int32_t step = prefill ? bsr::kPrefillRows : kMaxDecodeRows;
    for (int32_t h = 0; h < num_kv_heads; ++h)
      for (int32_t r0 = 0; r0 < rows; r0 += step) {
        const int32_t nr = std::min(step, rows - r0);
        int64_t kend = kv_len[b];
        if (causal)
          kend = std::min<int64_t>(kend, std::max<int64_t>(0, int64_t(qpos0) + (r0 + nr - 1) / group + 1));
        // sliding window: the first row (the earliest position) sees the oldest key;
        // the unit starts at the page (or 16-key stage) holding it, so pages wholly
        // before every row's window are never read (they may have been recycled)
        int64_t kbegin = 0;
        if (window_left > 0) {
          const int64_t align = std::max<int64_t>(page_size, kStageTokens);
          kbegin = std::max<int64_t>(0, int64_t(qpos0) + r0 / group - window_left + 1);
          kbegin = std::min(kbegin, kend) / align * align;
        }
        const Unit unit{b, h, r0, nr, int32_t(kend), indptr[b], q_row0[b], qpos0, int32_t(kbegin)};
        if (prefill) {
          punits.push_back(unit);
        } else {
          dunits.push_back(unit);
          max_rows = std::max(max_rows, nr);
        }
      }
  }
  // consecutive plans of a serving loop are alike: start from the last budget step
  thread_local int64_t dec_k = -1;
  const int64_t dec_workers = int64_t(num_sms) * dec_warps_per_sm;
  // the run-time pool: the shortest whole ranges up to kDynShare of the cost
  std::vector<Unit>& dyn = hp->dyn_units;
  dyn.clear();
  if (allow_dyn && page_size >= kStageTokens && !(rope_theta > 0.f)) {
    int64_t total = 0, longest = 0;
    for (const Unit& u : dunits) {
      total += u.kend - u.kbegin + kUnitOverhead;
      longest = std::max<int64_t>(longest, u.kend - u.kbegin);
    }
    if (total >= dec_workers * kDynMinWarpWork && longest >= kDynSkew * (total / dec_workers)) {
      const int64_t max_len = total / dec_workers / 4 - kUnitOverhead;
      const int64_t cap = int64_t(kDynShare * double(total));
      std::vector<uint8_t>& in_pool = hp->dyn_mark;
      in_pool.assign(dunits.size(), 0);
      if (max_len > 0 && max_len <= (int64_t(1) << 22)) {
        // shortest first, equal lengths in unit order: count by length, find the longest
        // length taken whole and how many of the next length still fit, then mark
        std::vector<int32_t>& cnt = hp->dyn_idx;
        cnt.assign(size_t(max_len) + 1, 0);
        for (const Unit& u : dunits) {
          const int64_t len = u.kend - u.kbegin;
          if (len > 0 && len <= max_len) ++cnt[size_t(len)];
        }
        int64_t pool = 0, cut_len = max_len + 1, cut_n = 0;
        for (int64_t len = 1; len <= max_len; ++len) {
          const int64_t c = len + kUnitOverhead, n = cnt[size_t(len)];
          if (n == 0) continue;
          if (pool + c * n <= cap) {
            pool += c * n;
            continue;
          }
          cut_len = len;
          cut_n = (cap - pool) / c;
          break;
        }
        for (size_t i = 0; i < dunits.size(); ++i) {
          const int64_t len = dunits[i].kend - dunits[i].kbegin;
          if (len <= 0 || len > max_len || len > cut_len) continue;
          if (len < cut_len) {
            in_pool[i] = 1;
          } else if (cut_n > 0) {
            in_pool[i] = 1;
            --cut_n;
          }
        }
      }
      size_t kept = 0;
      for (size_t i = 0; i < dunits.size(); ++i) {
        if (in_pool[i]) dyn.push_back(dunits[i]);
        else dunits[kept++] = dunits[i];
      }
      dunits.resize(kept);
    }
  }
  balance(dunits, dec_workers, std::max<int64_t>(page_size, kStageTokens), kUnitOverhead,
          kMinPiece, kMinWarpWork, &hp->dec, &dec_k, kMinPieceSmall, kSplitOverhead);
  hp->dec.n_dyn = 0;
  hp->dec.dyn_begin = int32_t(hp->dec.items.size());
  if (!dyn.empty()) {
    // every warp of the grid takes run-time units, including ones without a list
    WorkList& dl = hp->dec;
    while (dl.workers < dec_workers) {
      dl.ptr.push_back(dl.ptr.back());
      ++dl.workers;
    }
    // longest first, equal lengths in unit order (a counting sort: every length is at
    // most a quarter of a warp's share)
    int64_t lmax = 0;
    for (const Unit& u : dyn) lmax = std::max<int64_t>(lmax, u.kend - u.kbegin);
    std::vector<int32_t>& pos = hp->dyn_idx;
    pos.assign(size_t(lmax) + 2, 0);
    for (const Unit& u : dyn) ++pos[size_t(lmax - (u.kend - u.kbegin)) + 1];
    for (size_t k = 1; k < pos.size(); ++k) pos[k] += pos[k - 1];
    std::vector<Unit>& sorted = hp->dyn_sorted;
    sorted.resize(dyn.size());
    for (const Unit& u : dyn) sorted[size_t(pos[size_t(lmax - (u.kend - u.kbegin))]++)] = u;
    dyn.swap(sorted);
    // imbalance: the most planned (static) cost of a warp against the mean cost of all
    // decode work per warp, run-time units included (below 1: they fill the rest)
    int64_t mx = 0, all = 0;
    for (int32_t w = 0; w < dl.workers; ++w) {
      int64_t l = 0;
      for (int32_t i = dl.ptr[w]; i < dl.ptr[w + 1]; ++i)
        l += dl.items[i].tok1 - dl.items[i].tok0 + kUnitOverhead +
             (dl.items[i].nchunks > 1 ? kSplitOverhead : 0);
      mx = std::max(mx, l);
      all += l;
    }
    for (const Unit& u : dyn) {
      DecodeItem it{};
      it.req = u.req;
      it.kvh = u.kvh;
      it.row0 = u.row0;
      it.nrows = u.nrows;
      it.tok0 = u.kbegin;
      it.tok1 = u.kend;
      it.slot = -1;
      it.first_slot = -1;
      it.nchunks = 1;
      it.page_base = u.page_base;
      it.q_row0 = u.q_row0;
      it.qpos0 = u.qpos0;
      dl.items.push_back(it);
      all += u.kend - u.kbegin + kUnitOverhead;
    }
    dl.n_dyn = int32_t(dyn.size());
    const double mean = double(all) / dl.workers;
    dl.imbalance = mean > 0 ? double(mx) / mean : 1.0;
  }
  balance_gangs(punits, num_sms, std::max<int64_t>(page_size, bsr::kPrefillKeyTile),
                kPrefillOverhead, kPrefillMinPiece, kPrefillMinCtaWork, &hp->pre);
  hp->pmerge.clear();
  for (const DecodeItem& it : hp->pre.items)
    if (it.slot >= 0 && it.slot == it.first_slot) hp->pmerge.push_back(it);

  hp->dec_warps_per_cta = dec_warps_per_sm;
  hp->group = group;
  hp->sum_qo = sum_qo;
  hp->active = active;
  hp->max_len = max_len;
  hp->max_rows = max_rows;
  return BSR_OK;
}

}  // namespace

extern "C" int bsr_attn_plan(const int32_t* indptr, const int32_t* indices,
                             const int32_t* last_page_len, int32_t batch, int32_t num_qo_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                             const int32_t* qo_indptr, int32_t num_pages_in_pool, int32_t causal,
                             int32_t window_left, const int32_t* page_pos, int32_t kv_layout,
                             int32_t kv_dtype, float rope_theta, void* stream_v,
                             bsr_schedule_t* schedule) {
  if (kv_layout != BSR_KV_HND && kv_layout != BSR_KV_NHD) return BSR_ERR_INVALID_ARGUMENT;
  if (kv_dtype != BSR_KV_DTYPE_BF16 && kv_dtype != BSR_KV_DTYPE_E4M3) return BSR_ERR_INVALID_ARGUMENT;
  if (schedule == nullptr) return BSR_ERR_INVALID_ARGUMENT;
  const cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  const bool rope = rope_theta > 0.f;
  int device = 0, num_sms = 0;
  cudaError_t ce = cudaGetDevice(&device);
  if (ce != cudaSuccess) return fail_cuda(ce);
  ce = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device);
  if (ce != cudaSuccess) return fail_cuda(ce);
  if (*schedule != nullptr && (*schedule)->sm_budget > 0)
    num_sms = std::min(num_sms, int((*schedule)->sm_budget));
  thread_local HostPlan hp;   // reused: its vectors keep their memory between plans
  const int rc = make_host_plan(indptr, indices, last_page_len, batch, num_qo_heads, num_kv_heads,
                                head_dim, page_size, qo_indptr, num_pages_in_pool, causal,
                                window_left, page_pos, rope_theta, num_sms,
                                decode_warps_per_sm(kv_dtype, rope), kv_dtype == BSR_KV_DTYPE_BF16,
                                &hp);
  if (rc != BSR_OK) return rc;
  const int64_t nnz = indptr[batch];

  bsr_schedule* s = *schedule;
  const bool fresh = (s == nullptr);
  if (fresh) {
    s = new (std::nothrow) bsr_schedule();
    if (s == nullptr) return BSR_ERR_OUT_OF_MEMORY;
  } else if (s->device != device) {
    return BSR_ERR_SCHEDULE_MISMATCH;
  }
  auto bail = [&](int code) {
    if (fresh) bsr_schedule_destroy(s);
    return code;
  };

  // ---------------------------------------------------------------- RoPE tables (cached)
  const int64_t pos_end = std::max<int64_t>(hp.max_len, hp.max_pos_end);
  const int32_t need_rows =
      rope ? int32_t(align_up(size_t(pos_end), kStageTokens)) + kStageTokens : 0;
  if (rope && (s->h_rope == nullptr || s->rope_cache_theta != rope_theta ||
               s->rope_cache_D != head_dim || s->rope_cache_rows < need_rows)) {
    int64_t rows = 4096;
    while (rows < need_rows) rows *= 2;
    const size_t bytes = size_t(rows) * head_dim / 2 * sizeof(float) * 2;
    std::free(s->h_rope);
    s->rope_cache_rows = 0;
    s->d_rope_valid = false;
    s->h_rope = static_cast<uint8_t*>(std::malloc(2 * bytes));
    if (s->h_rope == nullptr) return bail(BSR_ERR_OUT_OF_MEMORY);
    build_rope_tables(reinterpret_cast<float*>(s->h_rope),
                      reinterpret_cast<float*>(s->h_rope + bytes), int32_t(rows), head_dim,
                      double(rope_theta));
    s->rope_cache_theta = rope_theta;
    s->rope_cache_D = head_dim;
    s->rope_cache_rows = int32_t(rows);
  }
  const size_t rope_bytes =
      rope ? size_t(s->rope_cache_rows) * head_dim / 2 * sizeof(float) * 2 : 0;
  if (rope && !s->d_rope_valid) {
    if (s->d_rope_cap < 2 * rope_bytes) {
      if (s->d_rope) {
        ce = cudaFree(s->d_rope);  // synchronizes: no kernel can still be reading it
        s->d_rope = nullptr;
        s->d_rope_cap = 0;
        if (ce != cudaSuccess) return bail(fail_cuda(ce));
      }
      ce = cudaMalloc(reinterpret_cast<void**>(&s->d_rope), 2 * rope_bytes);
      if (ce != cudaSuccess) return bail(fail_cuda(ce));
      s->d_rope_cap = 2 * rope_bytes;
    }
    // pageable source: returns once the bytes are staged; ordered on the stream
    ce = cudaMemcpyAsync(s->d_rope, s->h_rope, 2 * rope_bytes, cudaMemcpyHostToDevice, stream);
    if (ce != cudaSuccess) return bail(fail_cuda(ce));
    s->d_rope_valid = true;
  }

  // ---------------------------------------------------------------- workspace layout
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + std::max<size_t>(bytes, 1), kAlign);
    return o;
  };
  const size_t off_indices = take(size_t(std::max<int64_t>(nnz, 1)) * 4);
  const size_t off_items = take(hp.dec.items.size() * sizeof(DecodeItem));
  const size_t off_warp_ptr = take(hp.dec.ptr.size() * 4);
  const size_t off_counters = take(size_t(std::max(hp.dec.n_partials, 1)) * 4);
  const size_t off_pitems = take(hp.pre.items.size() * sizeof(DecodeItem));
  const size_t off_cta_ptr = take(hp.pre.ptr.size() * 4);
  const size_t off_pmerge = take(hp.pmerge.size() * sizeof(DecodeItem));
  const bool with_pos = page_pos != nullptr && rope;   // positions matter only for RoPE
  const size_t off_page_pos = take(with_pos ? size_t(std::max<int64_t>(nnz, 1)) * 4 : 0);
  const size_t off_qshift = take(with_pos ? size_t(std::max(batch, 1)) * 4 : 0);
  const size_t off_error = take(16);
  const size_t off_dyn_ctr = take(16);   // run-time queue: next unit, warps done (zeros)
  const size_t image_bytes = off;  // everything above is uploaded
  const size_t off_part_o = take(size_t(hp.dec.n_partials) * kMaxDecodeRows * head_dim * 4);
  const size_t off_part_lse = take(size_t(hp.dec.n_partials) * kMaxDecodeRows * 4);
  const size_t off_ppart_o = take(size_t(hp.pre.n_partials) * bsr::kPrefillRows * head_dim * 4);
  const size_t off_ppart_lse = take(size_t(hp.pre.n_partials) * bsr::kPrefillRows * 4);
  const size_t ws_bytes = off;

  // ---------------------------------------------------------------- staging + upload
  if (s->upload_pending) {
    ce = cudaEventSynchronize(s->upload_done);  // the staging buffer is about to be rewritten
    if (ce != cudaSuccess) return bail(fail_cuda(ce));
    s->upload_pending = false;
  }
  if (s->stage_cap < image_bytes) {
    if (s->h_stage) cudaFreeHost(s->h_stage);
    s->h_stage = nullptr;
    s->stage_cap = 0;
    ce = cudaMallocHost(reinterpret_cast<void**>(&s->h_stage), image_bytes);
    if (ce != cudaSuccess) return bail(fail_cuda(ce));
    s->stage_cap = image_bytes;
  }
  if (s->ws_cap < ws_bytes) {
    if (s->d_ws) {
      ce = cudaFree(s->d_ws);  // synchronizes: no kernel can still be reading it
      s->d_ws = nullptr;
      s->ws_cap = 0;
      if (ce != cudaSuccess) return bail(fail_cuda(ce));
    }
    ce = cudaMalloc(reinterpret_cast<void**>(&s->d_ws), ws_bytes);
    if (ce != cudaSuccess) return bail(fail_cuda(ce));
    s->ws_cap = ws_bytes;
  }
  if (s->upload_done == nullptr) {
    ce = cudaEventCreateWithFlags(&s->upload_done, cudaEventDisableTiming);
    if (ce != cudaSuccess) return bail(fail_cuda(ce));
  }
  uint8_t* h = s->h_stage;
  // every region is written below except the split-range counters and the status word
  std::memset(h + off_counters, 0, size_t(std::max(hp.dec.n_partials, 1)) * 4);
  std::memset(h + off_error, 0, 16);
  std::memset(h + off_dyn_ctr, 0, 16);
  if (nnz > 0) std::memcpy(h + off_indices, indices, size_t(nnz) * 4);
  if (!hp.dec.items.empty())
    std::memcpy(h + off_items, hp.dec.items.data(), hp.dec.items.size() * sizeof(DecodeItem));
  std::memcpy(h + off_warp_ptr, hp.dec.ptr.data(), hp.dec.ptr.size() * 4);
  if (with_pos) {
    if (nnz > 0) std::memcpy(h + off_page_pos, page_pos, size_t(nnz) * 4);
    if (batch > 0) std::memcpy(h + off_qshift, hp.qshift.data(), size_t(batch) * 4);
  }
  if (!hp.pre.items.empty())
    std::memcpy(h + off_pitems, hp.pre.items.data(), hp.pre.items.size() * sizeof(DecodeItem));
  std::memcpy(h + off_cta_ptr, hp.pre.ptr.data(), hp.pre.ptr.size() * 4);
  if (!hp.pmerge.empty())
    std::memcpy(h + off_pmerge, hp.pmerge.data(), hp.pmerge.size() * sizeof(DecodeItem));
  ce = cudaMemcpyAsync(s->d_ws, h, image_bytes, cudaMemcpyHostToDevice, stream);
  if (ce != cudaSuccess) return bail(fail_cuda(ce));
  ce = cudaEventRecord(s->upload_done, stream);
  if (ce != cudaSuccess) return bail(fail_cuda(ce));
  s->upload_pending = true;

  // ---------------------------------------------------------------- commit
  s->device = device;
  s->num_sms = num_sms;
  s->batch = batch;
  s->Hq = num_qo_heads;
  s->Hk = num_kv_heads;
  s->D = head_dim;
  s->P = page_size;
  s->group = hp.group;
  s->causal = causal;
  s->window_left = window_left;
  s->kv_layout = kv_layout;
  s->kv_dtype = kv_dtype;
  s->tm_k_ptr = s->tm_v_ptr = nullptr;      // the maps depend on the layout
  s->tm_k8_ptr = s->tm_v8_ptr = nullptr;
  s->rope_theta = rope_theta;
  s->num_pages = num_pages_in_pool;
  s->sum_qo = hp.sum_qo;
  s->active_tokens = hp.active;
  s->rope_rows = rope ? s->rope_cache_rows : 0;
  s->max_rows = hp.max_rows;
  s->n_items = int32_t(hp.dec.items.size());
  s->n_partials = hp.dec.n_partials;
  s->n_split = hp.dec.n_split;
  s->dec_warps = hp.dec.workers;
  s->dec_ctas = (hp.dec.workers + hp.dec_warps_per_cta - 1) / hp.dec_warps_per_cta;
  s->dec_warps_per_cta = hp.dec_warps_per_cta;
  s->dec_imbalance = hp.dec.imbalance;
  s->n_pitems = int32_t(hp.pre.items.size());
  s->n_ppartials = hp.pre.n_partials;
  s->n_psplit = hp.pre.n_split;
  s->pre_ctas = hp.pre.workers;
  s->pre_imbalance = hp.pre.imbalance;
  s->rope_bytes = rope_bytes;
  s->off_pitems = off_pitems;
  s->off_cta_ptr = off_cta_ptr;
  s->off_pmerge = off_pmerge;
  s->n_pmerge = int32_t(hp.pmerge.size());
  s->off_ppart_o = off_ppart_o;
  s->off_ppart_lse = off_ppart_lse;
  s->tm_q_ptr = nullptr;    // Q tensor map: encoded by run
  s->tm_pk_ptr = s->tm_pv_ptr = nullptr;   // prefill K/V maps depend on the page size
  s->ws_used = ws_bytes;
  s->upload_bytes = image_bytes;
  s->off_indices = off_indices;
  s->off_items = off_items;
  s->off_warp_ptr = off_warp_ptr;
  s->off_counters = off_counters;
  s->off_dyn_ctr = off_dyn_ctr;
  s->n_dyn = hp.dec.n_dyn;
  s->dyn_begin = hp.dec.dyn_begin;
  s->off_error = off_error;
  s->off_page_pos = with_pos ? off_page_pos : 0;
  s->off_qshift = with_pos ? off_qshift : 0;
  s->has_page_pos = with_pos;
  s->off_part_o = off_part_o;
  s->off_part_lse = off_part_lse;
  *schedule = s;
  return BSR_OK;
}

extern "C" int bsr_schedule_create(int32_t sm_budget, bsr_schedule_t* schedule) {
  if (schedule == nullptr || sm_budget < 0) return BSR_ERR_INVALID_ARGUMENT;
  int device = 0;
  const cudaError_t ce = cudaGetDevice(&device);
  if (ce != cudaSuccess) return fail_cuda(ce);
  bsr_schedule* s = new (std::nothrow) bsr_schedule();
  if (s == nullptr) return BSR_ERR_OUT_OF_MEMORY;
  s->device = device;
  s->sm_budget = sm_budget;
  *schedule = s;
  return BSR_OK;
}

extern "C" void bsr_schedule_destroy(bsr_schedule_t s) {
  if (s == nullptr) return;
  if (s->device >= 0) cudaSetDevice(s->device);
  if (s->d_ws) {
    cudaDeviceSynchronize();
    cudaFree(s->d_ws);
  }
  if (s->upload_done) cudaEventDestroy(s->upload_done);
  for (cudaEvent_t e : s->t_ev) cudaEventDestroy(e);
  if (s->h_stage) cudaFreeHost(s->h_stage);
  if (s->d_rope) cudaFree(s->d_rope);
  if (s->d_io) cudaFree(s->d_io);
  std::free(s->h_rope);
  cudaGetLastError();
  delete s;
}

extern "C" int bsr_schedule_get_info(bsr_schedule_t s, bsr_schedule_info_t* info) {
  if (s == nullptr || info == nullptr) return BSR_ERR_INVALID_ARGUMENT;
  std::memset(info, 0, sizeof(*info));
  info->batch = s->batch;
  info->num_qo_heads = s->Hq;
  info->num_kv_heads = s->Hk;
  info->head_dim = s->D;
  info->page_size = s->P;
  info->causal = s->causal;
  info->window_left = s->window_left;
  info->kv_layout = s->kv_layout;
  info->kv_dtype = s->kv_dtype;
  info->rope_theta = s->rope_theta;
  info->sum_qo = s->sum_qo;
  info->active_tokens = s->active_tokens;
  info->num_decode_items = s->n_items;
  info->num_prefill_items = s->n_pitems;
  info->num_split_streams = s->n_split + s->n_psplit;
  info->num_partials = s->n_partials + s->n_ppartials;
  info->decode_ctas = s->dec_ctas;
  info->decode_warps_per_cta = s->dec_warps_per_cta;
  info->prefill_ctas = s->pre_ctas;
  info->num_sms = s->num_sms;
  info->workspace_bytes = int64_t(s->ws_used);
  info->upload_bytes = int64_t(s->upload_bytes);
  info->decode_imbalance = s->dec_imbalance;
  info->prefill_imbalance = s->pre_imbalance;
  info->kernels_per_run = (s->n_items > 0 ? 1 : 0) + (s->n_pitems > 0 ? 1 : 0) +
                          (s->n_pmerge > 0 ? 1 : 0);
  return BSR_OK;
}

extern "C" int bsr_attn_plan_host(const int32_t* indptr, const int32_t* indices,
                                  const int32_t* last_page_len, int32_t batch,
                                  int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t page_size, const int32_t* qo_indptr,
                                  int32_t num_pages_in_pool, int32_t causal,
                                  int32_t window_left, const int32_t* page_pos,
                                  int32_t kv_layout, int32_t kv_dtype, float rope_theta,
                                  int32_t num_sms, bsr_schedule_info_t* info, int32_t* units,
                                  int64_t max_units) {
  if (kv_layout != BSR_KV_HND && kv_layout != BSR_KV_NHD) return BSR_ERR_INVALID_ARGUMENT;
  if (kv_dtype != BSR_KV_DTYPE_BF16 && kv_dtype != BSR_KV_DTYPE_E4M3) return BSR_ERR_INVALID_ARGUMENT;
  thread_local HostPlan hp;   // reused: its vectors keep their memory between plans
  const int rc = make_host_plan(indptr, indices, last_page_len, batch, num_qo_heads, num_kv_heads,
                                head_dim, page_size, qo_indptr, num_pages_in_pool, causal,
                                window_left, page_pos, rope_theta, num_sms,
                                decode_warps_per_sm(kv_dtype, rope_theta > 0.f),
                                kv_dtype == BSR_KV_DTYPE_BF16, &hp);
  if (rc != BSR_OK) return rc;
  if (info != nullptr) {
    std::memset(info, 0, sizeof(*info));
    info->batch = batch;
    info->num_qo_heads = num_qo_heads;
    info->num_kv_heads = num_kv_heads;
    info->head_dim = head_dim;
    info->page_size = page_size;
    info->causal = causal;
    info->window_left = window_left;
    info->kv_layout = kv_layout;
    info->kv_dtype = kv_dtype;
    info->rope_theta = rope_theta;
    info->sum_qo = hp.sum_qo;
    info->active_tokens = hp.active;
    info->num_decode_items = int32_t(hp.dec.items.size());
    info->num_prefill_items = int32_t(hp.pre.items.size());
    info->num_split_streams = hp.dec.n_split + hp.pre.n_split;
    info->num_partials = hp.dec.n_partials + hp.pre.n_partials;
    info->decode_ctas = (hp.dec.workers + hp.dec_warps_per_cta - 1) / hp.dec_warps_per_cta;
    info->decode_warps_per_cta = hp.dec_warps_per_cta;
    info->prefill_ctas = hp.pre.workers;
    info->num_sms = num_sms;
    info->decode_imbalance = hp.dec.imbalance;
    info->prefill_imbalance = hp.pre.imbalance;
    info->kernels_per_run = (hp.dec.items.empty() ? 0 : 1) + (hp.pre.items.empty() ? 0 : 1) +
                            (hp.pmerge.empty() ? 0 : 1);
  }
  const int64_t n = int64_t(hp.dec.items.size() + hp.pre.items.size());
  if (units != nullptr) {
    if (max_units < n) return BSR_ERR_INVALID_ARGUMENT;
    int64_t i_out = 0;
    auto put = [&](const DecodeItem& it, int32_t col) {
      int32_t* u = units + i_out * 8;
      u[0] = it.req; u[1] = it.kvh; u[2] = it.row0; u[3] = it.nrows;
      u[4] = it.tok0; u[5] = it.tok1; u[6] = it.slot; u[7] = col;
      ++i_out;
    };
    for (int pass = 0; pass < 2; ++pass) {
      const WorkList& wl = pass == 0 ? hp.dec : hp.pre;
      for (int32_t w = 0; w < wl.workers; ++w)
        for (int32_t i = wl.ptr[w]; i < wl.ptr[w + 1]; ++i) put(wl.items[i], pass == 0 ? w : -1 - w);
    }
    // run-time units: column decode warps + their place in the queue
    for (int32_t k = 0; k < hp.dec.n_dyn; ++k)
      put(hp.dec.items[size_t(hp.dec.dyn_begin + k)], hp.dec.workers + k);
  }
  return int(n);
}

extern "C" int bsr_last_device_error(bsr_schedule_t s) {
  if (s == nullptr || s->d_ws == nullptr) return BSR_ERR_INVALID_ARGUMENT;
  int32_t word = 0;
  cudaError_t ce = cudaSetDevice(s->device);
  if (ce == cudaSuccess) ce = cudaDeviceSynchronize();
  if (ce == cudaSuccess) ce = cudaMemcpy(&word, s->d_ws + s->off_error, 4, cudaMemcpyDeviceToHost);
  if (ce != cudaSuccess) return fail_cuda(ce);
  return word;
}

extern "C" const char* bsr_status_string(int status) {
  switch (status) {
    case BSR_OK: return "ok";
    case BSR_ERR_INVALID_ARGUMENT: return "invalid argument";
    case BSR_ERR_UNSUPPORTED: return "unsupported head_dim, page_size or head grouping";
    case BSR_ERR_PAGE_TABLE: return "malformed page table";
    case BSR_ERR_OUT_OF_MEMORY: return "out of memory";
    case BSR_ERR_CUDA: return "CUDA error";
    case BSR_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a bounded wait";
    case BSR_ERR_SCHEDULE_MISMATCH: return "arguments disagree with the schedule";
    default: return "unknown status";
  }
}
