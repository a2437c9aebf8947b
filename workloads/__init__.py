"""Seeded synthetic inputs for BSR (paged) KV-cache attention.

This module only draws random inputs and lays them out in the paged format;
it holds none of the attention arithmetic.  Both the oracle tests and the GPU
tests/bench take their inputs from here, so both sides see identical values.

Recipe (one ``torch.Generator`` seeded with ``1000 + config``; draws in this
fixed order: lengths, dropped pages, page permutation, q, k, v, then the
tokens to append):

* values: N(0, 1) in fp32, rounded to bf16 (round to nearest even);
* page table: request b owns ``ceil(len_b / P)`` logical pages; of its
  non-final pages ``floor(drop * (n_b - 1))`` are dropped (inactive blocks,
  absent from ``indices``) uniformly without replacement; the surviving pages
  take distinct physical ids from a random permutation of a pool of
  ``ceil(1.25 * demand)`` pages;
* poison: every pool page no request owns, every slot past
  ``last_page_len`` and every slot an append will fill is NaN (bf16 0x7FC0),
  so a stray read shows up as NaN in the output.

The five workloads follow the shapes of the pages' serving scenarios: a tiny
paged decode, a Llama-3-8B-shaped decode with RoPE, a skewed batch with
dropped blocks, a shared-prefix cascade and a chunked prefill with append.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

NAN_BF16 = 0x7FC0
NAN_E4M3 = 0x7F


@dataclass
class Paged:
    """One batch of requests over one paged KV pool (HND page layout)."""
    name: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    indptr: torch.Tensor          # int32 [B+1]
    indices: torch.Tensor         # int32 [indptr[B]]
    last_page_len: torch.Tensor   # int32 [B]
    qo_indptr: torch.Tensor       # int32 [B+1]
    kv_len: list                  # attended length per request (generator bookkeeping)
    q: torch.Tensor               # bf16 [sum_qo, Hq, D]
    k_pages: torch.Tensor         # bf16 [num_pages, Hk, P, D]
    v_pages: torch.Tensor
    sm_scale: float
    rope_theta: float = 0.0
    causal: bool = False
    append_indptr: torch.Tensor | None = None   # int32 [B+1]
    k_new: torch.Tensor | None = None           # bf16 [sum_append, Hk, D]
    v_new: torch.Tensor | None = None
    meta: dict = field(default_factory=dict)
    # FP8 KV cache (E4M3 codes, uint8, same layout as k_pages / v_pages): the keys and
    # values are k_scale * code and v_scale * code
    k_codes: torch.Tensor | None = None
    v_codes: torch.Tensor | None = None
    k_scale: float = 1.0
    v_scale: float = 1.0
    window_left: int = 0          # sliding window (0: none)
    # logical position of each page-table entry's first token (int32 [len(indices)]):
    # with dropped blocks the kept pages keep their original positions
    page_pos: torch.Tensor | None = None
    kv_layout: str = "HND"        # "NHD": pools are [num_pages, P, Hk, D]

    @property
    def batch(self) -> int:
        return len(self.indptr) - 1

    @property
    def active_tokens(self) -> int:
        """Keys some query attends: the whole history, or with a sliding window the
        union of the request's windows."""
        if self.window_left <= 0:
            return int(sum(self.kv_len))
        n = (self.qo_indptr[1:] - self.qo_indptr[:-1]).tolist()
        return int(sum(L - max(0, L - q - self.window_left + 1) for L, q in zip(self.kv_len, n)))


@dataclass
class Cascade:
    """Shared prefix (stored once) + per-request suffixes, merged by LSE."""
    name: str
    prefix: Paged     # batch 1; its query rows are all requests' queries
    suffix: Paged     # batch = number of requests


def _bf16(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.bfloat16)


def _poison(t: torch.Tensor):
    t.view(torch.int16).fill_(NAN_BF16)


def _pages_for(lens, page_size, drop, g):
    """Logical page lists after dropping; returns (active page counts, last lens, kept ords)."""
    kept, last = [], []
    for L in lens:
        n = (L + page_size - 1) // page_size
        if n == 0:
            kept.append([])
            last.append(0)
            continue
        k = int(math.floor(drop * (n - 1))) if n > 1 else 0
        dropped = set(torch.randperm(n - 1, generator=g)[:k].tolist()) if k > 0 else set()
        kept.append([j for j in range(n) if j not in dropped])
        last.append(L - (n - 1) * page_size)
    return kept, last


def _layout(lens, page_size, drop, g, pool_factor=1.25, pool_pages=None):
    kept, last = _pages_for(lens, page_size, drop, g)
    counts = [len(k) for k in kept]
    demand = sum(counts)
    pool = pool_pages if pool_pages is not None else max(int(math.ceil(pool_factor * demand)), 1)
    if pool < demand:
        raise ValueError("pool smaller than demand")
    perm = torch.randperm(pool, generator=g)[:demand].to(torch.int32)
    indptr = torch.zeros(len(lens) + 1, dtype=torch.int32)
    indptr[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int64), 0).to(torch.int32)
    last_page_len = torch.tensor([l if c > 0 else 0 for l, c in zip(last, counts)],
                                 dtype=torch.int32)
    attended = [(c - 1) * page_size + l if c > 0 else 0 for c, l in zip(counts, last)]
    _layout.kept = kept        # logical page ordinals of the last layout (for page_pos)
    return indptr, perm, last_page_len, pool, attended


def _fill_pool(pool, Hk, P, D, g):
    return _bf16(torch.randn(pool, Hk, P, D, generator=g))


def _poison_unused(w: Paged, fill_from: list | None = None):
    """NaN every slot no request owns (and, for append workloads, the slots to be filled)."""
    P = w.page_size
    valid = torch.zeros(w.num_pages, dtype=torch.int64)   # leading valid slots per page
    ind = w.indices.tolist()
    for b in range(w.batch):
        lo, hi = int(w.indptr[b]), int(w.indptr[b + 1])
        valid_to = w.kv_len[b] if fill_from is None else fill_from[b]
        for j, e in enumerate(range(lo, hi)):
            valid[ind[e]] = min(max(valid_to - j * P, 0), P)
    pools = [(w.k_pages.view(torch.int16), NAN_BF16), (w.v_pages.view(torch.int16), NAN_BF16)]
    if w.k_codes is not None:
        pools += [(w.k_codes, NAN_E4M3), (w.v_codes, NAN_E4M3)]
    for bits, nan in pools:
        empty = (valid == 0).nonzero().flatten()
        if len(empty):
            bits[empty] = nan
        for s in range(P):
            sel = ((valid <= s) & (valid > 0)).nonzero().flatten()
            if len(sel):
                bits[sel, :, s, :] = nan


def make_paged(name, seed, lens, *, Hq, Hk, D, P, qo_lens=None, drop=0.0, rope_theta=0.0,
               sm_scale=None, causal=False, append=False, pool_factor=1.25,
               pool_pages=None) -> Paged:
    """Build one paged batch.  ``lens`` are logical KV lengths (before drops).

    ``append=True``: the last ``qo_lens[b]`` tokens of each request are new —
    they are drawn into ``k_new``/``v_new`` and their slots in the pool are
    poisoned until an append writes them.
    """
    g = torch.Generator().manual_seed(seed)
    return _make_paged_g(name, g, lens, Hq=Hq, Hk=Hk, D=D, P=P, qo_lens=qo_lens, drop=drop,
                         rope_theta=rope_theta, sm_scale=sm_scale, causal=causal,
                         append=append, pool_factor=pool_factor, pool_pages=pool_pages)


def _make_paged_g(name, g, lens, *, Hq, Hk, D, P, qo_lens=None, drop=0.0, rope_theta=0.0,
                  sm_scale=None, causal=False, append=False, pool_factor=1.25,
                  pool_pages=None) -> Paged:
    B = len(lens)
    qo_lens = [1] * B if qo_lens is None else list(qo_lens)
    indptr, indices, last, pool, attended = _layout(lens, P, drop, g, pool_factor, pool_pages)
    qo_indptr = torch.zeros(B + 1, dtype=torch.int32)
    qo_indptr[1:] = torch.cumsum(torch.tensor(qo_lens, dtype=torch.int64), 0).to(torch.int32)
    q = _bf16(torch.randn(int(qo_indptr[-1]), Hq, D, generator=g))
    k = _fill_pool(pool, Hk, P, D, g)
    v = _fill_pool(pool, Hk, P, D, g)
    w = Paged(name=name, num_qo_heads=Hq, num_kv_heads=Hk, head_dim=D, page_size=P,
              num_pages=pool, indptr=indptr, indices=indices, last_page_len=last,
              qo_indptr=qo_indptr, kv_len=attended, q=q, k_pages=k, v_pages=v,
              sm_scale=sm_scale if sm_scale is not None else 1.0 / math.sqrt(D),
              rope_theta=rope_theta, causal=causal)
    if drop > 0:
        w.page_pos = torch.tensor([j * P for kept in _layout.kept for j in kept],
                                  dtype=torch.int32)
    if append:
        n_new = int(qo_indptr[-1])
        w.append_indptr = qo_indptr.clone()
        w.k_new = _bf16(torch.randn(n_new, Hk, D, generator=g))
        w.v_new = _bf16(torch.randn(n_new, Hk, D, generator=g))
        _poison_unused(w, fill_from=[attended[b] - qo_lens[b] for b in range(B)])
    else:
        _poison_unused(w)
    return w


# --------------------------------------------------------------------------------------
# The five workloads.  ``small=True`` gives a reduced case of the same structure that the
# oracle finishes in seconds (several tiles and a ragged tail), for parity tests.
# --------------------------------------------------------------------------------------

def config1() -> Paged:
    """Tiny paged decode: 4 requests, GQA 8/2, D 64, P 16, 64-page pool."""
    g = torch.Generator().manual_seed(1001)
    lens = [17, 64, 130, 255]
    return _make_paged_g("tiny_decode_b4_h8x2_d64_p16", g, lens, Hq=8, Hk=2, D=64, P=16,
                         sm_scale=1.0 / 8.0, pool_pages=64)


def config2(small: bool = False) -> Paged:
    """Llama-3-8B-shaped decode: 64 x 2048 tokens, 32/8 heads, D 128, RoPE 5e5."""
    g = torch.Generator().manual_seed(1002)
    if small:
        lens = torch.randint(1, 400, (7,), generator=g).tolist()
        name = "llama8b_decode_rope_small"
    else:
        lens = [2048] * 64
        name = "llama8b_decode_rope_b64_l2048"
    return _make_paged_g(name, g, lens, Hq=32, Hk=8, D=128, P=16, rope_theta=5e5)


def config3(small: bool = False) -> Paged:
    """Skewed block-sparse decode: 90% short, 10% long, 25% of non-final pages dropped."""
    g = torch.Generator().manual_seed(1003)
    if small:
        B, n_long, short, long_ = 20, 2, (1, 120), (900, 2500)
        name = "skewed_sparse_decode_small"
    else:
        B, n_long, short, long_ = 128, 13, (32, 512), (16384, 32768)
        name = "skewed_sparse_decode_b128"
    lens = torch.randint(short[0], short[1] + 1, (B,), generator=g)
    long_ids = torch.randperm(B, generator=g)[:n_long]
    lens[long_ids] = torch.randint(long_[0], long_[1] + 1, (n_long,), generator=g)
    return _make_paged_g(name, g, lens.tolist(), Hq=32, Hk=8, D=128, P=16, drop=0.25)


def config4(small: bool = False) -> Cascade:
    """Shared-prefix cascade: one prefix at P 256 stored once + suffixes at P 16."""
    g = torch.Generator().manual_seed(1004)
    if small:
        n_req, prefix_len, suf = 12, 704, (1, 90)
        name = "cascade_small"
    else:
        n_req, prefix_len, suf = 256, 8192, (64, 1024)
        name = "cascade_r256_prefix8192"
    Hq, Hk, D = 32, 8, 128
    suf_lens = torch.randint(suf[0], suf[1] + 1, (n_req,), generator=g).tolist()
    # page tables (no drops): prefix first, then suffixes
    p_indptr, p_indices, p_last, p_pool, p_att = _layout([prefix_len], 256, 0.0, g)
    s_indptr, s_indices, s_last, s_pool, s_att = _layout(suf_lens, 16, 0.0, g)
    q = _bf16(torch.randn(n_req, Hq, D, generator=g))
    pk = _fill_pool(p_pool, Hk, 256, D, g)
    sk = _fill_pool(s_pool, Hk, 16, D, g)
    pv = _fill_pool(p_pool, Hk, 256, D, g)
    sv = _fill_pool(s_pool, Hk, 16, D, g)
    scale = 1.0 / math.sqrt(D)
    prefix = Paged(name=name + ".prefix", num_qo_heads=Hq, num_kv_heads=Hk, head_dim=D,
                   page_size=256, num_pages=p_pool, indptr=p_indptr, indices=p_indices,
                   last_page_len=p_last, qo_indptr=torch.tensor([0, n_req], dtype=torch.int32),
                   kv_len=p_att, q=q, k_pages=pk, v_pages=pv, sm_scale=scale)
    suffix = Paged(name=name + ".suffix", num_qo_heads=Hq, num_kv_heads=Hk, head_dim=D,
                   page_size=16, num_pages=s_pool, indptr=s_indptr, indices=s_indices,
                   last_page_len=s_last,
                   qo_indptr=torch.arange(n_req + 1, dtype=torch.int32),
                   kv_len=s_att, q=q, k_pages=sk, v_pages=sv, sm_scale=scale)
    _poison_unused(prefix)
    _poison_unused(suffix)
    return Cascade(name=name, prefix=prefix, suffix=suffix)


@dataclass
class MultiCascade:
    """Several levels of shared KV segments: each level is a batch whose requests are
    that level's segments, every query row (all levels share ``q``) attending the one
    segment of each level its group points at; the levels' states are LSE-merged."""
    name: str
    levels: list      # [Paged]; level i's qo_indptr groups the query rows by segment


def multi_cascade(name, seed, level_lens, level_pages, groups, *, Hq=32, Hk=8, D=128):
    """``groups[i]``: number of segments of level i (the query rows are split evenly
    among them, in order); ``level_lens[i]``: (lo, hi) segment lengths (multiples of 16
    at the levels above the last); ``level_pages[i]``: page size of level i."""
    g = torch.Generator().manual_seed(seed)
    n_req = groups[-1]
    q = _bf16(torch.randn(n_req, Hq, D, generator=g))
    levels = []
    for i, (lens_, P, nseg) in enumerate(zip(level_lens, level_pages, groups)):
        lens = torch.randint(lens_[0], lens_[1] + 1, (nseg,), generator=g)
        if i < len(groups) - 1:
            lens = lens // 16 * 16
        indptr, indices, last, pool, att = _layout(lens.tolist(), P, 0.0, g)
        per = n_req // nseg
        qo = torch.arange(nseg + 1, dtype=torch.int32) * per
        w = Paged(name=f"{name}.level{i + 1}", num_qo_heads=Hq, num_kv_heads=Hk, head_dim=D,
                  page_size=P, num_pages=pool, indptr=indptr, indices=indices,
                  last_page_len=last, qo_indptr=qo, kv_len=att, q=q,
                  k_pages=_fill_pool(pool, Hk, P, D, g), v_pages=_fill_pool(pool, Hk, P, D, g),
                  sm_scale=1.0 / math.sqrt(D))
        _poison_unused(w)
        levels.append(w)
    return MultiCascade(name=name, levels=levels)


def config9(small: bool = False) -> MultiCascade:
    """Three-level cascade: one system prefix shared by every request, 8 group
    prefixes each shared by an eighth of the requests, per-request suffixes."""
    if small:
        return multi_cascade("cascade3_small", 1009, [(320, 320), (96, 208), (1, 90)],
                             [256, 64, 16], [1, 2, 16])
    return multi_cascade("cascade3_r256", 1009, [(4096, 4096), (1024, 2048), (64, 1024)],
                         [256, 64, 16], [1, 8, 256])


def _tokens(w: Paged, b: int, pool: torch.Tensor) -> torch.Tensor:
    """Request b's cached tokens [Hk, L, D] in order."""
    P, L = w.page_size, w.kv_len[b]
    pages = w.indices[int(w.indptr[b]):int(w.indptr[b + 1])].long()
    return pool[pages].permute(1, 0, 2, 3).reshape(w.num_kv_heads, -1, w.head_dim)[:, :L]


def flat_multi_cascade(c: MultiCascade) -> Paged:
    """Each query row's concatenation of its segments, laid out as one flat P-16 batch
    (used only to state "cascade == flat attention" as a check)."""
    base = c.levels[-1]
    Hq, Hk, D, P = base.num_qo_heads, base.num_kv_heads, base.head_dim, 16
    n_req = base.batch
    ks, vs, lens = [], [], []
    for r in range(n_req):
        kk, vv = [], []
        for w in c.levels:
            b = int(torch.searchsorted(w.qo_indptr, torch.tensor(r), right=True)) - 1
            kk.append(_tokens(w, b, w.k_pages))
            vv.append(_tokens(w, b, w.v_pages))
        ks.append(torch.cat(kk, 1))
        vs.append(torch.cat(vv, 1))
        lens.append(ks[-1].shape[1])
    npg = [(L + P - 1) // P for L in lens]
    pool = sum(npg)
    kp = torch.full((pool, Hk, P, D), float("nan"), dtype=torch.bfloat16)
    vp = kp.clone()
    indices, e = [], 0
    for r in range(n_req):
        for j in range(npg[r]):
            n = min(P, lens[r] - j * P)
            kp[e, :, :n] = ks[r][:, j * P:j * P + n]
            vp[e, :, :n] = vs[r][:, j * P:j * P + n]
            indices.append(e)
            e += 1
    indptr = torch.zeros(n_req + 1, dtype=torch.int32)
    indptr[1:] = torch.cumsum(torch.tensor(npg), 0).to(torch.int32)
    last = torch.tensor([L - (n - 1) * P for L, n in zip(lens, npg)], dtype=torch.int32)
    return Paged(name=c.name + ".flat", num_qo_heads=Hq, num_kv_heads=Hk, head_dim=D,
                 page_size=P, num_pages=pool, indptr=indptr,
                 indices=torch.tensor(indices, dtype=torch.int32), last_page_len=last,
                 qo_indptr=torch.arange(n_req + 1, dtype=torch.int32), kv_len=lens, q=base.q,
                 k_pages=kp, v_pages=vp, sm_scale=base.sm_scale)


def config5(small: bool = False) -> Paged:
    """Chunked prefill: append qo tokens after kv_len cached ones, causal, RoPE 5e5."""
    g = torch.Generator().manual_seed(1005)
    if small:
        B, qo, kv = 3, 150, (200, 700)
        name = "chunked_prefill_small"
    else:
        B, qo, kv = 16, 512, (1024, 8192)
        name = "chunked_prefill_b16_q512"
    kv_lens = torch.randint(kv[0], kv[1] + 1, (B,), generator=g).tolist()
    lens = [l + qo for l in kv_lens]
    return _make_paged_g(name, g, lens, Hq=32, Hk=8, D=128, P=16, qo_lens=[qo] * B,
                         rope_theta=5e5, causal=True, append=True)


def with_kv8(w: Paged, seed: int, spread: float = 16.0) -> Paged:
    """The same batch with an FP8 (E4M3) KV cache: fresh N(0, 1) keys and values
    drawn (generator seeded with ``seed``), multiplied by ``spread``, rounded to E4M3
    codes (round to nearest even, torch's conversion) and stored with scale
    1 / spread, so the cached values are N(0, 1)-like as in the bf16 workloads.
    Unowned slots hold the E4M3 NaN code."""
    g = torch.Generator().manual_seed(seed)
    shape = tuple(w.k_pages.shape)
    w.k_codes = (torch.randn(shape, generator=g) * spread).to(torch.float8_e4m3fn).view(torch.uint8)
    w.v_codes = (torch.randn(shape, generator=g) * spread).to(torch.float8_e4m3fn).view(torch.uint8)
    w.k_scale = w.v_scale = 1.0 / spread
    w.name = w.name + "_kv_e4m3"
    _poison_unused(w)
    for bf, codes in ((w.k_pages, w.k_codes), (w.v_pages, w.v_codes)):
        dead = torch.isnan(bf.float()).flatten(1).all(dim=1)    # wholly poisoned pages
        codes[dead] = NAN_E4M3
    return w


def sliding_window_decode(name, seed, lens, window, *, Hq, Hk, D, P, qo_lens=None,
                          causal=True) -> Paged:
    """Long requests attended through a sliding window of ``window`` keys.  Only the
    pages that hold a key some query may see get pool pages of their own (values
    N(0, 1) in bf16); every older page of a request points at one shared page poisoned
    with NaN, so the pool stays small and a read outside the window shows as NaN."""
    g = torch.Generator().manual_seed(seed)
    B = len(lens)
    qo_lens = [1] * B if qo_lens is None else list(qo_lens)
    counts, first_live, last = [], [], []
    for L, n in zip(lens, qo_lens):
        npg = (L + P - 1) // P
        lo = max(0, L - n - window + 1)             # first key any of the request's rows sees
        counts.append(npg)
        first_live.append(lo // P)
        last.append(L - (npg - 1) * P if npg else 0)
    live = sum(c - f for c, f in zip(counts, first_live))
    pool = live + 1                                 # page 0: the shared poisoned page
    perm = (torch.randperm(live, generator=g) + 1).to(torch.int32).tolist()
    indices, k = [], 0
    for c, f in zip(counts, first_live):
        indices += [0] * f + perm[k:k + c - f]
        k += c - f
    indptr = torch.zeros(B + 1, dtype=torch.int32)
    indptr[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int64), 0).to(torch.int32)
    qo_indptr = torch.zeros(B + 1, dtype=torch.int32)
    qo_indptr[1:] = torch.cumsum(torch.tensor(qo_lens, dtype=torch.int64), 0).to(torch.int32)
    q = _bf16(torch.randn(int(qo_indptr[-1]), Hq, D, generator=g))
    kp = _fill_pool(pool, Hk, P, D, g)
    vp = _fill_pool(pool, Hk, P, D, g)
    w = Paged(name=name, num_qo_heads=Hq, num_kv_heads=Hk, head_dim=D, page_size=P,
              num_pages=pool, indptr=indptr, indices=torch.tensor(indices, dtype=torch.int32),
              last_page_len=torch.tensor(last, dtype=torch.int32), qo_indptr=qo_indptr,
              kv_len=list(lens), q=q, k_pages=kp, v_pages=vp, sm_scale=1.0 / math.sqrt(D),
              causal=causal, window_left=window)
    _poison_unused(w)                 # unused slots of the last pages
    for t in (w.k_pages, w.v_pages):
        t.view(torch.int16)[0] = NAN_BF16
    return w


def config7(small: bool = False) -> Paged:
    """Sliding-window decode: long histories, each query sees its last 2048 keys."""
    g = torch.Generator().manual_seed(1007)
    if small:
        B, lens_, window = 12, (300, 2500), 257
        name = "sliding_window_decode_small"
    else:
        B, lens_, window = 64, (8192, 32768), 2048
        name = "sliding_window_decode_b64_w2048"
    lens = torch.randint(lens_[0], lens_[1] + 1, (B,), generator=g).tolist()
    return sliding_window_decode(name, 2007 if small else 3007, lens, window, Hq=32, Hk=8,
                                 D=128, P=16)


def config8(small: bool = False) -> Paged:
    """The skewed block-sparse decode with RoPE (theta 5e5) at the kept blocks' logical
    positions (``page_pos``): the same table and values as the skewed decode."""
    w = config3(small)
    w.rope_theta = 5e5
    w.name = w.name + "_rope_positions"
    return w


def to_nhd(w: Paged) -> Paged:
    """The same batch with token-major (NHD) page pools [num_pages, P, Hk, D]."""
    for name in ("k_pages", "v_pages", "k_codes", "v_codes"):
        t = getattr(w, name)
        if t is not None:
            setattr(w, name, t.permute(0, 2, 1, 3).contiguous())
    w.kv_layout = "NHD"
    w.name = w.name + "_nhd"
    return w


def config10(small: bool = False) -> Paged:
    """The skewed block-sparse decode over token-major (NHD) pages."""
    return to_nhd(config3(small))


def config6(small: bool = False) -> Paged:
    """The skewed block-sparse decode with an FP8 (E4M3) KV cache."""
    return with_kv8(config3(small), 1006)


def config11(small: bool = False) -> Paged:
    """The Llama-3-8B-shaped decode with RoPE over an FP8 (E4M3) KV cache."""
    return with_kv8(config2(small), 1011)


def by_name(cfg: int, small: bool = False):
    return {1: lambda: config1(), 2: lambda: config2(small), 3: lambda: config3(small),
            4: lambda: config4(small), 5: lambda: config5(small),
            6: lambda: config6(small), 7: lambda: config7(small),
            8: lambda: config8(small), 9: lambda: config9(small),
            10: lambda: config10(small), 11: lambda: config11(small)}[cfg]()


def flat_cascade(c: Cascade) -> Paged:
    """The cascade re-laid out as one flat P-16 table: prefix tokens then suffix tokens.

    Used only to state "cascade == flat attention" as a check: the prefix's
    pages are copied into extra P-16 pages appended to the suffix pool.
    """
    pre, suf = c.prefix, c.suffix
    P, Pp, Hk, D = suf.page_size, pre.page_size, suf.num_kv_heads, suf.head_dim
    L = pre.kv_len[0]
    if L % P:
        raise ValueError("flat_cascade needs a prefix length that is a multiple of 16")
    n16 = L // P
    # gather the prefix tokens [Hk, L, D] in order
    toks = []
    for j in range(int(pre.indptr[1])):
        page = int(pre.indices[j])
        n = min(Pp, L - j * Pp)
        toks.append(pre.k_pages[page, :, :n, :])
    kp = torch.cat(toks, dim=1)
    toks = []
    for j in range(int(pre.indptr[1])):
        page = int(pre.indices[j])
        n = min(Pp, L - j * Pp)
        toks.append(pre.v_pages[page, :, :n, :])
    vp = torch.cat(toks, dim=1)
    kp = kp.view(Hk, n16, P, D).permute(1, 0, 2, 3).contiguous()
    vp = vp.view(Hk, n16, P, D).permute(1, 0, 2, 3).contiguous()
    base = suf.num_pages
    k_all = torch.cat([suf.k_pages, kp], 0)
    v_all = torch.cat([suf.v_pages, vp], 0)
    indptr = [0]
    indices = []
    for b in range(suf.batch):
        indices += list(range(base, base + n16))
        indices += suf.indices[int(suf.indptr[b]):int(suf.indptr[b + 1])].tolist()
        indptr.append(len(indices))
    last = [int(suf.last_page_len[b]) if suf.kv_len[b] > 0 else P for b in range(suf.batch)]
    return Paged(name=c.name + ".flat", num_qo_heads=suf.num_qo_heads, num_kv_heads=Hk,
                 head_dim=D, page_size=P, num_pages=base + n16,
                 indptr=torch.tensor(indptr, dtype=torch.int32),
                 indices=torch.tensor(indices, dtype=torch.int32),
                 last_page_len=torch.tensor(last, dtype=torch.int32),
                 qo_indptr=suf.qo_indptr.clone(),
                 kv_len=[L + s for s in suf.kv_len], q=suf.q, k_pages=k_all, v_pages=v_all,
                 sm_scale=suf.sm_scale)


def algorithmic_bytes(w: Paged) -> int:
    """Bytes the attention must touch at least once: active K and V, q, out, lse, page table."""
    elt = 2                                            # q and out are bf16
    kv_elt = 1 if w.k_codes is not None else 2         # E4M3 or bf16 KV cache
    kv = w.active_tokens * 2 * w.num_kv_heads * w.head_dim * kv_elt
    rows = int(w.qo_indptr[-1]) * w.num_qo_heads
    qo = rows * w.head_dim * elt * 2 + rows * 4
    table = 4 * (len(w.indptr) + len(w.indices) + len(w.last_page_len) + len(w.qo_indptr))
    return kv + qo + table
