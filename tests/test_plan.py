"""Host planner: every key of every (request, kv head, row group) is covered exactly once,
split ranges are numbered in key order, and the load balances on skewed batches."""
import numpy as np
import pytest

import block_sparse_kv_bsr_gb300 as bsr
import workloads as wl
from block_sparse_kv_bsr_gb300 import _build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    bsr.load()


def plan_of(w: wl.Paged, num_sms=152):
    return bsr.bsr_attn_plan_host(
        w.indptr, w.indices, w.last_page_len, num_qo_heads=w.num_qo_heads,
        num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, page_size=w.page_size,
        num_pages=w.num_pages, num_sms=num_sms, qo_indptr=w.qo_indptr, causal=w.causal,
        rope_theta=w.rope_theta, window_left=w.window_left)


def is_prefill(w: wl.Paged, b: int) -> bool:
    g = w.num_qo_heads // w.num_kv_heads
    rows = int(w.qo_indptr[b + 1] - w.qo_indptr[b]) * g
    return w.page_size >= 16 and rows >= 64 and 128 % g == 0


def check_coverage(w: wl.Paged, units: np.ndarray):
    """Every key of every (request, kv head, row group) in exactly one unit, in key order.

    Decode units (warp >= 0) take 16-row groups; prefill units (warp < 0) 256 rows
    (two 128-row query tiles) with key ranges cut at multiples of 128 keys.
    """
    g = w.num_qo_heads // w.num_kv_heads
    ranges = {}
    for req, kvh, row0, nrows, tok0, tok1, slot, warp in units.tolist():
        step = 256 if warp < 0 else 16
        assert is_prefill(w, req) == (warp < 0)
        assert 1 <= nrows <= step
        # prefill cuts fall on 128-key tiles, a windowed start on its page (or 16 keys)
        align = max(w.page_size, 128 if warp < 0 and w.window_left == 0 else 16)
        assert tok0 % align == 0
        ranges.setdefault((req, kvh, row0, nrows), []).append((tok0, tok1, slot))
    for b in range(w.batch):
        L = w.kv_len[b]
        nq = int(w.qo_indptr[b + 1] - w.qo_indptr[b])
        rows = nq * g
        step = 256 if is_prefill(w, b) else 16
        for kvh in range(w.num_kv_heads):
            for r0 in range(0, rows, step):
                nr = min(step, rows - r0)
                kend = L
                if w.causal:
                    kend = min(L, max(0, (L - nq) + (r0 + nr - 1) // g + 1))
                pieces = sorted(ranges.pop((b, kvh, r0, nr)))
                if len(pieces) == 1:
                    assert pieces[0][2] == -1
                else:
                    slots = [p[2] for p in pieces]
                    assert slots == list(range(slots[0], slots[0] + len(slots)))
                # sliding window: from the oldest key the first row sees, aligned down
                kbegin = 0
                if w.window_left > 0:
                    align = max(w.page_size, 16)
                    kbegin = max(0, (L - nq) + r0 // g - w.window_left + 1)
                    kbegin = min(kbegin, kend) // align * align
                pos = kbegin
                for tok0, tok1, _ in pieces:
                    assert tok0 == pos and (tok1 > tok0 or kend == kbegin)
                    pos = tok1
                assert pos == kend
    assert not ranges, "units for ranges that do not exist"


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_small_configs_cover_every_key(cfg):
    w = wl.by_name(cfg, small=True)
    info, units = plan_of(w, num_sms=8)
    check_coverage(w, units)
    assert info["active_tokens"] == w.active_tokens


def test_cascade_levels_cover_every_key():
    c = wl.config4(small=True)
    for w in (c.prefix, c.suffix):
        info, units = plan_of(w, num_sms=8)
        check_coverage(w, units)


@pytest.mark.parametrize("P", [1, 2, 8, 32, 256])
def test_page_sizes(P):
    w = wl.make_paged("p", 3, [1, 15, 16, 17, 300, 513], Hq=8, Hk=2, D=64, P=P)
    info, units = plan_of(w, num_sms=2)
    check_coverage(w, units)


def test_empty_requests_get_a_unit():
    w = wl.make_paged("e", 4, [0, 40, 0], Hq=4, Hk=2, D=64, P=16)
    info, units = plan_of(w, num_sms=2)
    check_coverage(w, units)


def test_skewed_batch_is_balanced():
    w = wl.config3(small=False)
    info, units = plan_of(w, num_sms=152)
    check_coverage(w, units)
    assert info["decode_imbalance"] < 1.05
    assert info["num_split_streams"] >= 13 * 8     # every long (request, head) range is cut


@pytest.mark.parametrize("rope,warps", [(0.0, 12), (5e5, 8)])
def test_fp8_cache_plans_for_its_kernel_warps(rope, warps):
    """An FP8 (E4M3) schedule spreads the decode work over the FP8 kernel's warps per SM
    (12 without RoPE, 8 with), still covering every key once and balanced; bf16 keeps 8."""
    w = wl.config3(small=False)
    w.rope_theta = rope
    kw = dict(num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
              page_size=w.page_size, num_pages=w.num_pages, num_sms=152, rope_theta=rope)
    info, units = bsr.bsr_attn_plan_host(w.indptr, w.indices, w.last_page_len,
                                         kv_dtype="e4m3", **kw)
    check_coverage(w, units)
    assert info["kv_dtype"] == 1 and info["decode_warps_per_cta"] == warps
    assert info["decode_ctas"] == 152 and units[:, 7].max() < 152 * warps
    assert info["decode_imbalance"] < 1.05
    info16, _ = bsr.bsr_attn_plan_host(w.indptr, w.indices, w.last_page_len, **kw)
    assert info16["kv_dtype"] == 0 and info16["decode_warps_per_cta"] == 8
    with pytest.raises(ValueError):
        bsr.bsr_attn_plan_host(w.indptr, w.indices, w.last_page_len, kv_dtype="fp8", **kw)


def test_uniform_batch_is_balanced():
    w = wl.config2(small=False)
    info, units = plan_of(w, num_sms=152)
    check_coverage(w, units)
    assert info["decode_imbalance"] < 1.05


def test_prefill_configs_use_the_tensor_core_kernel():
    w = wl.config5(small=False)
    info, units = plan_of(w, num_sms=152)
    check_coverage(w, units)
    assert info["num_prefill_items"] > 0 and info["num_decode_items"] == 0
    assert info["prefill_imbalance"] < 1.10
    c = wl.config4(small=False)
    info, units = plan_of(c.prefix, num_sms=152)
    check_coverage(c.prefix, units)
    assert info["num_prefill_items"] >= 152          # 64 tiles cut to fill every SM
    assert info["num_split_streams"] > 0


def test_plan_is_deterministic():
    w = wl.config3(small=True)
    a = plan_of(w, num_sms=16)[1]
    b = plan_of(w, num_sms=16)[1]
    assert np.array_equal(a, b)


def test_sliding_window_plans_only_the_window():
    w = wl.config7(small=True)
    info, units = plan_of(w, num_sms=8)
    check_coverage(w, units)
    assert info["window_left"] == w.window_left
    assert info["active_tokens"] == w.active_tokens < sum(w.kv_len)
    planned = int((units[:, 5] - units[:, 4]).sum()) // w.num_kv_heads
    # at most one page (aligned down) more than the window per request
    assert planned <= w.active_tokens + w.batch * max(w.page_size, 16)
    # no planned key lies on the poisoned page every older page points at
    for req, kvh, row0, nrows, tok0, tok1, slot, warp in units.tolist():
        first = int(w.indptr[req]) + tok0 // w.page_size
        last = int(w.indptr[req]) + (tok1 - 1) // w.page_size
        assert (w.indices[first:last + 1] != 0).all()


def test_sliding_window_prefill_units():
    w = wl.make_paged("swpf", 31, [3000, 900], Hq=32, Hk=8, D=128, P=16, qo_lens=[300, 1],
                      causal=True)
    w.window_left = 700
    info, units = plan_of(w, num_sms=16)
    assert info["num_prefill_items"] > 0
    check_coverage(w, units)


def test_negative_window_is_refused():
    w = wl.config1()
    with pytest.raises(bsr.BsrError):
        bsr.bsr_attn_plan_host(w.indptr, w.indices, w.last_page_len, num_qo_heads=w.num_qo_heads,
                               num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                               page_size=w.page_size, num_pages=w.num_pages, num_sms=8,
                               qo_indptr=w.qo_indptr, window_left=-1)


def test_sliding_window_small_pages():
    w = wl.sliding_window_decode("swp4", 32, [300, 700, 45], 37, Hq=8, Hk=2, D=64, P=4)
    info, units = plan_of(w, num_sms=4)
    check_coverage(w, units)


def test_page_positions_validation():
    w = wl.make_paged("pp", 33, [100, 300], Hq=8, Hk=2, D=64, P=8, drop=0.3, rope_theta=1e4)
    kw = dict(num_qo_heads=8, num_kv_heads=2, head_dim=64, page_size=8, num_pages=w.num_pages,
              num_sms=4, qo_indptr=w.qo_indptr)
    # RoPE with positions needs pages of at least 16 keys
    with pytest.raises(bsr.BsrError):
        bsr.bsr_attn_plan_host(w.indptr, w.indices, w.last_page_len, rope_theta=1e4,
                               page_pos=w.page_pos, **kw)
    # without RoPE they are accepted (and unused); negative positions are refused
    bsr.bsr_attn_plan_host(w.indptr, w.indices, w.last_page_len, page_pos=w.page_pos, **kw)
    bad = w.page_pos.clone()
    bad[0] = -16
    with pytest.raises(bsr.BsrError):
        bsr.bsr_attn_plan_host(w.indptr, w.indices, w.last_page_len, page_pos=bad, **kw)


def test_plan_does_not_depend_on_earlier_plans():
    # the budget search starts from the last plan's step; the result must not depend on it
    a, b = wl.config3(small=False), wl.config2(small=False)
    first = plan_of(a, num_sms=152)[1]
    plan_of(b, num_sms=152)
    again = plan_of(a, num_sms=152)[1]
    assert np.array_equal(first, again)
    plan_of(wl.config1(), num_sms=152)
    assert np.array_equal(first, plan_of(a, num_sms=152)[1])


def test_host_array_forms_give_the_same_plan():
    # CPU int32 tensors and int32 numpy arrays go to the planner in place; other forms
    # (int64, non-contiguous, lists) are converted: every form plans the same batch
    import torch
    w = wl.config3(small=True)
    base = plan_of(w, num_sms=8)[1]
    kw = dict(num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
              page_size=w.page_size, num_pages=w.num_pages, num_sms=8)
    forms = [
        lambda t: t.numpy(),                                        # int32 numpy, in place
        lambda t: t.to(torch.int64),                                # converted
        lambda t: torch.stack([t, t], 1)[:, 0],                     # non-contiguous view
        lambda t: t.tolist(),                                       # a list
    ]
    for f in forms:
        _, units = bsr.bsr_attn_plan_host(f(w.indptr), f(w.indices), f(w.last_page_len),
                                          qo_indptr=f(w.qo_indptr), **kw)
        assert np.array_equal(units, base)


def test_ranges_are_cut_longest_first_in_unit_order():
    # The cut lays the key ranges end to end, longest first and equal lengths in unit
    # order (request, then kv head), so in worker order every range's pieces are
    # consecutive and the ranges appear by non-increasing length.  Lengths above 2^16
    # and 2^24 keys and many ties exercise every digit of the length sort.
    P, Hk = 16, 2
    lens = [1000, 300000, 70000, 0, 1000, 70000, 65541, 16, 17000000, 1000, 1, 65541]
    npages = [(n + P - 1) // P for n in lens]
    indptr = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
    indices = np.arange(indptr[-1], dtype=np.int32)
    last = np.array([n - (m - 1) * P if m else 0 for n, m in zip(lens, npages)], np.int32)
    info, units = bsr.bsr_attn_plan_host(indptr, indices, last, num_qo_heads=Hk, num_kv_heads=Hk,
                                         head_dim=128, page_size=P, num_pages=int(indptr[-1]),
                                         num_sms=4)
    assert info["num_split_streams"] > 0
    # ranges the plan leaves to run time (column >= the decode warps) come after every
    # warp's list, also longest first
    nwarps = info["decode_ctas"] * info["decode_warps_per_cta"]
    seen, late = [], set()
    for req, kvh, _, _, _, _, _, col in units.tolist():
        if col >= nwarps:
            late.add((req, kvh))
        if not seen or seen[-1] != (req, kvh):
            assert (req, kvh) not in seen, "a range's pieces are not consecutive"
            seen.append((req, kvh))
    expect = sorted(((b, h) for b in range(len(lens)) for h in range(Hk)),
                    key=lambda u: (u in late, -lens[u[0]], u))
    assert seen == expect


def test_skewed_batch_leaves_short_ranges_to_run_time():
    """On the skewed batch the shortest whole ranges (up to 15 % of the cost, each at most
    a quarter of a warp's share) are left out of the static cut: they come after every
    warp's list, unsplit, longest first.  Batches with RoPE, without a range several warps
    long, or over an FP8 cache keep a fully static plan."""
    w = wl.config3()
    kw = dict(num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
              page_size=w.page_size, num_pages=w.num_pages, num_sms=152)
    info, units = bsr.bsr_attn_plan_host(w.indptr, w.indices, w.last_page_len, **kw)
    check_coverage(w, units)
    nwarps = info["decode_ctas"] * info["decode_warps_per_cta"]
    late = units[units[:, 7] >= nwarps]
    assert len(late) > 0 and (late[:, 6] == -1).all()
    assert np.array_equal(late[:, 7], nwarps + np.arange(len(late)))       # queue order
    lens = late[:, 5] - late[:, 4]
    assert (np.diff(lens) <= 0).all() and lens.min() > 0
    static = units[units[:, 7] < nwarps]
    cost = lambda u: (u[:, 5] - u[:, 4] + 32).sum()
    assert cost(late) <= 0.15 * (cost(late) + cost(static)) + 1
    assert lens.max() <= (cost(late) + cost(static)) / nwarps / 4
    # the reported imbalance is the largest static share against the mean of all work
    assert info["decode_imbalance"] < 1.0
    for extra in (dict(rope_theta=1e4), dict(kv_dtype="e4m3")):
        info2, units2 = bsr.bsr_attn_plan_host(w.indptr, w.indices, w.last_page_len, **extra, **kw)
        n2 = info2["decode_ctas"] * info2["decode_warps_per_cta"]
        assert (units2[:, 7] < n2).all()
    u2 = wl.config2()
    info2, units2 = bsr.bsr_attn_plan_host(u2.indptr, u2.indices, u2.last_page_len,
                                           num_qo_heads=u2.num_qo_heads,
                                           num_kv_heads=u2.num_kv_heads, head_dim=u2.head_dim,
                                           page_size=u2.page_size, num_pages=u2.num_pages,
                                           num_sms=152)
    assert (units2[:, 7] < info2["decode_ctas"] * info2["decode_warps_per_cta"]).all()
