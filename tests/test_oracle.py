"""Pins for the fp64 oracle, against things other than the oracle itself.

The pages print no worked example, so the oracle is pinned by
  * brute-force dense attention through torch CPU fp64 library routines
    (``torch.softmax``, ``torch.logsumexp``; RoPE through complex exponentials),
  * closed forms (one key, zero query, identical keys, RoPE with D = 2),
  * invariances the BSR format promises ("FlashInfer: Block-Sparse KV 캐시로
    어텐션 병목을 해소하다", section "Block-Sparse 포맷": paged and contiguous
    layouts are instances of one format, inactive blocks are skipped, a shared
    prefix is stored once and composed with suffixes): page size, page
    permutation, dropping == masking, split + merge == unsplit,
    cascade == flat,
  * causal rows == decode at a shorter length.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

TOL = 1e-12


# ---------------------------------------------------------------- independent reference

def _rope_complex(x: torch.Tensor, pos: torch.Tensor, theta: float) -> torch.Tensor:
    """RoPE as multiplication of (x_i + i x_{i+D/2}) by exp(i pos omega_i)."""
    D = x.shape[-1]
    half = D // 2
    omega = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / D)
    z = torch.complex(x[..., :half], x[..., half:])
    rot = torch.polar(torch.ones_like(omega), pos[..., None].to(torch.float64) * omega)
    y = z * rot
    return torch.cat([y.real, y.imag], dim=-1)


def dense_reference(w: wl.Paged, drop_mask=None):
    """Attention by gathering each request's tokens with torch indexing, fp64."""
    Hq, Hk, D, P = w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size
    g = Hq // Hk
    q = w.q.to(torch.float64)
    kp = w.k_pages.to(torch.float64)
    vp = w.v_pages.to(torch.float64)
    outs, lses = [], []
    for b in range(w.batch):
        pages = w.indices[w.indptr[b]:w.indptr[b + 1]].long()
        L = w.kv_len[b]
        K = kp[pages].permute(1, 0, 2, 3).reshape(Hk, -1, D)[:, :L]
        V = vp[pages].permute(1, 0, 2, 3).reshape(Hk, -1, D)[:, :L]
        qb = q[w.qo_indptr[b]:w.qo_indptr[b + 1]]            # [n, Hq, D]
        n = qb.shape[0]
        qpos = torch.arange(L - n, L)
        if w.rope_theta > 0:
            qb = _rope_complex(qb, qpos[:, None].expand(n, Hq), w.rope_theta)
            K = _rope_complex(K, torch.arange(L)[None, :].expand(Hk, L), w.rope_theta)
        Kh = K.repeat_interleave(g, dim=0)                    # [Hq, L, D]
        Vh = V.repeat_interleave(g, dim=0)
        s = torch.einsum("nhd,hld->nhl", qb, Kh) * w.sm_scale
        if w.causal:
            keep = torch.arange(L)[None, :] <= qpos[:, None]
            s = s.masked_fill(~keep[:, None, :], -math.inf)
        if drop_mask is not None:
            s = s.masked_fill(~drop_mask[b][None, None, :], -math.inf)
        lse = torch.logsumexp(s, dim=-1)
        p = torch.softmax(s, dim=-1)
        p = torch.nan_to_num(p, nan=0.0)
        o = torch.einsum("nhl,hld->nhd", p, Vh)
        outs.append(o)
        lses.append(lse)
    return torch.cat(outs).numpy(), torch.cat(lses).numpy()


def run_oracle(w: wl.Paged, **kw):
    return oracle.attention(w.q, w.k_pages, w.v_pages, w.indptr, w.indices, w.last_page_len,
                            w.qo_indptr, num_qo_heads=w.num_qo_heads,
                            num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                            page_size=w.page_size, sm_scale=w.sm_scale,
                            rope_theta=w.rope_theta, causal=w.causal, **kw)


def _close(a, b, tol=TOL):
    a, b = np.asarray(a), np.asarray(b)
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    diff = np.where(both_inf, 0.0, np.abs(a - b))
    assert np.all(np.isfinite(diff)), "non-finite mismatch"
    assert diff.max(initial=0.0) <= tol, f"max diff {diff.max()}"


def tiny(seed=7, lens=(1, 7, 13, 30), Hq=4, Hk=2, D=8, P=4, **kw):
    return wl.make_paged("tiny", seed, list(lens), Hq=Hq, Hk=Hk, D=D, P=P, **kw)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("kw", [
    dict(),
    dict(rope_theta=10000.0),
    dict(qo_lens=[1, 3, 5, 2], causal=True),
    dict(qo_lens=[1, 3, 5, 2], causal=True, rope_theta=500.0),
    dict(qo_lens=[1, 2, 2, 4], causal=False),
    dict(Hq=6, Hk=3, D=6, P=3),
    dict(Hq=8, Hk=1, P=1),
])
def test_matches_dense_torch(kw):
    w = tiny(**kw)
    o, l = run_oracle(w)
    ro, rl = dense_reference(w)
    _close(o, ro)
    _close(l, rl)
    assert np.isfinite(o).all()


def test_matches_dense_torch_config1():
    w = wl.config1()
    o, l = run_oracle(w)
    ro, rl = dense_reference(w)
    _close(o, ro)
    _close(l, rl)


def test_selected_rows_match_full():
    w = tiny(qo_lens=[1, 3, 5, 2], causal=True, rope_theta=100.0)
    o, l = run_oracle(w)
    rng = np.random.default_rng(0)
    rows = rng.integers(0, int(w.qo_indptr[-1]), 9)
    heads = rng.integers(0, w.num_qo_heads, 9)
    so, sl = run_oracle(w, rows=rows, heads=heads)
    _close(so, o[rows, heads])
    _close(sl, l[rows, heads])


# ---------------------------------------------------------------- closed forms

def _single(seed, L, D=8, P=4, q_zero=False, k_equal=False):
    w = wl.make_paged("cf", seed, [L], Hq=2, Hk=1, D=D, P=P)
    if q_zero:
        w.q.zero_()
    if k_equal:
        page0 = int(w.indices[0])
        ref = w.k_pages[page0, :, 0, :].clone()
        for e in w.indices.tolist():
            w.k_pages[e, :, :, :] = ref[:, None, :]
    return w


def test_closed_form_single_key():
    w = _single(3, 1)
    o, l = run_oracle(w)
    page = int(w.indices[0])
    v0 = w.v_pages[page, 0, 0].double().numpy()
    k0 = w.k_pages[page, 0, 0].double().numpy()
    for h in range(2):
        _close(o[0, h], v0)
        _close(l[0, h], w.sm_scale * float(np.dot(w.q[0, h].double().numpy(), k0)))


@pytest.mark.parametrize("L", [2, 5, 16, 37])
def test_closed_form_zero_query(L):
    w = _single(4, L, q_zero=True)
    o, l = run_oracle(w)
    pages = w.indices.long()
    V = w.v_pages[pages, 0].reshape(-1, w.head_dim)[:L].double().numpy()
    for h in range(2):
        _close(o[0, h], V.mean(0))
        _close(l[0, h], math.log(L))


def test_closed_form_equal_keys():
    L = 23
    w = _single(5, L, k_equal=True)
    o, l = run_oracle(w)
    pages = w.indices.long()
    V = w.v_pages[pages, 0].reshape(-1, w.head_dim)[:L].double().numpy()
    k = w.k_pages[int(pages[0]), 0, 0].double().numpy()
    for h in range(2):
        s = w.sm_scale * float(np.dot(w.q[0, h].double().numpy(), k))
        _close(o[0, h], V.mean(0))
        _close(l[0, h], s + math.log(L), 1e-12)


def test_empty_request():
    w = wl.make_paged("e", 9, [0, 5], Hq=2, Hk=1, D=4, P=2)
    o, l = run_oracle(w)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(l[0]))
    assert np.all(np.isfinite(o[1]))


# ---------------------------------------------------------------- paging invariances

def _relayout(w: wl.Paged, P_new: int, seed: int, contiguous=False) -> wl.Paged:
    """Same token sequences, re-paged at P_new into a freshly permuted pool."""
    Hk, D = w.num_kv_heads, w.head_dim
    toks_k, toks_v, lens = [], [], []
    for b in range(w.batch):
        pages = w.indices[w.indptr[b]:w.indptr[b + 1]].long()
        L = w.kv_len[b]
        toks_k.append(w.k_pages[pages].permute(1, 0, 2, 3).reshape(Hk, -1, D)[:, :L])
        toks_v.append(w.v_pages[pages].permute(1, 0, 2, 3).reshape(Hk, -1, D)[:, :L])
        lens.append(L)
    if contiguous:
        P_new = max(max(lens), 1)
    counts = [(L + P_new - 1) // P_new for L in lens]
    pool = sum(counts) + 3
    perm = torch.randperm(pool, generator=torch.Generator().manual_seed(seed))
    kp = torch.full((pool, Hk, P_new, D), float("nan"), dtype=torch.bfloat16)
    vp = kp.clone()
    indices, indptr, last = [], [0], []
    c = 0
    for b, L in enumerate(lens):
        for j in range(counts[b]):
            page = int(perm[c]); c += 1
            n = min(P_new, L - j * P_new)
            kp[page, :, :n] = toks_k[b][:, j * P_new:j * P_new + n]
            vp[page, :, :n] = toks_v[b][:, j * P_new:j * P_new + n]
            indices.append(page)
        indptr.append(len(indices))
        last.append(L - (counts[b] - 1) * P_new if counts[b] else 0)
    return wl.Paged(name="relayout", num_qo_heads=w.num_qo_heads, num_kv_heads=Hk, head_dim=D,
                    page_size=P_new, num_pages=pool,
                    indptr=torch.tensor(indptr, dtype=torch.int32),
                    indices=torch.tensor(indices, dtype=torch.int32),
                    last_page_len=torch.tensor(last, dtype=torch.int32),
                    qo_indptr=w.qo_indptr, kv_len=list(lens), q=w.q, k_pages=kp, v_pages=vp,
                    sm_scale=w.sm_scale, rope_theta=w.rope_theta, causal=w.causal)


@pytest.mark.parametrize("kw", [dict(), dict(rope_theta=5e5, qo_lens=[2, 1, 3, 1], causal=True)])
def test_page_size_and_contiguous_invariance(kw):
    w = wl.make_paged("p16", 11, [5, 40, 77, 16], Hq=4, Hk=2, D=16, P=16, **kw)
    base_o, base_l = run_oracle(w)
    for P_new, contiguous in ((1, False), (4, False), (16, False), (0, True)):
        r = _relayout(w, P_new, seed=P_new + 1, contiguous=contiguous)
        o, l = run_oracle(r)
        _close(o, base_o)
        _close(l, base_l)


def test_page_permutation_invariance():
    w = wl.make_paged("perm", 12, [33, 64, 3], Hq=4, Hk=2, D=8, P=8)
    o0, l0 = run_oracle(w)
    for seed in (1, 2, 3):
        r = _relayout(w, 8, seed=100 + seed)
        o, l = run_oracle(r)
        _close(o, o0)
        _close(l, l0)


def test_poison_is_never_read():
    w = config3_small = wl.config3(small=True)
    o, l = run_oracle(config3_small)
    assert np.isfinite(o).all() and np.isfinite(l).all()
    # sanity: the pool really is poisoned somewhere
    assert torch.isnan(w.k_pages.float()).any()


# ---------------------------------------------------------------- block sparsity

def test_dropping_pages_equals_masking():
    P = 4
    full = wl.make_paged("full", 21, [29, 17, 40], Hq=4, Hk=2, D=8, P=P)
    rng = np.random.default_rng(5)
    indices, indptr, lens, masks = [], [0], [], []
    for b in range(full.batch):
        pages = full.indices[full.indptr[b]:full.indptr[b + 1]].tolist()
        n = len(pages)
        drop = set(rng.choice(n - 1, size=(n - 1) // 3, replace=False).tolist())
        keep = [j for j in range(n) if j not in drop]
        indices += [pages[j] for j in keep]
        indptr.append(len(indices))
        L = full.kv_len[b]
        mask = torch.ones(L, dtype=torch.bool)
        for j in drop:
            mask[j * P:(j + 1) * P] = False
        masks.append(mask)
        lens.append(int(mask.sum()))
    sparse = wl.Paged(name="sparse", num_qo_heads=4, num_kv_heads=2, head_dim=8, page_size=P,
                      num_pages=full.num_pages, indptr=torch.tensor(indptr, dtype=torch.int32),
                      indices=torch.tensor(indices, dtype=torch.int32),
                      last_page_len=full.last_page_len, qo_indptr=full.qo_indptr, kv_len=lens,
                      q=full.q, k_pages=full.k_pages, v_pages=full.v_pages,
                      sm_scale=full.sm_scale)
    o, l = run_oracle(sparse)
    ro, rl = dense_reference(full, drop_mask=masks)
    _close(o, ro)
    _close(l, rl)


# ---------------------------------------------------------------- merge states

def _split(w: wl.Paged, b: int, cut_pages: int):
    """Two single-request tables: the first cut_pages pages of b, and the rest."""
    pages = w.indices[w.indptr[b]:w.indptr[b + 1]]
    P = w.page_size
    q = w.q[w.qo_indptr[b]:w.qo_indptr[b + 1]]
    parts = []
    for sel, L in ((pages[:cut_pages], cut_pages * P),
                   (pages[cut_pages:], w.kv_len[b] - cut_pages * P)):
        parts.append(wl.Paged(name="part", num_qo_heads=w.num_qo_heads,
                              num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, page_size=P,
                              num_pages=w.num_pages,
                              indptr=torch.tensor([0, len(sel)], dtype=torch.int32),
                              indices=sel.clone(),
                              last_page_len=torch.tensor([P if sel is pages[:cut_pages] else
                                                          int(w.last_page_len[b])],
                                                         dtype=torch.int32),
                              qo_indptr=torch.tensor([0, q.shape[0]], dtype=torch.int32),
                              kv_len=[L], q=q, k_pages=w.k_pages, v_pages=w.v_pages,
                              sm_scale=w.sm_scale))
    parts[0].last_page_len = torch.tensor([P], dtype=torch.int32)
    return parts


@pytest.mark.parametrize("cut", [1, 3, 6])
def test_split_merge_equals_unsplit(cut):
    w = wl.make_paged("split", 31, [57], Hq=4, Hk=2, D=8, P=8)
    o, l = run_oracle(w)
    a, b = _split(w, 0, cut)
    oa, la = run_oracle(a)
    ob, lb = run_oracle(b)
    om, lm = oracle.merge_states(oa, la, ob, lb)
    _close(om, o)
    _close(lm, l)
    # commutative
    om2, lm2 = oracle.merge_states(ob, lb, oa, la)
    _close(om2, om)
    _close(lm2, lm)


def test_merge_with_empty_state_is_identity():
    w = wl.make_paged("m", 32, [20], Hq=4, Hk=2, D=8, P=4)
    o, l = run_oracle(w)
    empty_o = np.zeros_like(o)
    empty_l = np.full_like(l, -np.inf)
    om, lm = oracle.merge_states(o, l, empty_o, empty_l)
    _close(om, o)
    _close(lm, l)
    om, lm = oracle.merge_states(empty_o, empty_l, empty_o, empty_l)
    assert np.all(om == 0) and np.all(np.isneginf(lm))


def test_merge_matches_logsumexp_of_union():
    rng = np.random.default_rng(1)
    sa, sb = rng.normal(size=(3, 5)), rng.normal(size=(3, 7))
    va, vb = rng.normal(size=(5, 4)), rng.normal(size=(7, 4))
    t = torch.from_numpy
    la, lb = torch.logsumexp(t(sa), -1).numpy(), torch.logsumexp(t(sb), -1).numpy()
    oa = (torch.softmax(t(sa), -1) @ t(va)).numpy()
    ob = (torch.softmax(t(sb), -1) @ t(vb)).numpy()
    om, lm = oracle.merge_states(oa, la, ob, lb)
    s = np.concatenate([sa, sb], -1)
    v = np.concatenate([va, vb], 0)
    _close(lm, torch.logsumexp(t(s), -1).numpy())
    _close(om, (torch.softmax(t(s), -1) @ t(v)).numpy())


# ---------------------------------------------------------------- cascade

def test_cascade_equals_flat():
    c = wl.config4(small=True)
    op, lp = run_oracle(c.prefix)
    os_, ls = run_oracle(c.suffix)
    om, lm = oracle.merge_states(op, lp, os_, ls)
    f = wl.flat_cascade(c)
    of, lf = run_oracle(f)
    _close(om, of, 1e-11)
    _close(lm, lf, 1e-11)


# ---------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity_and_norm_preserving():
    rng = np.random.default_rng(2)
    x = rng.normal(size=16)
    _close(oracle.rope(x, 0.0, 5e5), x)
    for p in (1.0, 17.0, 2047.0, 30000.0):
        assert abs(np.linalg.norm(oracle.rope(x, p, 5e5)) - np.linalg.norm(x)) < 1e-12


def test_rope_matches_complex_rotation():
    rng = np.random.default_rng(3)
    for D, p, theta in ((8, 5.0, 10000.0), (128, 2047.0, 5e5), (64, 123.0, 500.0)):
        x = rng.normal(size=D)
        ref = _rope_complex(torch.from_numpy(x)[None], torch.tensor([p]), theta)[0].numpy()
        _close(oracle.rope(x, p, theta), ref, 1e-11)


def test_rope_d2_is_rotation_by_position_radians():
    x = np.array([0.3, -1.2])
    p = 0.7
    c, s = math.cos(p), math.sin(p)
    _close(oracle.rope(x, p, 5e5), np.array([0.3 * c + 1.2 * s, -1.2 * c + 0.3 * s]))


def test_rope_relative_position_shift_invariance():
    base = wl.make_paged("shift", 41, [50], Hq=2, Hk=1, D=16, P=8, rope_theta=1000.0,
                         qo_lens=[3], causal=True)
    o0, l0 = run_oracle(base)
    # prepend 16 tokens (two pages) that the causal mask cannot hide: instead compare
    # per-key scores: shifting both positions by c leaves every q.k unchanged.
    rng = np.random.default_rng(4)
    q, k = rng.normal(size=16), rng.normal(size=16)
    for c in (1.0, 8.0, 1000.0):
        d0 = np.dot(oracle.rope(q, 30.0, 1000.0), oracle.rope(k, 12.0, 1000.0))
        d1 = np.dot(oracle.rope(q, 30.0 + c, 1000.0), oracle.rope(k, 12.0 + c, 1000.0))
        assert abs(d0 - d1) < 1e-9
    assert np.isfinite(o0).all()


# ---------------------------------------------------------------- causal

def test_causal_single_query_equals_noncausal():
    w = tiny(rope_theta=100.0)
    o1, l1 = run_oracle(w)
    w.causal = True
    o2, l2 = run_oracle(w)
    _close(o1, o2)
    _close(l1, l2)


def test_causal_row_equals_decode_at_shorter_length():
    P = 4
    w = wl.make_paged("causal", 51, [30], Hq=4, Hk=2, D=8, P=P, qo_lens=[6], causal=True,
                      rope_theta=300.0)
    o, l = run_oracle(w)
    L = w.kv_len[0]
    pages = w.indices[:int(w.indptr[1])]
    for i in range(6):
        Li = L - 6 + i + 1
        n = (Li + P - 1) // P
        d = wl.Paged(name="d", num_qo_heads=4, num_kv_heads=2, head_dim=8, page_size=P,
                     num_pages=w.num_pages, indptr=torch.tensor([0, n], dtype=torch.int32),
                     indices=pages[:n].clone(),
                     last_page_len=torch.tensor([Li - (n - 1) * P], dtype=torch.int32),
                     qo_indptr=torch.tensor([0, 1], dtype=torch.int32), kv_len=[Li],
                     q=w.q[i:i + 1], k_pages=w.k_pages, v_pages=w.v_pages,
                     sm_scale=w.sm_scale, rope_theta=w.rope_theta)
        od, ld = run_oracle(d)
        _close(o[i], od[0])
        _close(l[i], ld[0])


# ---------------------------------------------------------------- append

def test_append_then_attend_equals_concatenation():
    w = wl.make_paged("app", 61, [20, 9, 33], Hq=4, Hk=2, D=8, P=4, qo_lens=[5, 3, 4],
                      causal=True, append=True)
    # before the append the new slots are poisoned
    assert torch.isnan(w.k_pages.float()).any()
    kp, vp = oracle.append_kv(w.k_new, w.v_new, w.append_indptr, w.indptr, w.indices,
                              w.last_page_len, w.k_pages, w.v_pages, num_kv_heads=2,
                              head_dim=8, page_size=4)
    # the appended tokens are the last n_b tokens of each request, in order
    kpt = torch.from_numpy(kp.view(np.int16)).view(torch.bfloat16)
    for b in range(w.batch):
        pages = w.indices[w.indptr[b]:w.indptr[b + 1]].long()
        L = w.kv_len[b]
        seq = kpt[pages].permute(1, 0, 2, 3).reshape(2, -1, 8)[:, :L]
        new = w.k_new[w.append_indptr[b]:w.append_indptr[b + 1]].permute(1, 0, 2)
        n = new.shape[1]
        assert torch.equal(seq[:, L - n:].view(torch.int16), new.view(torch.int16))
        assert not torch.isnan(seq.float()).any()
    # untouched slots keep their bits
    changed = (kp != oracle._bits(w.k_pages))
    assert changed.sum() == w.k_new.numel()
    w2 = wl.Paged(**{**w.__dict__})
    w2.k_pages = kpt
    w2.v_pages = torch.from_numpy(vp.view(np.int16)).view(torch.bfloat16)
    o, l = run_oracle(w2)
    ro, rl = dense_reference(w2)
    _close(o, ro)
    _close(l, rl)


def test_kv_len_and_malformed_tables():
    assert oracle.kv_len([0, 2, 2, 5], [3, 0, 1], 4).tolist() == [7, 0, 9]
    with pytest.raises(ValueError):
        oracle.kv_len([0, 2], [5], 4)          # last_page_len > P
    with pytest.raises(ValueError):
        oracle.kv_len([0, 2], [0], 4)          # last_page_len 0 with pages
    w = tiny()
    bad = w.indices.clone()
    bad[0] = w.num_pages
    with pytest.raises(ValueError):
        oracle.attention(w.q, w.k_pages, w.v_pages, w.indptr, bad, w.last_page_len,
                         w.qo_indptr, num_qo_heads=4, num_kv_heads=2, head_dim=8,
                         page_size=4, sm_scale=1.0)


def test_bf16_round_helper():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 0.0])
    r = oracle.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(r, ref)


# ---------------------------------------------------------------- FP8 (E4M3) KV cache

def test_e4m3_decoder_matches_torch_and_closed_forms():
    codes = np.arange(256, dtype=np.uint8)
    v = oracle.e4m3(codes)
    t = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(t)
    assert nan.sum() == 2 and np.array_equal(np.isnan(v), nan)       # S.1111.111 only
    assert np.array_equal(v[~nan], t[~nan])
    # the format's landmarks: 1 = 0.0111.000, -1, 448 = 0.1111.110 (largest), smallest
    # normal 2^-6 = 0.0001.000, smallest subnormal 2^-9 = 0.0000.001, +-0
    assert v[0x38] == 1.0 and v[0xB8] == -1.0 and v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9 and v[0x00] == 0.0 and v[0x80] == 0.0
    # every binade holds 8 evenly spaced values
    pos = v[0x08:0x7F]
    assert np.all(np.diff(pos) > 0)


def _kv8_pools_as_bf16(w: wl.Paged):
    """bf16 pools holding exactly the FP8 cache's values (an E4M3 value times a power of
    two is exact in bf16), via torch's own E4M3 conversion."""
    k = (w.k_codes.view(torch.float8_e4m3fn).to(torch.float64) * w.k_scale).to(torch.bfloat16)
    v = (w.v_codes.view(torch.float8_e4m3fn).to(torch.float64) * w.v_scale).to(torch.bfloat16)
    return k, v


def run_oracle_kv8(w: wl.Paged, **kw):
    return oracle.attention_kv8(w.q, w.k_codes, w.v_codes, w.k_scale, w.v_scale, w.indptr,
                                w.indices, w.last_page_len, w.qo_indptr,
                                num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads,
                                head_dim=w.head_dim, page_size=w.page_size,
                                sm_scale=w.sm_scale, rope_theta=w.rope_theta, causal=w.causal,
                                **kw)


@pytest.mark.parametrize("kw", [dict(), dict(qo_lens=[1, 3, 5, 2], causal=True),
                                dict(rope_theta=10000.0), dict(Hq=8, Hk=1, P=1)])
def test_kv8_equals_attention_over_the_decoded_values(kw):
    w = wl.with_kv8(tiny(**kw), 77)
    o8, l8 = run_oracle_kv8(w)
    k, v = _kv8_pools_as_bf16(w)
    w.k_pages, w.v_pages = k, v
    o, l = run_oracle(w)
    assert np.array_equal(o8, o) and np.array_equal(l8, l)
    ro, rl = dense_reference(w)
    _close(o8, ro)
    _close(l8, rl)
    assert np.isfinite(o8).all()


def test_kv8_scales_apply_to_keys_and_values():
    # doubling v_scale doubles the output; k_scale rescales the logits like sm_scale
    w = wl.with_kv8(tiny(), 78)
    o1, l1 = run_oracle_kv8(w)
    w.v_scale *= 2.0
    o2, l2 = run_oracle_kv8(w)
    assert np.array_equal(o2, 2.0 * o1) and np.array_equal(l2, l1)
    w.k_scale *= 2.0
    o3, l3 = run_oracle_kv8(w)
    w.k_scale /= 2.0
    w.sm_scale *= 2.0
    o4, l4 = run_oracle_kv8(w)
    _close(o3, o4)
    _close(l3, l4)


# ---------------------------------------------------------------- sliding window

def _windowed_dense(w: wl.Paged, W: int):
    """dense_reference with every key older than the window masked (a drop mask)."""
    masks = []
    for b in range(w.batch):
        L = w.kv_len[b]
        n = int(w.qo_indptr[b + 1] - w.qo_indptr[b])
        masks.append(None if n != 1 else torch.arange(L) >= L - W)
    return masks


def test_window_wider_than_every_request_changes_nothing():
    w = tiny(qo_lens=[1, 3, 5, 2], causal=True, rope_theta=300.0)
    o, l = run_oracle(w)
    o2, l2 = run_oracle(w, window_left=max(w.kv_len))
    assert np.array_equal(o, o2) and np.array_equal(l, l2)


def test_window_of_one_sees_only_its_own_key():
    w = tiny()                      # decode rows: position L - 1
    o, l = run_oracle(w, window_left=1)
    g = w.num_qo_heads // w.num_kv_heads
    for b in range(w.batch):
        L = w.kv_len[b]
        page = int(w.indices[w.indptr[b] + (L - 1) // w.page_size])
        for h in range(w.num_qo_heads):
            k = w.k_pages[page, h // g, (L - 1) % w.page_size].double()
            v = w.v_pages[page, h // g, (L - 1) % w.page_size].double()
            s = float(w.q[b, h].double() @ k) * w.sm_scale
            _close(o[b, h], v.numpy())
            _close(l[b, h], s)


@pytest.mark.parametrize("W", [2, 5, 9])
def test_window_equals_masking_older_keys(W):
    # decode rows: the window keeps keys L - W .. L - 1, i.e. drops the older ones
    w = tiny(lens=(1, 7, 13, 30, 41))
    o, l = run_oracle(w, window_left=W)
    ro, rl = dense_reference(w, drop_mask=_windowed_dense(w, W))
    _close(o, ro)
    _close(l, rl)


def test_window_causal_rows_equal_decode_with_window():
    # a causal row at position p with window W equals a decode of the first p + 1 keys
    w = tiny(qo_lens=[1, 3, 5, 2], causal=True, rope_theta=100.0)
    W = 4
    o, l = run_oracle(w, window_left=W)
    b, t = 2, int(w.qo_indptr[2]) + 3          # request 2, its 4th query
    L = w.kv_len[b]
    p = L - 5 + 3
    d = wl.make_paged("tiny", 7, [1], Hq=4, Hk=2, D=8, P=4)   # shape holder, replaced below
    d.indptr = torch.tensor([0, int(w.indptr[b + 1] - w.indptr[b])], dtype=torch.int32)
    d.indices = w.indices[w.indptr[b]:w.indptr[b + 1]].clone()
    d.last_page_len = torch.tensor([(p + 1) - ((p + 1 + w.page_size - 1) // w.page_size - 1)
                                    * w.page_size], dtype=torch.int32)
    n_pages = (p + 1 + w.page_size - 1) // w.page_size
    d.indptr[1] = n_pages
    d.indices = d.indices[:n_pages]
    d.kv_len = [p + 1]
    d.qo_indptr = torch.tensor([0, 1], dtype=torch.int32)
    d.q = w.q[t:t + 1].clone()
    d.k_pages, d.v_pages, d.num_pages = w.k_pages, w.v_pages, w.num_pages
    d.rope_theta = w.rope_theta
    od, ld = run_oracle(d, window_left=W)
    _close(o[t], od[0])
    _close(l[t], ld[0])


def test_window_workload_reads_nothing_outside_the_window():
    w = wl.config7(small=True)
    assert int((w.indices == 0).sum()) > 0          # pages aliased to the poisoned page
    o, l = run_oracle(w, window_left=w.window_left)
    assert np.isfinite(o).all() and np.isfinite(l).all()


# ---------------------------------------------------------------- per-page positions

def _dense_with_positions(w: wl.Paged):
    """Dense torch fp64 attention with RoPE at the logical positions w.page_pos gives."""
    Hq, Hk, D, P = w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size
    g = Hq // Hk
    q = w.q.to(torch.float64)
    kp, vp = w.k_pages.to(torch.float64), w.v_pages.to(torch.float64)
    outs, lses = [], []
    for b in range(w.batch):
        e0, e1 = int(w.indptr[b]), int(w.indptr[b + 1])
        pages = w.indices[e0:e1].long()
        L = w.kv_len[b]
        K = kp[pages].permute(1, 0, 2, 3).reshape(Hk, -1, D)[:, :L]
        V = vp[pages].permute(1, 0, 2, 3).reshape(Hk, -1, D)[:, :L]
        kpos = (w.page_pos[e0:e1].long()[:, None] + torch.arange(P)[None, :]).reshape(-1)[:L]
        qb = q[w.qo_indptr[b]:w.qo_indptr[b + 1]]
        n = qb.shape[0]
        qlog = int(w.page_pos[e1 - 1]) + int(w.last_page_len[b]) - n + torch.arange(n)
        qb = _rope_complex(qb, qlog[:, None].expand(n, Hq), w.rope_theta)
        K = _rope_complex(K, kpos[None, :].expand(Hk, L), w.rope_theta)
        s = torch.einsum("nhd,hld->nhl", qb, K.repeat_interleave(g, dim=0)) * w.sm_scale
        if w.causal:
            keep = torch.arange(L)[None, :] <= torch.arange(L - n, L)[:, None]
            s = s.masked_fill(~keep[:, None, :], -math.inf)
        outs.append(torch.einsum("nhl,hld->nhd", torch.softmax(s, -1),
                                 V.repeat_interleave(g, dim=0)))
        lses.append(torch.logsumexp(s, -1))
    return torch.cat(outs).numpy(), torch.cat(lses).numpy()


def test_identity_page_positions_change_nothing():
    w = tiny(rope_theta=300.0, qo_lens=[1, 3, 5, 2], causal=True)
    ident = torch.cat([torch.arange(int(w.indptr[b + 1] - w.indptr[b])) * w.page_size
                       for b in range(w.batch)]).to(torch.int32)
    o, l = run_oracle(w)
    o2, l2 = run_oracle(w, page_pos=ident)
    assert np.array_equal(o, o2) and np.array_equal(l, l2)


@pytest.mark.parametrize("kw", [dict(), dict(qo_lens=[1, 3, 2, 2, 4], causal=True)])
def test_page_positions_rotate_at_the_logical_positions(kw):
    w = tiny(lens=(30, 9, 41, 64, 70), rope_theta=500.0, drop=0.4, **kw)
    assert w.page_pos is not None and int(w.page_pos.max()) > 0
    o, l = run_oracle(w, page_pos=w.page_pos)
    ro, rl = _dense_with_positions(w)
    _close(o, ro, 1e-10)
    _close(l, rl, 1e-10)
    # and they matter: the cached order gives another result when blocks were dropped
    o0, _ = run_oracle(w)
    assert np.abs(o0 - o).max() > 1e-3


def test_page_positions_shift_invariance():
    # RoPE scores depend on position differences only: moving every page of a request
    # (and hence its queries) by the same amount changes nothing
    w = tiny(lens=(30, 9, 41), rope_theta=500.0, drop=0.4)
    o, l = run_oracle(w, page_pos=w.page_pos)
    shifted = w.page_pos.clone()
    e0, e1 = int(w.indptr[1]), int(w.indptr[2])
    shifted[e0:e1] += 1000
    o2, l2 = run_oracle(w, page_pos=shifted)
    _close(o, o2, 1e-9)
    _close(l, l2, 1e-9)


def test_three_level_cascade_equals_flat():
    # system prefix + group prefixes + suffixes, merged level by level == flat attention
    c = wl.config9(small=True)
    o, l = None, None
    for w in c.levels:
        ow, lw = run_oracle(w)
        o, l = (ow, lw) if o is None else oracle.merge_states(o, l, ow, lw)
    f = wl.flat_multi_cascade(c)
    ro, rl = run_oracle(f)
    _close(o, ro, 1e-10)
    _close(l, rl, 1e-10)


# ---------------------------------------------------------------- NHD pages

def test_nhd_pages_equal_hnd_pages():
    # token-major pools hold the same tokens: every result is identical
    for kw in (dict(), dict(qo_lens=[1, 3, 5, 2], causal=True, rope_theta=300.0),
               dict(Hq=6, Hk=3, D=6, P=3)):
        w = tiny(**kw)
        o, l = run_oracle(w)
        n = wl.to_nhd(tiny(**kw))
        o2, l2 = run_oracle(n, kv_layout="NHD")
        assert np.array_equal(o, o2) and np.array_equal(l, l2)


def test_nhd_append_writes_the_same_tokens():
    w = wl.make_paged("app", 11, [9, 20, 5], Hq=4, Hk=2, D=8, P=4, qo_lens=[3, 4, 2],
                      causal=True, append=True)
    kw = dict(num_kv_heads=2, head_dim=8, page_size=4)
    args = (w.k_new, w.v_new, w.append_indptr, w.indptr, w.indices, w.last_page_len)
    kp, vp = oracle.append_kv(*args, w.k_pages, w.v_pages, **kw)
    n = wl.to_nhd(w)
    kn, vn = oracle.append_kv(*args, n.k_pages, n.v_pages, kv_layout="NHD", **kw)
    shape = tuple(n.k_pages.shape)
    to_hnd = lambda a: np.ascontiguousarray(a.reshape(shape).transpose(0, 2, 1, 3))
    assert np.array_equal(to_hnd(kn), kp.reshape(to_hnd(kn).shape))
    assert np.array_equal(to_hnd(vn), vp.reshape(to_hnd(vn).shape))
