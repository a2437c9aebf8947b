"""GPU parity of the tensor-core (tcgen05/TMEM) prefill kernel against the fp64 oracle.

Requests whose packed (query, head) rows fill at least half of a 128-row tile
take this kernel; the cases cover causal and non-causal attention, RoPE,
ragged row tiles, key counts that are not multiples of the 128-key tile,
page sizes 16/32/256 and key ranges split over several CTAs and merged.
"""
import math

import numpy as np
import pytest
import torch

import block_sparse_kv_bsr_gb300 as bsr
import workloads as wl
from block_sparse_kv_bsr_gb300 import _build
from parity import (LSE_ATOL, assert_lse_close, assert_out_close, check_full, device_tensors,
                    oracle_full, plan, run)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    _build.build()
    bsr.load()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("P", [16, 32, 256])
def test_prefill_no_rope(causal, P):
    w = wl.make_paged(f"pf{P}", 40 + P, [700, 333, 1300], Hq=32, Hk=8, D=128, P=P,
                      qo_lens=[37, 16, 300], causal=causal)
    out, lse, s = run(w)
    info = s.info()
    assert info["num_prefill_items"] > 0
    check_full(w, out, lse)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_prefill_rope_causal(out_dtype):
    w = wl.make_paged("pfrope", 51, [900, 1500], Hq=32, Hk=8, D=128, P=16,
                      qo_lens=[100, 257], causal=True, rope_theta=5e5)
    out, lse, s = run(w, out_dtype=out_dtype)
    assert s.info()["num_prefill_items"] > 0
    check_full(w, out, lse)


def test_prefill_split_ranges_merge():
    # few row tiles against many keys: the planner cuts key ranges to fill the SMs
    w = wl.make_paged("pfsplit", 52, [20000], Hq=32, Hk=8, D=128, P=16, qo_lens=[64])
    out, lse, s = run(w)
    info = s.info()
    assert info["num_prefill_items"] > info["num_split_streams"] > 0
    check_full(w, out, lse)


def test_prefill_rows_at_the_class_boundary():
    # 16 queries x group 4 = 64 rows (prefill) next to 15 x 4 = 60 rows (decode groups)
    w = wl.make_paged("pfmix", 53, [400, 401], Hq=32, Hk=8, D=128, P=16, qo_lens=[16, 15],
                      causal=True)
    out, lse, s = run(w)
    info = s.info()
    assert info["num_prefill_items"] > 0 and info["num_decode_items"] > 0
    check_full(w, out, lse)


def test_prefill_rope_short_keys_within_rounding_bound():
    """RoPE with very few keys per query: the rotated q and k are fp16 MMA operands
    (scaled by 2^-4), so each rotated element carries a rounding error of at most
    2^-11 of itself plus 2^-21 (half the fp16 subnormal spacing, unscaled).  A score
    then moves by at most sm_scale * (2^-10 * sum_f |q_f| |k_f| + 2^-21 * sum_d (|q_d| +
    |k_d|)) with |x_f| the norm of rotation pair f (rotation keeps it).  lse and out
    are checked against that bound (plus the usual bars) instead of the bare 1e-3,
    which long key ranges meet by averaging."""
    w = wl.make_paged("pfshort", 54, [70, 130], Hq=32, Hk=8, D=128, P=16, qo_lens=[64, 64],
                      causal=True, rope_theta=1e4)
    out, lse, _ = run(w)
    ro, rl = oracle_full(w)
    q = w.q.double()
    bound = 0.0
    for b in range(w.batch):
        pages = w.indices[w.indptr[b]:w.indptr[b + 1]].long()
        K = w.k_pages[pages].permute(1, 0, 2, 3).reshape(w.num_kv_heads, -1, 128)[:, :w.kv_len[b]]
        qb = q[w.qo_indptr[b]:w.qo_indptr[b + 1]]
        # pair norms bound the rotated elements and products
        qa = qb.abs().view(qb.shape[0], qb.shape[1], 2, 64).pow(2).sum(2).sqrt()
        ka = K.double().abs().view(K.shape[0], K.shape[1], 2, 64).pow(2).sum(2).sqrt()
        kh = ka.repeat_interleave(w.num_qo_heads // w.num_kv_heads, 0)
        s_abs = torch.einsum("nhf,hlf->nhl", qa, kh)
        sums = qa.sum(-1)[:, :, None] * 2 ** 0.5 + kh.sum(-1)[None, :, :] * 2 ** 0.5
        b_all = (s_abs * 2.0 ** -10 + sums * 2.0 ** -21) * w.sm_scale
        bound = max(bound, float(b_all.max()))
    err_l = np.abs(lse.cpu().numpy() - rl)
    assert err_l.max() <= LSE_ATOL + bound, (err_l.max(), bound)
    err_o = np.abs(out.float().cpu().numpy() - ro)
    assert err_o.max() <= 5e-3 + 2 * bound * np.abs(w.v_pages.float().nan_to_num()).max()


def test_prefill_rope_operand_range_sets_status():
    """A rotated key beyond the fp16 operand range (|x| >= 2^20) sets status bit 1;
    planning again clears the word."""
    w = wl.make_paged("pfrange", 55, [300], Hq=32, Hk=8, D=128, P=16, qo_lens=[64],
                      causal=True, rope_theta=1e4)
    q, k, v = device_tensors(w)
    k = k.clone()
    k[int(w.indices[0]), 0, 0, :] = 3.0e6       # key 0 of request 0, kv head 0
    s = plan(w)
    assert s.info()["num_prefill_items"] > 0
    bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, rope_theta=w.rope_theta, causal=w.causal)
    torch.cuda.synchronize()
    assert bsr.bsr_last_device_error(s) & 2
    s = plan(w, s)
    bsr.bsr_attn_run(s, q, *device_tensors(w)[1:], sm_scale=w.sm_scale, rope_theta=w.rope_theta,
                     causal=w.causal)
    torch.cuda.synchronize()
    assert bsr.bsr_last_device_error(s) == 0


@pytest.mark.parametrize("Hq,rope", [(8, 0.0), (16, 0.0), (64, 1e4), (128, 0.0)])
def test_prefill_group_sizes(Hq, rope):
    """A query tile is 128 / group whole queries of one kv head's group (one TMA box)."""
    g = Hq // 8
    w = wl.make_paged(f"pfg{g}", 60 + g, [500, 900], Hq=Hq, Hk=8, D=128, P=16, qo_lens=[200, 77],
                      causal=True, rope_theta=rope)
    out, lse, s = run(w)
    assert s.info()["num_prefill_items"] > 0
    check_full(w, out, lse)


def test_prefill_group_not_dividing_the_tile_takes_decode():
    # group 3 does not divide a 128-row tile: every row goes to the decode kernel
    w = wl.make_paged("pfg3", 70, [400, 260], Hq=24, Hk=8, D=128, P=16, qo_lens=[100, 64],
                      causal=True, rope_theta=1e4)
    out, lse, s = run(w)
    info = s.info()
    assert info["num_prefill_items"] == 0 and info["num_decode_items"] > 0
    check_full(w, out, lse)


def test_stage_timing_hook():
    """Per-stage events of bsr_attn_run: RoPE pre-pass, prefill and (with split ranges)
    merge are timed for the kept runs; a run that was not kept is refused."""
    w = wl.make_paged("pftime", 57, [20000], Hq=32, Hk=8, D=128, P=16, qo_lens=[64],
                      causal=True, rope_theta=1e4)
    q, k, v = device_tensors(w)
    s = plan(w)
    info = s.info()
    assert info["kernels_per_run"] == 3 and info["num_split_streams"] > 0
    bsr.bsr_schedule_set_stage_timing(s, 2)
    for _ in range(3):
        bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, rope_theta=w.rope_theta, causal=True)
    for call in range(2):
        t = bsr.bsr_schedule_stage_times(s, call)
        assert set(t) == {"rope_prepass", "prefill", "merge"} and all(x > 0 for x in t.values())
    with pytest.raises(bsr.BsrError):
        bsr.bsr_schedule_stage_times(s, 2)
    bsr.bsr_schedule_set_stage_timing(s, 0)
    with pytest.raises(bsr.BsrError):
        bsr.bsr_schedule_stage_times(s, 0)


def test_replan_grow_then_shrink_keeps_rope_tables():
    # One schedule re-planned for longer, then shorter requests: the cos/sin tables it
    # keeps (grown once, reused after) must serve the decode kernel and the prefill
    # RoPE pre-pass alike.
    short = wl.make_paged("rp_short", 54, [900, 40], Hq=32, Hk=8, D=128, P=16,
                          qo_lens=[100, 1], causal=True, rope_theta=5e5)
    long_ = wl.make_paged("rp_long", 55, [6000, 77], Hq=32, Hk=8, D=128, P=16,
                          qo_lens=[150, 1], causal=True, rope_theta=5e5)
    s = None
    for w in (short, long_, short):
        out, lse, s = run(w, schedule=s)
        info = s.info()
        assert info["num_prefill_items"] > 0 and info["num_decode_items"] > 0
        check_full(w, out, lse)
