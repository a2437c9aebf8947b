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
from parity import check_full, device_tensors, plan, run

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


def test_prefill_rope_short_keys():
    """RoPE prefill rows that see very few keys (the first queries of a chunk appended
    after a 6-key history): the rotated q and k enter the products with rounding that
    cannot average out over many keys, and the rows are still held to the plain bars
    (out 5e-3, lse 1e-3)."""
    w = wl.make_paged("pfshort", 54, [70, 130], Hq=32, Hk=8, D=128, P=16, qo_lens=[64, 64],
                      causal=True, rope_theta=1e4)
    out, lse, _ = run(w)
    e_out, e_lse = check_full(w, out, lse)
    print(f"prefill RoPE short keys: out max err {e_out:.3e}, lse max err {e_lse:.3e}")


@pytest.mark.parametrize("rope", [0.0, 5e5])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_prefill_fresh_prompt_rows_with_few_keys(rope, out_dtype):
    """A prompt with no history (kv_len == qo_len, causal): query row i sees i + 1 keys,
    so the first rows of each request weigh a handful of keys, where neither the
    rounding of P nor (with RoPE) that of the rotated q and k averages out.  Held to the
    plain bars (out 5e-3, lse 1e-3)."""
    w = wl.make_paged("pffresh", 77, [256, 300, 129], Hq=32, Hk=8, D=128, P=16,
                      qo_lens=[256, 300, 129], causal=True, rope_theta=rope)
    out, lse, s = run(w, out_dtype=out_dtype)
    assert s.info()["num_prefill_items"] > 0 and s.info()["num_decode_items"] == 0
    e_out, e_lse = check_full(w, out, lse)
    print(f"fresh prompt rope={rope} {out_dtype}: out max err {e_out:.3e}, lse {e_lse:.3e}")


@pytest.mark.parametrize("rope", [0.0, 5e5])
def test_prefill_one_tile_units_between_two_tile_units(rope):
    """600 packed rows per (request, kv head) make units of 256, 256 and 88 rows, so a
    CTA's list mixes units of two query tiles with units of one, whose second-tile
    warps have no rows but still take their share of every V tile in ring order."""
    w = wl.make_paged("pfmixtiles", 78, [350, 700, 500, 160], Hq=32, Hk=8, D=128, P=16,
                      qo_lens=[150, 150, 150, 150], causal=True, rope_theta=rope)
    out, lse, s = run(w)
    assert s.info()["num_prefill_items"] > 0
    check_full(w, out, lse)


@pytest.mark.parametrize("causal,P,rope", [(False, 16, 0.0), (True, 16, 1e4), (True, 32, 5e5),
                                            (True, 256, 0.0)])
def test_prefill_head_dim_64(causal, P, rope):
    """head_dim 64 on the tensor-core kernel: the 128-wide tile program with the upper
    64 dimensions of q, k and v landing as zeros, RoPE pairs 32 apart."""
    w = wl.make_paged(f"pf64_{P}", 90 + P, [700, 333, 1300], Hq=16, Hk=4, D=64, P=P,
                      qo_lens=[37, 16, 300], causal=causal, rope_theta=rope)
    out, lse, s = run(w)
    assert s.info()["num_prefill_items"] > 0
    e_out, e_lse = check_full(w, out, lse)
    print(f"head_dim 64 causal={causal} P={P} rope={rope}: out {e_out:.3e}, lse {e_lse:.3e}")


@pytest.mark.parametrize("rope", [0.0, 1e4])
def test_prefill_head_dim_64_split_ranges_and_nhd(rope):
    """head_dim 64: key ranges split over CTAs and merged (fp32 out), and token-major
    (NHD) pages, against the oracle."""
    w = wl.make_paged("pf64split", 95, [20000], Hq=32, Hk=8, D=64, P=16, qo_lens=[64],
                      causal=True, rope_theta=rope)
    out, lse, s = run(w, out_dtype=torch.float32)
    assert s.info()["num_prefill_items"] > s.info()["num_split_streams"] > 0
    check_full(w, out, lse)
    n = wl.to_nhd(wl.make_paged("pf64nhd", 96, [500, 900], Hq=16, Hk=4, D=64, P=16,
                                qo_lens=[200, 129], causal=True, rope_theta=rope))
    out, lse, s = run(n)
    assert s.info()["num_prefill_items"] > 0
    check_full(n, out, lse)


@pytest.mark.parametrize("rope", [0.0, 1e4])
def test_prefill_head_dim_64_sliding_window(rope):
    """head_dim 64 with a 150-key sliding window (the windowed kernel variants, RoPE pairs
    32 apart included): units start at the page holding their oldest visible key."""
    w = wl.make_paged("pf64win", 98, [900, 400], Hq=16, Hk=4, D=64, P=16,
                      qo_lens=[200, 100], causal=True, rope_theta=rope)
    w.window_left = 150
    out, lse, s = run(w)
    assert s.info()["num_prefill_items"] > 0 and s.info()["window_left"] == 150
    check_full(w, out, lse)


def test_prefill_head_dim_64_fresh_prompt():
    """A head_dim 64 prompt with no history: its first rows see a handful of keys.
    Plain bars, with RoPE."""
    w = wl.make_paged("pf64fresh", 97, [256, 300], Hq=16, Hk=4, D=64, P=16,
                      qo_lens=[256, 300], causal=True, rope_theta=1e4)
    out, lse, s = run(w)
    assert s.info()["num_prefill_items"] > 0 and s.info()["num_decode_items"] == 0
    e_out, e_lse = check_full(w, out, lse)
    print(f"head_dim 64 fresh prompt: out {e_out:.3e}, lse {e_lse:.3e}")


def test_prefill_v_beyond_fp16_range_sets_status():
    """P and V enter P.V as fp16: a V value beyond 65504 on the tensor-core path sets
    status bit 1 instead of passing silently; planning again clears the word."""
    w = wl.make_paged("pfvrange", 56, [300], Hq=32, Hk=8, D=128, P=16, qo_lens=[64],
                      causal=True)
    q, k, v = device_tensors(w)
    v = v.clone()
    v[int(w.indices[1]), 3, 2, 7] = 1.0e5       # key 18 of request 0, kv head 3
    s = plan(w)
    assert s.info()["num_prefill_items"] > 0
    bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, causal=w.causal)
    torch.cuda.synchronize()
    assert bsr.bsr_last_device_error(s) & 2
    s = plan(w, s)
    bsr.bsr_attn_run(s, *device_tensors(w), sm_scale=w.sm_scale, causal=w.causal)
    torch.cuda.synchronize()
    assert bsr.bsr_last_device_error(s) == 0


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
    """Per-stage events of bsr_attn_run: prefill (RoPE fused in) and, with split ranges,
    merge are timed for the kept runs; a run that was not kept is refused."""
    w = wl.make_paged("pftime", 57, [20000], Hq=32, Hk=8, D=128, P=16, qo_lens=[64],
                      causal=True, rope_theta=1e4)
    q, k, v = device_tensors(w)
    s = plan(w)
    info = s.info()
    assert info["kernels_per_run"] == 2 and info["num_split_streams"] > 0
    bsr.bsr_schedule_set_stage_timing(s, 2)
    for _ in range(3):
        bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, rope_theta=w.rope_theta, causal=True)
    for call in range(2):
        t = bsr.bsr_schedule_stage_times(s, call)
        assert set(t) == {"prefill", "merge"} and all(x > 0 for x in t.values())
    with pytest.raises(bsr.BsrError):
        bsr.bsr_schedule_stage_times(s, 2)
    bsr.bsr_schedule_set_stage_timing(s, 0)
    with pytest.raises(bsr.BsrError):
        bsr.bsr_schedule_stage_times(s, 0)


def test_replan_grow_then_shrink_keeps_rope_tables():
    # One schedule re-planned for longer, then shorter requests: the cos/sin tables it
    # keeps (grown once, reused after) must serve the decode kernel and the prefill
    # kernel's in-tile rotation alike.
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
