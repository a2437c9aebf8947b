"""GPU parity of the FP8 (E4M3) KV-cache decode path against the fp64 oracle.

The cache holds E4M3 codes with one scale per pool; the oracle decodes the
codes from the format definition.  Cases: the skewed block-sparse decode
(small, element by element; full size, sampled rows), ragged tails and split
ranges, a 16-row GQA group, causal multi-query decode rows, page sizes 16 to
256, fp32 output, NaN codes in unowned slots, and the schedules the path does
not cover (refused, not run).
"""
import numpy as np
import pytest
import torch

import block_sparse_kv_bsr_gb300 as bsr
import oracle
import workloads as wl
from block_sparse_kv_bsr_gb300 import _build
from parity import assert_lse_close, assert_out_close, plan, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    _build.build()
    bsr.load()


def run_kv8(w: wl.Paged, out_dtype=torch.bfloat16):
    dev = "cuda:0"
    s = plan(w)
    out, lse = bsr.bsr_attn_run_kv8(s, w.q.to(dev), w.k_codes.to(dev), w.v_codes.to(dev),
                                    k_scale=w.k_scale, v_scale=w.v_scale, sm_scale=w.sm_scale,
                                    rope_theta=w.rope_theta, causal=w.causal, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert bsr.bsr_last_device_error(s) == 0
    return out, lse, s


def oracle_kv8(w: wl.Paged, rows=None, heads=None):
    return oracle.attention_kv8(w.q, w.k_codes, w.v_codes, w.k_scale, w.v_scale, w.indptr,
                                w.indices, w.last_page_len, w.qo_indptr,
                                num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads,
                                head_dim=w.head_dim, page_size=w.page_size,
                                sm_scale=w.sm_scale, rope_theta=w.rope_theta, causal=w.causal,
                                page_pos=w.page_pos, rows=rows, heads=heads)


def check_full_kv8(w, out, lse):
    ro, rl = oracle_kv8(w)
    bf16 = out.dtype == torch.bfloat16
    assert_out_close(out.float().cpu().numpy(), ro, bf16, w.name)
    assert_lse_close(lse.cpu().numpy(), rl, w.name)


def test_kv8_skewed_small():
    w = wl.config6(small=True)
    out, lse, s = run_kv8(w)
    assert s.info()["num_split_streams"] > 0
    check_full_kv8(w, out, lse)


def test_kv8_skewed_full_size_sampled():
    w = wl.config6()
    out, lse, _ = run_kv8(w)
    rows, heads = sample_rows(w, 1536)
    ro, rl = oracle_kv8(w, rows, heads)
    assert_out_close(out.float().cpu().numpy()[rows, heads], ro, True, w.name)
    assert_lse_close(lse.cpu().numpy()[rows, heads], rl, w.name)


@pytest.mark.parametrize("P", [16, 32, 256])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_kv8_page_sizes_and_ragged_tails(P, out_dtype):
    w = wl.with_kv8(wl.make_paged(f"kv8p{P}", 60 + P, [1, 15, 17, 300, 1000, 2600], Hq=32, Hk=8,
                                  D=128, P=P, drop=0.2), 601 + P)
    out, lse, _ = run_kv8(w, out_dtype)
    check_full_kv8(w, out, lse)


def test_kv8_sixteen_row_group_and_long_split():
    # GQA group 16 (two 8-row halves in one MMA row tile), one long request cut into chunks
    w = wl.with_kv8(wl.make_paged("kv8g16", 71, [9000, 40, 333], Hq=32, Hk=2, D=128, P=16), 701)
    out, lse, s = run_kv8(w)
    assert s.info()["num_split_streams"] > 0
    check_full_kv8(w, out, lse)


def test_kv8_causal_multi_query_rows():
    w = wl.with_kv8(wl.make_paged("kv8causal", 72, [50, 400, 1200], Hq=32, Hk=8, D=128, P=16,
                                  qo_lens=[3, 1, 2], causal=True), 702)
    out, lse, s = run_kv8(w)
    assert s.info()["num_prefill_items"] == 0
    check_full_kv8(w, out, lse)


def test_kv8_run_with_host_buffers_matches_the_device_run():
    """bsr_attn_run_host on a schedule planned for E4M3 runs the FP8 kernel with the given
    scales and returns the bits of bsr_attn_run_kv8."""
    dev = "cuda:0"
    w = wl.config11(small=True)
    s = plan(w)
    k, v = w.k_codes.to(dev), w.v_codes.to(dev)
    out, lse = bsr.bsr_attn_run_kv8(s, w.q.to(dev), k, v, k_scale=w.k_scale, v_scale=w.v_scale,
                                    sm_scale=w.sm_scale, rope_theta=w.rope_theta,
                                    causal=w.causal)
    out_h, lse_h = bsr.bsr_attn_run_host(s, w.q.pin_memory(), k, v, k_scale=w.k_scale,
                                         v_scale=w.v_scale, sm_scale=w.sm_scale,
                                         rope_theta=w.rope_theta, causal=w.causal)
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int16), out.cpu().view(torch.int16))
    assert torch.equal(lse_h, lse.cpu())


def test_schedule_planned_for_the_other_cache_type_is_refused():
    """bsr_attn_run_kv8 needs a schedule planned with kv_dtype "e4m3" (its decode work is
    spread over the FP8 kernel's warps), bsr_attn_run one planned for "bf16"."""
    dev = "cuda:0"
    w = wl.with_kv8(wl.make_paged("kv8mis", 74, [100, 200], Hq=32, Hk=8, D=128, P=16), 704)
    kw = dict(num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
              page_size=w.page_size, num_pages=w.num_pages)
    s16 = bsr.bsr_attn_plan(w.indptr, w.indices, w.last_page_len, kv_dtype="bf16", **kw)
    with pytest.raises(bsr.BsrError) as e:
        bsr.bsr_attn_run_kv8(s16, w.q.to(dev), w.k_codes.to(dev), w.v_codes.to(dev),
                             k_scale=w.k_scale, v_scale=w.v_scale, sm_scale=w.sm_scale)
    assert e.value.code == -7
    s8 = bsr.bsr_attn_plan(w.indptr, w.indices, w.last_page_len, kv_dtype="e4m3", **kw)
    assert s8.info()["decode_warps_per_cta"] == 12
    with pytest.raises(bsr.BsrError) as e:
        bsr.bsr_attn_run(s8, w.q.to(dev), w.k_pages.to(dev), w.v_pages.to(dev),
                         sm_scale=w.sm_scale)
    assert e.value.code == -7


def test_kv8_unsupported_schedules_are_refused():
    dev = "cuda:0"
    cases = [
        wl.make_paged("kv8d64", 73, [100, 200], Hq=8, Hk=2, D=64, P=16),          # head_dim 64
        wl.make_paged("kv8pf", 75, [700], Hq=32, Hk=8, D=128, P=16, qo_lens=[300],
                      causal=True),                                                # prefill class
        wl.make_paged("kv8p8", 76, [100, 200], Hq=32, Hk=8, D=128, P=8),            # P < 16
    ]
    for w in cases:
        w = wl.with_kv8(w, 703)
        s = plan(w)
        with pytest.raises(bsr.BsrError):
            bsr.bsr_attn_run_kv8(s, w.q.to(dev), w.k_codes.to(dev), w.v_codes.to(dev),
                                 k_scale=w.k_scale, v_scale=w.v_scale, sm_scale=w.sm_scale,
                                 rope_theta=w.rope_theta, causal=w.causal)


# ---------------------------------------------------------------- FP8 cache with RoPE

def test_kv8_rope_llama8b_small():
    w = wl.config11(small=True)
    out, lse, _ = run_kv8(w)
    check_full_kv8(w, out, lse)


def test_kv8_rope_llama8b_full_size_sampled():
    w = wl.config11()
    out, lse, _ = run_kv8(w)
    rows, heads = sample_rows(w, 1536)
    ro, rl = oracle_kv8(w, rows, heads)
    assert_out_close(out.float().cpu().numpy()[rows, heads], ro, True, w.name)
    assert_lse_close(lse.cpu().numpy()[rows, heads], rl, w.name)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_kv8_rope_short_keys_and_causal_rows(out_dtype):
    """Rows that see a handful of keys (the rotated operands' rounding does not average
    out), several query rows per request, a 16-row group: the plain bars."""
    w = wl.with_kv8(wl.make_paged("kv8ropeshort", 81, [5, 17, 40, 300, 2100], Hq=32, Hk=2,
                                  D=128, P=16, qo_lens=[1, 3, 1, 2, 1], causal=True,
                                  rope_theta=1e4), 811)
    out, lse, _ = run_kv8(w, out_dtype)
    check_full_kv8(w, out, lse)


@pytest.mark.parametrize("P", [16, 64])
def test_kv8_rope_at_logical_positions(P):
    """Dropped blocks keep the logical positions of the kept ones (page_pos)."""
    w = wl.with_kv8(wl.make_paged(f"kv8ropepos{P}", 82 + P, [900, 3000, 40], Hq=32, Hk=8, D=128,
                                  P=P, drop=0.25, rope_theta=5e5), 821 + P)
    assert w.page_pos is not None
    out, lse, _ = run_kv8(w)
    check_full_kv8(w, out, lse)


def test_kv8_rope_query_beyond_operand_range_sets_status():
    """A rotated query element of magnitude 2^20 or more does not fit its fp16 operand:
    status bit 1."""
    dev = "cuda:0"
    w = wl.with_kv8(wl.make_paged("kv8roperange", 83, [300, 200], Hq=32, Hk=8, D=128, P=16,
                                  rope_theta=1e4), 831)
    q = w.q.clone()
    q[0, 0, 3] = 3.0e6
    s = plan(w)
    bsr.bsr_attn_run_kv8(s, q.to(dev), w.k_codes.to(dev), w.v_codes.to(dev), k_scale=w.k_scale,
                         v_scale=w.v_scale, sm_scale=w.sm_scale, rope_theta=w.rope_theta)
    torch.cuda.synchronize()
    assert bsr.bsr_last_device_error(s) & 2
