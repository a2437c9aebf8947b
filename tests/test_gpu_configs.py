"""GPU parity on the five workloads: small cases element by element, full sizes on
sampled (query row, head) outputs that the oracle computes one by one."""
import numpy as np
import pytest
import torch

import block_sparse_kv_bsr_gb300 as bsr
import oracle
import workloads as wl
from block_sparse_kv_bsr_gb300 import _build
from parity import (assert_lse_close, assert_out_close, bits, check_full, check_sampled,
                    device_tensors, oracle_full, oracle_rows, plan, run, sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    _build.build()
    bsr.load()


def test_config2_full_size_sampled():
    w = wl.config2()
    out, lse, _ = run(w)
    check_sampled(w, out, lse, n=1536)


def test_config3_full_size_sampled():
    w = wl.config3()
    out, lse, s = run(w)
    info = s.info()
    assert info["decode_imbalance"] < 1.05
    check_sampled(w, out, lse, n=1536)


# ---------------------------------------------------------------- cascade

def run_cascade(c: wl.Cascade, level_dtype):
    dev = "cuda:0"
    q = c.suffix.q.to(dev)
    pk, pv = c.prefix.k_pages.to(dev), c.prefix.v_pages.to(dev)
    sk, sv = c.suffix.k_pages.to(dev), c.suffix.v_pages.to(dev)
    op, lp, _ = run(c.prefix, (q, pk, pv), out_dtype=level_dtype)
    os_, ls, _ = run(c.suffix, (q, sk, sv), out_dtype=level_dtype)
    o, l = bsr.bsr_merge_states(op, lp, os_, ls)
    torch.cuda.synchronize()
    return o, l


@pytest.mark.parametrize("level_dtype", [torch.float32, torch.bfloat16])
def test_cascade_small_equals_flat(level_dtype):
    c = wl.config4(small=True)
    o, l = run_cascade(c, level_dtype)
    f = wl.flat_cascade(c)
    ro, rl = oracle_full(f)
    assert_out_close(o.float().cpu().numpy(), ro, level_dtype == torch.bfloat16, "cascade")
    assert_lse_close(l.cpu().numpy(), rl, "cascade")


def test_cascade_levels_side_by_side():
    """The prefix level planned on a share of the SMs (bsr_schedule_create) and run on a
    second stream while the suffix level runs on the other SMs, then merged: the result
    equals flat attention over prefix + suffix, and each schedule kept to its SMs."""
    c = wl.config4(small=True)
    dev = "cuda:0"
    n = torch.cuda.get_device_properties(0).multi_processor_count
    sp = plan(c.prefix, bsr.bsr_schedule_create(n // 3))
    ss = plan(c.suffix, bsr.bsr_schedule_create(n - n // 3))
    assert sp.info()["num_sms"] == n // 3 and ss.info()["num_sms"] == n - n // 3
    assert sp.info()["prefill_ctas"] <= n // 3
    assert ss.info()["decode_ctas"] <= n - n // 3
    q = c.suffix.q.to(dev)
    pk, pv = c.prefix.k_pages.to(dev), c.prefix.v_pages.to(dev)
    sk, sv = c.suffix.k_pages.to(dev), c.suffix.v_pages.to(dev)
    side = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    fork, join = torch.cuda.Event(), torch.cuda.Event()
    fork.record(main)
    side.wait_event(fork)
    op, lp = bsr.bsr_attn_run(sp, q, pk, pv, sm_scale=c.prefix.sm_scale, out_dtype=torch.float32,
                              stream=side)
    join.record(side)
    os_, ls = bsr.bsr_attn_run(ss, q, sk, sv, sm_scale=c.suffix.sm_scale,
                               out_dtype=torch.float32)
    main.wait_event(join)
    o, l = bsr.bsr_merge_states(op, lp, os_, ls)
    torch.cuda.synchronize()
    assert bsr.bsr_last_device_error(sp) == 0 and bsr.bsr_last_device_error(ss) == 0
    ro, rl = oracle_full(wl.flat_cascade(c))
    assert_out_close(o.float().cpu().numpy(), ro, False, "cascade side by side")
    assert_lse_close(l.cpu().numpy(), rl, "cascade side by side")


def test_cascade_full_size_sampled():
    c = wl.config4()
    o, l = run_cascade(c, torch.float32)
    f = wl.flat_cascade(c)
    rows, heads = sample_rows(f, 768)
    ro, rl = oracle_rows(f, rows, heads)
    assert_out_close(o.float().cpu().numpy()[rows, heads], ro, False, "cascade")
    assert_lse_close(l.cpu().numpy()[rows, heads], rl, "cascade")


# ---------------------------------------------------------------- chunked prefill

def append_then_attend(w: wl.Paged):
    dev = "cuda:0"
    q, k, v = device_tensors(w)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    bsr.bsr_append_kv(w.k_new.to(dev), w.v_new.to(dev), w.append_indptr.to(dev),
                      w.indptr.to(dev), w.indices.to(dev), w.last_page_len.to(dev), k, v,
                      device_status=status)
    out, lse, _ = run(w, (q, k, v))
    assert int(status.item()) == 0
    kp, vp = oracle.append_kv(w.k_new, w.v_new, w.append_indptr, w.indptr, w.indices,
                              w.last_page_len, w.k_pages, w.v_pages,
                              num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                              page_size=w.page_size)
    assert np.array_equal(bits(k).view(np.uint16), kp)
    assert np.array_equal(bits(v).view(np.uint16), vp)
    return out, lse, kp, vp


def test_chunked_prefill_small():
    w = wl.config5(small=True)
    out, lse, kp, vp = append_then_attend(w)
    check_full(w, out, lse, kp, vp)


def test_chunked_prefill_full_size_sampled():
    w = wl.config5()
    out, lse, kp, vp = append_then_attend(w)
    check_sampled(w, out, lse, n=512, k_pages=kp, v_pages=vp)
