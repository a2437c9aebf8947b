"""GPU parity of the sliding-window variant against the fp64 oracle.

Every page a request holds outside all of its rows' windows points at one
NaN-poisoned page (workloads.sliding_window_decode), so a kernel that reads
outside the window returns NaN.  Cases: windowed decode (small element by
element, full size sampled), causal multi-query decode rows, the tensor-core
prefill kernel (with and without RoPE), the FP8 cache path, and a window wider
than every request (identical to no window).
"""
import numpy as np
import pytest
import torch

import block_sparse_kv_bsr_gb300 as bsr
import oracle
import workloads as wl
from block_sparse_kv_bsr_gb300 import _build
from parity import assert_lse_close, assert_out_close, plan, run, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    _build.build()
    bsr.load()


def oracle_w(w: wl.Paged, rows=None, heads=None):
    kw = dict(num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
              page_size=w.page_size, sm_scale=w.sm_scale, rope_theta=w.rope_theta,
              causal=w.causal, window_left=w.window_left, rows=rows, heads=heads)
    table = (w.indptr, w.indices, w.last_page_len, w.qo_indptr)
    if w.k_codes is not None:
        return oracle.attention_kv8(w.q, w.k_codes, w.v_codes, w.k_scale, w.v_scale, *table, **kw)
    return oracle.attention(w.q, w.k_pages, w.v_pages, *table, **kw)


def check(w, out, lse, rows=None, heads=None):
    ro, rl = oracle_w(w, rows, heads)
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    if rows is not None:
        o, l = o[rows, heads], l[rows, heads]
    assert_out_close(o, ro, out.dtype == torch.bfloat16, w.name)
    assert_lse_close(l, rl, w.name)


def test_window_decode_small():
    w = wl.config7(small=True)
    out, lse, s = run(w)
    assert s.info()["window_left"] == w.window_left
    check(w, out, lse)


def test_window_decode_full_size_sampled():
    w = wl.config7()
    out, lse, _ = run(w)
    rows, heads = sample_rows(w, 1536)
    check(w, out, lse, rows, heads)


def test_window_causal_multi_query_decode_rows():
    w = wl.sliding_window_decode("swq", 81, [400, 1500, 77], 130, Hq=32, Hk=8, D=128, P=16,
                                 qo_lens=[3, 7, 2])
    out, lse, s = run(w)
    assert s.info()["num_prefill_items"] == 0
    check(w, out, lse)


@pytest.mark.parametrize("rope", [0.0, 5e5])
def test_window_prefill(rope):
    w = wl.sliding_window_decode("swpf", 82, [3000, 900], 700, Hq=32, Hk=8, D=128, P=16,
                                 qo_lens=[300, 1])
    w.rope_theta = rope
    out, lse, s = run(w, out_dtype=torch.float32)
    assert s.info()["num_prefill_items"] > 0
    check(w, out, lse)


def test_window_fp8_cache():
    w = wl.with_kv8(wl.config7(small=True), 83)
    dev = "cuda:0"
    s = plan(w)
    out, lse = bsr.bsr_attn_run_kv8(s, w.q.to(dev), w.k_codes.to(dev), w.v_codes.to(dev),
                                    k_scale=w.k_scale, v_scale=w.v_scale, sm_scale=w.sm_scale,
                                    causal=w.causal)
    torch.cuda.synchronize()
    assert bsr.bsr_last_device_error(s) == 0
    check(w, out, lse)


@pytest.mark.parametrize("P", [4, 8, 32])
def test_window_page_sizes(P):
    # pages below 16 keys: a 16-key stage spans pages that lie wholly before the window
    w = wl.sliding_window_decode(f"swp{P}", 84 + P, [300, 700, 45, 1200], 37, Hq=8, Hk=2, D=64,
                                 P=P)
    out, lse, _ = run(w)
    check(w, out, lse)


def test_window_wider_than_every_request_is_no_window():
    w = wl.config3(small=True)
    out0, lse0, _ = run(w)
    w.window_left = max(w.kv_len) + 5
    out1, lse1, _ = run(w)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
