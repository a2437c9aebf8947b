"""bsr_attn_decode_noalloc: decode for callers that cannot allocate device memory.

Such callers (a serving runtime that hands out all device memory from its own
pool, a host that forbids allocation while it executes a step) pass every
buffer themselves; the library keeps its scratch in a fixed static device array.
Here the entry point is called through the C ABI and its output is checked
against the planned entry point (bsr_attn_plan + bsr_attn_run) on the same
inputs, with the parity tolerances, on two calls in a row (the second call
reuses the scratch the first one left behind).  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_sparse_kv_bsr_gb300 as bsr
import workloads as wl
from block_sparse_kv_bsr_gb300 import _build
from parity import assert_lse_close, assert_out_close, check_full, device_tensors, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    _build.build()
    bsr.load()


def call_noalloc(w, tensors, out, lse, status):
    """Call the C entry point directly (ctypes), every buffer preallocated by the caller."""
    lib = bsr.load()
    q, k, v = tensors
    dev_tab = [w.indptr.to(q.device), w.indices.to(q.device), w.last_page_len.to(q.device)]
    code = lib.bsr_attn_decode_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(dev_tab[0].data_ptr()),
        ctypes.c_void_p(dev_tab[1].data_ptr()), ctypes.c_void_p(dev_tab[2].data_ptr()),
        w.batch, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, w.num_pages,
        ctypes.c_float(w.sm_scale), ctypes.c_void_p(out.data_ptr()),
        1 if out.dtype == torch.float32 else 0, ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(status.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return code


CASES = {
    "tiny_d64": lambda: wl.config1(),
    "skewed_small_d128": lambda: wl.config3(small=True),
    "page1_gqa8": lambda: wl.make_paged("p1", 31, [1, 40, 0, 333], Hq=16, Hk=2, D=128, P=1),
    "page256": lambda: wl.make_paged("p256", 32, [300, 5, 1000], Hq=8, Hk=8, D=64, P=256),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_planned_entry_point_twice(name, out_dtype):
    w = CASES[name]()
    tensors = device_tensors(w)
    ref_out, ref_lse, _ = run(w, tensors, out_dtype=out_dtype)
    ref_o = ref_out.float().cpu().numpy().astype(np.float64)
    ref_l = ref_lse.cpu().numpy().astype(np.float64)
    bf16 = out_dtype == torch.bfloat16
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device=ref_out.device)
        assert call_noalloc(w, tensors, out, lse, status) == 0
        assert int(status.item()) == 0
        assert_out_close(out.float().cpu().numpy(), ref_o, bf16, f"{name} call {call}")
        assert_lse_close(lse.cpu().numpy(), ref_l, f"{name} call {call}")
        check_full(w, out, lse)      # and against the fp64 oracle


def test_noalloc_refuses_batches_beyond_its_scratch():
    w = wl.make_paged("big", 33, [16] * 257, Hq=8, Hk=8, D=64, P=16)   # 2056 > 2048 units
    tensors = device_tensors(w)
    out = torch.empty_like(tensors[0])
    lse = torch.empty(tensors[0].shape[:2], dtype=torch.float32, device=out.device)
    status = torch.zeros(1, dtype=torch.int32, device=out.device)
    assert call_noalloc(w, tensors, out, lse, status) == -2     # BSR_ERR_UNSUPPORTED


@pytest.mark.parametrize("bad_entry", [0, 2])
def test_noalloc_reports_pages_outside_the_pool(bad_entry):
    """A request naming a page outside the pool is dropped as a whole: every chunk of
    it (the range of 40 keys is cut into several chunks, the bad page sits in the first
    or the last), so its out rows are 0 and its lse -inf; the other request is
    unaffected and still matches the planned entry point."""
    w = wl.make_paged("badpage", 34, [40, 20], Hq=8, Hk=2, D=128, P=16)
    tensors = device_tensors(w)
    ref_out, ref_lse, _ = run(w, tensors, out_dtype=torch.float32)
    bad = w.indices.clone()
    bad[bad_entry] = w.num_pages + 3          # entries 0..2 belong to request 0
    w.indices = bad
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=out.device)
    for call in range(2):
        assert call_noalloc(w, tensors, out, lse, status) == 0
        assert int(status.item()) & 2
        assert torch.equal(out[0].cpu(), torch.zeros_like(out[0].cpu()))
        assert torch.isneginf(lse[0]).all()
        assert_out_close(out[1:].cpu().numpy(), ref_out[1:].cpu().numpy().astype(np.float64),
                         False, "good request beside a bad one")
        assert_lse_close(lse[1:].cpu().numpy(), ref_lse[1:].cpu().numpy().astype(np.float64),
                         "good request beside a bad one")


@pytest.mark.parametrize("fault", ["last_page_len", "huge_count"])
def test_noalloc_malformed_lengths_are_empty(fault):
    """A last_page_len beyond the page size, or a page count whose key count passes
    2^31 - 1 (which also leaves the next request with a negative count), makes only
    the requests concerned empty (status bit 1), and nothing outside the table is read."""
    w = wl.make_paged("badlen", 39, [40, 20, 33], Hq=8, Hk=2, D=128, P=16)
    tensors = device_tensors(w)
    ref_out, ref_lse, _ = run(w, tensors, out_dtype=torch.float32)
    if fault == "last_page_len":
        lpl = w.last_page_len.clone()
        lpl[1] = 17
        w.last_page_len = lpl
        empty, good = [1], [0, 2]
    else:
        ip = w.indptr.clone()
        ip[2] = 1 << 28                        # request 1: 2^28 pages of 16 keys
        w.indptr = ip
        empty, good = [1, 2], [0]
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=out.device)
    assert call_noalloc(w, tensors, out, lse, status) == 0
    assert int(status.item()) & 2
    for r in empty:
        assert torch.equal(out[r].cpu(), torch.zeros_like(out[r].cpu()))
        assert torch.isneginf(lse[r]).all()
    for r in good:
        assert_out_close(out[r].cpu().numpy(), ref_out[r].cpu().numpy().astype(np.float64), False,
                         f"request {r}")
        assert_lse_close(lse[r].cpu().numpy(), ref_lse[r].cpu().numpy().astype(np.float64),
                         f"request {r}")


@pytest.mark.parametrize("P", [16, 32])
def test_noalloc_fp8_cache_matches_the_oracle_twice(P):
    import oracle
    w = wl.with_kv8(wl.make_paged(f"na8p{P}", 35 + P, [300, 17, 0, 1500, 64], Hq=32, Hk=8,
                                  D=128, P=P), 36 + P)
    dev = "cuda:0"
    q, kc, vc = w.q.to(dev), w.k_codes.to(dev), w.v_codes.to(dev)
    tab = [w.indptr.to(dev), w.indices.to(dev), w.last_page_len.to(dev)]
    ro, rl = oracle.attention_kv8(w.q, w.k_codes, w.v_codes, w.k_scale, w.v_scale, w.indptr,
                                  w.indices, w.last_page_len, w.qo_indptr,
                                  num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads,
                                  head_dim=w.head_dim, page_size=w.page_size, sm_scale=w.sm_scale)
    for call in range(2):
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=dev)
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        bsr.bsr_attn_decode_noalloc_kv8(q, kc, vc, *tab, sm_scale=w.sm_scale, k_scale=w.k_scale,
                                        v_scale=w.v_scale, out=out, lse=lse, device_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_out_close(out.cpu().numpy(), ro, False, f"noalloc fp8 P{P} call {call}")
        assert_lse_close(lse.cpu().numpy(), rl, f"noalloc fp8 P{P} call {call}")


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_noalloc_sliding_window(kv_dtype):
    # pages wholly older than every window point at one NaN-poisoned page: a read there
    # would show as NaN
    import oracle
    w = wl.sliding_window_decode("naw", 37, [900, 3000, 40, 1700], 300, Hq=32, Hk=8, D=128,
                                 P=16, causal=False)
    if kv_dtype == "e4m3":
        w = wl.with_kv8(w, 38)
    dev = "cuda:0"
    q = w.q.to(dev)
    k, v = ((w.k_codes, w.v_codes) if kv_dtype == "e4m3" else (w.k_pages, w.v_pages))
    tab = [w.indptr.to(dev), w.indices.to(dev), w.last_page_len.to(dev)]
    kw = dict(num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
              page_size=w.page_size, sm_scale=w.sm_scale, window_left=w.window_left)
    table = (w.indptr, w.indices, w.last_page_len, w.qo_indptr)
    if kv_dtype == "e4m3":
        ro, rl = oracle.attention_kv8(w.q, w.k_codes, w.v_codes, w.k_scale, w.v_scale, *table, **kw)
    else:
        ro, rl = oracle.attention(w.q, w.k_pages, w.v_pages, *table, **kw)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    bsr.bsr_attn_decode_noalloc_ex(q, k.to(dev), v.to(dev), *tab, sm_scale=w.sm_scale, out=out,
                                   kv_dtype=kv_dtype, k_scale=w.k_scale, v_scale=w.v_scale,
                                   window_left=w.window_left, lse=lse, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_out_close(out.cpu().numpy(), ro, False, f"noalloc window {kv_dtype}")
    assert_lse_close(lse.cpu().numpy(), rl, f"noalloc window {kv_dtype}")
