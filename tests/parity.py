"""Shared helpers for the GPU parity tests: run the library, run the oracle, compare.

Tolerances (stated once, used everywhere):
  * out: max-abs 5e-3 against the fp64 oracle.  A bf16 output cannot be closer
    to the exact value than half a bf16 ulp, which exceeds 5e-3 once
    |out| >= 2; there the bar is that half ulp plus 1e-3 (the kernel's own
    error budget).  fp32 outputs are held to 5e-3 everywhere.
  * lse: max-abs 1e-3; an empty row must give -inf on both sides.
  * append_kv: bit exact.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import block_sparse_kv_bsr_gb300 as bsr
import oracle
import workloads as wl

OUT_ATOL = 5e-3
LSE_ATOL = 1e-3


def device_tensors(w: wl.Paged, dev="cuda:0"):
    return (w.q.to(dev), w.k_pages.to(dev), w.v_pages.to(dev))


def plan(w: wl.Paged, schedule=None):
    return bsr.bsr_attn_plan(w.indptr, w.indices, w.last_page_len,
                             num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads,
                             head_dim=w.head_dim, page_size=w.page_size, num_pages=w.num_pages,
                             qo_indptr=w.qo_indptr, causal=w.causal, rope_theta=w.rope_theta,
                             window_left=w.window_left, page_pos=w.page_pos,
                             kv_layout=w.kv_layout,
                             kv_dtype="e4m3" if w.k_codes is not None else "bf16",
                             schedule=schedule)


def run(w: wl.Paged, tensors=None, out_dtype=torch.bfloat16, schedule=None):
    q, k, v = tensors if tensors is not None else device_tensors(w)
    s = plan(w, schedule)
    out, lse = bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, rope_theta=w.rope_theta,
                                causal=w.causal, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert bsr.bsr_last_device_error(s) == 0
    return out, lse, s


def oracle_full(w: wl.Paged, k_pages=None, v_pages=None):
    return oracle.attention(w.q, w.k_pages if k_pages is None else k_pages,
                            w.v_pages if v_pages is None else v_pages, w.indptr, w.indices,
                            w.last_page_len, w.qo_indptr, num_qo_heads=w.num_qo_heads,
                            num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                            page_size=w.page_size, sm_scale=w.sm_scale,
                            rope_theta=w.rope_theta, causal=w.causal,
                            window_left=w.window_left, page_pos=w.page_pos,
                            kv_layout=w.kv_layout)


def oracle_rows(w: wl.Paged, rows, heads, k_pages=None, v_pages=None):
    return oracle.attention(w.q, w.k_pages if k_pages is None else k_pages,
                            w.v_pages if v_pages is None else v_pages, w.indptr, w.indices,
                            w.last_page_len, w.qo_indptr, num_qo_heads=w.num_qo_heads,
                            num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                            page_size=w.page_size, sm_scale=w.sm_scale,
                            rope_theta=w.rope_theta, causal=w.causal,
                            window_left=w.window_left, page_pos=w.page_pos,
                            kv_layout=w.kv_layout, rows=rows, heads=heads)


def sample_rows(w: wl.Paged, n: int, seed: int = 0):
    """n (query row, qo head) pairs: every request's last row and head 0/last, plus random."""
    rng = np.random.default_rng(seed)
    sum_qo = int(w.qo_indptr[-1])
    rows = list(rng.integers(0, sum_qo, n))
    heads = list(rng.integers(0, w.num_qo_heads, n))
    for b in range(w.batch):
        if w.qo_indptr[b + 1] > w.qo_indptr[b]:
            rows += [int(w.qo_indptr[b + 1]) - 1] * 2
            heads += [0, w.num_qo_heads - 1]
    return np.array(rows, dtype=np.int64), np.array(heads, dtype=np.int32)


def out_tolerance(ref: np.ndarray, bf16: bool) -> np.ndarray:
    tol = np.full(ref.shape, OUT_ATOL)
    if bf16:
        mag = np.abs(ref)
        big = mag >= 2.0
        if big.any():
            e = np.floor(np.log2(mag[big]))
            tol[big] = np.maximum(OUT_ATOL, np.exp2(e - 8) + 1e-3)
    return tol


def assert_out_close(gpu: np.ndarray, ref: np.ndarray, bf16: bool, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    assert np.isfinite(gpu).all(), f"{what}: non-finite output"
    err = np.abs(gpu - ref)
    tol = out_tolerance(ref, bf16)
    bad = err > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs off; max err {err.max():.3e} "
                           f"at ref {ref.flat[np.argmax(err)]:.4f}")
    return float(err.max()) if err.size else 0.0


def assert_lse_close(gpu: np.ndarray, ref: np.ndarray, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    neg = np.isneginf(ref)
    assert np.array_equal(np.isneginf(gpu), neg), f"{what}: -inf rows differ"
    fin = ~neg
    assert np.isfinite(gpu[fin]).all(), f"{what}: non-finite lse"
    err = np.abs(gpu[fin] - ref[fin])
    assert err.size == 0 or err.max() <= LSE_ATOL, f"{what}: lse max err {err.max():.3e}"
    return float(err.max()) if err.size else 0.0


def check_full(w: wl.Paged, out: torch.Tensor, lse: torch.Tensor, k_pages=None, v_pages=None):
    ro, rl = oracle_full(w, k_pages, v_pages)
    bf16 = out.dtype == torch.bfloat16
    e1 = assert_out_close(out.float().cpu().numpy(), ro, bf16, w.name)
    e2 = assert_lse_close(lse.cpu().numpy(), rl, w.name)
    return e1, e2


def check_sampled(w: wl.Paged, out: torch.Tensor, lse: torch.Tensor, n=1024, seed=0,
                  k_pages=None, v_pages=None):
    rows, heads = sample_rows(w, n, seed)
    ro, rl = oracle_rows(w, rows, heads, k_pages, v_pages)
    o = out.float().cpu().numpy()[rows, heads]
    l = lse.cpu().numpy()[rows, heads]
    bf16 = out.dtype == torch.bfloat16
    return (assert_out_close(o, ro, bf16, w.name), assert_lse_close(l, rl, w.name))


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy()
