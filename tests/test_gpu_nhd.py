"""GPU parity over token-major (NHD) page pools [pages, P, Hk, D]: the same batches as
the head-major tests, with the pools transposed, through every kernel path (decode
with TMA stages and with pages below 16 keys, FP8 decode, tensor-core prefill with
page-sized and whole-tile K boxes, RoPE rotated in the prefill kernel, append_kv) against the oracle
reading the same NHD pools."""
import numpy as np
import pytest
import torch

import block_sparse_kv_bsr_gb300 as bsr
import oracle
import workloads as wl
from block_sparse_kv_bsr_gb300 import _build
from parity import bits, check_full, check_sampled, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    _build.build()
    bsr.load()


def test_nhd_decode_small():
    w = wl.config10(small=True)
    out, lse, s = run(w)
    assert s.info()["kv_layout"] == bsr.BSR_KV_NHD
    check_full(w, out, lse)


def test_nhd_decode_full_size_sampled():
    w = wl.config10()
    out, lse, _ = run(w)
    check_sampled(w, out, lse, n=1536)


@pytest.mark.parametrize("P,D", [(4, 64), (8, 128), (32, 128), (16, 64)])
def test_nhd_decode_page_sizes(P, D):
    w = wl.to_nhd(wl.make_paged(f"nhd{P}", 101 + P, [1, 40, 333, 1200], Hq=16, Hk=4, D=D, P=P,
                                qo_lens=[1, 2, 3, 1], causal=True))
    out, lse, _ = run(w, out_dtype=torch.float32)
    check_full(w, out, lse)


@pytest.mark.parametrize("P,rope", [(16, 0.0), (16, 5e5), (128, 0.0), (256, 1e4)])
def test_nhd_prefill(P, rope):
    w = wl.to_nhd(wl.make_paged(f"nhdpf{P}", 111 + P, [900, 1700], Hq=32, Hk=8, D=128, P=P,
                                qo_lens=[200, 90], causal=True, rope_theta=rope))
    out, lse, s = run(w)
    assert s.info()["num_prefill_items"] > 0
    check_full(w, out, lse)


def test_nhd_fp8_decode():
    w = wl.to_nhd(wl.with_kv8(wl.config3(small=True), 121))
    dev = "cuda:0"
    from parity import plan
    s = plan(w)
    out, lse = bsr.bsr_attn_run_kv8(s, w.q.to(dev), w.k_codes.to(dev), w.v_codes.to(dev),
                                    k_scale=w.k_scale, v_scale=w.v_scale, sm_scale=w.sm_scale)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_kv8(w.q, w.k_codes, w.v_codes, w.k_scale, w.v_scale, w.indptr,
                                  w.indices, w.last_page_len, w.qo_indptr,
                                  num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads,
                                  head_dim=w.head_dim, page_size=w.page_size,
                                  sm_scale=w.sm_scale, kv_layout="NHD")
    from parity import assert_lse_close, assert_out_close
    assert_out_close(out.float().cpu().numpy(), ro, True, w.name)
    assert_lse_close(lse.cpu().numpy(), rl, w.name)


def test_nhd_append_then_chunked_prefill():
    w = wl.to_nhd(wl.config5(small=True))
    dev = "cuda:0"
    k, v = w.k_pages.to(dev), w.v_pages.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    bsr.bsr_append_kv(w.k_new.to(dev), w.v_new.to(dev), w.append_indptr.to(dev),
                      w.indptr.to(dev), w.indices.to(dev), w.last_page_len.to(dev), k, v,
                      kv_layout="NHD", device_status=status)
    kp, vp = oracle.append_kv(w.k_new, w.v_new, w.append_indptr, w.indptr, w.indices,
                              w.last_page_len, w.k_pages, w.v_pages, kv_layout="NHD",
                              num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                              page_size=w.page_size)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(k).view(np.uint16).ravel(), kp.ravel())
    assert np.array_equal(bits(v).view(np.uint16).ravel(), vp.ravel())
    out, lse, _ = run(w, (w.q.to(dev), k, v), out_dtype=torch.float32)
    check_full(w, out, lse, kp.reshape(w.k_pages.shape), vp.reshape(w.v_pages.shape))
