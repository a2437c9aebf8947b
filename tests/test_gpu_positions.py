"""GPU parity of RoPE at per-page logical positions (caches whose inactive blocks were
dropped keep their tokens' positions) against the fp64 oracle: the decode kernel
(the stage's cos/sin row follows its page's position, queries follow the last logical
key), the RoPE rotation inside the tensor-core prefill kernel, and identity positions."""
import pytest
import torch

import block_sparse_kv_bsr_gb300 as bsr
import workloads as wl
from block_sparse_kv_bsr_gb300 import _build
from parity import check_full, check_sampled, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    _build.build()
    bsr.load()


def test_positions_decode_small():
    w = wl.config8(small=True)
    assert w.page_pos is not None
    out, lse, _ = run(w)
    check_full(w, out, lse)


def test_positions_decode_full_size_sampled():
    w = wl.config8()
    out, lse, _ = run(w)
    check_sampled(w, out, lse, n=1536)


@pytest.mark.parametrize("P", [16, 64])
def test_positions_decode_multi_query_and_groups(P):
    w = wl.make_paged(f"posq{P}", 91 + P, [40, 700, 1500, 3000], Hq=32, Hk=2, D=128, P=P,
                      qo_lens=[1, 3, 2, 5], causal=True, drop=0.3, rope_theta=1e4)
    out, lse, _ = run(w, out_dtype=torch.float32)
    check_full(w, out, lse)


def test_positions_prefill():
    w = wl.make_paged("pospf", 92, [2000, 900], Hq=32, Hk=8, D=128, P=16, qo_lens=[300, 100],
                      causal=True, drop=0.3, rope_theta=5e5)
    out, lse, s = run(w)
    assert s.info()["num_prefill_items"] > 0
    check_full(w, out, lse)


def test_identity_positions_change_nothing():
    w = wl.config2(small=True)
    out0, lse0, _ = run(w)
    w.page_pos = torch.cat([torch.arange(int(w.indptr[b + 1] - w.indptr[b])) * w.page_size
                            for b in range(w.batch)]).to(torch.int32)
    out1, lse1, _ = run(w)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)
