"""GPU parity of a three-level cascade (system prefix shared by all requests, group
prefixes, per-request suffixes): every level through plan/run (prefix levels on the
tensor-core kernel, suffixes on the decode kernel), merged level by level with
bsr_merge_states, against the oracle over the flat layout (small) or the oracle's
own level-by-level composition (full size, sampled rows; pinned to flat on CPU)."""
import numpy as np
import pytest
import torch

import block_sparse_kv_bsr_gb300 as bsr
import oracle
import workloads as wl
from block_sparse_kv_bsr_gb300 import _build
from parity import assert_lse_close, assert_out_close, oracle_full, oracle_rows, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    _build.build()
    bsr.load()


def run_levels(c: wl.MultiCascade):
    dev = "cuda:0"
    q = c.levels[0].q.to(dev)
    o = l = None
    kinds = []
    for w in c.levels:
        ow, lw, s = run(w, (q, w.k_pages.to(dev), w.v_pages.to(dev)), out_dtype=torch.float32)
        kinds.append(s.info()["num_prefill_items"] > 0)
        o, l = (ow, lw) if o is None else bsr.bsr_merge_states(o, l, ow, lw)
    torch.cuda.synchronize()
    return o, l, kinds


def test_cascade3_small_equals_flat():
    c = wl.config9(small=True)
    o, l, kinds = run_levels(c)
    ro, rl = oracle_full(wl.flat_multi_cascade(c))
    assert_out_close(o.cpu().numpy(), ro, False, c.name)
    assert_lse_close(l.cpu().numpy(), rl, c.name)


def test_cascade3_full_size_sampled():
    c = wl.config9()
    o, l, kinds = run_levels(c)
    assert kinds == [True, True, False]      # prefixes on tensor cores, suffixes decode
    rng = np.random.default_rng(5)
    n_req = c.levels[-1].batch
    rows = rng.integers(0, n_req, 384).astype(np.int64)
    heads = rng.integers(0, c.levels[0].num_qo_heads, 384).astype(np.int32)
    ro = rl = None
    for w in c.levels:
        ow, lw = oracle_rows(w, rows, heads)
        ro, rl = (ow, lw) if ro is None else oracle.merge_states(ro, rl, ow, lw)
    assert_out_close(o.cpu().numpy()[rows, heads], ro, False, c.name)
    assert_lse_close(l.cpu().numpy()[rows, heads], rl, c.name)
