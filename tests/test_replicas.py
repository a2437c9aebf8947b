"""The N > 1 path of bench.py is replicas only (the attention path has no exchange):
one process per GPU, a barrier, and the slowest rank's step time.  Checked here on CPU
with gloo ranks on 127.0.0.1."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    results[rank] = bench.max_over_ranks(10.0 + rank, world)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), results), nprocs=2, join=True,
                           start_method="spawn")
        assert dict(results) == {0: 11.0, 1: 11.0}


def test_max_over_ranks_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5


def test_reference_arm_under_torchrun_prints_once():
    """Two ranks (gloo, no GPU): rank 0 alone times the oracle and prints one JSON line."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--small"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["value"] > 0


def test_reference_step_samples_cover_the_batch():
    """A sampled reference step (every k-th request) is the same attention on those
    requests; the k offsets together cover the batch once."""
    import bench
    import oracle
    import workloads as wl
    w = wl.config8(small=True)          # drops and per-page positions
    kw = dict(num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
              page_size=w.page_size, sm_scale=w.sm_scale, rope_theta=w.rope_theta,
              causal=w.causal)
    full_o, full_l = oracle.attention(w.q, w.k_pages, w.v_pages, w.indptr, w.indices,
                                      w.last_page_len, w.qo_indptr, page_pos=w.page_pos, **kw)
    qo = w.qo_indptr.tolist()
    seen = []
    for off in range(3):
        reqs = list(range(off, w.batch, 3))
        s = bench.sub_batch(w, reqs)
        o, l = oracle.attention(s.q, s.k_pages, s.v_pages, s.indptr, s.indices,
                                s.last_page_len, s.qo_indptr, page_pos=s.page_pos, **kw)
        rows = [r for b in reqs for r in range(qo[b], qo[b + 1])]
        assert np.array_equal(o, full_o[rows]) and np.array_equal(l, full_l[rows])
        seen += reqs
    assert sorted(seen) == list(range(w.batch))
