"""GPU parity of the decode path (plan + run through the C ABI) against the fp64 oracle,
element by element, on seeded inputs that span several tiles and ragged tails."""
import numpy as np
import pytest
import torch

import block_sparse_kv_bsr_gb300 as bsr
import oracle
import workloads as wl
from block_sparse_kv_bsr_gb300 import _build
from parity import (assert_lse_close, assert_out_close, bits, check_full, device_tensors, plan,
                    run, sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_device):
    _build.build()
    bsr.load()


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_tiny_decode(out_dtype):
    w = wl.config1()
    out, lse, _ = run(w, out_dtype=out_dtype)
    check_full(w, out, lse)


@pytest.mark.parametrize("cfg", [2, 3])
def test_small_configs(cfg):
    w = wl.by_name(cfg, small=True)
    out, lse, s = run(w)
    check_full(w, out, lse)
    out32, lse32, _ = run(w, out_dtype=torch.float32)
    check_full(w, out32, lse32)


@pytest.mark.parametrize("P", [1, 2, 4, 8, 16, 32, 64, 256])
@pytest.mark.parametrize("D", [64, 128])
def test_page_sizes(P, D):
    lens = [1, P, P + 1, 3 * P - 1, 37, 300, 777]
    w = wl.make_paged(f"p{P}d{D}", 100 + P, lens, Hq=8, Hk=2, D=D, P=P)
    out, lse, _ = run(w)
    check_full(w, out, lse)


@pytest.mark.parametrize("Hq,Hk", [(8, 8), (8, 2), (16, 2), (32, 8), (16, 1)])
def test_gqa_groups(Hq, Hk):
    w = wl.make_paged(f"g{Hq}x{Hk}", 7, [5, 64, 200, 513], Hq=Hq, Hk=Hk, D=128, P=16)
    out, lse, _ = run(w)
    check_full(w, out, lse)


@pytest.mark.parametrize("rope", [0.0, 5e5])
@pytest.mark.parametrize("causal", [False, True])
def test_multi_query_rows(rope, causal):
    # qo_len * group spans one and several 16-row groups, with ragged row tails
    w = wl.make_paged("mq", 9, [40, 130, 17, 600], Hq=16, Hk=2, D=128, P=16,
                      qo_lens=[1, 2, 3, 5], causal=causal, rope_theta=rope)
    out, lse, _ = run(w)
    check_full(w, out, lse)


def test_rope_long_positions():
    w = wl.make_paged("ropelong", 11, [5000, 1, 33, 4097], Hq=32, Hk=8, D=128, P=16,
                      rope_theta=5e5)
    out, lse, _ = run(w)
    check_full(w, out, lse)


def test_rope_d64():
    w = wl.make_paged("rope64", 12, [1, 77, 300], Hq=8, Hk=2, D=64, P=16, rope_theta=1e4,
                      qo_lens=[1, 2, 4], causal=True)
    out, lse, _ = run(w)
    check_full(w, out, lse)


def test_empty_and_edge_lengths():
    w = wl.make_paged("edges", 13, [0, 1, 16, 17, 31, 32, 0], Hq=8, Hk=2, D=128, P=16)
    out, lse, _ = run(w)
    check_full(w, out, lse)
    o = out.float().cpu().numpy()
    assert np.all(o[0] == 0) and np.all(o[6] == 0)
    assert np.all(np.isneginf(lse.cpu().numpy()[[0, 6]]))


def test_dropped_blocks_are_skipped():
    w = wl.make_paged("drop", 14, [2000, 50, 900, 16], Hq=32, Hk=8, D=128, P=16, drop=0.5)
    out, lse, _ = run(w)
    check_full(w, out, lse)


def test_long_sequence_split_and_merged():
    # one long request: the planner must cut it over many warps and merge the pieces
    w = wl.make_paged("long", 15, [60000], Hq=32, Hk=8, D=128, P=16)
    out, lse, s = run(w)
    assert s.info()["num_split_streams"] == 8
    check_full(w, out, lse)


def test_run_is_deterministic_and_replan_in_place():
    w = wl.config3(small=True)
    t = device_tensors(w)
    out1, lse1, s = run(w, t)
    out2, lse2, s2 = run(w, t, schedule=s)   # re-plan into the same schedule
    assert s2 is s
    assert torch.equal(bits_t(out1), bits_t(out2)) and torch.equal(lse1, lse2)


def bits_t(x):
    return x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32)


def test_run_time_units_match_the_oracle_and_repeat_bit_exact():
    """A skewed batch large enough that the plan leaves its short ranges to run time
    (warps take them from a queue once their own list is done): every output matches
    the oracle, and repeated runs -- each with its own assignment of the queued ranges
    to warps, the queue reset by the kernel between launches -- give the same bits."""
    lens = [20000, 23000, 17500, 26000] + [16 + (37 * i) % 280 for i in range(160)]
    w = wl.make_paged("dynq", 77, lens, Hq=32, Hk=8, D=128, P=16)
    q, k, v = device_tensors(w)
    s = plan(w)
    info = s.info()
    nwarps = info["decode_ctas"] * info["decode_warps_per_cta"]
    ip, ix, lp = [np.ascontiguousarray(np.asarray(x).astype(np.int32))
                  for x in (w.indptr, w.indices, w.last_page_len)]
    _, units = bsr.bsr_attn_plan_host(ip, ix, lp, num_qo_heads=32, num_kv_heads=8, head_dim=128,
                                      page_size=16, num_pages=w.num_pages,
                                      num_sms=info["num_sms"])
    assert (units[:, 7] >= nwarps).sum() > 500          # the queue is in use
    outs = []
    for _ in range(4):
        out, lse = bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale)
        torch.cuda.synchronize()
        outs.append((bits_t(out).clone(), lse.clone()))
    assert bsr.bsr_last_device_error(s) == 0
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    check_full(w, out, lse)


def _queued_batch(kind):
    short = [16 + (37 * i) % 280 for i in range(160)]
    if kind == "d64":
        return wl.make_paged("dynq64", 78, [40000, 46000, 35000, 52000] + short * 2,
                             Hq=16, Hk=4, D=64, P=16)
    if kind == "nhd":
        return wl.to_nhd(wl.make_paged("dynqn", 79, [20000, 23000, 17500, 26000] + short,
                                       Hq=32, Hk=8, D=128, P=16))
    if kind == "window":
        return wl.sliding_window_decode("dynqw", 80, [20000, 23000, 17500, 26000] + short + short[:40],
                                        4096, Hq=32, Hk=8, D=128, P=16)
    return wl.make_paged("dynq64p", 81, [20000, 23000, 17500, 26000] + short, Hq=32, Hk=8,
                         D=128, P=64)


@pytest.mark.parametrize("kind", ["d64", "nhd", "window", "p64"])
def test_run_time_units_in_every_kernel_variant(kind):
    """The run-time unit queue with head_dim 64, token-major pages, a sliding window and
    64-key pages: the plan queues ranges, results match the oracle and repeat bit-exact."""
    w = _queued_batch(kind)
    q, k, v = device_tensors(w)
    s = plan(w)
    info = s.info()
    nwarps = info["decode_ctas"] * info["decode_warps_per_cta"]
    _, units = bsr.bsr_attn_plan_host(w.indptr, w.indices, w.last_page_len,
                                      num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads,
                                      head_dim=w.head_dim, page_size=w.page_size,
                                      num_pages=w.num_pages, num_sms=info["num_sms"],
                                      window_left=w.window_left, kv_layout=w.kv_layout)
    assert (units[:, 7] >= nwarps).sum() > 50
    out1, lse1 = bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, causal=w.causal)
    out2, lse2 = bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, causal=w.causal)
    torch.cuda.synchronize()
    assert bsr.bsr_last_device_error(s) == 0
    assert torch.equal(bits_t(out1), bits_t(out2)) and torch.equal(lse1, lse2)
    check_full(w, out2, lse2)


def test_cuda_graph_capture_replays_identically():
    w = wl.config2(small=True)
    q, k, v = device_tensors(w)
    s = plan(w)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, rope_theta=w.rope_theta, out=out,
                         lse=lse)   # warm-up: tensor maps, function attributes
    torch.cuda.synchronize()
    ref_out, ref_lse = out.clone(), lse.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, rope_theta=w.rope_theta, out=out,
                         lse=lse, stream=stream)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(bits_t(out), bits_t(ref_out)) and torch.equal(lse, ref_lse)


@pytest.mark.parametrize("cfg", ["decode", "prefill"])
def test_run_with_host_buffers_matches_the_device_run(cfg):
    """bsr_attn_run_host (host q in, host out / lse back, one call) gives the bits of
    bsr_attn_run on the same schedule, for a decode and a prefill batch."""
    if cfg == "decode":
        w = wl.config2(small=True)
    else:
        w = wl.make_paged("hostpf", 58, [700, 333], Hq=32, Hk=8, D=128, P=16, qo_lens=[100, 64],
                          causal=True, rope_theta=1e4)
    q, k, v = device_tensors(w)
    s = plan(w)
    out, lse = bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, rope_theta=w.rope_theta,
                                causal=w.causal)
    q_host = w.q.pin_memory()
    out_h, lse_h = bsr.bsr_attn_run_host(s, q_host, k, v, sm_scale=w.sm_scale,
                                         rope_theta=w.rope_theta, causal=w.causal)
    torch.cuda.synchronize()
    assert not out_h.is_cuda and out_h.is_pinned()
    assert torch.equal(bits_t(out_h), bits_t(out.cpu())) and torch.equal(lse_h, lse.cpu())
    # fp32 output, no lse, and pageable host memory
    out_f, lse_f = bsr.bsr_attn_run_host(s, w.q.clone(), k, v, sm_scale=w.sm_scale,
                                         rope_theta=w.rope_theta, causal=w.causal,
                                         out=torch.empty(w.q.shape, dtype=torch.float32),
                                         want_lse=False)
    torch.cuda.synchronize()
    assert lse_f is None
    check_full(w, out_f, lse.cpu())


def test_mismatched_run_arguments_are_rejected():
    w = wl.config2(small=True)
    q, k, v = device_tensors(w)
    s = plan(w)
    with pytest.raises(bsr.BsrError) as e:
        bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, rope_theta=0.0)
    assert e.value.code == -7
    with pytest.raises(bsr.BsrError) as e:
        bsr.bsr_attn_run(s, q, k, v, sm_scale=-1.0, rope_theta=w.rope_theta)
    assert e.value.code == -1


# ---------------------------------------------------------------- merge_states

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
def test_merge_states(dtype, D):
    g = torch.Generator().manual_seed(5)
    rows, heads = 37, 6
    oa = torch.randn(rows, heads, D, generator=g).to(dtype)
    ob = torch.randn(rows, heads, D, generator=g).to(dtype)
    la = (torch.randn(rows, heads, generator=g) * 3).float()
    lb = (torch.randn(rows, heads, generator=g) * 3).float()
    la[0, 0] = -float("inf")            # one side empty
    la[1, :] = -float("inf")
    lb[1, :] = -float("inf")            # both sides empty
    oa[1] = float("nan")                # an empty state's o must not leak
    ob[1] = float("nan")
    ro, rl = oracle.merge_states(oa.double().numpy(), la.double().numpy(),
                                 ob.double().numpy(), lb.double().numpy())
    dev = "cuda:0"
    o, l = bsr.bsr_merge_states(oa.to(dev), la.to(dev), ob.to(dev), lb.to(dev))
    torch.cuda.synchronize()
    assert_out_close(o.float().cpu().numpy(), ro, dtype == torch.bfloat16, "merge")
    assert_lse_close(l.cpu().numpy(), rl, "merge")
    # in place into o_a / lse_a
    a, al = oa.to(dev), la.to(dev)
    bsr.bsr_merge_states(a, al, ob.to(dev), lb.to(dev), o_out=a, lse_out=al)
    torch.cuda.synchronize()
    assert torch.equal(bits_t(a), bits_t(o)) and torch.equal(al, l)


# ---------------------------------------------------------------- append_kv

@pytest.mark.parametrize("P,D", [(16, 128), (1, 64), (256, 128), (8, 128)])
def test_append_kv_is_bit_exact(P, D):
    w = wl.make_paged("app", 21, [40, 9, 300, 1], Hq=8, Hk=2, D=D, P=P, qo_lens=[5, 9, 17, 1],
                      causal=True, append=True)
    kp, vp = oracle.append_kv(w.k_new, w.v_new, w.append_indptr, w.indptr, w.indices,
                              w.last_page_len, w.k_pages, w.v_pages, num_kv_heads=2, head_dim=D,
                              page_size=P)
    dev = "cuda:0"
    k, v = w.k_pages.to(dev), w.v_pages.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    bsr.bsr_append_kv(w.k_new.to(dev), w.v_new.to(dev), w.append_indptr.to(dev),
                      w.indptr.to(dev), w.indices.to(dev), w.last_page_len.to(dev), k, v,
                      device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(k).view(np.uint16), kp)
    assert np.array_equal(bits(v).view(np.uint16), vp)


def test_append_rejects_out_of_range_page_on_device():
    w = wl.make_paged("appbad", 22, [40], Hq=8, Hk=2, D=128, P=16, qo_lens=[3], causal=True,
                      append=True)
    dev = "cuda:0"
    bad = w.indices.clone()
    bad[-1] = w.num_pages + 5
    k, v = w.k_pages.to(dev), w.v_pages.to(dev)
    before = bits(k).copy()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    bsr.bsr_append_kv(w.k_new.to(dev), w.v_new.to(dev), w.append_indptr.to(dev),
                      w.indptr.to(dev), bad.to(dev), w.last_page_len.to(dev), k, v,
                      device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert np.array_equal(bits(k), before)


def test_decode_rope_short_keys():
    """RoPE decode rows with few keys: the rotated q and k are fp16 MMA operands (11
    significant bits), so even a handful of keys keeps lse within 1e-3."""
    w = wl.make_paged("decropeshort", 82, [5, 17, 40, 300], Hq=32, Hk=8, D=128, P=16,
                      rope_theta=1e4)
    out, lse, _ = run(w)
    check_full(w, out, lse)


def test_decode_rope_operand_range_sets_status():
    """A rotated key beyond the fp16 operand range (|x| >= 2^20) on the decode path
    sets status bit 1."""
    w = wl.make_paged("decrange", 81, [300, 200], Hq=32, Hk=8, D=128, P=16, rope_theta=1e4)
    q, k, v = device_tensors(w)
    k = k.clone()
    k[int(w.indices[0]), 0, 5, :] = 3.0e6       # key 5 of request 0, kv head 0
    s = plan(w)
    assert s.info()["num_decode_items"] > 0 and s.info()["num_prefill_items"] == 0
    bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, rope_theta=w.rope_theta, causal=w.causal)
    torch.cuda.synchronize()
    assert bsr.bsr_last_device_error(s) & 2


@pytest.mark.parametrize("kv8", [False, True])
def test_repeated_launches_bit_exact(kv8):
    # Full-size skewed batch: every unit is computed exactly once per launch (outputs
    # start as NaN each time) and the split-range counters end each launch at zero,
    # so repeated launches of one schedule are bit-identical and match the oracle.
    w = wl.config3(small=False)
    if kv8:
        w = wl.with_kv8(w, 91)
    s = plan(w)
    dev = "cuda:0"
    q = w.q.to(dev)
    k, v = ((w.k_codes, w.v_codes) if kv8 else (w.k_pages, w.v_pages))
    k, v = k.to(dev), v.to(dev)
    outs = []
    for _ in range(4):
        out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=dev)
        if kv8:
            bsr.bsr_attn_run_kv8(s, q, k, v, k_scale=w.k_scale, v_scale=w.v_scale,
                                 sm_scale=w.sm_scale, causal=w.causal, out=out, lse=lse)
        else:
            bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, causal=w.causal, out=out, lse=lse)
        torch.cuda.synchronize()
        assert bsr.bsr_last_device_error(s) == 0
        assert not torch.isnan(out).any() and not torch.isnan(lse).any()
        outs.append((bits_t(out).clone(), lse.clone()))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    rows, heads = sample_rows(w, 512)
    kw = dict(num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
              page_size=w.page_size, sm_scale=w.sm_scale, causal=w.causal, rows=rows, heads=heads)
    table = (w.indptr, w.indices, w.last_page_len, w.qo_indptr)
    if kv8:
        ro, rl = oracle.attention_kv8(w.q, w.k_codes, w.v_codes, w.k_scale, w.v_scale, *table, **kw)
    else:
        ro, rl = oracle.attention(w.q, w.k_pages, w.v_pages, *table, **kw)
    o = outs[0][0].view(torch.bfloat16).float().cpu().numpy()[rows, heads]
    assert_out_close(o, ro, True, w.name)
    assert_lse_close(outs[0][1].cpu().numpy()[rows, heads], rl, w.name)


def test_longest_context_one_request():
    # one request of 262,144 keys (16,384 pages, 1 GB of K/V): every kv head's range is
    # cut over ~150 warps and merged in the kernel from that many partial states
    w = wl.make_paged("long256k", 16, [262144], Hq=32, Hk=8, D=128, P=16)
    out, lse, s = run(w)
    info = s.info()
    assert info["num_split_streams"] == 8 and info["num_partials"] >= 8 * 100
    check_full(w, out, lse)


def test_bounded_wait_gives_up_and_reports():
    # failure detection without a fault: a wait on a barrier nothing arrives on gives up
    # after its limit, sets bit 0 of the status word, and the context stays usable
    status = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    bsr.bsr_selftest_bounded_wait(status, 20_000_000)   # 20 ms
    t1.record()
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    assert t0.elapsed_time(t1) >= 19.0
    w = wl.config1()
    out, lse, s = run(w)
    check_full(w, out, lse)
