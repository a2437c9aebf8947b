"""Benchmark: skewed block-sparse BSR decode attention on one GB300 (per rank).

Workload (one "step" = one plan-free bsr_attn_run over the whole batch):
  batch 128, 32 qo / 8 kv heads, head_dim 128, page_size 16; kv_len 90%
  uniform[32, 512], 10% uniform[16384, 32768]; 25% of each request's
  non-final pages dropped (absent from indices); bf16 N(0, 1); no RoPE.
Inputs are synthetic (seeded, see workloads/) and larger than L2 (about 1 GB
of active KV against 129 MB of L2), so consecutive steps read KV from HBM.

value     = algorithmic bytes (active K+V, q, out, lse, page table) / device time per step.
e2e       = the same bytes / time of the call a user makes with HOST buffers:
            re-plan from host page-table arrays, H2D of q, run, D2H of out and lse.
roofline  = the decode kernel's algorithmic bytes / its mean CUDA-event duration,
            against the measured HBM copy bandwidth.
cpu_baseline = the fp64 oracle on this host's cores (a bounded sample of the batch).

--impl reference times the oracle (the only reference this method has here) on the
same workload.  Under torchrun each rank runs an independent replica (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "BSR decode attention achieved HBM GB/s & % of GB300 peak; µs/call (skewed)"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "bsr_decode_skewed_b128.md")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--small", action="store_true", help="small case (profiling, smoke)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons around the timed region.

    The sampler is started (and its first sample awaited) before the timed
    region; samples that arrive inside the region are summarized.  A region
    shorter than the sampling period gets the nearest sample, marked as such.
    """
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.samples = []          # (host time, sm_mhz, max_mhz, reasons)
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        threading.Thread(target=self._read, daemon=True).start()
        deadline = time.time() + 10.0
        while not self.samples and time.time() < deadline:
            time.sleep(0.01)
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = {n for n, v in zip(self.NAMES, parts[5:9]) if v.lower().startswith("active")}
            self.samples.append((time.time(), sm, mx, reasons))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()
        time.sleep(2 * self.period / 1000.0)   # let a sample that straddles the end arrive

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.samples or self.t0 is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [x for x in self.samples if self.t0 <= x[0] <= self.t1 + self.period / 1000.0]
        how = "inside timed region"
        if not inside:
            mid = 0.5 * (self.t0 + self.t1)
            inside = [min(self.samples, key=lambda x: abs(x[0] - mid))]
            how = "nearest sample (timed region shorter than the sampling period)"
        reasons = set()
        for x in inside:
            reasons |= x[3]
        return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": inside[0][2],
                "reasons": sorted(reasons), "samples": len(inside), "period_ms": self.period,
                "window": how}


def traffic_from_profile(digest: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches this build."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s*\(build\s+([0-9a-f]+)\)", text)
    if not m or m.group(2) != digest:
        return None
    return float(m.group(1))


def cpu_baseline(w, budget_s=10.0, min_passes=1):
    """Time the fp64 oracle over whole passes of the batch until `budget_s` is spent."""
    import oracle
    import workloads as wl
    threads = oracle.default_threads()
    alg = wl.algorithmic_bytes(w)
    passes, spent = 0, 0.0
    while passes < min_passes or spent < budget_s:
        t0 = time.perf_counter()
        oracle.attention(w.q, w.k_pages, w.v_pages, w.indptr, w.indices, w.last_page_len,
                         w.qo_indptr, num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads,
                         head_dim=w.head_dim, page_size=w.page_size, sm_scale=w.sm_scale,
                         rope_theta=w.rope_theta, causal=w.causal, threads=threads)
        spent += time.perf_counter() - t0
        passes += 1
    return {"value": round(alg * passes / spent / 1e9, 3), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{passes} full pass(es) of the {w.batch}-request batch "
                      f"({w.active_tokens} keys, all heads), fp64 C oracle, {spent:.1f} s"}


def main():
    args = parse()
    rank, world, local = dist_env()
    import torch
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import workloads as wl
    import block_sparse_kv_bsr_gb300 as bsr
    from block_sparse_kv_bsr_gb300 import _build
    _build.build()
    bsr.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    w = wl.config3(small=args.small)
    alg_bytes = wl.algorithmic_bytes(w)
    q = w.q.to(dev)
    k = w.k_pages.to(dev)
    v = w.v_pages.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    s = bsr.bsr_attn_plan(w.indptr, w.indices, w.last_page_len, num_qo_heads=w.num_qo_heads,
                          num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                          page_size=w.page_size, num_pages=w.num_pages, qo_indptr=w.qo_indptr)
    info = s.info()

    def step():
        bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, out=out, lse=lse)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- device-timed steps: one event pair per launch (kernel duration) + the whole region
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local).start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks.mark_start()
    t_start.record(stream)
    for a, b in evs:
        a.record(stream)
        step()
        b.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    total_ms = t_start.elapsed_time(t_end)
    kernel_ms = [a.elapsed_time(b) for a, b in evs]
    ms_step = total_ms / args.steps
    if world > 1:
        t = torch.tensor([ms_step], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms_step = float(t.item())
    assert bsr.bsr_last_device_error(s) == 0

    # ---- end to end through the public API with host buffers
    q_host = w.q.pin_memory()
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_host = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    q_dev = torch.empty_like(q)

    def e2e_step():
        bsr.bsr_attn_plan(w.indptr, w.indices, w.last_page_len, num_qo_heads=w.num_qo_heads,
                          num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                          page_size=w.page_size, num_pages=w.num_pages, qo_indptr=w.qo_indptr,
                          schedule=s)
        q_dev.copy_(q_host, non_blocking=True)
        bsr.bsr_attn_run(s, q_dev, k, v, sm_scale=w.sm_scale, out=out, lse=lse)
        out_host.copy_(out, non_blocking=True)
        lse_host.copy_(lse, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(max(1, args.warmup)):
        e2e_step()
    e2e_steps = max(3, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / e2e_steps
    info = s.info()
    h2d = q.numel() * 2 + int(info["upload_bytes"])
    d2h = out.numel() * 2 + lse.numel() * 4

    peak, peak_kind = peaks()
    kern_mean_ms = sum(kernel_ms) / len(kernel_ms)
    achieved = alg_bytes / (kern_mean_ms * 1e-3) / 1e9
    value = alg_bytes * world / (ms_step * 1e-3) / 1e9
    res = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "us_per_call": round(ms_step * 1e3, 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, page table drawn per workloads/)",
        "config": {"workload": w.name, "batch": w.batch, "num_qo_heads": w.num_qo_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "page_size": w.page_size, "active_kv_tokens": w.active_tokens,
                   "algorithmic_bytes": alg_bytes, "drop": "25% of non-final pages",
                   "l2": "inputs larger than L2 (active KV >> 129 MB), no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "peak_kind": f"{peak_kind} hbm_gbs (copy)",
                     "traffic": traffic_from_profile(_build._digest()),
                     "kernel": "bsr_decode_kernel<128,false,false,false>",
                     "kernel_us_mean": round(kern_mean_ms * 1e3, 2),
                     "kernel_us_min": round(min(kernel_ms) * 1e3, 2)},
        "e2e": {"value": round(alg_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "includes": "re-plan from host page table + H2D q + run + D2H out/lse"},
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
        "schedule": {"warps": info["decode_ctas"] * info["decode_warps_per_cta"],
                     "items": info["num_decode_items"],
                     "split_ranges": info["num_split_streams"],
                     "imbalance": round(info["decode_imbalance"], 4)},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(res))
    s.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args, rank, world):
    """The oracle as it stands, on this host's cores: one step = one pass over the batch."""
    if rank != 0:
        return
    import workloads as wl
    w = wl.config3(small=args.small)
    for _ in range(args.warmup):
        cpu_baseline(w, budget_s=0.0)
    t0 = time.perf_counter()
    r = cpu_baseline(w, budget_s=0.0, min_passes=args.steps)
    elapsed = time.perf_counter() - t0
    res = {"impl": "reference", "metric": METRIC, "value": r["value"], "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(elapsed * 1e3 / args.steps, 2), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": w.name},
           "cpu_baseline": {"value": r["value"], "unit": "GB/s", "cores": r["cores"],
                            "kind": "oracle", "sample": r["sample"]},
           "e2e": {"value": r["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


if __name__ == "__main__":
    main()
