"""Benchmark: skewed block-sparse BSR decode attention on one GB300 (per rank).

Workload (one "step" = one plan-free bsr_attn_run over the whole batch):
  batch 128, 32 qo / 8 kv heads, head_dim 128, page_size 16; kv_len 90%
  uniform[32, 512], 10% uniform[16384, 32768]; 25% of each request's
  non-final pages dropped (absent from indices); bf16 N(0, 1); no RoPE.
Inputs are synthetic (seeded, see workloads/) and larger than L2 (about 1 GB
of active KV against 129 MB of L2), so consecutive steps read KV from HBM.

value     = algorithmic bytes (active K+V, q, out, lse, page table) / device time per step
            (K steps, CUDA events at the ends of the region only).
hot, cold = the same steps timed one by one: back to back, and after a write of twice the
            L2 before each step (outside its events), so that every step starts cold.
graph     = (single-call decode workloads) K steps captured in one CUDA graph and replayed:
            the device time per step without the host's per-call launch cost.
e2e       = the same bytes / time of the call a user makes with HOST buffers: per step the
            plan of the page table (on the host, overlapping the previous step's kernel as
            a serving loop would), H2D of q and the plan, run, D2H of out and lse, and the
            host's wait for them; the serialised form is reported beside it.
roofline  = the dominant kernel's algorithmic bytes (or FLOPs) / its mean launch duration,
            against the measured HBM copy bandwidth (or bf16 dense peak).  A step of one
            kernel launch is timed as K back-to-back steps with CUDA events at their ends
            only; steps of several kernels by the library's stage events around each
            kernel (which also give p10 / median / p90 per call for every workload).  The
            DRAM traffic comes from the committed ncu summary of the same build.
cpu_baseline = the fp64 oracle on this host's cores over whole passes for ~10 s (decode
            workloads; configs 1 and 2 add a one-thread figure).
clocks    = SM clock and clock-event reasons polled through NVML every ~0.5 ms during the
            first timed region (nvidia-smi samples where NVML does not load).
configs   = after the headline, the other workloads (--configs), each with hot and cold
            timings, its kernels, its roofline and (decode) its e2e figure.

--config selects the headline workload (2: Llama-3-8B-shaped decode with RoPE,
4: shared-prefix cascade, 5: chunked prefill with append, reported in TFLOP/s, 6: the
skewed decode over an FP8 (E4M3) KV cache, 7: sliding-window decode over long histories,
8: the skewed decode with RoPE at the kept blocks' logical positions, 9: a three-level
cascade of shared prefixes, 10: the skewed decode over token-major (NHD) pages, 11: the
Llama-3-8B-shaped decode with RoPE over an FP8 cache);
the default is the skewed decode above.  --impl reference times the oracle (the only
reference this method has here) on the same workload, each step one pass over the batch
or, when K passes would take more than ~90 s, over every k-th request.  Under torchrun each
rank runs an independent replica (weak scaling).
"""
from __future__ import annotations

import argparse
import gc
import itertools
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
PROFILES = os.path.join(ROOT, "profiles")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--small", action="store_true", help="small case (profiling, smoke)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11],
                    help="workload; 3 (skewed block-sparse decode) is the headline")
    ap.add_argument("--configs", default="1,2,4,5,6,7,8,9,10,11",
                    help="further workloads measured after the headline (comma list; '' for none)")
    ap.add_argument("--time-budget", type=float, default=240.0,
                    help="seconds after which further workloads are skipped (and listed as such)")
    args = ap.parse_args()
    args.configs = [int(x) for x in args.configs.split(",") if x.strip()]
    return args


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (the slowest replica sets the job's time)."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


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


class NvmlClocks:
    """SM clock and clock-event reasons polled through NVML (the driver's own library,
    loaded with ctypes) in a background thread every ~0.5 ms, so that even a timed region
    of a few milliseconds holds several samples.  Same interface as ClockSampler; the
    device is matched to the CUDA device by UUID, then by PCI bus id."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int, period_s: float = 0.0005):
        import ctypes
        import torch
        self.period = period_s
        self.samples = []
        self.t0 = self.t1 = None
        self._stop = False
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(cuda_index)
        ok = False
        try:
            ok = lib.nvmlDeviceGetHandleByUUID(f"GPU-{props.uuid}".encode(), ctypes.byref(self.h)) == 0
        except Exception:
            ok = False
        if not ok:
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) == 0
        if not ok:
            raise RuntimeError("no NVML handle for the CUDA device")
        try:
            self._reasons_fn = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self._reasons_fn = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = (float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0
                        else None)

    def _sample(self):
        import ctypes
        sm = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(sm)) != 0:
            return
        reasons = set()
        if self._reasons_fn(self.h, ctypes.byref(rs)) == 0:
            reasons = {n for bit, n in self.REASONS.items() if rs.value & bit}
        self.samples.append((time.time(), float(sm.value), self.max_mhz, reasons))

    def _loop(self):
        while not self._stop:
            self._sample()
            time.sleep(self.period)

    def start(self):
        self._sample()
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        self._stop = True
        self.thread.join(timeout=1.0)

    def summary(self):
        inside = [x for x in self.samples if self.t0 is not None and self.t0 <= x[0] <= self.t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml"}
        reasons = set()
        for x in inside:
            reasons |= x[3]
        return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(x[1] for x in inside), "reasons": sorted(reasons),
                "samples": len(inside), "period_ms": self.period * 1e3,
                "window": "inside timed region", "source": "nvml"}


def clock_sampler(local: int):
    """NVML polling when the driver library loads, else nvidia-smi samples."""
    try:
        return NvmlClocks(local).start()
    except Exception:
        return ClockSampler(local).start()


def traffic_from_profile(name: str, digest: str):
    """DRAM bytes per launch from a committed ncu summary under profiles/, if it was
    captured on the kernel built from the current sources (digest of those sources)."""
    try:
        text = open(os.path.join(PROFILES, name)).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s*\(build\s+([0-9a-f]+)\)", text)
    if not m or m.group(2) != digest:
        return None
    return float(m.group(1))


def cpu_baseline(w, budget_s=10.0, min_passes=1, threads=None):
    """Time the fp64 oracle over whole passes of the batch until `budget_s` is spent
    (all host cores unless `threads` is given)."""
    import oracle
    import workloads as wl
    threads = oracle.default_threads() if threads is None else threads
    alg = wl.algorithmic_bytes(w)
    passes, spent = 0, 0.0
    while passes < min_passes or spent < budget_s:
        t0 = time.perf_counter()
        table = (w.indptr, w.indices, w.last_page_len, w.qo_indptr)
        kw = dict(num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                  page_size=w.page_size, sm_scale=w.sm_scale, rope_theta=w.rope_theta,
                  causal=w.causal, window_left=w.window_left, page_pos=w.page_pos,
                  kv_layout=w.kv_layout, threads=threads)
        if w.k_codes is not None:
            oracle.attention_kv8(w.q, w.k_codes, w.v_codes, w.k_scale, w.v_scale, *table, **kw)
        else:
            oracle.attention(w.q, w.k_pages, w.v_pages, *table, **kw)
        spent += time.perf_counter() - t0
        passes += 1
    return {"value": round(alg * passes / spent / 1e9, 3), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{passes} full pass(es) of the {w.batch}-request batch "
                      f"({w.active_tokens} keys, all heads), fp64 C oracle, {spent:.1f} s"}


class Part:
    """One library call of a step, timed with its own CUDA events.

    For bsr_attn_run calls `sched`/`stage` name the schedule and the stage whose
    kernel the roofline is about (timed by the library's stage events); `family`
    and `profile` select the committed ncu summary holding its DRAM traffic.
    """

    def __init__(self, label, fn, kernel, bound, work, work_unit, launches=1, sched=None,
                 stage=None, family=None, profile=None):
        self.label, self.fn, self.kernel, self.bound = label, fn, kernel, bound
        self.work, self.work_unit = work, work_unit      # algorithmic bytes or FLOPs per call
        self.launches, self.sched, self.stage = launches, sched, stage
        self.family, self.profile = family, profile
        self.ms = []          # whole call
        self.kernel_ms = []   # the stage's kernel alone
        self.stage_ms = {}    # every kernel the call launched, by stage


def attention_flops(w) -> int:
    """4*D FLOPs (QK^T and PV) per attended (query, qo head, key) pair."""
    total = 0
    for b in range(w.batch):
        n = int(w.qo_indptr[b + 1] - w.qo_indptr[b])
        L = w.kv_len[b]
        keys = sum(min(L, L - n + i + 1) for i in range(n)) if w.causal else n * L
        total += keys
    return total * w.num_qo_heads * 4 * w.head_dim


def cascade_prefix_sms(num_sms: int, prefix_flops: float, suffix_bytes: float,
                       prefix_levels: int = 1) -> int:
    """SMs for a cascade's tensor-core prefix level when it runs beside the HBM-bound
    suffix level on the other SMs: the split that evens out the two levels' times, from
    rates measured on GB300 with the levels side by side (the prefill kernel ~5.2 TFLOP/s
    per SM plus ~12 us per prefix level for merging its split ranges; the decode kernel
    streams ~58 GB/s per SM, ~6.3 TB/s at most over the whole GPU)."""
    best = (float("inf"), num_sms // 2)
    for s1 in range(8, num_sms - 7):
        t = max(prefix_flops / (s1 * 5.2e12) + 12e-6 * prefix_levels,
                suffix_bytes / min((num_sms - s1) * 58e9, 6.3e12))
        if t < best[0]:
            best = (t, s1)
    return best[1]


def build_job(cfg: int, dev, small: bool):
    """Device tensors, schedules and the per-step calls of one workload."""
    import torch
    import block_sparse_kv_bsr_gb300 as bsr
    import workloads as wl

    def plan(w, schedule=None, stream=None):
        return bsr.bsr_attn_plan(w.indptr, w.indices, w.last_page_len,
                                 num_qo_heads=w.num_qo_heads, num_kv_heads=w.num_kv_heads,
                                 head_dim=w.head_dim, page_size=w.page_size,
                                 num_pages=w.num_pages, qo_indptr=w.qo_indptr, causal=w.causal,
                                 rope_theta=w.rope_theta, window_left=w.window_left,
                                 page_pos=w.page_pos, kv_layout=w.kv_layout,
                                 kv_dtype="e4m3" if w.k_codes is not None else "bf16",
                                 schedule=schedule, stream=stream)

    job = {"parts": [], "schedules": []}
    if cfg in (1, 2, 3, 7, 8, 10):
        w = wl.by_name(cfg, small)
        q, k, v = w.q.to(dev), w.k_pages.to(dev), w.v_pages.to(dev)
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        s = plan(w)
        run = lambda: bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, rope_theta=w.rope_theta,
                                       causal=w.causal, out=out, lse=lse)
        alg = wl.algorithmic_bytes(w)
        kname = f"bsr_decode_kernel<{w.head_dim},{int(w.rope_theta > 0)},0,0>"
        prof = {2: "bsr_decode_rope_llama8b_b64.md", 3: "bsr_decode_skewed_b128.md",
                7: "bsr_decode_window_b64_w2048.md",
                8: "bsr_decode_rope_positions_b128.md",
                10: "bsr_decode_skewed_b128_nhd.md"}.get(cfg)
        job["parts"] = [Part("decode", run, kname, "hbm", alg, "B",
                             launches=s.info()["kernels_per_run"], sched=s, stage="decode",
                             family="decode", profile=None if small else prof)]
        job["schedules"] = [s]
        job["graphable"] = True
        job.update(workload=w, metric=METRIC, unit="GB/s", numerator=alg, scale=1e9,
                   config={"workload": w.name, "batch": w.batch, "num_qo_heads": w.num_qo_heads,
                           "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                           "page_size": w.page_size, "active_kv_tokens": w.active_tokens,
                           "algorithmic_bytes": alg, "rope_theta": w.rope_theta,
                           "l2": "inputs larger than L2, no flush" if alg > 2e8 else
                                 "inputs smaller than L2: L2-warm"})
        if cfg in (3, 8, 10):
            job["config"]["drop"] = "25% of non-final pages"
        if cfg == 10:
            job["config"]["kv_layout"] = "NHD (token-major pages)"
        if cfg == 8:
            job["config"]["rope_positions"] = "logical (per-page positions of the kept blocks)"
        if cfg == 7:
            job["config"]["window_left"] = w.window_left
            job["config"]["kv_tokens_held"] = int(sum(w.kv_len))
        q_host = w.q.pin_memory()
        out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_host = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

        def e2e_step(sched):
            # host q in, host out / lse back: one library call queues the copies and the run
            bsr.bsr_attn_run_host(sched, q_host, k, v, sm_scale=w.sm_scale,
                                  rope_theta=w.rope_theta, causal=w.causal, out=out_host,
                                  lse=lse_host)

        job["e2e"] = (lambda: plan(w, s), lambda: e2e_step(s))
        job["e2e_bytes"] = lambda: (q.numel() * 2 + int(s.info()["upload_bytes"]),
                                    out.numel() * 2 + lse.numel() * 4)
    elif cfg in (6, 11):
        w = wl.config6(small) if cfg == 6 else wl.config11(small)
        q = w.q.to(dev)
        k, v = w.k_codes.to(dev), w.v_codes.to(dev)
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        s = plan(w)
        run = lambda: bsr.bsr_attn_run_kv8(s, q, k, v, k_scale=w.k_scale, v_scale=w.v_scale,
                                           sm_scale=w.sm_scale, rope_theta=w.rope_theta,
                                           causal=w.causal, out=out, lse=lse)
        alg = wl.algorithmic_bytes(w)
        job["parts"] = [Part("decode", run, "bsr_decode_kv8_kernel", "hbm", alg, "B",
                             launches=s.info()["kernels_per_run"], sched=s, stage="decode",
                             family="decode_kv8",
                             profile=None if small else
                             "bsr_decode_kv8_skewed_b128.md" if cfg == 6 else
                             "bsr_decode_kv8_rope_llama8b_b64.md")]
        job["schedules"] = [s]
        job["graphable"] = True
        job["dtype"] = "f16 MMA on E4M3 codes, fp32 accumulate"
        job.update(workload=w, metric=METRIC, unit="GB/s", numerator=alg, scale=1e9,
                   config={"workload": w.name, "batch": w.batch, "num_qo_heads": w.num_qo_heads,
                           "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                           "page_size": w.page_size, "active_kv_tokens": w.active_tokens,
                           "kv_cache": "E4M3 codes + per-pool scales (q, out bf16)",
                           "algorithmic_bytes": alg, "rope_theta": w.rope_theta,
                           "drop": "25% of non-final pages" if cfg == 6 else "none",
                           "l2": "inputs larger than L2, no flush"})
        q_host = w.q.pin_memory()
        out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_host = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

        def e2e_step(sched):
            bsr.bsr_attn_run_host(sched, q_host, k, v, k_scale=w.k_scale, v_scale=w.v_scale,
                                  sm_scale=w.sm_scale, rope_theta=w.rope_theta, causal=w.causal,
                                  out=out_host, lse=lse_host)

        job["e2e"] = (lambda: plan(w, s), lambda: e2e_step(s))
        job["e2e_bytes"] = lambda: (q.numel() * 2 + int(s.info()["upload_bytes"]),
                                    out.numel() * 2 + lse.numel() * 4)
    elif cfg == 4:
        c = wl.config4(small)
        pre, suf = c.prefix, c.suffix
        q = suf.q.to(dev)
        pk, pv = pre.k_pages.to(dev), pre.v_pages.to(dev)
        sk, sv = suf.k_pages.to(dev), suf.v_pages.to(dev)
        o_p = torch.empty(q.shape, dtype=torch.float32, device=dev)
        o_s = torch.empty_like(o_p)
        l_p = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        l_s = torch.empty_like(l_p)
        o = torch.empty_like(o_p)
        l = torch.empty_like(l_p)
        kv_p = pre.active_tokens * 2 * pre.num_kv_heads * pre.head_dim * 2
        kv_s = suf.active_tokens * 2 * suf.num_kv_heads * suf.head_dim * 2
        qo = q.numel() * 2
        st = o.numel() * 4 + l.numel() * 4                  # one fp32 state
        # the two levels side by side: the prefix level (tensor cores) on its own stream
        # and share of the SMs, the suffix level (HBM) on the rest; the merge waits for both
        n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
        s_pre = cascade_prefix_sms(n_sms, attention_flops(pre), kv_s + qo + st)
        sp = plan(pre, bsr.bsr_schedule_create(s_pre))
        ss = plan(suf, bsr.bsr_schedule_create(n_sms - s_pre))
        side = torch.cuda.Stream(dev)
        fork, join = torch.cuda.Event(), torch.cuda.Event()

        def prefix_level():
            main = torch.cuda.current_stream()
            fork.record(main)
            side.wait_event(fork)
            bsr.bsr_attn_run(sp, q, pk, pv, sm_scale=pre.sm_scale, out=o_p, lse=l_p, stream=side)
            join.record(side)

        def merge_levels():
            torch.cuda.current_stream().wait_event(join)
            bsr.bsr_merge_states(o_p, l_p, o_s, l_s, o_out=o, lse_out=l)

        job["parts"] = [
            Part("prefix", prefix_level,
                 "bsr_prefill_kernel<0>", "tensor", attention_flops(pre), "FLOP",
                 launches=sp.info()["kernels_per_run"], sched=sp, stage="prefill",
                 family="prefill", profile=None if small else "bsr_prefill_cascade_prefix8192.md"),
            Part("suffix", lambda: bsr.bsr_attn_run(ss, q, sk, sv, sm_scale=suf.sm_scale,
                                                    out=o_s, lse=l_s),
                 "bsr_decode_kernel<128,0,0,0>", "hbm", kv_s + qo + st, "B",
                 launches=ss.info()["kernels_per_run"], sched=ss, stage="decode",
                 family="decode", profile=None if small else "bsr_decode_cascade_suffix.md"),
            Part("merge", merge_levels, "merge_states_kernel<128,1>", "hbm", 3 * st, "B"),
        ]
        job["schedules"] = [sp, ss]
        alg = kv_p + kv_s + qo + st
        job.update(workload=suf, metric="BSR shared-prefix cascade decode: achieved GB/s; us/call",
                   unit="GB/s", numerator=alg, scale=1e9,
                   config={"workload": c.name, "requests": suf.batch,
                           "prefix_tokens": pre.kv_len[0], "prefix_page_size": pre.page_size,
                           "suffix_tokens": suf.active_tokens, "algorithmic_bytes": alg,
                           "levels": "prefix (tensor cores) beside suffix (decode), then LSE merge",
                           "sm_split": {"prefix": s_pre, "suffix": n_sms - s_pre}})
    elif cfg == 9:
        c = wl.config9(small)
        q = c.levels[0].q.to(dev)
        st = q.shape[0] * q.shape[1] * (q.shape[2] + 1) * 4          # one fp32 state
        n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
        # levels on the tensor-core kernel run one after the other on a second stream and
        # an SM share, beside the decode level on the other SMs (as for the cascade above)
        is_pre = [plan(w).info()["num_prefill_items"] > 0 for w in c.levels]
        kvb = [w.active_tokens * 2 * w.num_kv_heads * w.head_dim * 2 for w in c.levels]
        s_pre = cascade_prefix_sms(
            n_sms, sum(attention_flops(w) for w, pr in zip(c.levels, is_pre) if pr),
            sum(kv + q.numel() * 2 + st for kv, pr in zip(kvb, is_pre) if not pr),
            prefix_levels=sum(is_pre))
        side = torch.cuda.Stream(dev)
        fork, join = torch.cuda.Event(), torch.cuda.Event()
        parts, scheds, outs, alg = [], [], [], 0
        for i, w in enumerate(c.levels):
            k, v = w.k_pages.to(dev), w.v_pages.to(dev)
            o_i = torch.empty(q.shape, dtype=torch.float32, device=dev)
            l_i = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
            pre = is_pre[i]
            s = plan(w, bsr.bsr_schedule_create(s_pre if pre else n_sms - s_pre))
            first_pre = pre and not any(is_pre[:i])

            def fn(s=s, k=k, v=v, w=w, o_i=o_i, l_i=l_i, pre=pre, first_pre=first_pre):
                if pre and first_pre:
                    fork.record(torch.cuda.current_stream())
                    side.wait_event(fork)
                bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale, out=o_i, lse=l_i,
                                 stream=side if pre else None)

            parts.append(Part(f"level{i + 1}", fn,
                              "bsr_prefill_kernel<0>" if pre else "bsr_decode_kernel<128,0,0,0>",
                              "tensor" if pre else "hbm",
                              attention_flops(w) if pre else kvb[i] + q.numel() * 2 + st,
                              "FLOP" if pre else "B", launches=s.info()["kernels_per_run"],
                              sched=s, stage="prefill" if pre else "decode",
                              family="prefill" if pre else "decode",
                              profile=None if small or pre else "bsr_decode_cascade3_suffix.md"))
            scheds.append(s)
            outs.append((o_i, l_i))
            alg += kvb[i]
        acc_o = torch.empty(q.shape, dtype=torch.float32, device=dev)
        acc_l = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        # the two shared levels merge on the second stream; the result joins the last level
        pair_stream = side if is_pre[0] and is_pre[1] else None

        def merge12():
            bsr.bsr_merge_states(outs[0][0], outs[0][1], outs[1][0], outs[1][1], o_out=acc_o,
                                 lse_out=acc_l, stream=pair_stream)
            if pair_stream is not None:
                join.record(side)

        def merge123():
            if pair_stream is not None:
                torch.cuda.current_stream().wait_event(join)
            bsr.bsr_merge_states(acc_o, acc_l, outs[2][0], outs[2][1], o_out=acc_o,
                                 lse_out=acc_l)

        parts.append(Part("merge12", merge12, "merge_states_kernel<128,1>", "hbm", 3 * st, "B"))
        parts.append(Part("merge123", merge123, "merge_states_kernel<128,1>", "hbm", 3 * st, "B"))
        job["parts"] = parts
        job["schedules"] = scheds
        alg += q.numel() * 2 + st
        job.update(workload=c.levels[-1], metric="BSR multi-level cascade decode: achieved GB/s; us/call",
                   unit="GB/s", numerator=alg, scale=1e9,
                   config={"workload": c.name, "requests": c.levels[-1].batch,
                           "levels": [{"segments": w.batch, "tokens": w.active_tokens,
                                       "page_size": w.page_size} for w in c.levels],
                           "algorithmic_bytes": alg,
                           "composition": "system prefix + group prefixes (tensor cores, one "
                                          "after the other on a second stream) beside the "
                                          "suffixes (decode), LSE-merged level by level",
                           "sm_split": {"prefix_levels": s_pre, "decode_level": n_sms - s_pre}})
    elif cfg == 5:
        w = wl.config5(small)
        q, k, v = w.q.to(dev), w.k_pages.to(dev), w.v_pages.to(dev)
        kn, vn = w.k_new.to(dev), w.v_new.to(dev)
        tab = [t.to(dev) for t in (w.append_indptr, w.indptr, w.indices, w.last_page_len)]
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        s = plan(w)
        flops = attention_flops(w)
        app_bytes = 2 * 2 * kn.numel() * 2
        job["parts"] = [
            Part("append", lambda: bsr.bsr_append_kv(kn, vn, *tab, k, v), "append_kv_kernel",
                 "hbm", app_bytes, "B"),
            Part("prefill", lambda: bsr.bsr_attn_run(s, q, k, v, sm_scale=w.sm_scale,
                                                     rope_theta=w.rope_theta, causal=True,
                                                     out=out, lse=lse),
                 "bsr_prefill_kernel<1>", "tensor", flops, "FLOP",
                 launches=s.info()["kernels_per_run"], sched=s, stage="prefill",
                 family="prefill", profile=None if small else "bsr_prefill_chunked_b16_q512.md"),
        ]
        job["schedules"] = [s]
        job.update(workload=w, metric="BSR chunked-prefill attention (causal, RoPE): TFLOP/s",
                   unit="TFLOP/s", numerator=flops, scale=1e12,
                   config={"workload": w.name, "batch": w.batch, "qo_len": 512,
                           "kv_tokens_after_append": w.active_tokens,
                           "algorithmic_flops": flops, "rope_theta": w.rope_theta})
    return job


def region_steps(step, steps, stream):
    """Device time per step (ms) of `steps` back-to-back steps, CUDA events at the ends."""
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def timed_steps(step, steps, stream, flush=None):
    """Device time (ms) of each of `steps` steps, CUDA events around each on `stream`.
    With `flush` (an int32 tensor over twice the L2), every step is preceded, outside
    its events, by a write of the whole buffer, so the step starts with a cold L2."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i, (a, b) in enumerate(evs):
        if flush is not None:
            flush.fill_(i + 1)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def graph_steps(step, steps):
    """Device time per step (ms) of `steps` steps captured in one CUDA graph: the
    launches are queued without the host's per-call cost, as a serving loop that
    replays a captured step issues them.  One replay warms up; one more is timed with
    CUDA events around it on the replaying stream."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for _ in range(steps):
            step()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(side):
        g.replay()
        a.record(side)
        g.replay()
        b.record(side)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    del g
    return ms


def graph_result(job, step, steps):
    ms = graph_steps(step, steps)
    return {"us_per_step": round(ms * 1e3, 2),
            "value": round(job["numerator"] / (ms * 1e-3) / job["scale"], 1),
            "note": f"{steps} steps captured in one CUDA graph, replayed (no host launch cost)"}


def kernel_pass(parts, steps, stream, bsr):
    """K more steps with CUDA events around each library call and the library's own
    stage events around each kernel of a bsr_attn_run call (records that sit between
    kernels, which is why the whole-job region has none)."""
    import torch
    for pt in parts:
        pt.ms, pt.kernel_ms, pt.stage_ms = [], [], {}
        if pt.sched is not None:
            bsr.bsr_schedule_set_stage_timing(pt.sched, steps)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in parts] for _ in range(steps)]
    for row in evs:
        for pt, (a, b) in zip(parts, row):
            a.record(stream)
            pt.fn()
            b.record(stream)
    torch.cuda.synchronize()
    for row in evs:
        for pt, (a, b) in zip(parts, row):
            pt.ms.append(a.elapsed_time(b))
    for pt in parts:
        if pt.sched is not None:
            for call in range(steps):
                t = bsr.bsr_schedule_stage_times(pt.sched, call)
                if pt.stage in t:
                    pt.kernel_ms.append(t[pt.stage])
                for name, ms in t.items():
                    pt.stage_ms.setdefault(name, []).append(ms)
            bsr.bsr_schedule_set_stage_timing(pt.sched, 0)


def spread(ms):
    """mean / median / p10 / p90 of a list of milliseconds, in microseconds."""
    dec = statistics.quantiles(ms, n=10, method="inclusive") if len(ms) > 1 else [ms[0]] * 9
    return {"us_mean": round(sum(ms) / len(ms) * 1e3, 2),
            "us_median": round(statistics.median(ms) * 1e3, 2),
            "us_p10": round(dec[0] * 1e3, 2), "us_p90": round(dec[-1] * 1e3, 2)}


def roofline_of(parts, _build, whole_ms=None, whole_by=None):
    """Roofline of the call that takes the most time in a step (among the attention
    kernels' calls): its algorithmic bytes or FLOPs over its kernel's mean duration.
    When a step is one call launching one kernel, `whole_ms` -- the per-step time of K
    back-to-back steps timed with events only at their ends (or replayed from a CUDA
    graph) -- is that kernel's mean launch duration, without the event records the
    per-kernel pass inserts between launches (a few us each); the per-kernel figures are
    reported beside it."""
    peak_hbm, hbm_kind = peaks()
    peak_tensor, tensor_kind = tensor_peak()
    dom = max([pt for pt in parts if pt.family is not None] or parts, key=lambda pt: sum(pt.ms))
    call_ms = sum(dom.ms) / len(dom.ms)
    kms = dom.kernel_ms if dom.kernel_ms else dom.ms
    dom_ms = sum(kms) / len(kms)
    one_kernel = whole_ms is not None and len(parts) == 1 and dom.launches == 1
    if one_kernel:
        dom_ms = whole_ms
    sources = {"decode": _build.DECODE_KERNEL_SOURCES,
               "decode_kv8": _build.DECODE_KV8_KERNEL_SOURCES,
               "prefill": _build.PREFILL_KERNEL_SOURCES}.get(dom.family)
    build_digest = _build.kernel_digest(sources) if sources else None
    traffic = traffic_from_profile(dom.profile, build_digest) if dom.profile is not None else None
    if dom.bound == "hbm":
        achieved, peak, unit = dom.work / (dom_ms * 1e-3) / 1e9, peak_hbm, "GB/s"
        kind = f"{hbm_kind} hbm_gbs (copy)"
    else:
        achieved, peak, unit = dom.work / (dom_ms * 1e-3) / 1e12, peak_tensor, "TFLOP/s"
        kind = f"{tensor_kind} bf16 dense (cuBLAS GEMM)"
    sp = spread(kms)
    return {"bound": dom.bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
            "frac": round(achieved / peak, 4), "peak_kind": kind, "traffic": traffic,
            "traffic_source": f"profiles/{dom.profile}" if traffic is not None else None,
            "kernel": dom.kernel, "kernel_build": build_digest,
            "kernel_us_mean": sp["us_mean"], "kernel_us_min": round(min(kms) * 1e3, 2),
            "kernel_us_p10": sp["us_p10"], "kernel_us_median": sp["us_median"],
            "kernel_us_p90": sp["us_p90"],
            "kernel_us_launch": round(dom_ms * 1e3, 2),
            "timed_by": whole_by if one_kernel else
                        ("library stage events around the kernel" if dom.kernel_ms
                         else "CUDA events around the call") + ", a separate timed pass of K steps",
            "kernel_us_by": "library stage events around each kernel, a separate pass of K steps",
            "call_us_mean": round(call_ms * 1e3, 2)}


def l2_flush_buffer(dev):
    """An int32 buffer over twice the L2 (written before each cold step)."""
    import torch
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (129 << 20)
    return torch.empty(2 * l2 // 4 + 1024, dtype=torch.int32, device=dev), l2


def e2e_run(job, steps, warmup, stream):
    """The same metric through the public API with host buffers, every step: H2D of q
    from pinned memory, bsr_attn_run, D2H of out and lse, and a host wait for them.
    Pipelined as a serving loop would run it: the page table of step i + 1 depends only
    on the lengths, so it is planned on the host while the GPU runs step i (its image
    upload queued behind step i's read-back, which is all the host waits for); q of step
    i + 1 is uploaded after the result of step i has been read back.  The serialised
    form (plan, then copy, run, read) is timed too."""
    plan, launch = job["e2e"]
    for _ in range(max(1, warmup)):
        plan()
        launch()
        stream.synchronize()
    gc.collect()
    n = max(3, min(5 * steps, 100))
    done = None
    plan()
    t0 = time.perf_counter()
    for _ in range(n):
        launch()
        done = stream.record_event(done)   # this step's out / lse are on the host then
        plan()                   # the next step's table, while the GPU runs this one
        done.synchronize()       # (the next table's upload, queued behind, need not be waited for)
    stream.synchronize()
    piped_ms = (time.perf_counter() - t0) * 1e3 / n
    serial = []
    for _ in range(n):
        t = time.perf_counter()
        plan()
        launch()
        stream.synchronize()
        serial.append((time.perf_counter() - t) * 1e3)
    h2d, d2h = job["e2e_bytes"]()
    return {"value": round(job["numerator"] / (piped_ms * 1e-3) / job["scale"], 1),
            "unit": job["unit"], "ms_per_step": round(piped_ms, 4), "steps": n,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "includes": "per step: bsr_attn_plan of the page table (overlapping the previous "
                        "step's kernel; its image goes up with one H2D copy), then "
                        "bsr_attn_run_host with host q / out / lse (H2D of q, run, D2H of out "
                        "and lse), host wait for the read-back",
            "serial": {"value": round(job["numerator"] / (statistics.mean(serial) * 1e-3) / job["scale"], 1),
                       "ms_per_step": round(statistics.mean(serial), 4),
                       "ms_per_step_median": round(statistics.median(serial), 4),
                       "includes": "plan, then H2D q + run + D2H out/lse, host wait"}}


def measure_config(cfg, dev, args, stream, flush, bsr, _build):
    """Hot and cold-L2 timings, per-kernel times and the roofline of one more workload."""
    import torch
    job = build_job(cfg, dev, False)
    parts = job["parts"]

    def step():
        for pt in parts:
            pt.fn()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    region_ms = region_steps(step, args.steps, stream)
    hot = timed_steps(step, args.steps, stream)
    cold = timed_steps(step, args.steps, stream, flush)
    kernel_pass(parts, args.steps, stream, bsr)
    for s in job["schedules"]:
        assert bsr.bsr_last_device_error(s) == 0
    unit, num, scale = job["unit"], job["numerator"], job["scale"]
    res = {"workload": job["config"]["workload"], "metric": job["metric"], "unit": unit,
           "hot": dict(spread(hot), value=round(num / (statistics.median(hot) * 1e-3) / scale, 1)),
           "cold": dict(spread(cold), value=round(num / (statistics.median(cold) * 1e-3) / scale, 1)),
           "region": {"us_per_step": round(region_ms * 1e3, 2),
                      "value": round(num / (region_ms * 1e-3) / scale, 1),
                      "note": "K back-to-back steps, CUDA events at their ends only"},
           "roofline": roofline_of(parts, _build, whole_ms=region_ms,
                                   whole_by="K back-to-back steps of one kernel launch each, "
                                            "CUDA events at their ends only"),
           "kernels_us": {f"{pt.label}.{name}": round(sum(v) / len(v) * 1e3, 2)
                          for pt in parts for name, v in pt.stage_ms.items()},
           "config": job["config"]}
    if job.get("graphable"):
        res["graph"] = graph_result(job, step, args.steps)
    if "e2e" in job:
        res["e2e"] = e2e_run(job, args.steps, args.warmup, stream)
    if cfg in (1, 2) and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(job["workload"], budget_s=2.0)
        one = cpu_baseline(job["workload"], budget_s=2.0, threads=1)
        res["cpu_baseline"]["single_thread"] = {"value": one["value"], "unit": one["unit"],
                                                "sample": one["sample"]}
    del job, parts
    gc.collect()
    torch.cuda.empty_cache()
    return res


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

    import block_sparse_kv_bsr_gb300 as bsr
    from block_sparse_kv_bsr_gb300 import _build
    _build.build()
    bsr.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    t_begin = time.time()

    job = build_job(args.config, dev, args.small)
    parts = job["parts"]
    stream = torch.cuda.current_stream()

    def step():
        for pt in parts:
            pt.fn()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- region 1: K steps with events only at its ends (whole-job time, clocks)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = clock_sampler(local)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks.mark_start()
    t_start.record(stream)
    for _ in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.mark_end()
    clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    total_ms = t_start.elapsed_time(t_end)

    # ---- region 2: per call and per kernel (library stage events)
    kernel_pass(parts, args.steps, stream, bsr)
    ms_step = max_over_ranks(total_ms / args.steps, world, dev)
    for s in job["schedules"]:
        assert bsr.bsr_last_device_error(s) == 0

    # ---- the same steps one by one, hot and after an L2 flush
    flush, l2_bytes = l2_flush_buffer(dev)
    hot = timed_steps(step, args.steps, stream)
    cold = timed_steps(step, args.steps, stream, flush)

    graph = graph_result(job, step, args.steps) if job.get("graphable") else None

    # ---- end to end through the public API with host buffers
    e2e = e2e_run(job, args.steps, args.warmup, stream) if "e2e" in job else None

    value = job["numerator"] * world / (ms_step * 1e-3) / job["scale"]
    unit, num, scale = job["unit"], job["numerator"], job["scale"]
    res = {
        "metric": job["metric"],
        "value": round(value, 1),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "us_per_call": round(ms_step * 1e3, 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": job.get("dtype", "bf16"),
        "data": "synthetic (seeded N(0,1) bf16, page table drawn per workloads/)",
        "config": dict(job["config"], parallelism=f"replicas x{world}" if world > 1 else "1 GPU"),
        "roofline": roofline_of(parts, _build, whole_ms=ms_step,
                                whole_by="region 1: CUDA events at the ends of K back-to-back "
                                         "steps of one kernel launch each"),
        "hot": dict(spread(hot), value=round(num / (statistics.median(hot) * 1e-3) / scale, 1)),
        "cold": dict(spread(cold), value=round(num / (statistics.median(cold) * 1e-3) / scale, 1),
                     flush=f"write of {2 * l2_bytes >> 20} MiB (2x L2) before each step, "
                           "outside its events"),
        "parts_us": {pt.label: round(sum(pt.ms) / len(pt.ms) * 1e3, 2) for pt in parts},
        "kernels_us": {f"{pt.label}.{name}": round(sum(v) / len(v) * 1e3, 2)
                       for pt in parts for name, v in pt.stage_ms.items()},
        "gpu_launches": args.steps * sum(pt.launches for pt in parts),
        "gpu_launches_note": "kernels launched in the whole-job timed region (region 1)",
        "clocks": clocks.summary(),
    }
    if graph is not None:
        res["graph"] = graph
    if e2e is not None:
        res["e2e"] = e2e
    info = job["schedules"][-1].info()
    res["schedule"] = {"decode_warps": info["decode_ctas"] * info["decode_warps_per_cta"],
                       "decode_items": info["num_decode_items"],
                       "prefill_ctas": info["prefill_ctas"],
                       "prefill_items": info["num_prefill_items"],
                       "split_ranges": info["num_split_streams"],
                       "imbalance": round(max(info["decode_imbalance"], info["prefill_imbalance"]), 4)}
    # the oracle on the host cores, for the decode workloads (a pass takes well under a
    # second there); on the tiny and the Llama-8B-shaped ones also on one thread
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.config in (1, 2, 3, 6, 7, 8, 10, 11):
        res["cpu_baseline"] = cpu_baseline(job["workload"])
        if args.config in (1, 2):
            one = cpu_baseline(job["workload"], budget_s=3.0, threads=1)
            res["cpu_baseline"]["single_thread"] = {"value": one["value"], "unit": one["unit"],
                                                    "sample": one["sample"]}
    del job, parts
    gc.collect()
    torch.cuda.empty_cache()

    # ---- the other workloads (the five headline configurations first, then the extended
    # ones), each hot and cold, on rank 0 of a single-GPU run
    if world == 1 and args.configs:
        res["configs"] = {}
        for cfg in args.configs:
            if cfg == args.config:
                continue
            if time.time() - t_begin > args.time_budget:
                res["configs"][str(cfg)] = {"skipped": f"bench time budget of {args.time_budget} s spent"}
                continue
            res["configs"][str(cfg)] = measure_config(cfg, dev, args, stream, flush, bsr, _build)
    res["bench_wall_s"] = round(time.time() - t_begin, 1)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


def sub_batch(w, reqs):
    """The same pools with only requests `reqs` (page-table slicing, no attention math)."""
    import dataclasses
    import torch
    ip, qo = w.indptr.tolist(), w.qo_indptr.tolist()
    pages = [torch.arange(ip[b], ip[b + 1]) for b in reqs]
    rows = [torch.arange(qo[b], qo[b + 1]) for b in reqs]
    sel_p = torch.cat(pages) if pages else torch.zeros(0, dtype=torch.int64)
    sel_q = torch.cat(rows) if rows else torch.zeros(0, dtype=torch.int64)
    def cum(lens):
        return torch.tensor([0] + list(itertools.accumulate(lens)), dtype=torch.int32)

    return dataclasses.replace(
        w, indptr=cum([ip[b + 1] - ip[b] for b in reqs]), indices=w.indices[sel_p].contiguous(),
        last_page_len=w.last_page_len[list(reqs)].contiguous(),
        qo_indptr=cum([qo[b + 1] - qo[b] for b in reqs]), q=w.q[sel_q].contiguous(),
        kv_len=[w.kv_len[b] for b in reqs],
        page_pos=None if w.page_pos is None else w.page_pos[sel_p].contiguous())


def run_reference(args, rank, world):
    """The oracle as it stands, on this host's cores.  One step is one pass over the
    batch, or, when K such passes would take more than ~90 s, over every k-th request
    (a bounded sample; the offset turns with the step, so all requests take part)."""
    if rank != 0:
        return
    import workloads as wl
    w = wl.by_name(args.config if args.config in (1, 2, 3, 6, 7, 8, 10, 11) else 3, args.small)
    t_pass = 0.0
    for _ in range(max(args.warmup, 1)):
        t = time.perf_counter()
        cpu_baseline(w, budget_s=0.0)
        t_pass = time.perf_counter() - t
    stride = max(1, math.ceil(args.steps * t_pass / 90.0))
    stride = min(stride, w.batch)
    steps = [sub_batch(w, list(range(i % stride, w.batch, stride))) if stride > 1 else w
             for i in range(min(args.steps, stride))]
    t0 = time.perf_counter()
    work, cores = 0, None
    for i in range(args.steps):
        r = cpu_baseline(steps[i % len(steps)], budget_s=0.0)
        work += wl.algorithmic_bytes(steps[i % len(steps)])
        cores = r["cores"]
    elapsed = time.perf_counter() - t0
    value = round(work / elapsed / 1e9, 3)
    sample = (f"{args.steps} step(s), each a full pass of the {w.batch}-request batch"
              if stride == 1 else
              f"{args.steps} step(s), each every {stride}-th request of the {w.batch}-request "
              f"batch (offset turning per step)") + f", fp64 C oracle, {elapsed:.1f} s"
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(elapsed * 1e3 / args.steps, 2), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": w.name},
           "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


if __name__ == "__main__":
    main()
