"""Benchmark of the paged-attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  prefill 8x16K (default): the 65 ubatches of 8 x 16384-token prompts, each
      ubatch = per-token expansion -> reshape-and-cache -> plan -> prefill
      (tcgen05) + decode (split-KV + reduce) for one Qwen3-8B-shaped layer
      (32/8 heads, d 128, page 128).  value = causal attention TFLOP/s.
  decode (reported beside it): 8 sequences, KV length U[1024, 4096], one query
      token each; expansion + plan once, then 36 layers of append + decode over
      36 distinct pools (4 GB > L2).  value = algorithmic KV GB/s.

Prints ONE JSON line (rank 0).  --impl reference times the CPU fp64 oracle on
the same workload (bounded sample per step).  Under torchrun every rank runs its
own replica (weak scaling; no data-path collective); timings are max-reduced.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s + prefill TFLOP/s, Qwen3-8B-shape paged attn, 8×16K, 1 GB300"

# DRAM bytes (read + write) per launch from ncu captures of the same workloads, with a
# digest of the kernel's sources at capture time: a kernel changed since then reports
# traffic null.  k_prefill / k_prefill_fp8: one launch of `profile_case prefill
# --ubatch 48` / `prefill_fp8 --ubatch 48`, scaled to the 8x16K step's mean work per
# launch (16,258 of ubatch 48's 16,640 key-block units); k_decode: one decode_8seq
# launch (`profile_case decode`); k_decode_longtail: `profile_case longtail`;
# k_decode_span: one masked launch of `profile_case span`; k_decode_fp8 /
# k_decode_fp8_longtail: one FP8 launch of `profile_case fp8` / `fp8_longtail`; k_copy_pages: one launch of `profile_case copy` (writes still
# in L2 at the end of the launch are not counted).  Summaries and commands: profiles/.
TRAFFIC = {
    "k_prefill": {"bytes": 397.60e6, "files": ["k_prefill.cu"], "digest": "d64645999e60d5cd"},
    "k_prefill_fp8": {"bytes": 216.40e6, "files": ["k_prefill.cu"], "digest": "d64645999e60d5cd"},
    "k_decode": {"bytes": 86.21e6, "files": ["k_decode.cu"], "digest": "7c09222e8332d9bc"},
    "k_decode_longtail": {"bytes": 1081.85e6, "files": ["k_decode.cu"], "digest": "7c09222e8332d9bc"},
    "k_decode_span": {"bytes": 116.18e6, "files": ["k_decode.cu"], "digest": "7c09222e8332d9bc"},
    "k_decode_fp8": {"bytes": 43.68e6, "files": ["k_decode.cu"], "digest": "7c09222e8332d9bc"},
    "k_decode_fp8_longtail": {"bytes": 559.86e6, "files": ["k_decode.cu"], "digest": "7c09222e8332d9bc"},
    "k_copy_pages": {"bytes": 488.15e6, "files": ["k_small.cu"], "digest": "8ffc91b37d609dbd"},
}
_TRAFFIC_HEADERS = ["common.cuh", "tc.cuh", "tmap.cuh", "kernels.cuh"]


def traffic_of(kernel: str):
    """Recorded DRAM bytes per launch of `kernel`, or None if its sources changed."""
    import hashlib
    rec = TRAFFIC.get(kernel)
    if rec is None:
        return None
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "paged_kv_cache_pages_gb300",
                        "csrc")
    h = hashlib.sha256()
    for f in rec["files"] + _TRAFFIC_HEADERS:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return rec["bytes"] if h.hexdigest()[:16] == rec["digest"] else None
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DECODE_LAYERS = 36


# ----------------------------------------------------------------------------- helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        mhz = sorted(r[0] for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3])
                          if v.lower() == "active"})
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(rows),
                "reasons": reasons}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(units_per_rank: float, seconds_max: float, world: int) -> float:
    """Whole-job throughput: units all ranks processed / max-over-ranks time."""
    return units_per_rank * world / seconds_max


def measure_f16_peak(torch, dev, gpu_index, n=8192, sustain_s=4.0):
    """Dense f16 tensor peak on this GPU, measured like the bf16 entries of the peak
    file: torch.matmul of two n x n f16 matrices (2 n^3 FLOP), best of 10 launches
    timed by CUDA events (burst), and launches back to back for sustain_s seconds
    (sustained, under the power cap), with the SM clocks sampled during each."""
    a = torch.randn(n, n, dtype=torch.float16, device=dev)
    b = torch.randn(n, n, dtype=torch.float16, device=dev)
    c = torch.empty(n, n, dtype=torch.float16, device=dev)
    flop = 2.0 * n ** 3
    for _ in range(5):
        torch.matmul(a, b, out=c)
    torch.cuda.synchronize()
    best = float("inf")
    with ClockSampler(gpu_index) as clk_b:
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) / 1e3)
    with ClockSampler(gpu_index) as clk_s:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        count = 0
        t_end = time.perf_counter() + sustain_s
        e0.record()
        while time.perf_counter() < t_end:
            for _ in range(16):
                torch.matmul(a, b, out=c)
            count += 16
            torch.cuda.synchronize()
        e1.record()
        torch.cuda.synchronize()
        sus = e0.elapsed_time(e1) / 1e3
    del a, b, c
    return {"burst": round(flop / best / 1e12, 1), "sustained": round(flop * count / sus / 1e12, 1),
            "burst_clocks": clk_b.summary(), "sustained_clocks": clk_s.summary(),
            "how": f"torch.matmul f16 {n}^3: best of 10 (burst); back to back for "
                   f"{sustain_s:.0f} s (sustained)"}


def clock_matched_peak(clocks, burst, sustained):
    """The peak that a kernel timed under `clocks` can earn: the burst figure when its
    median SM clock sat at the maximum (a power-cap sample with the clock still at the
    maximum does not lower it), else the sustained one."""
    mhz, top = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    at_max = bool(mhz and top and mhz >= 0.97 * top)
    if at_max:
        return burst, "burst (kernel's median SM clock at the maximum)"
    return sustained, "sustained (kernel's median SM clock below the maximum)"


# ----------------------------------------------------------------------------- prefill leg

class PrefillBench:
    def __init__(self, pa, torch, dev, seed=0):
        import workloads
        self.pa, self.torch, self.dev = pa, torch, dev
        self.wl = wl = workloads.Prefill8x16K(seed)
        t = torch
        self.spt = t.from_numpy(wl.seq_page_table).to(dev)
        self.kp = t.full((wl.num_pages, wl.Hkv, wl.P, wl.d), float("nan"), dtype=t.float16,
                         device=dev)
        self.vp = t.full_like(self.kp, float("nan"))
        self.ub = []
        self.host = []
        for u in range(len(wl.ubatches)):
            ts, tp, q, k, v = wl.ubatch(u)
            h = dict(tok_seq=t.from_numpy(ts).pin_memory(), tok_pos=t.from_numpy(tp).pin_memory(),
                     q=t.from_numpy(q.view(np.float16)).pin_memory(),
                     k=t.from_numpy(np.ascontiguousarray(k).view(np.float16)).pin_memory(),
                     v=t.from_numpy(np.ascontiguousarray(v).view(np.float16)).pin_memory())
            self.host.append(h)
            d = {k_: x.to(dev) for k_, x in h.items()}
            T = ts.shape[0]
            d["T"] = T
            d["out"] = t.empty((T, wl.Hq, wl.d), dtype=t.float16, device=dev)
            d["tpt"] = t.empty((T, wl.max_pages), dtype=t.int32, device=dev)
            d["kv"] = t.empty(T, dtype=t.int32, device=dev)
            d["slot"] = t.empty(T, dtype=t.int64, device=dev)
            d["flops"] = 4.0 * wl.d * wl.Hq * float((tp.astype(np.int64) + 1).sum())
            self.ub.append(d)
        self.host_out = [t.empty((d["T"], wl.Hq, wl.d), dtype=t.float16).pin_memory()
                         for d in self.ub]
        Tmax = max(d["T"] for d in self.ub)
        self.ws = pa.new_workspace(Tmax, wl.Hq, wl.Hkv, wl.d, dev)
        self.flops = sum(d["flops"] for d in self.ub)
        self.launches_per_step = 6 * len(self.ub)   # expand, append, plan x2, prefill, decode

    def _ubatch(self, d, ev=None):
        pa, wl = self.pa, self.wl
        pa.expand_ubatch(self.spt, d["tok_seq"], d["tok_pos"], wl.P, out=(d["tpt"], d["kv"], d["slot"]))
        pa.kv_append(d["k"], d["v"], d["slot"], self.kp, self.vp)
        pa.plan(d["tpt"], d["kv"], wl.Hq, wl.Hkv, wl.P, wl.d, self.ws)
        if ev is not None:
            ev[0].record()
        pa.prefill(d["q"], self.kp, self.vp, d["tpt"], d["kv"], wl.scale, d["out"], self.ws)
        if ev is not None:
            ev[1].record()
        pa.decode(d["q"], self.kp, self.vp, d["tpt"], d["kv"], wl.scale, d["out"], self.ws)

    def step(self, events=None):
        for i, d in enumerate(self.ub):
            self._ubatch(d, None if events is None else events[i])

    def step_e2e(self):
        """Same step from pinned host buffers: H2D of each ubatch's inputs, D2H of its
        output.  The uploads run on one copy stream and the downloads on another, so the
        copies of other ubatches overlap the attention of this one; ubatch i's kernels
        wait (event) for its own upload, and its download waits for its kernels.  Every
        ubatch has its own device buffers, and the step ends when the last download has
        landed (the compute stream waits for the download stream)."""
        t = self.torch
        cur = t.cuda.current_stream()
        if not hasattr(self, "_e2e_streams"):
            self._e2e_streams = (t.cuda.Stream(), t.cuda.Stream())
            n = len(self.ub)
            self._e2e_in = [t.cuda.Event() for _ in range(n)]
            self._e2e_done = [t.cuda.Event() for _ in range(n)]
        up, down = self._e2e_streams
        h2d = d2h = 0
        up.wait_stream(cur)
        with t.cuda.stream(up):
            for d, h, ev in zip(self.ub, self.host, self._e2e_in):
                for k_ in ("tok_seq", "tok_pos", "q", "k", "v"):
                    d[k_].copy_(h[k_], non_blocking=True)
                    h2d += h[k_].numel() * h[k_].element_size()
                ev.record(up)
        down.wait_stream(cur)
        for d, ev_in, ev_done in zip(self.ub, self._e2e_in, self._e2e_done):
            cur.wait_event(ev_in)
            self._ubatch(d)
            ev_done.record(cur)
        with t.cuda.stream(down):
            for d, ho, ev in zip(self.ub, self.host_out, self._e2e_done):
                down.wait_event(ev)
                ho.copy_(d["out"], non_blocking=True)
                d2h += ho.numel() * ho.element_size()
        cur.wait_stream(down)
        return h2d, d2h


# ----------------------------------------------------------------------------- decode leg

class DecodeBench:
    def __init__(self, pa, torch, dev, seed=0, layers=DECODE_LAYERS, case=None):
        import workloads
        self.pa, self.torch = pa, torch
        self.case = c = workloads.decode(seed) if case is None else case
        t = torch
        self.spt = t.from_numpy(c.seq_page_table()).to(dev)
        self.tok_seq = t.from_numpy(c.tok_seq).to(dev)
        self.tok_pos = t.from_numpy(c.tok_pos).to(dev)
        kp = t.from_numpy(c.k_pool.view(np.float16)).to(dev)
        vp = t.from_numpy(c.v_pool.view(np.float16)).to(dev)
        self.pools = [(kp.clone(), vp.clone()) for _ in range(layers)]
        self.q = [t.from_numpy(c.q.view(np.float16)).to(dev) for _ in range(layers)]
        self.kn = t.from_numpy(c.k_new.view(np.float16)).to(dev)
        self.vn = t.from_numpy(c.v_new.view(np.float16)).to(dev)
        self.out = [t.empty_like(self.q[0]) for _ in range(layers)]
        self.ws = pa.new_workspace(c.T, c.Hq, c.Hkv, c.d, dev)
        self.tpt = t.empty((c.T, c.max_pages), dtype=t.int32, device=dev)
        self.kv = t.empty(c.T, dtype=t.int32, device=dev)
        self.slot = t.empty(c.T, dtype=t.int64, device=dev)
        self.bytes_per_layer = float(c.seq_len.astype(np.int64).sum()) * c.Hkv * c.d * 2 * 2
        self.layers = layers
        self.launches_per_step = 3 + layers   # expand, plan x2; per layer one fused launch

    def step(self, events=None):
        """One decode step: expansion and plan once, then per layer one launch that
        appends the layer's new K/V rows and runs the split-KV decode."""
        pa, c = self.pa, self.case
        pa.expand_ubatch(self.spt, self.tok_seq, self.tok_pos, c.P, out=(self.tpt, self.kv, self.slot))
        pa.plan(self.tpt, self.kv, c.Hq, c.Hkv, c.P, c.d, self.ws)
        for l in range(self.layers):
            kp, vp = self.pools[l]
            if events is not None:
                events[l][0].record()
            pa.decode_append(self.q[l], self.kn, self.vn, self.slot, kp, vp, self.tpt, self.kv,
                             c.scale, self.out[l], self.ws)
            if events is not None:
                events[l][1].record()

    def attention_only(self):
        """The step's decode launches back to back (the same pools, queries and plan as
        the last step): times the attention kernel without the appends between."""
        pa, c = self.pa, self.case
        for l in range(self.layers):
            kp, vp = self.pools[l]
            pa.decode(self.q[l], kp, vp, self.tpt, self.kv, c.scale, self.out[l], self.ws)


# ----------------------------------------------------------------------------- timing

SPIN_CYCLES = 4_000_000   # about 2 ms at the maximum SM clock


def time_steps(torch, fn, steps, warmup, world, per_launch=None):
    """Warm up, then time exactly `steps` calls of fn between barrier+sync pairs.
    per_launch: number of (start, end) event pairs to record per step (kernel timing).
    In that mode each step is queued behind a short device-side spin, so the host has
    queued the whole step before the GPU reaches it and the event pairs time the
    kernels, not the host's launch rate."""
    for _ in range(warmup):
        fn(None) if per_launch else fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev_pairs = []
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        if per_launch:
            pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(per_launch)]
            ev_pairs.append(pairs)
            torch.cuda._sleep(SPIN_CYCLES)
            fn(pairs)
        else:
            fn()
    stop.record()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    total_ms = start.elapsed_time(stop)
    kern_ms = None
    if per_launch:
        kern_ms = sum(a.elapsed_time(b) for pairs in ev_pairs for (a, b) in pairs)
    return total_ms, kern_ms


def time_launches(torch, fn, n_pairs, steps, warmup, world):
    """Average device time of the launches that fn brackets with its (start, end)
    event pairs.  Preferred: the step is captured as a CUDA graph with the event
    records as graph nodes, so the pairs time each kernel inside the same graph
    replay as the timed step (no host launch gaps).  If this PyTorch cannot put
    event records in a graph, the pairs are timed in an eager pass instead.
    Returns (total ms over all pairs of all steps, how it was timed)."""
    try:
        pairs = [(torch.cuda.Event(enable_timing=True, external=True),
                  torch.cuda.Event(enable_timing=True, external=True)) for _ in range(n_pairs)]
        graph = capture_step(torch, lambda: fn(pairs))
    except (TypeError, RuntimeError):
        _, ms = time_steps(torch, fn, steps, warmup, world, per_launch=n_pairs)
        return ms, "eager pass, event pairs around each launch"
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    total = 0.0
    for _ in range(steps):
        graph.replay()
        torch.cuda.synchronize()
        total += sum(a.elapsed_time(b) for a, b in pairs)
    barrier(world)
    return total, "event-record nodes around each launch inside a CUDA graph of the step"


def capture_step(torch, fn):
    """One step captured as a CUDA graph (the same launches, replayed without
    host launch overhead)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def cpu_baseline_prefill(wl, budget_s=12.0, keep=False):
    """The oracle as it stands on host cores: sampled tokens of the middle
    ubatches of the 8x16K prefill, growing the sample until ~budget_s of work.
    keep=True also returns the oracle's outputs [(ubatch, tokens, out)], which the
    benchmark compares with the GPU outputs of the same ubatches."""
    import oracle
    kp, vp = wl.pool_final()
    mids = list(range(len(wl.ubatches) // 2, len(wl.ubatches)))
    flops = 0.0
    secs = 0.0
    n_tok = 0
    stride = 64
    i = 0
    kept = []
    while secs < budget_s and i < len(mids):
        u = mids[i]
        ts, tp, q, _, _ = wl.ubatch(u)
        tpt, kv, _ = oracle.expand_ubatch(wl.seq_page_table, ts, tp, wl.P)
        sel = np.arange(0, ts.shape[0], stride, dtype=np.int32)
        t0 = time.perf_counter()
        ref = oracle.paged_attention(q, kp, vp, tpt, kv, wl.scale, tokens=sel)
        secs += time.perf_counter() - t0
        if keep:
            kept.append((u, sel, ref))
        flops += 4.0 * wl.d * wl.Hq * float(kv[sel].astype(np.int64).sum())
        n_tok += len(sel)
        i += 1
    res = {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
           "kind": "oracle",
           "sample": f"{n_tok} tokens (every {stride}th) of {i} late ubatches of the 8x16K "
                     f"prefill, all 32 heads, fp64; {secs:.1f} s of CPU work"}
    return (res, kept) if keep else res


ATOL, RTOL = 2e-3, 1e-2   # |gpu - oracle| <= ATOL + RTOL |oracle|, elementwise


def parity_check(kept, gpu_rows):
    """Element-wise comparison of GPU outputs with the oracle's on the sampled
    tokens.  gpu_rows(u, tokens) -> float array [n][Hq][d].  Returns a record; the
    benchmark refuses to print a number whose check failed."""
    n_tok = n_bad = 0
    max_abs = 0.0
    finite = True
    for u, sel, ref in kept:
        got = np.asarray(gpu_rows(u, sel), np.float64)
        finite &= bool(np.all(np.isfinite(got)))
        err = np.abs(got - ref)
        n_bad += int((err > ATOL + RTOL * np.abs(ref)).sum())
        max_abs = max(max_abs, float(np.nanmax(err)) if err.size else 0.0)
        n_tok += len(sel)
    return {"tokens": n_tok, "ubatches": len(kept), "max_abs": max_abs,
            "out_of_tolerance": n_bad, "finite": finite,
            "ok": bool(finite and n_bad == 0 and n_tok > 0),
            "tolerance": f"|gpu - oracle| <= {ATOL} + {RTOL} |oracle| elementwise"}


def cpu_baseline_decode(case, reps_budget_s=3.0):
    """The oracle as it stands on host cores, on the whole decode layer (all 8 tokens,
    all heads): KV bytes the layer reads per second of oracle time."""
    import oracle
    tpt, kv, slot = oracle.expand_ubatch(case.seq_page_table(), case.tok_seq, case.tok_pos, case.P)
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    oracle.kv_append(case.k_new, case.v_new, slot, kp, vp)
    nbytes = float(kv.astype(np.int64).sum()) * case.Hkv * case.d * 2 * 2
    secs, reps = 0.0, 0
    while secs < reps_budget_s:
        t0 = time.perf_counter()
        oracle.paged_attention(case.q, kp, vp, tpt, kv, case.scale)
        secs += time.perf_counter() - t0
        reps += 1
    return {"value": round(nbytes * reps / secs / 1e9, 3), "unit": "GB/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"the whole decode layer (8 tokens, 32 heads, fp64), {reps} runs in "
                      f"{secs:.1f} s"}


# ----------------------------------------------------------------------------- arms

def bench_copy_pages(pa, torch, dev, steps, warmup, world, hbm, with_cpu, seed=0):
    """Page copy of copy-on-write forks: 512 random pages of a decode-shaped pool
    (8 KV heads x 128 rows x d 128, K and V: 512 KB a page) copied to 512 other
    pages per launch (256 MB read + 256 MB written, more than L2).  GB/s counts
    bytes read + written, like the HBM copy peak."""
    import workloads
    N, Hkv, P, d, n = 1280, 8, 128, 128, 512
    rng = np.random.default_rng(seed + 7000)
    ids = rng.permutation(N).astype(np.int32)
    src_h, dst_h = ids[:n].copy(), ids[n:2 * n].copy()
    kp = torch.empty((N, Hkv, P, d), dtype=torch.float16, device=dev).normal_()
    vp = torch.empty_like(kp).normal_()
    src, dst = torch.from_numpy(src_h).to(dev), torch.from_numpy(dst_h).to(dev)
    g = capture_step(torch, lambda: pa.copy_pages(src, dst, kp, vp))
    total_ms, _ = time_steps(torch, g.replay, steps, warmup, world)
    t = max_over_ranks(total_ms / 1e3 / steps, world)
    nbytes = 2.0 * 2 * n * Hkv * P * d * 2  # K and V, read and written
    gbs = aggregate(nbytes, t, world) / 1e9
    res = {"workload": "fork_copy_512_pages", "value": round(gbs, 1), "unit": "GB/s",
           "bytes_per_launch": nbytes,
           "roofline": {"bound": "hbm", "kernel": "k_copy_pages", "achieved": round(gbs / world, 1),
                        "peak": hbm, "unit": "GB/s", "frac": round(gbs / world / hbm, 4),
                        "traffic": traffic_of("k_copy_pages")}}
    if with_cpu:
        import oracle
        k_h = workloads.randn_f16(rng, (N, Hkv, P, d))
        v_h = workloads.randn_f16(rng, (N, Hkv, P, d))
        oracle.copy_pages(src_h, dst_h, k_h, v_h)
        reps, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < 1.0:
            oracle.copy_pages(src_h, dst_h, k_h, v_h)
            reps += 1
        secs = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": round(nbytes * reps / secs / 1e9, 2), "unit": "GB/s",
                               "cores": 1, "kind": "oracle",
                               "sample": f"the same 512 page pairs, {reps} copies in {secs:.1f} s"}
    return res


def span_roofline(logical_gbs, ms_layer, hbm):
    """The masked span kernel reads each token's whole span (the logical bytes), but
    the 8 tokens re-read one pool that fits in L2: DRAM sees about one pool per launch
    and L2 serves the rest.  So the HBM roofline is taken on the DRAM bytes (the ncu
    record), and the logical rate is reported beside it."""
    traffic = traffic_of("k_decode_span")
    dram = traffic / (ms_layer / 1e3) / 1e9 if traffic else None
    return {"bound": "l2 (DRAM sees one pool per launch)", "kernel": "k_decode (masked)",
            "achieved": round(dram, 1) if dram else None, "peak": hbm, "unit": "GB/s",
            "frac": round(dram / hbm, 4) if dram else None, "traffic": traffic,
            "logical_gbs": round(logical_gbs, 1),
            "note": "achieved = DRAM bytes per launch (ncu) / time; logical_gbs counts the span "
                    "bytes every token reads, most of them served by L2"}


def bench_unified_span(pa, torch, db, steps, warmup, world, hbm, paged_ms_per_layer):
    """The unified-span baseline on the decode workload: the same 36 layers, each
    pool seen as one span shared by the 8 sequences (every token streams the whole
    pool, free cells included, under a per-cell mask), against the paged decode."""
    import workloads
    c = db.case
    tpt, kv, cs, cp, ts, tp = workloads.span_view(c)
    dev = db.q[0].device
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    tpt, kv, cs, cp, ts, tp = t(tpt), t(kv), t(cs), t(cp), t(ts), t(tp)
    ws = pa.new_workspace(c.T, c.Hq, c.Hkv, c.d, dev)
    out = torch.empty_like(db.q[0])

    def step():
        pa.plan_decode(tpt, kv, c.Hq, c.Hkv, c.P, c.d, ws)
        for l in range(db.layers):
            kp, vp = db.pools[l]
            pa.masked_decode(db.q[l], kp, vp, tpt, kv, c.scale, cs, cp, ts, tp, out, ws)

    g = capture_step(torch, step)
    total_ms, _ = time_steps(torch, g.replay, steps, warmup, world)
    ms_layer = max_over_ranks(total_ms / steps / db.layers, world)
    span_bytes = float(c.T) * c.num_pages * c.Hkv * c.P * c.d * 2 * 2  # K+V of the span, per token
    if pa.read_error(ws):
        raise RuntimeError("device error word set in the unified-span baseline")
    gbs = span_bytes / (ms_layer / 1e3) / 1e9
    return {"workload": "decode_8seq_unified_span", "unit": "GB/s", "value": round(gbs * world, 1),
            "ms_per_layer": round(ms_layer, 4), "bytes_per_layer": span_bytes,
            "paged_ms_per_layer": round(paged_ms_per_layer, 4),
            "paged_speedup": round(ms_layer / paged_ms_per_layer, 2),
            "bytes_ratio": round(span_bytes / db.bytes_per_layer, 2),
            "roofline": span_roofline(gbs, ms_layer, hbm),
            "timing": "CUDA graph of one plan and 36 masked decode launches (one per layer)"}


def bench_unified_span_prefill(pa, torch, pb, steps, warmup, world, paged_ms_per_step):
    """The unified-span baseline of the headline prefill: every ubatch of the 8x16K step
    attends over the span of the whole pool (every token's row names all 1280 pages,
    kv_len = the span) under the per-cell (sequence, position) mask, on the same tcgen05
    tiles; against the paged step.  Runs on the pool after the timed paged steps (every
    owned cell written); the cell map is the final one (positions past a token's own
    are masked as in the paged kernel)."""
    wl, dev = pb.wl, pb.kp.device
    N, P = wl.num_pages, wl.P
    cs = np.full(N * P, -1, np.int32)
    cp = np.full(N * P, -1, np.int32)
    for s_ in range(wl.n_seq):
        pos = np.arange(wl.seq_len)
        slots = wl.seq_page_table[s_][pos // P].astype(np.int64) * P + pos % P
        cs[slots], cp[slots] = s_, pos
    Tmax = max(d["T"] for d in pb.ub)
    tpt = torch.arange(N, dtype=torch.int32, device=dev).repeat(Tmax, 1).contiguous()
    kv = torch.full((Tmax,), N * P, dtype=torch.int32, device=dev)
    cs_d, cp_d = torch.from_numpy(cs).to(dev), torch.from_numpy(cp).to(dev)
    ws = pa.new_workspace(Tmax, wl.Hq, wl.Hkv, wl.d, dev)
    out = torch.empty((Tmax, wl.Hq, wl.d), dtype=torch.float16, device=dev)

    def step():
        for d in pb.ub:
            T = d["T"]
            pa.plan_prefill(tpt[:T], kv[:T], wl.Hq, wl.Hkv, P, wl.d, ws)
            pa.masked_prefill(d["q"], pb.kp, pb.vp, tpt[:T], kv[:T], wl.scale, cs_d, cp_d,
                              d["tok_seq"], d["tok_pos"], out[:T], ws)

    g = capture_step(torch, step)
    n_steps = max(1, min(steps, 3))
    total_ms, _ = time_steps(torch, g.replay, n_steps, min(warmup, 1), world)
    ms = max_over_ranks(total_ms / n_steps, world)
    if pa.read_error(ws):
        raise RuntimeError("device error word set in the unified-span prefill")
    # the last ubatch of the span step against the paged output of the same ubatch
    last = pb.ub[-1]
    diff = (out[:last["T"]].float() - last["out"].float()).abs()
    tol = 2e-3 + 1e-2 * last["out"].float().abs()
    agree = bool((diff <= 2 * tol).all())
    # K/V bytes each kernel streams and the MMA work it does: a tile item reads every key
    # block up to its longest kv_len (paged) or the whole span (unified)
    G = wl.Hq // wl.Hkv
    items_per_tile = wl.Hkv * max(1, G // 2)
    blk_bytes = 128 * wl.d * 2 * 2
    paged_blocks = span_blocks = 0
    for u in range(len(pb.ub)):
        ts_, tp_ = wl.ubatches[u]
        cut = np.flatnonzero(np.diff(ts_)) + 1
        for a_, b_ in zip(np.concatenate([[0], cut]), np.concatenate([cut, [len(ts_)]])):
            n = b_ - a_
            nt = -(-n // 128)
            for i in range(nt):
                lo, hi = a_ + n * i // nt, a_ + n * (i + 1) // nt
                paged_blocks += items_per_tile * -(-int(tp_[lo:hi].max() + 1) // 128)
        span_blocks += items_per_tile * -(-len(ts_) // 128) * (N * P // 128)
    return {"workload": "prefill_8x16k_unified_span", "unit": "ms", "value": round(ms, 3),
            "higher_is_better": False, "ms_per_step": round(ms, 3),
            "paged_ms_per_step": round(paged_ms_per_step, 3),
            "paged_speedup": round(ms / paged_ms_per_step, 2),
            "kv_bytes_per_step": {"span": span_blocks * blk_bytes, "paged": paged_blocks * blk_bytes},
            "bytes_ratio": round(span_blocks / paged_blocks, 2),
            "tflops_equiv": round(pb.flops / (ms / 1e3) / 1e12, 2),
            "agrees_with_paged_on_last_ubatch": agree,
            "timing": f"CUDA graph of 65 x (plan + masked tcgen05 prefill), {n_steps} step(s)",
            "note": "the span is every cell of the pool (free cells masked, their V rows zeroed); "
                    "llama.cpp's unified cache reads the span the same way"}


def bench_fp8_decode(pa, torch, db, steps, warmup, world, hbm, f16_ms_per_layer,
                     workload="decode_8seq_fp8_pages", traffic_key="k_decode_fp8"):
    """FP8 KV pages on a decode workload: the same layers with every cached row
    quantised (E4M3 codes, one scale per row) by the library's quantising append;
    one plan, then the FP8 decode launches back to back."""
    c = db.case
    dev = db.q[0].device
    rows_k, rows_v, slots = [], [], []
    for s_, pages in enumerate(c.seq_pages):
        L = int(c.seq_len[s_])
        pos = np.arange(L)
        slots.append(np.asarray(pages, np.int64)[pos // c.P] * c.P + pos % c.P)
        rows_k.append(c.k_ctx[s_][:L])
        rows_v.append(c.v_ctx[s_][:L])
    kr = torch.from_numpy(np.concatenate(rows_k).view(np.float16)).to(dev)
    vr = torch.from_numpy(np.concatenate(rows_v).view(np.float16)).to(dev)
    sl = torch.from_numpy(np.concatenate(slots)).to(dev)
    base = pa.new_fp8_pool(c.num_pages, c.Hkv, c.P, c.d, dev)
    pa.kv_append_fp8(kr, vr, sl, *base)
    pools = [base] + [tuple(t.clone() for t in base) for _ in range(db.layers - 1)]
    ws = pa.new_workspace(c.T, c.Hq, c.Hkv, c.d, dev)
    out = torch.empty_like(db.q[0])

    def step():
        pa.plan_decode(db.tpt, db.kv, c.Hq, c.Hkv, c.P, c.d, ws)
        for l in range(db.layers):
            pa.decode_fp8(db.q[l], *pools[l], db.tpt, db.kv, c.scale, out, ws)

    g = capture_step(torch, step)
    total_ms, _ = time_steps(torch, g.replay, steps, warmup, world)
    ms_layer = max_over_ranks(total_ms / steps / db.layers, world)
    if pa.read_error(ws):
        raise RuntimeError("device error word set in the FP8 decode")
    nbytes = float(c.seq_len.astype(np.int64).sum()) * c.Hkv * (2 * c.d + 2 * 4)
    gbs = nbytes / (ms_layer / 1e3) / 1e9
    return {"workload": workload, "unit": "GB/s", "value": round(gbs * world, 1),
            "ms_per_layer": round(ms_layer, 4), "bytes_per_layer": nbytes,
            "f16_ms_per_layer": round(f16_ms_per_layer, 4),
            "speedup_vs_f16": round(f16_ms_per_layer / ms_layer, 2),
            "roofline": {"bound": "hbm", "kernel": "k_decode (FP8 pages)",
                         "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbs / hbm, 4), "traffic": traffic_of(traffic_key)},
            "timing": f"CUDA graph of one plan and {db.layers} FP8 decode launches (one per layer)"}


def bench_fp8_prefill(pa, torch, pb, steps, warmup, world, peak, f16_ms_per_step,
                      f16_ms_per_launch, with_cpu):
    """The 8x16K prefill step over FP8 pages: the same ubatches, each one expansion,
    quantising append (E4M3 codes, one scale per row), plan, tensor-core prefill (the
    codes widened to binary16 in shared memory) and decode launch, over a pool of
    codes (half the K/V bytes of the binary16 pool)."""
    wl, dev = pb.wl, pb.dev
    pool = pa.new_fp8_pool(wl.num_pages, wl.Hkv, wl.P, wl.d, dev)
    ws = pa.new_workspace(max(d["T"] for d in pb.ub), wl.Hq, wl.Hkv, wl.d, dev)
    outs = [torch.empty_like(d["out"]) for d in pb.ub]

    def ubatch(d, out, ev=None):
        pa.expand_ubatch(pb.spt, d["tok_seq"], d["tok_pos"], wl.P,
                         out=(d["tpt"], d["kv"], d["slot"]))
        pa.kv_append_fp8(d["k"], d["v"], d["slot"], *pool)
        pa.plan(d["tpt"], d["kv"], wl.Hq, wl.Hkv, wl.P, wl.d, ws)
        if ev is not None:
            ev[0].record()
        pa.prefill_fp8(d["q"], *pool, d["tpt"], d["kv"], wl.scale, out, ws)
        if ev is not None:
            ev[1].record()
        pa.decode_fp8(d["q"], *pool, d["tpt"], d["kv"], wl.scale, out, ws)

    def step(events=None):
        for i, (d, out) in enumerate(zip(pb.ub, outs)):
            ubatch(d, out, None if events is None else events[i])

    n_ub = len(pb.ub)
    g = capture_step(torch, step)
    total, _ = time_steps(torch, g.replay, steps, warmup, world)
    kern, how = time_launches(torch, step, n_ub, steps, warmup, world)
    if pa.read_error(ws):
        raise RuntimeError("device error word set in the FP8 prefill")
    t_step = max_over_ranks(total / 1e3 / steps, world)
    t_kern = kern / 1e3 / (steps * n_ub)
    ach = pb.flops / n_ub / t_kern / 1e12
    res = {"workload": "prefill_8x16k_fp8_pages", "unit": "TFLOP/s",
           "value": round(aggregate(pb.flops, t_step, world) / 1e12, 3),
           "ms_per_step": round(t_step * 1e3, 3),
           "f16_ms_per_step": round(f16_ms_per_step, 3),
           "f16_ms_per_prefill_launch": round(f16_ms_per_launch, 4),
           "ms_per_prefill_launch": round(t_kern * 1e3, 4),
           "gpu_launches": 5 * n_ub * steps,
           "roofline": {"bound": "tensor", "kernel": "k_prefill (FP8 pages)",
                        "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s",
                        "frac": round(ach / peak, 4), "timing": how,
                        "traffic": traffic_of("k_prefill_fp8")},
           "timing": "value: CUDA graph of the 65 ubatches x (expand, append_fp8, plan, "
                     "prefill_fp8, decode_fp8)"}
    if with_cpu:
        import oracle
        u = n_ub - 1
        d = pb.ub[u]
        q = d["q"].cpu().numpy().view(np.uint16)
        rng = np.random.default_rng(11)
        sel = np.sort(rng.choice(d["T"], min(24, d["T"]), replace=False)).astype(np.int32)
        host = [x.cpu().numpy() for x in pool]
        tpt_h, kv_h = d["tpt"].cpu().numpy(), d["kv"].cpu().numpy()
        t0 = time.perf_counter()
        ref = oracle.paged_attention_fp8(q, *host, tpt_h, kv_h, wl.scale, tokens=sel)
        secs = time.perf_counter() - t0
        f_s = 4.0 * wl.d * wl.Hq * float(kv_h[sel].astype(np.int64).sum())
        res["cpu_baseline"] = {"value": f_s / secs / 1e12, "unit": "TFLOP/s",
                               "cores": oracle.num_threads(), "kind": "oracle",
                               "sample": f"{len(sel)} tokens of the last ubatch, all heads, "
                                         f"fp64 over the FP8 pool, {secs:.1f} s"}
        res["parity"] = parity_check(
            [(u, sel, ref)],
            lambda u_, s_: outs[u_][torch.from_numpy(s_).long().to(dev)].float().cpu().numpy())
        if not res["parity"]["ok"]:
            raise RuntimeError(f"FP8 prefill outputs differ from the oracle: {res['parity']}")
    return res


LONGTAIL_LAYERS = 4


def bench_longtail(pa, torch, dev, steps, warmup, world, hbm, with_cpu, seed=0):
    """Long-tail decode: 64 sequences, KV lengths lognormal (median 2048, clipped to
    256..32768), 30% free pages; about 0.85 GB of K/V per layer, so 4 layers over 4
    distinct pools exceed L2 many times over.  One expansion and plan, then per layer
    append + decode (the split-KV path with its fused reduce)."""
    import workloads
    db = DecodeBench(pa, torch, dev, seed=seed, layers=LONGTAIL_LAYERS,
                     case=workloads.longtail(seed))
    g = capture_step(torch, db.step)
    total, _ = time_steps(torch, g.replay, steps, warmup, world)
    a_graph = capture_step(torch, db.attention_only)
    kern, _ = time_steps(torch, a_graph.replay, steps, warmup, world)
    if pa.read_error(db.ws):
        raise RuntimeError("device error word set in the long-tail decode")
    t_step = max_over_ranks(total / 1e3 / steps, world)
    t_kern = kern / 1e3 / (steps * db.layers)
    ach = db.bytes_per_layer / t_kern / 1e9
    c = db.case
    res = {"workload": "decode_longtail_64seq", "unit": "GB/s",
           "value": round(aggregate(db.bytes_per_layer * db.layers, t_step, world) / 1e9, 1),
           "layers": db.layers, "kv_bytes_per_layer": db.bytes_per_layer,
           "ms_per_step": round(t_step * 1e3, 4), "ms_per_layer_decode": round(t_kern * 1e3, 4),
           "seq_len": {"min": int(c.seq_len.min()), "median": float(np.median(c.seq_len)),
                       "max": int(c.seq_len.max())},
           "gpu_launches": db.launches_per_step * steps,
           "roofline": {"bound": "hbm", "kernel": "k_decode", "achieved": round(ach, 1),
                        "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
                        "timing": "CUDA events around a graph of the 4 decode launches back to "
                                  "back (appends left out)",
                        "traffic": traffic_of("k_decode_longtail")},
           "timing": "value: CUDA graph of expansion, plan and 4 x (append + decode)"}
    # FP8 pages on the same long-tail layer: half the bytes, where streaming dominates
    res["fp8_pages"] = bench_fp8_decode(pa, torch, db, steps, warmup, world, hbm, t_kern * 1e3,
                                        workload="decode_longtail_64seq_fp8_pages",
                                        traffic_key="k_decode_fp8_longtail")
    if with_cpu:
        res["cpu_baseline"] = cpu_baseline_decode(c, reps_budget_s=3.0)
        res["cpu_baseline"]["sample"] = res["cpu_baseline"]["sample"].replace(
            "8 tokens", f"{c.T} tokens")
    return res


MIXED_LAYERS = 8


def mixed_unique_bytes(case):
    """K/V bytes of the distinct (page, KV head) blocks a ubatch reads, each counted
    once, only the rows below each reader's kv_len (the shared prefix counts once),
    against the logical bytes (every token's own sequence K/V)."""
    P, row = case.P, case.Hkv * case.d * 2 * 2     # K + V bytes of one cached row
    rows_of_page = {}
    logical = 0
    for s, p in zip(case.tok_seq, case.tok_pos):
        if s < 0:
            continue
        L = int(p) + 1
        logical += L * row
        pages = case.seq_pages[int(s)]
        for j in range(-(-L // P)):
            pg = int(pages[j])
            rows_of_page[pg] = max(rows_of_page.get(pg, 0), min(P, L - j * P))
    return float(sum(rows_of_page.values()) * row), float(logical)


def bench_mixed(pa, torch, dev, steps, warmup, world, hbm, tensor_peak, with_cpu, seed=0):
    """The shared-prefix mixed ubatch: 16 sequences share 64 prefix pages (8192 tokens);
    12 decode tokens plus 4 x 256 prefill tokens in one ubatch.  One expansion and
    plan (prefill tiles and decode items in the same plan), then per layer append +
    run (the tcgen05 prefill launch, then the split-KV decode launch), over 8 distinct
    pools.  Roofline: the time the ubatch needs at least, max(unique K/V bytes / HBM
    peak, FLOPs / tensor peak), over the measured time."""
    import workloads
    c = workloads.shared_prefix(seed)
    t = torch
    spt = t.from_numpy(c.seq_page_table()).to(dev)
    ts, tp = t.from_numpy(c.tok_seq).to(dev), t.from_numpy(c.tok_pos).to(dev)
    kp = t.from_numpy(c.k_pool.view(np.float16)).to(dev)
    vp = t.from_numpy(c.v_pool.view(np.float16)).to(dev)
    pools = [(kp.clone(), vp.clone()) for _ in range(MIXED_LAYERS)]
    qs = [t.from_numpy(c.q.view(np.float16)).to(dev) for _ in range(MIXED_LAYERS)]
    kn, vn = t.from_numpy(c.k_new.view(np.float16)).to(dev), t.from_numpy(c.v_new.view(np.float16)).to(dev)
    outs = [t.empty_like(qs[0]) for _ in range(MIXED_LAYERS)]
    ws = pa.new_workspace(c.T, c.Hq, c.Hkv, c.d, dev)
    tpt = t.empty((c.T, c.max_pages), dtype=t.int32, device=dev)
    kv = t.empty(c.T, dtype=t.int32, device=dev)
    slot = t.empty(c.T, dtype=t.int64, device=dev)

    def step():
        pa.expand_ubatch(spt, ts, tp, c.P, out=(tpt, kv, slot))
        pa.plan(tpt, kv, c.Hq, c.Hkv, c.P, c.d, ws)
        for l in range(MIXED_LAYERS):
            pa.kv_append(kn, vn, slot, *pools[l])
            pa.run(qs[l], *pools[l], tpt, kv, c.scale, outs[l], ws)

    g = capture_step(torch, step)
    total, _ = time_steps(torch, g.replay, steps, warmup, world)
    if pa.read_error(ws):
        raise RuntimeError("device error word set in the mixed shared-prefix ubatch")
    t_step = max_over_ranks(total / 1e3 / steps, world)
    t_layer = t_step / MIXED_LAYERS
    kv_len = c.tok_pos.astype(np.int64) + 1
    flops = 4.0 * c.d * c.Hq * float(kv_len.sum())
    uniq, logical = mixed_unique_bytes(c)
    t_min = max(uniq / (hbm * 1e9), flops / (tensor_peak * 1e12))
    res = {"workload": "mixed_shared_prefix_12dec_1024pf", "unit": "TFLOP/s",
           "value": round(aggregate(flops * MIXED_LAYERS, t_step, world) / 1e12, 2),
           "layers": MIXED_LAYERS, "ms_per_layer": round(t_layer * 1e3, 4),
           "flops_per_layer": flops, "unique_kv_bytes_per_layer": uniq,
           "logical_kv_bytes_per_layer": logical,
           "unique_gbs": round(uniq / t_layer / 1e9, 1),
           "logical_gbs": round(logical / t_layer / 1e9, 1),
           "roofline": {"bound": "tensor" if flops / (tensor_peak * 1e12) >= uniq / (hbm * 1e9)
                        else "hbm",
                        "kernel": "k_prefill + k_decode (one layer of the ubatch)",
                        "achieved": round(flops / t_layer / 1e12, 2), "peak": tensor_peak,
                        "unit": "TFLOP/s", "frac": round(t_min / t_layer, 4),
                        "hbm_peak_gbs": hbm, "t_min_ms": round(t_min * 1e3, 4),
                        "note": "frac = max(unique bytes / HBM peak, FLOPs / tensor peak) "
                                "/ measured time per layer (append, prefill and decode launches)",
                        "traffic": None},
           "gpu_launches": (2 + 3 * MIXED_LAYERS + 1) * steps,
           "timing": "CUDA graph of expansion, plan and 8 x (append + prefill + decode)"}
    if with_cpu:
        import oracle
        tpt_h, kv_h, slot_h = oracle.expand_ubatch(c.seq_page_table(), c.tok_seq, c.tok_pos, c.P)
        kph, vph = c.k_pool.copy(), c.v_pool.copy()
        oracle.kv_append(c.k_new, c.v_new, slot_h, kph, vph)
        sel = np.concatenate([np.arange(12), np.arange(12, c.T, 16)]).astype(np.int32)
        t0 = time.perf_counter()
        ref = oracle.paged_attention(c.q, kph, vph, tpt_h, kv_h, c.scale, tokens=sel)
        secs = time.perf_counter() - t0
        f_s = 4.0 * c.d * c.Hq * float(kv_h[sel].astype(np.int64).sum())
        res["cpu_baseline"] = {"value": f_s / secs / 1e12, "unit": "TFLOP/s",
                               "cores": oracle.num_threads(), "kind": "oracle",
                               "sample": f"the 12 decode tokens and every 16th prefill token "
                                         f"({len(sel)} tokens, all heads, fp64), {secs:.1f} s"}
        res["parity"] = parity_check(
            [(0, sel, ref)],
            lambda u, s_: outs[-1][t.from_numpy(s_).long().to(dev)].float().cpu().numpy())
        if not res["parity"]["ok"]:
            raise RuntimeError(f"mixed ubatch outputs differ from the oracle: {res['parity']}")
    return res


def run_ours(args):
    import torch
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import paged_kv_cache_pages_gb300 as pa

    peaks, peak_src = load_peaks()
    pb = PrefillBench(pa, torch, dev, seed=args.seed)
    n_ub = len(pb.ub)

    # correctness guard: the run must not report device errors
    pb.step()
    torch.cuda.synchronize()
    if pa.read_error(pb.ws):
        raise RuntimeError("device error word set during the prefill warm-up")

    graph = capture_step(torch, pb.step)
    with ClockSampler(local) as clk:
        total_ms, _ = time_steps(torch, graph.replay, args.steps, args.warmup, world)
        kern_ms, kern_how = time_launches(torch, pb.step, n_ub, args.steps, args.warmup, world)
    clocks = clk.summary()
    t_step = max_over_ranks(total_ms / 1e3 / args.steps, world)
    value = aggregate(pb.flops, t_step, world) / 1e12
    t_kern = kern_ms / 1e3 / (args.steps * n_ub)             # average prefill launch
    achieved = pb.flops / n_ub / t_kern / 1e12
    f16 = measure_f16_peak(torch, dev, local)
    peak, peak_how = clock_matched_peak(clocks, f16["burst"], f16["sustained"])

    # end to end: pinned host buffers, copies inside the timed region
    for _ in range(args.warmup):
        pb.step_e2e()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(args.steps):
        h2d, d2h = pb.step_e2e()
    s1.record()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(s0.elapsed_time(s1) / 1e3 / args.steps, world)

    # decode leg
    db = DecodeBench(pa, torch, dev, seed=args.seed)
    d_graph = capture_step(torch, db.step)
    d_total, _ = time_steps(torch, d_graph.replay, args.steps, args.warmup, world)
    d_kern_node, _ = time_launches(torch, db.step, db.layers, args.steps, args.warmup, world)
    a_graph = capture_step(torch, db.attention_only)
    d_kern, _ = time_steps(torch, a_graph.replay, args.steps, args.warmup, world)
    d_step = max_over_ranks(d_total / 1e3 / args.steps, world)
    d_value = aggregate(db.bytes_per_layer * db.layers, d_step, world) / 1e9
    d_kt = d_kern / 1e3 / (args.steps * db.layers)
    d_ach = db.bytes_per_layer / d_kt / 1e9
    d_ach_node = db.bytes_per_layer / (d_kern_node / 1e3 / (args.steps * db.layers)) / 1e9
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    if pa.read_error(db.ws) or pa.read_error(pb.ws):
        raise RuntimeError("device error word set during the timed region")

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": "prefill_8x16k", "n_seq": 8, "prompt_tokens": 16384,
                   "ubatches": n_ub, "ubatch_tokens_max": 2048, "slots": 4,
                   "q_heads": 32, "kv_heads": 8, "head_dim": 128, "page_size": 128,
                   "pool_pages": pb.wl.num_pages, "flops_per_step": pb.flops,
                   "l2": "inputs larger than L2 (KV pool 655 MB, q 1 GB per step)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "kernel": "k_prefill", "achieved": round(achieved, 2),
                     "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"measured in this run: f16 {peak_how}",
                     "peak_f16_burst": f16["burst"], "peak_f16_sustained": f16["sustained"],
                     "frac_vs_f16_burst": round(achieved / f16["burst"], 4),
                     "frac_vs_f16_sustained": round(achieved / f16["sustained"], 4),
                     "f16_peak": f16,
                     "peak_file_bf16": {"burst": peaks.get("bf16_tflops"),
                                        "sustained": peaks.get("bf16_tflops_sustained"),
                                        "source": peak_src},
                     "per_step_frac": round(value / world / peak, 4),
                     "traffic": traffic_of("k_prefill")},
        "e2e": {"value": round(aggregate(pb.flops, e2e_s, world) / 1e12, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": pb.launches_per_step * args.steps,
        "timing": "value: CUDA-graph replay of whole steps; roofline: " + kern_how,
        "clocks": clocks,
        "decode": {"workload": "decode_8seq", "value": round(d_value, 1), "unit": "GB/s",
                   "layers": db.layers, "kv_bytes_per_layer": db.bytes_per_layer,
                   "ms_per_step": round(d_step * 1e3, 3),
                   "step": "expansion and plan, then per layer one launch: the layer's K/V "
                           "append fused into the split-KV decode",
                   "gpu_launches": db.launches_per_step * args.steps,
                   "roofline": {"bound": "hbm", "kernel": "k_decode",
                                "achieved": round(d_ach, 1), "peak": hbm, "unit": "GB/s",
                                "frac": round(d_ach / hbm, 4),
                                "timing": "CUDA events around a graph of 36 decode launches "
                                          "back to back (no append); the step's fused "
                                          "append + decode launches timed between "
                                          "event-record nodes inside the step graph: "
                                          "%.1f GB/s" % d_ach_node,
                                "peak_source": f"{peak_src} hbm copy",
                                "traffic": traffic_of("k_decode")}},
    }
    # rows beyond the headline, same bar: page copy of copy-on-write forks
    line["next"] = {
        "copy_pages": bench_copy_pages(
            pa, torch, dev, args.steps, args.warmup, world, hbm,
            with_cpu=rank == 0 and world == 1 and not args.no_cpu_baseline, seed=args.seed),
        "unified_span": bench_unified_span(pa, torch, db, args.steps, args.warmup, world, hbm,
                                           d_kt * 1e3),
        "unified_span_prefill": bench_unified_span_prefill(pa, torch, pb, args.steps,
                                                           args.warmup, world, t_step * 1e3),
        "fp8_pages": bench_fp8_decode(pa, torch, db, args.steps, args.warmup, world, hbm,
                                      d_kt * 1e3),
        "fp8_pages_prefill": bench_fp8_prefill(
            pa, torch, pb, args.steps, args.warmup, world, peak, t_step * 1e3, t_kern * 1e3,
            with_cpu=rank == 0 and world == 1 and not args.no_cpu_baseline),
    }
    line["longtail"] = bench_longtail(pa, torch, dev, args.steps, args.warmup, world, hbm,
                                      with_cpu=rank == 0 and world == 1 and not args.no_cpu_baseline,
                                      seed=args.seed)
    line["mixed_shared_prefix"] = bench_mixed(
        pa, torch, dev, args.steps, args.warmup, world, hbm, peak,
        with_cpu=rank == 0 and world == 1 and not args.no_cpu_baseline, seed=args.seed)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"], kept = cpu_baseline_prefill(pb.wl, budget_s=args.cpu_budget,
                                                          keep=True)
        line["decode"]["cpu_baseline"] = cpu_baseline_decode(db.case)
        # the outputs the timed steps left in each ubatch's buffer, against the oracle
        line["parity"] = parity_check(
            kept, lambda u, sel: pb.ub[u]["out"][torch.from_numpy(sel).long().to(dev)]
            .float().cpu().numpy())
        if not line["parity"]["ok"]:
            raise RuntimeError(f"8x16K outputs differ from the oracle: {line['parity']}")
    else:
        line["parity"] = None
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The CPU fp64 oracle as the reference arm (rank 0 only)."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import workloads
    wl = workloads.Prefill8x16K(args.seed)
    for _ in range(args.warmup):
        cpu_baseline_prefill(wl, budget_s=1.0)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline_prefill(wl, budget_s=args.cpu_budget / max(args.steps, 1)))
    wall = time.perf_counter() - t0
    v = float(np.median([x["value"] for x in vals]))
    line = {"metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(wall / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": "prefill_8x16k", "n_seq": 8, "prompt_tokens": 16384,
                       "q_heads": 32, "kv_heads": 8, "head_dim": 128, "page_size": 128,
                       "parallelism": "host cores"},
            "cpu_baseline": {"kind": "oracle", "cores": vals[0]["cores"], "value": v,
                             "unit": "TFLOP/s", "sample": vals[0]["sample"]},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
