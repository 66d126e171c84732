"""Small, self-contained cases for kernel profiling (ncu) and quick timing.

  python -m paged_kv_cache_pages_gb300.profile_case prefill [--ubatch U] [--reps R]
      one ubatch of the 8 x 16K prefill (default: a late one, long contexts):
      expand -> append -> plan -> prefill -> decode, R times.  Device memory:
      the 655 MB KV pool (larger than L2) plus one ubatch.
  python -m paged_kv_cache_pages_gb300.profile_case prefill_fp8 [--ubatch U] [--reps R]
      the same ubatch over FP8 pages (every row of the 8 sequences quantised by the
      library's append: 336 MB of codes), the prefill call alone, R times.
  python -m paged_kv_cache_pages_gb300.profile_case decode [--reps R] [--pools N]
      the 8-sequence decode layer: expand -> plan -> append -> decode, over N
      copies of the 82 MB pool used in turn (default 8: 660 MB, larger than L2,
      so every call streams its pool from HBM).

  python -m paged_kv_cache_pages_gb300.profile_case longtail [--reps R] [--pools N]
      the long-tail decode layer (64 sequences, lognormal lengths, 1.06 GB of K/V):
      expand -> plan -> append -> decode over N pool copies in turn (use 2: 3 GB).

  python -m paged_kv_cache_pages_gb300.profile_case span [--reps R]
      the unified-span baseline on the decode layer: every token reads the whole
      pool under a per-cell mask (one plan + masked decode per call).
  python -m paged_kv_cache_pages_gb300.profile_case fp8 [--reps R] [--pools N]
      the decode layer over FP8 pages (every cached row quantised by the
      library's append), N pool copies in turn (default 8).
  python -m paged_kv_cache_pages_gb300.profile_case fp8_longtail [--reps R] [--pools N]
      the long-tail layer over FP8 pages (0.55 GB of codes and scales), N copies in
      turn (use 2).
  python -m paged_kv_cache_pages_gb300.profile_case copy [--reps R]
      page copy of copy-on-write forks: 512 of 1280 pages (8 KV heads x 128 rows
      x d 128, K and V) copied to 512 others per call.

Prints the average time of the call (CUDA events) and exits 0.
"""
import argparse
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import paged_kv_cache_pages_gb300 as pa  # noqa: E402
import workloads  # noqa: E402


def _time(fn, reps):
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fn()
    torch.cuda.synchronize()
    s.record()
    for _ in range(reps):
        fn()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / reps


def prefill(ubatch: int, reps: int):
    wl = workloads.Prefill8x16K(0)
    kp_h, vp_h = wl.pool_final()
    dev = "cuda"
    kp = torch.from_numpy(kp_h.view(np.float16)).to(dev)
    vp = torch.from_numpy(vp_h.view(np.float16)).to(dev)
    ts, tp, q, k, v = wl.ubatch(ubatch)
    spt = torch.from_numpy(wl.seq_page_table).to(dev)
    ts_d, tp_d = torch.from_numpy(ts).to(dev), torch.from_numpy(tp).to(dev)
    q_d = torch.from_numpy(q.view(np.float16)).to(dev)
    k_d = torch.from_numpy(np.ascontiguousarray(k).view(np.float16)).to(dev)
    v_d = torch.from_numpy(np.ascontiguousarray(v).view(np.float16)).to(dev)
    out = torch.empty_like(q_d)
    ws = pa.new_workspace(ts.shape[0], wl.Hq, wl.Hkv, wl.d, dev)
    tpt, kv, slot = pa.expand_ubatch(spt, ts_d, tp_d, wl.P)
    pa.kv_append(k_d, v_d, slot, kp, vp)
    pa.plan(tpt, kv, wl.Hq, wl.Hkv, wl.P, wl.d, ws)

    def fn():
        pa.prefill(q_d, kp, vp, tpt, kv, wl.scale, out, ws)
        pa.decode(q_d, kp, vp, tpt, kv, wl.scale, out, ws)

    ms = _time(fn, reps)
    if pa.read_error(ws):
        raise SystemExit("device error word set")
    flops = 4.0 * wl.d * wl.Hq * float((tp.astype(np.int64) + 1).sum())
    print(f"prefill ubatch {ubatch}: T={ts.shape[0]} {ms * 1e3:.1f} us/call "
          f"{flops / ms / 1e9:.1f} TFLOP/s (prefill+decode calls)")


def decode(reps: int, n_pools: int, longtail: bool = False):
    c = workloads.longtail(0) if longtail else workloads.decode(0)
    dev = "cuda"
    spt = torch.from_numpy(c.seq_page_table()).to(dev)
    kp = torch.from_numpy(c.k_pool.view(np.float16)).to(dev)
    vp = torch.from_numpy(c.v_pool.view(np.float16)).to(dev)
    q = torch.from_numpy(c.q.view(np.float16)).to(dev)
    tpt, kv, slot = pa.expand_ubatch(spt, torch.from_numpy(c.tok_seq).to(dev),
                                     torch.from_numpy(c.tok_pos).to(dev), c.P)
    pa.kv_append(torch.from_numpy(c.k_new.view(np.float16)).to(dev),
                 torch.from_numpy(c.v_new.view(np.float16)).to(dev), slot, kp, vp)
    ws = pa.new_workspace(c.T, c.Hq, c.Hkv, c.d, dev)
    out = torch.empty_like(q)
    pa.plan(tpt, kv, c.Hq, c.Hkv, c.P, c.d, ws)
    pools = [(kp, vp)] + [(kp.clone(), vp.clone()) for _ in range(n_pools - 1)]
    turn = [0]

    def fn():
        k_, v_ = pools[turn[0] % len(pools)]
        turn[0] += 1
        pa.decode(q, k_, v_, tpt, kv, c.scale, out, ws)

    ms = _time(fn, reps)
    if pa.read_error(ws):
        raise SystemExit("device error word set")
    nbytes = float(c.seq_len.astype(np.int64).sum()) * c.Hkv * c.d * 4
    print(f"{c.name}: {ms * 1e3:.1f} us/call {nbytes / ms / 1e6:.1f} GB/s "
          f"({len(pools)} pools in turn, eager launches)")


def span(reps: int):
    c = workloads.decode(0)
    dev = "cuda"
    tpt0, kv0, slot = pa.expand_ubatch(
        torch.from_numpy(c.seq_page_table()).to(dev), torch.from_numpy(c.tok_seq).to(dev),
        torch.from_numpy(c.tok_pos).to(dev), c.P)
    kp = torch.from_numpy(c.k_pool.view(np.float16)).to(dev)
    vp = torch.from_numpy(c.v_pool.view(np.float16)).to(dev)
    pa.kv_append(torch.from_numpy(c.k_new.view(np.float16)).to(dev),
                 torch.from_numpy(c.v_new.view(np.float16)).to(dev), slot, kp, vp)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    tpt, kv, cs, cp, ts, tp = (t(a) for a in workloads.span_view(c))
    q = torch.from_numpy(c.q.view(np.float16)).to(dev)
    out = torch.empty_like(q)
    ws = pa.new_workspace(c.T, c.Hq, c.Hkv, c.d, dev)
    pa.plan_decode(tpt, kv, c.Hq, c.Hkv, c.P, c.d, ws)
    ms = _time(lambda: pa.masked_decode(q, kp, vp, tpt, kv, c.scale, cs, cp, ts, tp, out, ws),
               reps)
    if pa.read_error(ws):
        raise SystemExit("device error word set")
    nbytes = float(c.T) * c.num_pages * c.Hkv * c.P * c.d * 4
    print(f"span: {ms * 1e3:.1f} us/call {nbytes / ms / 1e6:.1f} GB/s of span reads "
          f"({c.num_pages} pages read by each of {c.T} tokens)")


def prefill_fp8(ubatch: int, reps: int):
    wl = workloads.Prefill8x16K(0)
    K, V = wl._draw_kv()
    dev = "cuda"
    pos = np.arange(wl.seq_len)
    slots = np.concatenate([wl.seq_page_table[s][pos // wl.P].astype(np.int64) * wl.P + pos % wl.P
                            for s in range(wl.n_seq)])
    pool = pa.new_fp8_pool(wl.num_pages, wl.Hkv, wl.P, wl.d, dev)
    pa.kv_append_fp8(torch.from_numpy(K.reshape(-1, wl.Hkv, wl.d).view(np.float16)).to(dev),
                     torch.from_numpy(V.reshape(-1, wl.Hkv, wl.d).view(np.float16)).to(dev),
                     torch.from_numpy(slots).to(dev), *pool)
    ts, tp, q, _, _ = wl.ubatch(ubatch)
    spt = torch.from_numpy(wl.seq_page_table).to(dev)
    q_d = torch.from_numpy(q.view(np.float16)).to(dev)
    out = torch.empty_like(q_d)
    ws = pa.new_workspace(ts.shape[0], wl.Hq, wl.Hkv, wl.d, dev)
    tpt, kv, _ = pa.expand_ubatch(spt, torch.from_numpy(ts).to(dev), torch.from_numpy(tp).to(dev),
                                  wl.P)
    pa.plan(tpt, kv, wl.Hq, wl.Hkv, wl.P, wl.d, ws)

    def fn():
        pa.prefill_fp8(q_d, *pool, tpt, kv, wl.scale, out, ws)

    ms = _time(fn, reps)
    if pa.read_error(ws):
        raise SystemExit("device error word set")
    flops = 4.0 * wl.d * wl.Hq * float((tp.astype(np.int64) + 1).sum())
    print(f"prefill_fp8 ubatch {ubatch}: T={ts.shape[0]} {ms * 1e3:.1f} us/call "
          f"{flops / ms / 1e9:.1f} TFLOP/s (prefill call; FP8 pool of every row)")


def fp8(reps: int, n_pools: int, longtail: bool = False):
    c = workloads.longtail(0) if longtail else workloads.decode(0)
    dev = "cuda"
    tpt, kv, _ = pa.expand_ubatch(
        torch.from_numpy(c.seq_page_table()).to(dev), torch.from_numpy(c.tok_seq).to(dev),
        torch.from_numpy(c.tok_pos).to(dev), c.P)
    rows_k, rows_v, slots = [], [], []
    for s, pages in enumerate(c.seq_pages):
        L = int(c.seq_len[s])
        pos = np.arange(L)
        slots.append(np.asarray(pages, np.int64)[pos // c.P] * c.P + pos % c.P)
        rows_k.append(c.k_ctx[s][:L])
        rows_v.append(c.v_ctx[s][:L])
    base = pa.new_fp8_pool(c.num_pages, c.Hkv, c.P, c.d, dev)
    pa.kv_append_fp8(torch.from_numpy(np.concatenate(rows_k).view(np.float16)).to(dev),
                     torch.from_numpy(np.concatenate(rows_v).view(np.float16)).to(dev),
                     torch.from_numpy(np.concatenate(slots)).to(dev), *base)
    pools = [base] + [tuple(t.clone() for t in base) for _ in range(n_pools - 1)]
    q = torch.from_numpy(c.q.view(np.float16)).to(dev)
    out = torch.empty_like(q)
    ws = pa.new_workspace(c.T, c.Hq, c.Hkv, c.d, dev)
    pa.plan_decode(tpt, kv, c.Hq, c.Hkv, c.P, c.d, ws)
    turn = [0]

    def fn():
        p_ = pools[turn[0] % len(pools)]
        turn[0] += 1
        pa.decode_fp8(q, *p_, tpt, kv, c.scale, out, ws)

    ms = _time(fn, reps)
    if pa.read_error(ws):
        raise SystemExit("device error word set")
    nbytes = float(c.seq_len.astype(np.int64).sum()) * c.Hkv * (2 * c.d + 8)
    print(f"fp8 {c.name}: {ms * 1e3:.1f} us/call {nbytes / ms / 1e6:.1f} GB/s "
          f"({len(pools)} pools in turn)")


def copy(reps: int):
    dev = "cuda"
    N, Hkv, P, d, n = 1280, 8, 128, 128, 512
    rng = np.random.default_rng(7000)
    ids = rng.permutation(N).astype(np.int32)
    src = torch.from_numpy(ids[:n].copy()).to(dev)
    dst = torch.from_numpy(ids[n:2 * n].copy()).to(dev)
    kp = torch.empty((N, Hkv, P, d), dtype=torch.float16, device=dev).normal_()
    vp = torch.empty_like(kp).normal_()
    ms = _time(lambda: pa.copy_pages(src, dst, kp, vp), reps)
    nbytes = 2.0 * 2 * n * Hkv * P * d * 2
    print(f"copy_pages: {ms * 1e3:.1f} us/call {nbytes / ms / 1e6:.1f} GB/s (read + written)")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["prefill", "prefill_fp8", "decode", "longtail", "copy",
                                     "span", "fp8", "fp8_longtail"])
    ap.add_argument("--ubatch", type=int, default=48)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--pools", type=int, default=8)
    a = ap.parse_args()
    if a.case == "prefill":
        prefill(a.ubatch, a.reps)
    elif a.case == "prefill_fp8":
        prefill_fp8(a.ubatch, a.reps)
    elif a.case == "decode":
        decode(a.reps, a.pools)
    elif a.case == "longtail":
        decode(a.reps, a.pools, longtail=True)
    elif a.case == "span":
        span(a.reps)
    elif a.case == "fp8":
        fp8(a.reps, a.pools)
    elif a.case == "fp8_longtail":
        fp8(a.reps, a.pools, longtail=True)
    else:
        copy(a.reps)


if __name__ == "__main__":
    main()
