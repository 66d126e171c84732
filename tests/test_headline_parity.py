"""GPU parity on the 8 x 16K prefill schedule itself, the workload the headline
TFLOP/s is quoted on (UA-PagedAttention page, sections 作品简介 and 关键性能数据:
16K-token prompts at 8-way concurrency, per-token page rows and true lengths).

All 65 ubatches run in order on one pool, each through expand -> append ->
forward (plan + tcgen05 prefill + split-KV decode), exactly as the benchmark
issues them.  Checked against the fp64 oracle, element by element at
2e-3 + 1e-2 |ref|, on sampled tokens x all 32 query heads of:
  - ubatch 0 (empty prefixes),
  - ubatch 30 (every slot at a ~15K-token prefix),
  - ubatch 32 (slots 1-3 cross from sequence k to k + 4: seven runs),
  - ubatch 62 (second sequences of each slot at ~15K),
  - the last ubatch (only the tail of the staggered slots).
The sample holds each run's first and last token and the tokens on both sides of
every 128-token boundary (the tensor-core tile edges), so every tile edge of the
planner's near-equal split is covered.  After the last ubatch the whole pool is
compared bit for bit with the pool the oracle's append builds.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import workloads
from tests._gpu import assert_attn_close

pytestmark = pytest.mark.gpu

CHECK = (0, 30, 32, 62, 64)


def runs_of(tok_seq):
    """(start, length) of each maximal span of consecutive tokens of one sequence."""
    cut = np.flatnonzero(np.diff(tok_seq)) + 1
    starts = np.concatenate([[0], cut])
    ends = np.concatenate([cut, [len(tok_seq)]])
    return list(zip(starts.tolist(), (ends - starts).tolist()))


def sample_tokens(tok_seq):
    sel = set()
    for a, n in runs_of(tok_seq):
        sel |= {a, a + n - 1}
        for b in range(128, n, 128):          # 128-token boundaries from the run start
            sel |= {a + b - 1, a + b}
        nt = -(-n // 128)                     # near-equal split of the run into tiles
        for i in range(1, nt):
            b = n * i // nt
            sel |= {a + b - 1, a + b}
    return np.array(sorted(sel), np.int32)


def test_prefill_8x16k_schedule_matches_oracle():
    import paged_kv_cache_pages_gb300 as pa
    wl = workloads.Prefill8x16K(0)
    assert len(wl.ubatches) == 65
    assert len(runs_of(wl.ubatches[32][0])) == 7   # the k -> k + 4 crossing ubatch
    dev = "cuda"
    spt = torch.from_numpy(wl.seq_page_table).to(dev)
    kp = torch.full((wl.num_pages, wl.Hkv, wl.P, wl.d), float("nan"), dtype=torch.float16,
                    device=dev)
    vp = torch.full_like(kp, float("nan"))
    Tmax = max(ts.shape[0] for ts, _ in wl.ubatches)
    ws = pa.new_workspace(Tmax, wl.Hq, wl.Hkv, wl.d, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    got = {}
    for u in range(len(wl.ubatches)):
        ts, tp, q, k, v = wl.ubatch(u)
        f16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).to(dev)  # noqa
        tpt, kv, slot = pa.expand_ubatch(spt, torch.from_numpy(ts).to(dev),
                                         torch.from_numpy(tp).to(dev), wl.P, err=err)
        pa.kv_append(f16(k), f16(v), slot, kp, vp, err=err)
        out = pa.forward(f16(q), kp, vp, tpt, kv, wl.scale, workspace=ws)
        if u in CHECK:
            sel = sample_tokens(ts)
            got[u] = (sel, out[torch.from_numpy(sel).long().to(dev)].float().cpu().numpy())
            assert pa.read_error(ws) == 0, f"device error word set in ubatch {u}"
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    kf, vf = wl.pool_final()
    assert np.array_equal(kp.cpu().numpy().view(np.uint16), kf)
    assert np.array_equal(vp.cpu().numpy().view(np.uint16), vf)

    for u in CHECK:
        ts, tp, q, _, _ = wl.ubatch(u)
        tpt, kv, _ = oracle.expand_ubatch(wl.seq_page_table, ts, tp, wl.P)
        sel, g = got[u]
        ref = oracle.paged_attention(q, kf, vf, tpt, kv, wl.scale, tokens=sel)
        assert_attn_close(g, ref, f"8x16K ubatch {u} ({len(sel)} tokens x {wl.Hq} heads)")


def test_prefill_8x16k_schedule_over_fp8_pages_matches_oracle():
    """The same 65 ubatches over FP8 pages: each through expand -> quantising append ->
    forward_fp8 (plan + tensor-core prefill over widened codes + split-KV decode).  The
    final FP8 pool is compared bit for bit with the oracle's quantising append of every
    row; the checked ubatches' sampled tokens x all heads with the oracle's attention over
    the dequantised codes."""
    import paged_kv_cache_pages_gb300 as pa
    wl = workloads.Prefill8x16K(0)
    dev = "cuda"
    spt = torch.from_numpy(wl.seq_page_table).to(dev)
    nan_codes = lambda shape: np.full(shape, 0x7F, np.uint8)  # noqa: E731
    N, Hkv, P, d = wl.num_pages, wl.Hkv, wl.P, wl.d
    host = [nan_codes((N, Hkv, P, d)), nan_codes((N, Hkv, d, P)),
            np.full((N, Hkv, P), np.nan, np.float32), np.full((N, Hkv, P), np.nan, np.float32)]
    pool = [torch.from_numpy(x).to(dev) for x in host]
    Tmax = max(ts.shape[0] for ts, _ in wl.ubatches)
    ws = pa.new_workspace(Tmax, wl.Hq, Hkv, d, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    got = {}
    for u in range(len(wl.ubatches)):
        ts, tp, q, k, v = wl.ubatch(u)
        f16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).to(dev)  # noqa
        tpt, kv, slot = pa.expand_ubatch(spt, torch.from_numpy(ts).to(dev),
                                         torch.from_numpy(tp).to(dev), P, err=err)
        pa.kv_append_fp8(f16(k), f16(v), slot, *pool, err=err)
        out = pa.forward_fp8(f16(q), *pool, tpt, kv, wl.scale, workspace=ws)
        if u in CHECK:
            sel = sample_tokens(ts)
            got[u] = (sel, out[torch.from_numpy(sel).long().to(dev)].float().cpu().numpy())
            assert pa.read_error(ws) == 0, f"device error word set in ubatch {u}"
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    # the oracle's quantising append of every row of the 8 sequences
    K, V = wl._draw_kv()
    pos = np.arange(wl.seq_len)
    slots = np.concatenate([wl.seq_page_table[s][pos // P].astype(np.int64) * P + pos % P
                            for s in range(wl.n_seq)])
    oracle.kv_append_fp8(K.reshape(-1, Hkv, d), V.reshape(-1, Hkv, d), slots, *host)
    for g_, h_ in zip(pool, host):
        assert np.array_equal(g_.cpu().numpy().view(np.uint8), h_.view(np.uint8))

    for u in CHECK:
        ts, tp, q, _, _ = wl.ubatch(u)
        tpt, kv, _ = oracle.expand_ubatch(wl.seq_page_table, ts, tp, P)
        sel, g = got[u]
        ref = oracle.paged_attention_fp8(q, *host, tpt, kv, wl.scale, tokens=sel)
        assert_attn_close(g, ref, f"8x16K FP8 ubatch {u} ({len(sel)} tokens x {wl.Hq} heads)")
