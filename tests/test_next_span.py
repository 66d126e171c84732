"""Unified-span baseline (UA-PagedAttention page, section 作品简介: the original
cache is one span of cells shared by every sequence; attention reads the whole
span under a mask).  The oracle's masked attention is pinned to the paged
definition (the mask keeps exactly a token's own cells) and to a numpy brute
force; on the GPU the masked decode kernel (split-KV) and the masked prefill
kernel (tcgen05 tiles) are checked against it."""
import numpy as np
import pytest

import oracle
import workloads
from tests._gpu import ATOL, RTOL


def paged_ref(case, tokens=None):
    tpt, kv, slot = oracle.expand_ubatch(case.seq_page_table(), case.tok_seq, case.tok_pos, case.P)
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    oracle.kv_append(case.k_new, case.v_new, slot, kp, vp)
    return oracle.paged_attention(case.q, kp, vp, tpt, kv, case.scale, tokens), kp, vp


def brute_masked(q, kp, vp, tpt, kv, scale, cs, cp, ts, tp):
    """numpy: every slot of the token's row, mask, softmax (float64)."""
    T, Hq, d = q.shape
    N, Hkv, P, _ = kp.shape
    G = Hq // Hkv
    qf = q.view(np.float16).astype(np.float64)
    kf = kp.view(np.float16).astype(np.float64)
    vf = vp.view(np.float16).astype(np.float64)
    out = np.zeros((T, Hq, d))
    for t in range(T):
        j = np.arange(kv[t])
        pages = tpt[t][j // P]
        slots = pages * P + j % P
        keep = (cs[slots] == ts[t]) & (cp[slots] <= tp[t])
        if not keep.any():
            continue
        pk, rk = pages[keep], (j % P)[keep]
        for h in range(Hq):
            K = kf[pk, h // G, rk]
            V = vf[pk, h // G, rk]
            s = scale * (K @ qf[t, h])
            w = np.exp(s - s.max())
            out[t, h] = (w / w.sum()) @ V
    return out


@pytest.mark.parametrize("make", [workloads.tiny, workloads.decode])
def test_masked_oracle_equals_paged_oracle_on_the_span_view(make):
    case = make(0)
    ref, kp, vp = paged_ref(case)
    tpt, kv, cs, cp, ts, tp = workloads.span_view(case)
    got = oracle.masked_attention(case.q, kp, vp, tpt, kv, case.scale, cs, cp, ts, tp)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_masked_oracle_matches_numpy_brute_force():
    rng = np.random.default_rng(11)
    N, Hkv, P, d, Hq, T = 6, 2, 16, 32, 4, 5
    kp = workloads.randn_f16(rng, (N, Hkv, P, d))
    vp = workloads.randn_f16(rng, (N, Hkv, P, d))
    q = workloads.randn_f16(rng, (T, Hq, d))
    cs = rng.integers(-1, 3, N * P).astype(np.int32)   # cells of 3 sequences, some free
    cp = rng.integers(0, 60, N * P).astype(np.int32)
    ts = rng.integers(0, 3, T).astype(np.int32)
    tp = rng.integers(20, 60, T).astype(np.int32)
    tpt = np.stack([rng.permutation(N) for _ in range(T)]).astype(np.int32)
    kv = rng.integers(P, N * P + 1, T).astype(np.int32)
    got = oracle.masked_attention(q, kp, vp, tpt, kv, 0.2, cs, cp, ts, tp)
    np.testing.assert_allclose(got, brute_masked(q, kp, vp, tpt, kv, 0.2, cs, cp, ts, tp),
                               rtol=1e-12, atol=1e-12)


def test_masked_oracle_position_bound_matters_and_empty_mask_is_zero():
    case = workloads.tiny(0)
    ref, kp, vp = paged_ref(case)
    tpt, kv, cs, cp, ts, tp = workloads.span_view(case)
    # sensitivity: without the position bound the tokens see their sequence's later cells
    late = oracle.masked_attention(case.q, kp, vp, tpt, kv, case.scale, cs, cp, ts,
                                   np.full_like(tp, 1 << 30))
    assert not np.allclose(late, ref)
    # a token of a sequence that owns no cell keeps nothing: zero row
    ts2 = ts.copy()
    ts2[0] = 7
    got = oracle.masked_attention(case.q, kp, vp, tpt, kv, case.scale, cs, cp, ts2, tp)
    assert np.all(got[0] == 0.0) and np.allclose(got[1:], ref[1:], rtol=1e-12, atol=1e-12)


def test_span_view_refuses_shared_pages():
    with pytest.raises(ValueError):
        workloads.span_view(workloads.shared_prefix(0))


# ------------------------------------------------------------------ GPU

@pytest.fixture(scope="module")
def pa():
    torch = pytest.importorskip("torch")
    import paged_kv_cache_pages_gb300 as m
    assert torch.cuda.is_available()
    return m


def run_masked(pa, case, kp, vp, kind="decode", view=None):
    """The masked kernel of `kind` (decode: split-KV, prefill: tcgen05 tiles) on the
    span view of the case (or on the given tables)."""
    import torch
    tpt, kv, cs, cp, ts, tp = workloads.span_view(case) if view is None else view
    dev = "cuda"
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    T = tpt.shape[0]
    out = torch.full((T, case.Hq, case.d), float("nan"), dtype=torch.float16, device=dev)
    ws = pa.new_workspace(T, case.Hq, case.Hkv, case.d, dev)
    plan = pa.plan_decode if kind == "decode" else pa.plan_prefill
    run = pa.masked_decode if kind == "decode" else pa.masked_prefill
    plan(t(tpt), t(kv), case.Hq, case.Hkv, case.P, case.d, ws)
    run(t(case.q.view(np.float16)), t(kp.view(np.float16)), t(vp.view(np.float16)),
        t(tpt), t(kv), case.scale, t(cs), t(cp), t(ts), t(tp), out, ws)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    return out.float().cpu().numpy(), (tpt, kv, cs, cp, ts, tp)


@pytest.mark.gpu
@pytest.mark.parametrize("make", [workloads.tiny, workloads.decode])
def test_masked_decode_matches_oracle(pa, make):
    from tests._gpu import assert_attn_close
    case = make(0)
    ref, kp, vp = paged_ref(case)
    got, (tpt, kv, cs, cp, ts, tp) = run_masked(pa, case, kp, vp)
    mref = oracle.masked_attention(case.q, kp, vp, tpt, kv, case.scale, cs, cp, ts, tp)
    assert_attn_close(got, mref, f"masked {case.name}")
    assert_attn_close(got, ref, f"masked vs paged {case.name}")


@pytest.mark.gpu
def test_masked_decode_long_tail_sampled(pa):
    """64 sequences up to 32K keys: every token streams the whole 0.9 GB span."""
    from tests._gpu import assert_attn_close
    case = workloads.longtail(0)
    tpt0, kv0, slot = oracle.expand_ubatch(case.seq_page_table(), case.tok_seq, case.tok_pos,
                                           case.P)
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    oracle.kv_append(case.k_new, case.v_new, slot, kp, vp)
    got, _ = run_masked(pa, case, kp, vp)
    toks = np.array([0, 9, int(np.argmax(case.seq_len)), int(np.argmin(case.seq_len))], np.int32)
    ref = oracle.paged_attention(case.q, kp, vp, tpt0, kv0, case.scale, toks)
    assert_attn_close(got[toks], ref, "masked long tail")


@pytest.mark.gpu
def test_masked_decode_padding_token_gets_zero_row(pa):
    case = workloads.tiny(0)
    case.tok_seq = case.tok_seq.copy()
    case.tok_seq[3] = -1  # a padding token: kv_len 0 in the span view, zero output
    _, kp, vp = paged_ref(workloads.tiny(0))
    got, (tpt, kv, cs, cp, ts, tp) = run_masked(pa, case, kp, vp)
    assert kv[3] == 0 and np.all(got[3] == 0.0)
    mref = oracle.masked_attention(case.q, kp, vp, tpt, kv, case.scale, cs, cp, ts, tp)
    from tests._gpu import assert_attn_close
    assert_attn_close(got, mref, "masked with padding")


@pytest.mark.gpu
@pytest.mark.parametrize("make", [
    workloads.tiny, workloads.decode,
    lambda s: workloads.small_prefill(s, P=128, d=128, Hq=8, Hkv=2),
    lambda s: workloads.small_prefill(s, P=16, d=64, Hq=4, Hkv=2),
    lambda s: workloads.small_prefill(s, P=64, d=128, Hq=4, Hkv=4)],
    ids=["tiny", "decode", "prefill_P128_d128", "prefill_P16_d64", "prefill_G1"])
def test_masked_prefill_matches_oracle(pa, make):
    """The unified-span baseline on the tcgen05 tiles: tiles of 128 consecutive tokens of
    any sequences, each streaming the whole span (free cells hold NaN)."""
    from tests._gpu import assert_attn_close
    case = make(0)
    ref, kp, vp = paged_ref(case)
    got, (tpt, kv, cs, cp, ts, tp) = run_masked(pa, case, kp, vp, kind="prefill")
    mref = oracle.masked_attention(case.q, kp, vp, tpt, kv, case.scale, cs, cp, ts, tp)
    assert_attn_close(got, mref, f"masked prefill {case.name}")
    assert_attn_close(got, ref, f"masked prefill vs paged {case.name}")


@pytest.mark.gpu
def test_masked_prefill_random_cells(pa):
    """Random cell owners and positions (three sequences, free cells holding NaN), random
    rows and lengths: against the oracle and the numpy brute force."""
    from tests._gpu import assert_attn_close
    rng = np.random.default_rng(12)
    N, Hkv, P, d, Hq, T = 24, 2, 16, 64, 4, 150
    case = workloads.tiny(0)
    case.Hq, case.Hkv, case.P, case.d, case.scale = Hq, Hkv, P, d, 0.125
    kp = workloads.randn_f16(rng, (N, Hkv, P, d))
    vp = workloads.randn_f16(rng, (N, Hkv, P, d))
    case.q = workloads.randn_f16(rng, (T, Hq, d))
    cs = rng.integers(-1, 3, N * P).astype(np.int32)
    cp = rng.integers(0, 300, N * P).astype(np.int32)
    free = np.flatnonzero(cs < 0)
    kp[free // P, :, free % P, :] = 0x7E00
    vp[free // P, :, free % P, :] = 0x7E00
    ts = rng.integers(0, 3, T).astype(np.int32)
    tp = rng.integers(100, 300, T).astype(np.int32)
    row = rng.permutation(N).astype(np.int32)
    tpt = np.tile(row, (T, 1))        # one row for all: tiles of 128 mixed tokens
    kv = np.full(T, N * P, np.int32)
    kv[:7] = rng.integers(1, N * P, 7)  # ...and a few short ones
    got, _ = run_masked(pa, case, kp, vp, kind="prefill", view=(tpt, kv, cs, cp, ts, tp))
    mref = oracle.masked_attention(case.q, kp, vp, tpt, kv, case.scale, cs, cp, ts, tp)
    assert_attn_close(got, mref, "masked prefill, random cells")
    assert_attn_close(got, brute_masked(case.q, kp, vp, tpt, kv, case.scale, cs, cp, ts, tp),
                      "masked prefill vs brute force")


@pytest.mark.gpu
def test_masked_prefill_8x16k_ubatch_sampled(pa):
    """One late ubatch of the 8 x 16K schedule over the span of the whole 1280-page pool:
    every tile streams the pool (the baseline the page's TTFT claim is measured against)."""
    from tests._gpu import assert_attn_close
    wl = workloads.Prefill8x16K(0)
    u = 40
    ts, tp, q, _, _ = wl.ubatch(u)
    kf, vf = wl.pool_final()
    N, P = wl.num_pages, wl.P
    cs = np.full(N * P, -1, np.int32)
    cp = np.full(N * P, -1, np.int32)
    for s_ in range(wl.n_seq):
        pos = np.arange(wl.seq_len)
        slots = wl.seq_page_table[s_][pos // P].astype(np.int64) * P + pos % P
        cs[slots], cp[slots] = s_, pos
    T = ts.shape[0]
    tpt = np.tile(np.arange(N, dtype=np.int32), (T, 1))
    kv = np.full(T, N * P, np.int32)

    class C:  # the shape fields run_masked reads
        Hq, Hkv, d, scale = wl.Hq, wl.Hkv, wl.d, wl.scale
    C.P, C.q = P, q
    got, _ = run_masked(pa, C, kf, vf, kind="prefill", view=(tpt, kv, cs, cp, ts, tp))
    sel = np.array([0, 127, 128, 700, 1300, T - 1], np.int32)
    tpt_p, kv_p, _ = oracle.expand_ubatch(wl.seq_page_table, ts, tp, P)
    ref = oracle.paged_attention(q, kf, vf, tpt_p, kv_p, wl.scale, tokens=sel)
    assert_attn_close(got[sel], ref, "masked prefill 8x16K ubatch vs paged oracle")
