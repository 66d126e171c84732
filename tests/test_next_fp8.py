"""FP8 (E4M3) KV pages with one scale per cached row: the oracle's codec pinned
to torch's float8_e4m3fn and to the format's special cases, the quantising append
and the dequantised attention pinned to numpy; on the GPU the quantising append is
bit-exact against the oracle and the FP8 decode matches the oracle's attention
over the same codes."""
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")


def torch_e4m3_values():
    codes = np.arange(256, dtype=np.uint8)
    return torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


# ------------------------------------------------------------------ codec pins

def test_e4m3_decode_matches_torch_for_every_code():
    ref = torch_e4m3_values()
    mine = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    assert np.array_equal(ref[~np.isnan(ref)], mine[~np.isnan(mine)])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and np.isnan(mine[0x7F])


def test_e4m3_encode_matches_torch_for_every_binary16_in_range():
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) <= 448.0)]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([oracle.f32_to_e4m3(v) for v in x], np.uint8)
    assert np.array_equal(mine, ref)


def test_e4m3_encode_saturates_and_breaks_ties_to_even():
    assert oracle.f32_to_e4m3(500.0) == 0x7E and oracle.f32_to_e4m3(-1e30) == 0xFE
    assert oracle.f32_to_e4m3(float("nan")) == 0x7F
    # 1.0 (0x38) and 1.125 (0x39): the midpoint goes to the even code
    assert oracle.f32_to_e4m3(1.0625) == 0x38
    # 1.125 (0x39) and 1.25 (0x3A): the midpoint goes to the even code 0x3A
    assert oracle.f32_to_e4m3(1.1875) == 0x3A
    # half the smallest subnormal (2^-10) rounds to zero, a hair more to 2^-9
    assert oracle.f32_to_e4m3(2.0 ** -10) == 0x00
    assert oracle.f32_to_e4m3(np.nextafter(np.float32(2.0 ** -10), np.float32(1))) == 0x01


# ------------------------------------------------------------------ append + attention pins

def fp8_pool(N, Hkv, P, d):
    return (np.zeros((N, Hkv, P, d), np.uint8), np.zeros((N, Hkv, d, P), np.uint8),
            np.ones((N, Hkv, P), np.float32), np.ones((N, Hkv, P), np.float32))


def test_quantising_append_error_bound_and_layout():
    rng = np.random.default_rng(21)
    N, Hkv, P, d, T = 4, 2, 16, 32, 9
    k = workloads.randn_f16(rng, (T, Hkv, d))
    v = workloads.randn_f16(rng, (T, Hkv, d))
    k[3] = 0  # an all-zero row: scale 1, codes 0
    slot = rng.permutation(N * P)[:T].astype(np.int64)
    k8, v8t, ks, vs = fp8_pool(N, Hkv, P, d)
    oracle.kv_append_fp8(k, v, slot, k8, v8t, ks, vs)
    val = torch_e4m3_values()
    for t in range(T):
        pg, off = divmod(int(slot[t]), P)
        for h in range(Hkv):
            for src, codes, sc in ((k, k8[pg, h, off], ks[pg, h, off]),
                                   (v, v8t[pg, h, :, off], vs[pg, h, off])):
                x = src[t, h].view(np.float16).astype(np.float64)
                amax = np.abs(x).max()
                if amax == 0:
                    assert sc == 1.0 and not codes.any()
                    continue
                assert sc == np.float32(np.float32(amax) / np.float32(448.0))
                deq = val[codes] * float(sc)
                # 3 mantissa bits: half an ulp is 1/16 of the value (normal range),
                # half the subnormal step below 2^-6 of the scaled range
                bound = np.maximum(np.abs(x) / 16.0, 2.0 ** -10 * float(sc)) * (1 + 1e-6)
                assert np.all(np.abs(deq - x) <= bound)
                assert np.max(np.abs(val[codes])) == 448.0  # the row's amax lands on 448


def test_fp8_attention_matches_numpy():
    rng = np.random.default_rng(22)
    N, Hkv, P, d, Hq, T = 5, 2, 16, 32, 4, 3
    k8 = rng.integers(0, 0x7E, (N, Hkv, P, d)).astype(np.uint8)
    k8 |= (rng.random(k8.shape) < 0.5).astype(np.uint8) << 7  # random signs
    v8t = rng.integers(0, 0x7E, (N, Hkv, d, P)).astype(np.uint8)
    ks = rng.uniform(0.001, 0.01, (N, Hkv, P)).astype(np.float32)
    vs = rng.uniform(0.001, 0.01, (N, Hkv, P)).astype(np.float32)
    q = workloads.randn_f16(rng, (T, Hq, d))
    tpt = np.stack([rng.permutation(N) for _ in range(T)]).astype(np.int32)
    kv = np.array([1, 37, N * P], np.int32)
    got = oracle.paged_attention_fp8(q, k8, v8t, ks, vs, tpt, kv, 0.3)
    val = torch_e4m3_values()
    G = Hq // Hkv
    for t in range(T):
        j = np.arange(kv[t])
        pg, off = tpt[t][j // P], j % P
        for h in range(Hq):
            g = h // G
            K = val[k8[pg, g, off]] * ks[pg, g, off][:, None].astype(np.float64)
            V = val[v8t[pg, g, :, off]] * vs[pg, g, off][:, None].astype(np.float64)
            s = 0.3 * (K @ q[t, h].view(np.float16).astype(np.float64))
            w = np.exp(s - s.max())
            np.testing.assert_allclose(got[t, h], (w / w.sum()) @ V, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ GPU

@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_pages_gb300 as m
    assert torch.cuda.is_available()
    return m


def fill_slots(case):
    """Every cached row of every sequence: (k, v rows, slots) to append."""
    ks, vs, sl = [], [], []
    for s, pages in enumerate(case.seq_pages):
        L = int(case.seq_len[s])
        pos = np.arange(L)
        sl.append(np.asarray(pages, np.int64)[pos // case.P] * case.P + pos % case.P)
        ks.append(case.k_ctx[s][:L])
        vs.append(case.v_ctx[s][:L])
    return np.concatenate(ks), np.concatenate(vs), np.concatenate(sl)


@pytest.mark.gpu
def test_append_fp8_bit_exact(pa):
    rng = np.random.default_rng(31)
    N, Hkv, P, d, T = 40, 8, 128, 128, 300
    k = workloads.randn_f16(rng, (T, Hkv, d))
    v = workloads.randn_f16(rng, (T, Hkv, d))
    k[5] = 0
    v[7, 3] = np.float16(200.0).view(np.uint16)  # a large row: the scale moves
    slot = rng.permutation(N * P)[:T].astype(np.int64)
    slot[11] = -1  # padding token: skipped
    ref = fp8_pool(N, Hkv, P, d)
    oracle.kv_append_fp8(k, v, slot, *ref)
    dev = "cuda"
    pool = pa.new_fp8_pool(N, Hkv, P, d, dev)
    pa.kv_append_fp8(torch.from_numpy(k.view(np.float16)).to(dev),
                     torch.from_numpy(v.view(np.float16)).to(dev),
                     torch.from_numpy(slot).to(dev), *pool)
    torch.cuda.synchronize()
    for got, want in zip(pool, ref):
        assert np.array_equal(got.cpu().numpy(), want)


@pytest.mark.gpu
@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (64, 8)])
def test_decode_fp8_matches_oracle(pa, Hq, Hkv):
    from tests._gpu import assert_attn_close
    rng = np.random.default_rng(40 + Hq)
    lens = rng.integers(100, 3000, 6)
    case = workloads.build_case("fp8", 3, lens, [(s, int(L) - 1) for s, L in enumerate(lens)],
                                P=128, Hq=Hq, Hkv=Hkv, d=128)
    k, v, slot = fill_slots(case)
    N = case.num_pages
    ref = fp8_pool(N, Hkv, 128, 128)
    oracle.kv_append_fp8(k, v, slot, *ref)
    tpt, kv, _ = oracle.expand_ubatch(case.seq_page_table(), case.tok_seq, case.tok_pos, 128)
    want = oracle.paged_attention_fp8(case.q, *ref, tpt, kv, case.scale)
    dev = "cuda"
    pool = pa.new_fp8_pool(N, Hkv, 128, 128, dev)
    pa.kv_append_fp8(torch.from_numpy(k.view(np.float16)).to(dev),
                     torch.from_numpy(v.view(np.float16)).to(dev),
                     torch.from_numpy(slot).to(dev), *pool)
    q = torch.from_numpy(case.q.view(np.float16)).to(dev)
    out = torch.empty_like(q)
    ws = pa.new_workspace(case.T, Hq, Hkv, 128, dev)
    tpt_d, kv_d = torch.from_numpy(tpt).to(dev), torch.from_numpy(kv).to(dev)
    pa.plan_decode(tpt_d, kv_d, Hq, Hkv, 128, 128, ws)
    pa.decode_fp8(q, *pool, tpt_d, kv_d, case.scale, out, ws)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    assert_attn_close(out.float().cpu().numpy(), want, f"fp8 G={Hq // Hkv}")


def _fp8_setup(pa, seed=50, Hq=32, Hkv=8):
    rng = np.random.default_rng(seed)
    lens = rng.integers(100, 2000, 4)
    case = workloads.build_case("fp8e", seed, lens, [(s, int(L) - 1) for s, L in enumerate(lens)],
                                P=128, Hq=Hq, Hkv=Hkv, d=128)
    k, v, slot = fill_slots(case)
    dev = "cuda"
    pool = pa.new_fp8_pool(case.num_pages, Hkv, 128, 128, dev)
    pa.kv_append_fp8(torch.from_numpy(k.view(np.float16)).to(dev),
                     torch.from_numpy(v.view(np.float16)).to(dev),
                     torch.from_numpy(slot).to(dev), *pool)
    tpt, kv, _ = oracle.expand_ubatch(case.seq_page_table(), case.tok_seq, case.tok_pos, 128)
    return case, pool, tpt, kv


def _fp8_run(pa, case, pool, tpt, kv):
    dev = "cuda"
    q = torch.from_numpy(case.q.view(np.float16)).to(dev)
    out = torch.full_like(q, float("nan"))
    ws = pa.new_workspace(case.T, case.Hq, case.Hkv, 128, dev)
    tpt_d, kv_d = torch.from_numpy(tpt).to(dev), torch.from_numpy(kv).to(dev)
    pa.plan_decode(tpt_d, kv_d, case.Hq, case.Hkv, 128, 128, ws)
    pa.decode_fp8(q, *pool, tpt_d, kv_d, case.scale, out, ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), pa.read_error(ws)


@pytest.mark.gpu
def test_decode_fp8_bad_page_and_empty_rows(pa):
    case, pool, tpt, kv = _fp8_setup(pa)
    tpt = tpt.copy()
    kv = kv.copy()
    tpt[1, 0] = case.num_pages + 3  # out of the pool: flagged, that block skipped, no fault
    kv[2] = 0                       # no key: a zero row
    out, err = _fp8_run(pa, case, pool, tpt, kv)
    assert err & pa.PA_ERR_PAGE_RANGE
    assert np.all(out[2] == 0.0)
    # the context stays usable and the untouched tokens are right
    tpt2, kv2 = _fp8_setup(pa)[2:]
    out2, err2 = _fp8_run(pa, case, pool, tpt2, kv2)
    assert err2 == 0 and np.all(np.isfinite(out2))


@pytest.mark.gpu
def test_decode_fp8_is_bitwise_deterministic(pa):
    case, pool, tpt, kv = _fp8_setup(pa, seed=51)
    a, _ = _fp8_run(pa, case, pool, tpt, kv)
    b, _ = _fp8_run(pa, case, pool, tpt, kv)
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ GPU: prefill tiles over FP8

def nan_fp8_pool(N, Hkv, P=128, d=128):
    """A pool whose unwritten cells hold NaN codes (0x7F) and NaN scales: only the
    cells below a token's kv_len may reach its output."""
    return (np.full((N, Hkv, P, d), 0x7F, np.uint8), np.full((N, Hkv, d, P), 0x7F, np.uint8),
            np.full((N, Hkv, P), np.nan, np.float32), np.full((N, Hkv, P), np.nan, np.float32))


def unique_rows(case):
    """Every cached row once (pages shared by several sequences are written once)."""
    filled = np.zeros(case.num_pages * case.P, bool)
    ks, vs, sl = [], [], []
    for s, pages in enumerate(case.seq_pages):
        L = int(case.seq_len[s])
        pos = np.arange(L)
        slots = np.asarray(pages, np.int64)[pos // case.P] * case.P + pos % case.P
        new = ~filled[slots]
        filled[slots] = True
        sl.append(slots[new])
        ks.append(case.k_ctx[s][:L][new])
        vs.append(case.v_ctx[s][:L][new])
    return np.concatenate(ks), np.concatenate(vs), np.concatenate(sl)


def fp8_on_gpu(pa, case):
    """Quantise every cached row into a NaN-filled FP8 pool, on the host (oracle) and on
    the device (checked bit-exact); returns (oracle pool, device pool, tpt, kv)."""
    k, v, slot = unique_rows(case)
    ref = nan_fp8_pool(case.num_pages, case.Hkv)
    oracle.kv_append_fp8(k, v, slot, *ref)
    dev = "cuda"
    pool = [torch.from_numpy(x).to(dev) for x in nan_fp8_pool(case.num_pages, case.Hkv)]
    pa.kv_append_fp8(torch.from_numpy(k.view(np.float16)).to(dev),
                     torch.from_numpy(v.view(np.float16)).to(dev),
                     torch.from_numpy(slot).to(dev), *pool)
    torch.cuda.synchronize()
    for got, want in zip(pool, ref):
        assert np.array_equal(got.cpu().numpy().view(np.uint8), want.view(np.uint8))
    tpt, kv, _ = oracle.expand_ubatch(case.seq_page_table(), case.tok_seq, case.tok_pos, case.P)
    return ref, pool, tpt, kv


def run_forward_fp8(pa, case, pool, tpt, kv, min_run=16):
    dev = "cuda"
    old = pa.set_prefill_min_run(min_run)
    try:
        q = torch.from_numpy(case.q.view(np.float16)).to(dev)
        out = torch.full_like(q, float("nan"))
        ws = pa.new_workspace(case.T, case.Hq, case.Hkv, 128, dev)
        pa.forward_fp8(q, *pool, torch.from_numpy(tpt).to(dev), torch.from_numpy(kv).to(dev),
                       case.scale, out=out, workspace=ws)
        torch.cuda.synchronize()
        return out.float().cpu().numpy(), pa.read_error(ws)
    finally:
        pa.set_prefill_min_run(old)


def tiny128(seed=0):
    """The tiny workload's sequences and tokens (lengths 37 and 100; tokens 32..36 of
    the first, 97..99 of the second) at the page size and head dimension FP8 pages
    support (128, 128)."""
    tokens = [(0, p) for p in range(32, 37)] + [(1, p) for p in range(97, 100)]
    return workloads.build_case("tiny128", seed, [37, 100], tokens, P=128, Hq=4, Hkv=2, d=128,
                                num_pages=8, scale=1.0 / np.sqrt(128.0))


@pytest.mark.gpu
@pytest.mark.parametrize("min_run", [1, 16, 1 << 30], ids=["all_prefill", "default", "all_decode"])
def test_forward_fp8_tiny(pa, min_run):
    from tests._gpu import assert_attn_close
    case = tiny128(0)
    ref, pool, tpt, kv = fp8_on_gpu(pa, case)
    want = oracle.paged_attention_fp8(case.q, *ref, tpt, kv, case.scale)
    got, err = run_forward_fp8(pa, case, pool, tpt, kv, min_run)
    assert err == 0
    assert_attn_close(got, want, "fp8 tiny128")


@pytest.mark.gpu
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (32, 8), (8, 8), (16, 8), (64, 8)])
@pytest.mark.parametrize("min_run", [1, 16], ids=["all_prefill", "default"])
def test_forward_fp8_small_mixed(pa, Hq, Hkv, min_run):
    from tests._gpu import assert_attn_close
    case = workloads.small_prefill(5, P=128, d=128, Hq=Hq, Hkv=Hkv)
    ref, pool, tpt, kv = fp8_on_gpu(pa, case)
    want = oracle.paged_attention_fp8(case.q, *ref, tpt, kv, case.scale)
    got, err = run_forward_fp8(pa, case, pool, tpt, kv, min_run)
    assert err == 0
    assert_attn_close(got, want, f"fp8 small mixed {Hq}/{Hkv}")


@pytest.mark.gpu
def test_forward_fp8_long_chunks_split_items(pa):
    """Chunks of several key blocks: items are cut across CTAs (stream-K parts,
    combined by the last one) and tiles end on ragged key counts."""
    from tests._gpu import assert_attn_close
    case = workloads.small_prefill(6, P=128, d=128, Hq=32, Hkv=8,
                                   chunks=((0, 2000, 700), (1, 0, 300), (2, 5000, 129)),
                                   extra_decode=3)
    ref, pool, tpt, kv = fp8_on_gpu(pa, case)
    rng = np.random.default_rng(7)
    toks = sorted(set(rng.choice(case.T, 96, replace=False).tolist()) | {0, case.T - 1})
    want = oracle.paged_attention_fp8(case.q, *ref, tpt, kv, case.scale, tokens=toks)
    got, err = run_forward_fp8(pa, case, pool, tpt, kv, 16)
    assert err == 0
    assert np.all(np.isfinite(got))
    assert_attn_close(got[toks], want, "fp8 long chunks")


@pytest.mark.gpu
def test_forward_fp8_shared_prefix(pa):
    from tests._gpu import assert_attn_close
    case = workloads.shared_prefix(0)
    ref, pool, tpt, kv = fp8_on_gpu(pa, case)
    rng = np.random.default_rng(2)
    pre = rng.choice(np.arange(12, case.T), 24, replace=False).tolist()
    toks = list(range(12)) + sorted(pre) + [case.T - 1]
    want = oracle.paged_attention_fp8(case.q, *ref, tpt, kv, case.scale, tokens=toks)
    got, err = run_forward_fp8(pa, case, pool, tpt, kv, 16)
    assert err == 0
    assert np.all(np.isfinite(got))
    assert_attn_close(got[toks], want, "fp8 shared prefix")


@pytest.mark.gpu
def test_prefill_fp8_bad_page_and_repeat(pa):
    case = workloads.small_prefill(8, P=128, d=128, Hq=8, Hkv=2)
    ref, pool, tpt, kv = fp8_on_gpu(pa, case)
    a, err_a = run_forward_fp8(pa, case, pool, tpt, kv, 1)
    b, err_b = run_forward_fp8(pa, case, pool, tpt, kv, 1)
    assert err_a == 0 and err_b == 0
    assert np.array_equal(a, b)  # bitwise deterministic
    bad = tpt.copy()
    bad[0, 0] = case.num_pages + 5  # a prefill tile's first page is out of the pool
    c, err_c = run_forward_fp8(pa, case, pool, bad, kv, 1)
    assert err_c & pa.PA_ERR_PAGE_RANGE
    # the context stays usable
    d_, err_d = run_forward_fp8(pa, case, pool, tpt, kv, 1)
    assert err_d == 0 and np.array_equal(a, d_)


@pytest.mark.gpu
def test_prefill_fp8_refuses_other_shapes(pa):
    case = workloads.tiny(0)  # page size 16, d 64
    dev = "cuda"
    N = case.num_pages
    pool = [torch.from_numpy(x).to(dev) for x in nan_fp8_pool(N, case.Hkv, case.P, case.d)]
    tpt, kv, _ = oracle.expand_ubatch(case.seq_page_table(), case.tok_seq, case.tok_pos, case.P)
    q = torch.from_numpy(case.q.view(np.float16)).to(dev)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.forward_fp8(q, *pool, torch.from_numpy(tpt).to(dev), torch.from_numpy(kv).to(dev),
                       case.scale)
    assert e.value.status == pa.PA_EUNSUPPORTED


@pytest.mark.gpu
def test_prefill_fp8_and_decode_fp8_split_a_mixed_plan(pa):
    """prefill_fp8 and decode_fp8 on one mixed plan write disjoint tokens: together
    they give forward_fp8's output bit for bit."""
    case = workloads.small_prefill(9, P=128, d=128, Hq=32, Hkv=8)
    ref, pool, tpt, kv = fp8_on_gpu(pa, case)
    full, err = run_forward_fp8(pa, case, pool, tpt, kv, 16)
    assert err == 0
    dev = "cuda"
    q = torch.from_numpy(case.q.view(np.float16)).to(dev)
    out = torch.full_like(q, float("nan"))
    ws = pa.new_workspace(case.T, case.Hq, case.Hkv, 128, dev)
    tpt_d, kv_d = torch.from_numpy(tpt).to(dev), torch.from_numpy(kv).to(dev)
    old = pa.set_prefill_min_run(16)
    try:
        pa.plan(tpt_d, kv_d, case.Hq, case.Hkv, 128, 128, ws)
    finally:
        pa.set_prefill_min_run(old)
    pa.prefill_fp8(q, *pool, tpt_d, kv_d, case.scale, out, ws)
    part = out.float().cpu().numpy()
    pf_rows = ~np.isnan(part).any(axis=(1, 2))
    assert pf_rows.any() and not pf_rows.all()  # both paths have tokens
    pa.decode_fp8(q, *pool, tpt_d, kv_d, case.scale, out, ws)
    torch.cuda.synchronize()
    assert pa.read_error(ws) == 0
    both = out.float().cpu().numpy()
    assert np.array_equal(both, full)


@pytest.mark.gpu
def test_forward_fp8_zero_kv_rows_and_empty_ubatch(pa):
    """kv_len 0 gives zero rows on both paths (a whole prefill tile of them too), and an
    empty ubatch is a no-op."""
    from tests._gpu import assert_attn_close
    case = workloads.small_prefill(10, P=128, d=128, Hq=32, Hkv=8,
                                   chunks=((0, 300, 181), (1, 0, 130)), extra_decode=3)
    ref, pool, tpt, kv = fp8_on_gpu(pa, case)
    kv = kv.copy()
    zero = np.r_[np.arange(181, 181 + 130), case.T - 1]  # the second run, a decode token
    kv[zero] = 0
    want = oracle.paged_attention_fp8(case.q, *ref, tpt, kv, case.scale)
    assert np.all(want[zero] == 0.0)
    got, err = run_forward_fp8(pa, case, pool, tpt, kv, 16)
    assert err == 0
    assert np.all(got[zero] == 0.0)
    assert_attn_close(got, want, "fp8 zero kv rows")
    dev = "cuda"
    q0 = torch.empty((0, case.Hq, 128), dtype=torch.float16, device=dev)
    t0 = torch.empty((0, tpt.shape[1]), dtype=torch.int32, device=dev)
    k0 = torch.empty((0,), dtype=torch.int32, device=dev)
    out = pa.forward_fp8(q0, *pool, t0, k0, case.scale,
                         workspace=pa.new_workspace(1, case.Hq, case.Hkv, 128, dev))
    assert out.shape == (0, case.Hq, 128)
