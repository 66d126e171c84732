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
