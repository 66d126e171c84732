"""Page copy for copy-on-write forks (CacheFlow page, section 核心架构 2 and 3):
the oracle's page copy pinned against numpy indexing, the host fork logic, and
(GPU) the copy kernel bit-exact against the oracle plus a fork -> copy -> append
-> attention scenario checked against the oracle."""
import numpy as np
import pytest

import oracle
import workloads

NAN16 = np.uint16(0x7E00)


def random_pool(rng, N=24, Hkv=2, P=16, d=64):
    k = workloads.randn_f16(rng, (N, Hkv, P, d))
    v = workloads.randn_f16(rng, (N, Hkv, P, d))
    k[rng.random(N) < 0.2] = NAN16  # some pages hold NaN payloads: copied as bits
    return k, v


def copy_pairs(rng, N, n):
    ids = rng.permutation(N)
    return ids[:n].astype(np.int32), ids[n:2 * n].astype(np.int32)


# ------------------------------------------------------------------ oracle pins

def test_oracle_copy_matches_numpy_indexing():
    rng = np.random.default_rng(5)
    k, v = random_pool(rng)
    src, dst = copy_pairs(rng, k.shape[0], 7)
    ek, ev = k.copy(), v.copy()
    ek[dst] = k[src]
    ev[dst] = v[src]
    assert oracle.copy_pages(src, dst, k, v) == 0
    assert np.array_equal(k, ek) and np.array_equal(v, ev)


def test_oracle_copy_skips_out_of_range_pairs():
    rng = np.random.default_rng(6)
    k, v = random_pool(rng)
    N = k.shape[0]
    k0, v0 = k.copy(), v.copy()
    src = np.array([3, -1, 4, 5], np.int32)
    dst = np.array([N, 7, 8, 9], np.int32)
    assert oracle.copy_pages(src, dst, k, v) == 2
    ek, ev = k0.copy(), v0.copy()
    ek[[8, 9]] = k0[[4, 5]]
    ev[[8, 9]] = v0[[4, 5]]
    assert np.array_equal(k, ek) and np.array_equal(v, ev)


def test_oracle_copy_touches_only_destinations_and_both_pools():
    # sensitivity: a copy that forgot V, or wrote a neighbour page, fails here
    rng = np.random.default_rng(7)
    k, v = random_pool(rng)
    k0, v0 = k.copy(), v.copy()
    src, dst = np.array([2], np.int32), np.array([11], np.int32)
    oracle.copy_pages(src, dst, k, v)
    changed_k = np.where((k != k0).reshape(k.shape[0], -1).any(1))[0]
    changed_v = np.where((v != v0).reshape(v.shape[0], -1).any(1))[0]
    assert changed_k.tolist() == [11] and changed_v.tolist() == [11]
    assert np.array_equal(k[11], k0[2]) and np.array_equal(v[11], v0[2])


# ------------------------------------------------------------------ host fork

@pytest.fixture(scope="module")
def pa_host():
    torch = pytest.importorskip("torch")  # noqa: F841  (the binding imports torch)
    import paged_kv_cache_pages_gb300 as m
    return m


def test_fork_shares_full_pages_and_copies_the_partial_one(pa_host):
    pool = pa_host.PagePool(8)
    parent = pool.alloc(3)
    child, pair = pool.fork(parent, 2 * 16 + 5, 16)
    assert child[:2] == parent[:2] and child[2] not in parent
    assert pair == (parent[2], child[2])
    assert [pool.refcount(p) for p in parent] == [2, 2, 1]
    assert pool.refcount(child[2]) == 1 and pool.num_free == 4


def test_fork_of_whole_pages_copies_nothing(pa_host):
    pool = pa_host.PagePool(4)
    parent = pool.alloc(2)
    child, pair = pool.fork(parent, 32, 16)
    assert child == parent and pair is None
    assert [pool.refcount(p) for p in parent] == [2, 2] and pool.num_free == 2
    pool.release(parent)  # the parent finishes: the child keeps the pages
    assert [pool.refcount(p) for p in child] == [1, 1] and pool.num_free == 2


def test_fork_without_a_free_page_changes_nothing(pa_host):
    pool = pa_host.PagePool(2)
    parent = pool.alloc(2)
    with pytest.raises(pa_host.PagedAttnError):
        pool.fork(parent, 20, 16)
    assert [pool.refcount(p) for p in parent] == [1, 1] and pool.num_free == 0


def test_fork_of_a_free_page_is_rejected(pa_host):
    pool = pa_host.PagePool(4)
    with pytest.raises(pa_host.PagedAttnError):
        pool.fork([0], 5, 16)
    assert pool.num_free == 4


# ------------------------------------------------------------------ GPU

@pytest.fixture(scope="module")
def pa():
    torch = pytest.importorskip("torch")
    import paged_kv_cache_pages_gb300 as m
    assert torch.cuda.is_available()
    return m


@pytest.mark.gpu
@pytest.mark.parametrize("Hkv,P,d", [(2, 16, 64), (8, 128, 128), (1, 32, 64)])
def test_copy_pages_bit_exact(pa, Hkv, P, d):
    import torch
    rng = np.random.default_rng(100 + P)
    k, v = random_pool(rng, N=40, Hkv=Hkv, P=P, d=d)
    src, dst = copy_pairs(rng, 40, 12)
    src[3], dst[5] = -2, 40  # two invalid pairs: skipped and flagged
    kd = torch.from_numpy(k.view(np.float16)).cuda()
    vd = torch.from_numpy(v.view(np.float16)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.copy_pages(torch.from_numpy(src).cuda(), torch.from_numpy(dst).cuda(), kd, vd, err=err)
    torch.cuda.synchronize()
    assert oracle.copy_pages(src, dst, k, v) == 2
    assert np.array_equal(kd.cpu().numpy().view(np.uint16), k)
    assert np.array_equal(vd.cpu().numpy().view(np.uint16), v)
    assert int(err.item()) & pa.PA_ERR_PAGE_RANGE


@pytest.mark.gpu
def test_fork_copy_append_attention(pa):
    """A parent with a partly filled last page is forked; parent and child then
    each append a different next token into their own last page.  Both tokens'
    attention must match the oracle run on the same operations, and the child's
    write must not reach the parent."""
    import torch
    from tests._gpu import assert_attn_close
    rng = np.random.default_rng(42)
    N, Hkv, P, d, Hq = 16, 2, 16, 64, 4
    L = 37  # 2 full pages + 5 rows
    pool = pa.PagePool(N)
    parent = pool.alloc(3)
    k = np.full((N, Hkv, P, d), NAN16, np.uint16)
    v = np.full((N, Hkv, P, d), NAN16, np.uint16)
    kk = workloads.randn_f16(rng, (L, Hkv, d))
    vv = workloads.randn_f16(rng, (L, Hkv, d))
    for pos in range(L):
        k[parent[pos // P], :, pos % P] = kk[pos]
        v[parent[pos // P], :, pos % P] = vv[pos]
    child, pair = pool.fork(parent, L, P)
    assert pair is not None
    # the next token of each sequence (position L), appended after the copy
    k_new = workloads.randn_f16(rng, (2, Hkv, d))
    v_new = workloads.randn_f16(rng, (2, Hkv, d))
    q = workloads.randn_f16(rng, (2, Hq, d))
    seq_pt = np.full((2, 4), -1, np.int32)
    seq_pt[0, :3], seq_pt[1, :3] = parent, child
    tok_seq = np.array([0, 1], np.int32)
    tok_pos = np.array([L, L], np.int32)
    scale = 1.0 / np.sqrt(d)

    # oracle: copy, expand, append, attention
    ok_, ov_ = k.copy(), v.copy()
    oracle.copy_pages(np.array([pair[0]], np.int32), np.array([pair[1]], np.int32), ok_, ov_)
    tpt, kv, slot = oracle.expand_ubatch(seq_pt, tok_seq, tok_pos, P)
    oracle.kv_append(k_new, v_new, slot, ok_, ov_)
    ref = oracle.paged_attention(q, ok_, ov_, tpt, kv, scale)

    # GPU through the C ABI
    dev = "cuda"
    kd = torch.from_numpy(k.view(np.float16)).to(dev)
    vd = torch.from_numpy(v.view(np.float16)).to(dev)
    pa.copy_pages(torch.tensor([pair[0]], dtype=torch.int32, device=dev),
                  torch.tensor([pair[1]], dtype=torch.int32, device=dev), kd, vd)
    tpt_d, kv_d, slot_d = pa.expand_ubatch(torch.from_numpy(seq_pt).to(dev),
                                           torch.from_numpy(tok_seq).to(dev),
                                           torch.from_numpy(tok_pos).to(dev), P)
    pa.kv_append(torch.from_numpy(k_new.view(np.float16)).to(dev),
                 torch.from_numpy(v_new.view(np.float16)).to(dev), slot_d, kd, vd)
    out = pa.forward(torch.from_numpy(q.view(np.float16)).to(dev), kd, vd, tpt_d, kv_d, scale)
    torch.cuda.synchronize()
    assert np.array_equal(kd.cpu().numpy().view(np.uint16), ok_)
    assert np.array_equal(vd.cpu().numpy().view(np.uint16), ov_)
    assert_attn_close(out.float().cpu().numpy(), ref, "fork")
    # the two sequences share their first 37 keys and differ only in the last one
    assert not np.allclose(ref[0], ref[1])


@pytest.mark.gpu
def test_copy_pages_of_nothing_is_a_no_op(pa):
    import torch
    k = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device="cuda")
    v = torch.zeros_like(k)
    e = torch.empty(0, dtype=torch.int32, device="cuda")
    pa.copy_pages(e, e, k, v)
    torch.cuda.synchronize()
    assert not k.any() and not v.any()
