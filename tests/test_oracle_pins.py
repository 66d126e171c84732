"""Pins of the CPU fp64 oracle to things other than itself (no GPU).

* binary16 decoding vs numpy's float16 (library routine), all 65536 patterns;
* hand-derived closed-form cases (tests/golden/closed_form.json);
* brute-force unpaged attention from each sequence's contiguous K/V, written
  here with numpy, on the tiny workload and random small cases;
* torch scaled_dot_product_attention in float64 on one contiguous sequence;
* invariants: physical page permutation, NaN in free / tail cells, constant V,
  kv_len = 1, q = 0, shared prefix pages vs private copies;
* sensitivity: plausible mistakes (K/V swapped, wrong GQA mapping, another
  sequence's table, an off-by-one kv_len) must fail the brute-force pin.
"""
import math

import numpy as np
import pytest

import workloads
from tests import _golden


def f64(bits):
    return bits.view(np.float16).astype(np.float64)


def oracle_after_append(orc, case, q=None, tokens=None):
    """expand + append + attention through the oracle for a workloads.Case."""
    tpt, kv, slot = orc.expand_ubatch(case.seq_page_table(), case.tok_seq, case.tok_pos, case.P)
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    orc.kv_append(case.k_new, case.v_new, slot, kp, vp)
    out = orc.paged_attention(case.q if q is None else q, kp, vp, tpt, kv, case.scale, tokens)
    return out, (tpt, kv, slot, kp, vp)


def brute_force(case, q=None):
    """Unpaged attention from the contiguous per-sequence K/V (before paging)."""
    q = case.q if q is None else q
    G = case.Hq // case.Hkv
    out = np.zeros((case.T, case.Hq, case.d))
    for t in range(case.T):
        s, p = int(case.tok_seq[t]), int(case.tok_pos[t])
        if s < 0:
            continue
        K = f64(case.k_ctx[s][:p + 1])          # [L][Hkv][d]
        V = f64(case.v_ctx[s][:p + 1])
        for h in range(case.Hq):
            sc = case.scale * (K[:, h // G, :] @ f64(q[t, h]))
            w = np.exp(sc - sc.max())
            w /= w.sum()
            out[t, h] = w @ V[:, h // G, :]
    return out


# --------------------------------------------------------------------------- f16

def test_f16_decode_matches_numpy_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# --------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("case", _golden.load_cases(), ids=lambda c: c["name"])
def test_closed_form_cases(oracle_mod, case):
    g = _golden.materialise(case)
    tpt, kv, slot = oracle_mod.expand_ubatch(g["seq_page_table"], g["tok_seq"], g["tok_pos"], g["P"])
    out = oracle_mod.paged_attention(g["q"], g["k_pages"], g["v_pages"], tpt, kv, g["scale"])
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out, g["expected"], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- brute force

def test_tiny_matches_brute_force(oracle_mod):
    case = workloads.tiny(0)
    out, (tpt, kv, slot, kp, vp) = oracle_after_append(oracle_mod, case)
    assert list(kv) == [33, 34, 35, 36, 37, 98, 99, 100]
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out, brute_force(case), rtol=0, atol=1e-12)


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("P,d,Hq,Hkv", [(16, 64, 4, 2), (128, 128, 8, 2), (16, 128, 6, 3)])
def test_random_mixed_matches_brute_force(oracle_mod, seed, P, d, Hq, Hkv):
    case = workloads.small_prefill(seed, P=P, d=d, Hq=Hq, Hkv=Hkv,
                                   chunks=((0, 40, 37), (1, 0, 21), (2, 150, 3)), extra_decode=3)
    out, _ = oracle_after_append(oracle_mod, case)
    np.testing.assert_allclose(out, brute_force(case), rtol=0, atol=1e-12)


def test_sdpa_fp64_single_sequence(oracle_mod):
    torch = pytest.importorskip("torch")
    L, P, Hq, Hkv, d = 70, 16, 4, 2, 64
    case = workloads.build_case("sdpa", 11, [L], [(0, p) for p in range(L)], P, Hq, Hkv, d)
    out, _ = oracle_after_append(oracle_mod, case)
    G = Hq // Hkv
    q = torch.from_numpy(f64(case.q)).permute(1, 0, 2)                       # [Hq][L][d]
    k = torch.from_numpy(f64(case.k_ctx[0])).permute(1, 0, 2).repeat_interleave(G, 0)
    v = torch.from_numpy(f64(case.v_ctx[0])).permute(1, 0, 2).repeat_interleave(G, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                           scale=case.scale)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- invariants

def test_page_permutation_invariance(oracle_mod):
    case = workloads.small_prefill(5, P=16, d=64, Hq=4, Hkv=2)
    out, (tpt, kv, slot, kp, vp) = oracle_after_append(oracle_mod, case)
    rng = np.random.default_rng(99)
    perm = rng.permutation(case.num_pages).astype(np.int32)   # old id -> new id
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    tpt2 = np.where(tpt >= 0, perm[np.maximum(tpt, 0)], -1).astype(np.int32)
    out2 = oracle_mod.paged_attention(case.q, kp2, vp2, tpt2, kv, case.scale)
    assert np.array_equal(out, out2)


def test_nan_free_cells_never_reach_output(oracle_mod):
    case = workloads.tiny(0)
    nan_cells = np.isnan(case.k_pool.view(np.float16)).sum()
    assert nan_cells > 0
    out, _ = oracle_after_append(oracle_mod, case)
    assert np.all(np.isfinite(out))


def test_constant_v_gives_v(oracle_mod):
    case = workloads.tiny(3)
    c = np.float16(0.7109375).view(np.uint16)   # exact in binary16
    for arr in [case.v_new, *case.v_ctx]:
        arr[...] = c
    valid = ~np.isnan(case.v_pool.view(np.float16))
    case.v_pool[valid] = c
    out, _ = oracle_after_append(oracle_mod, case)
    np.testing.assert_allclose(out, 0.7109375, rtol=0, atol=1e-13)


def test_kv_len_one_gives_first_value(oracle_mod):
    case = workloads.build_case("kv1", 4, [1, 1, 1], [(0, 0), (1, 0), (2, 0)], 16, 4, 2, 64)
    out, _ = oracle_after_append(oracle_mod, case)
    for t in range(3):
        for h in range(4):
            assert np.array_equal(out[t, h], f64(case.v_ctx[t][0, h // 2]))


def test_zero_q_gives_mean_of_valid_values(oracle_mod):
    case = workloads.small_prefill(6, P=16, d=64, Hq=4, Hkv=2)
    q0 = np.zeros_like(case.q)
    out, _ = oracle_after_append(oracle_mod, case, q=q0)
    for t in range(case.T):
        s, p = int(case.tok_seq[t]), int(case.tok_pos[t])
        mean = f64(case.v_ctx[s][:p + 1]).mean(axis=0)            # [Hkv][d]
        np.testing.assert_allclose(out[t], np.repeat(mean, 2, axis=0), rtol=0, atol=1e-12)


def test_shared_prefix_pages_equal_private_copies(oracle_mod):
    pref = 64
    lens = [pref + 20, pref + 37, pref + 5]
    toks = [(0, pref + 19), (1, pref + 30), (1, pref + 31), (2, pref + 4)]
    shared = workloads.build_case("sh", 8, lens, toks, 16, 4, 2, 64, shared_prefix_tokens=pref)
    assert all(np.array_equal(shared.seq_pages[0][:4], p[:4]) for p in shared.seq_pages)
    out_sh, (tpt, kv, slot, kp, vp) = oracle_after_append(oracle_mod, shared)
    # private copies: give every sequence but the first its own copy of the prefix pages
    n_extra = 4 * (len(lens) - 1)
    N = shared.num_pages + n_extra
    kp2 = np.full((N,) + kp.shape[1:], np.uint16(0x7E00), np.uint16)
    vp2 = kp2.copy()
    kp2[:shared.num_pages] = kp
    vp2[:shared.num_pages] = vp
    spt = shared.seq_page_table()
    nxt = shared.num_pages
    for s in range(1, len(lens)):
        for i in range(4):
            kp2[nxt] = kp[spt[s, i]]
            vp2[nxt] = vp[spt[s, i]]
            spt[s, i] = nxt
            nxt += 1
    tpt2 = spt[shared.tok_seq]
    out_priv = oracle_mod.paged_attention(shared.q, kp2, vp2, tpt2, kv, shared.scale)
    assert np.array_equal(out_sh, out_priv)
    np.testing.assert_allclose(out_sh, brute_force(shared), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- expand + append

def test_append_reproduces_generator_layout(oracle_mod):
    """expand + append of the ubatch rows must give exactly the pool the generator
    lays out when it writes every position (its own layout code, not the oracle's)."""
    for case in (workloads.tiny(0), workloads.small_prefill(2, P=16, d=64, Hq=4, Hkv=2)):
        _, (tpt, kv, slot, kp, vp) = oracle_after_append(oracle_mod, case)
        full_k = np.full_like(case.k_pool, np.uint16(0x7E00))
        full_v = full_k.copy()
        for s, L in enumerate(case.seq_len):
            workloads._fill_pool(full_k, case.seq_pages[s], case.k_ctx[s], case.P, int(L))
            workloads._fill_pool(full_v, case.seq_pages[s], case.v_ctx[s], case.P, int(L))
        assert np.array_equal(kp, full_k) and np.array_equal(vp, full_v)
        assert np.array_equal(kv, case.tok_pos + 1)


def test_expand_padding_and_unallocated(oracle_mod):
    spt = np.array([[5, 2, -1], [7, -1, -1]], np.int32)
    tpt, kv, slot = oracle_mod.expand_ubatch(spt, [0, -1, 1, 0], [17, 0, 3, 40], 16)
    assert list(kv) == [18, 0, 4, 41]
    assert list(slot) == [2 * 16 + 1, -1, 7 * 16 + 3, -1]
    assert np.array_equal(tpt[1], [-1, -1, -1])
    assert np.array_equal(tpt[3], spt[0])
    with pytest.raises(ValueError):
        oracle_mod.expand_ubatch(spt, [2], [0], 16)


def test_append_skips_negative_slots(oracle_mod):
    kp = np.zeros((2, 1, 4, 8), np.uint16)
    vp = np.zeros_like(kp)
    k = np.arange(3 * 8, dtype=np.uint16).reshape(3, 1, 8) + 1
    v = k + 100
    oracle_mod.kv_append(k, v, np.array([5, -1, 0], np.int64), kp, vp)
    assert np.array_equal(kp[1, 0, 1], k[0, 0]) and np.array_equal(kp[0, 0, 0], k[2, 0])
    assert np.count_nonzero(kp) == 16 and np.array_equal(vp[1, 0, 1], v[0, 0])
    with pytest.raises(ValueError):
        oracle_mod.kv_append(k[:1], v[:1], np.array([8], np.int64), kp, vp)


# --------------------------------------------------------------------------- sensitivity

def test_pins_detect_plausible_mistakes(oracle_mod):
    """Feeding the oracle a plausibly wrong input (the effect of a dropped term,
    swapped operand or wrong index) must break the brute-force pin."""
    case = workloads.small_prefill(7, P=16, d=64, Hq=4, Hkv=2)
    ref = brute_force(case)
    tpt, kv, slot = oracle_mod.expand_ubatch(case.seq_page_table(), case.tok_seq, case.tok_pos, case.P)
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    oracle_mod.kv_append(case.k_new, case.v_new, slot, kp, vp)

    def off(*args):
        try:
            out = oracle_mod.paged_attention(*args)
        except ValueError:
            return True                      # rejected: also a detection
        return np.nanmax(np.abs(out - ref)) > 1e-3 or not np.all(np.isfinite(out))

    assert not off(case.q, kp, vp, tpt, kv, case.scale)
    # K and V swapped
    assert off(case.q, vp, kp, tpt, kv, case.scale)
    # GQA interleaved instead of contiguous: swap KV heads in the pool
    assert off(case.q, kp[:, ::-1].copy(), vp[:, ::-1].copy(), tpt, kv, case.scale)
    # kv_len off by one (position instead of position + 1)
    assert off(case.q, kp, vp, tpt, np.maximum(kv - 1, 1), case.scale)
    # another sequence's table row
    assert off(case.q, kp, vp, np.roll(tpt, 1, axis=0), kv, case.scale)
    # scale dropped
    assert off(case.q, kp, vp, tpt, kv, 1.0)
