"""Decode with the append fused into the same launch (paged_attn_decode_append): the
pool after the call must equal the oracle's append bit for bit (NaN payloads of every
other cell included), and the attention must match the oracle; a slot other than the
token's last key is flagged and not written."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
import workloads
from tests._gpu import assert_attn_close, f16_dev, i32_dev, oracle_case

pytestmark = pytest.mark.gpu


def one_token_per_sequence(seed, P, d, Hq, Hkv, n_seq=12):
    rng = np.random.default_rng(seed + 6000)
    lens = rng.integers(1, 700, size=n_seq, endpoint=True)
    return workloads.build_case(f"decode_P{P}_d{d}", seed, lens,
                                [(s, int(L) - 1) for s, L in enumerate(lens)],
                                P=P, Hq=Hq, Hkv=Hkv, d=d, free_frac=0.3)


def run_fused(pa, case, slot_override=None):
    dev = "cuda"
    kp, vp = f16_dev(case.k_pool), f16_dev(case.v_pool)
    tpt, kv, slot = pa.expand_ubatch(i32_dev(case.seq_page_table()), i32_dev(case.tok_seq),
                                     i32_dev(case.tok_pos), case.P)
    if slot_override is not None:
        slot = slot_override(slot)
    q = f16_dev(case.q)
    out = torch.full_like(q, float("nan"))
    ws = pa.new_workspace(case.T, case.Hq, case.Hkv, case.d, dev)
    pa.plan(tpt, kv, case.Hq, case.Hkv, case.P, case.d, ws)
    pa.decode_append(q, f16_dev(case.k_new), f16_dev(case.v_new), slot, kp, vp, tpt, kv,
                     case.scale, out, ws)
    torch.cuda.synchronize()
    return out, kp, vp, ws


@pytest.mark.parametrize("make", [
    lambda: workloads.decode(0),
    lambda: one_token_per_sequence(1, P=16, d=64, Hq=4, Hkv=2),
    lambda: one_token_per_sequence(2, P=64, d=128, Hq=8, Hkv=1),
    lambda: one_token_per_sequence(3, P=128, d=128, Hq=8, Hkv=8)],
    ids=["decode", "P16_d64", "P64_G8", "P128_G1"])
def test_fused_append_matches_oracle(make):
    import paged_kv_cache_pages_gb300 as pa
    case = make()
    out, kp, vp, ws = run_fused(pa, case)
    assert pa.read_error(ws) == 0
    ref, _, _, _, rk, rv = oracle_case(case)
    assert np.array_equal(kp.cpu().numpy().view(np.uint16), rk)
    assert np.array_equal(vp.cpu().numpy().view(np.uint16), rv)
    assert_attn_close(out.float().cpu().numpy(), ref, f"decode_append {case.name}")


def test_fused_append_long_tail_sampled():
    import paged_kv_cache_pages_gb300 as pa
    case = workloads.longtail(0)
    out, kp, vp, ws = run_fused(pa, case)
    assert pa.read_error(ws) == 0
    toks = [0, 9, int(np.argmax(case.seq_len)), int(np.argmin(case.seq_len)), case.T - 1]
    ref, _, _, _, rk, rv = oracle_case(case, tokens=toks)
    assert np.array_equal(kp.cpu().numpy().view(np.uint16), rk)
    assert_attn_close(out.float().cpu().numpy()[toks], ref, "decode_append long tail")


def test_fused_append_flags_a_slot_that_is_not_the_last_key():
    import paged_kv_cache_pages_gb300 as pa
    case = workloads.decode(2)

    def bad(slot):
        s = slot.clone()
        s[3] = s[3] - 1          # the key before the token's own
        s[5] = -1                # a padding token: skipped, not flagged
        return s
    out, kp, vp, ws = run_fused(pa, case, slot_override=bad)
    assert pa.read_error(ws) == pa.PA_ERR_SLOT_RANGE
    # every row except tokens 3 and 5 is written; those two cells keep the pool's NaN
    _, tpt, kv, slot, rk, _ = oracle_case(case, tokens=[0])
    got = kp.cpu().numpy().view(np.uint16)
    for t in range(case.T):
        page, off = divmod(int(slot[t]), case.P)
        cell = got[page, :, off]
        if t in (3, 5):
            assert np.all(cell == 0x7E00)
        else:
            assert np.array_equal(cell, rk[page, :, off])
