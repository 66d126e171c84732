"""GPU parity: the CUDA path (through the C-ABI) against the CPU fp64 oracle.

Bit-exact for the expansion (tables, kv_len, slot mapping) and for the whole
pool after append (NaN payloads of untouched cells included); attention within
|gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads
from tests import _golden
from tests._gpu import GpuCase, assert_attn_close, f16_dev, i32_dev, oracle_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    import paged_kv_cache_pages_gb300 as m
    assert torch.cuda.is_available()
    return m


@pytest.fixture
def routing(pa):
    """Set the prefill threshold for one test, restore afterwards."""
    old = pa.set_prefill_min_run(16)
    pa.set_prefill_min_run(old)
    yield pa.set_prefill_min_run
    pa.set_prefill_min_run(old)


ALL_DECODE = 1 << 30


def check_expand_append(g, ref):
    _, tpt, kv, slot, kp, vp = ref
    assert np.array_equal(g.tpt.cpu().numpy(), tpt)
    assert np.array_equal(g.kv.cpu().numpy(), kv)
    assert np.array_equal(g.slot.cpu().numpy(), slot)
    assert np.array_equal(g.kp.cpu().numpy().view(np.uint16), kp)
    assert np.array_equal(g.vp.cpu().numpy().view(np.uint16), vp)
    assert int(g.err.item()) == 0


# ----------------------------------------------------------------- expand + append

@pytest.mark.parametrize("make", [workloads.tiny, workloads.decode, workloads.shared_prefix],
                         ids=["tiny", "decode", "shared_prefix"])
def test_expand_append_bit_exact(pa, make):
    case = make(0)
    g = GpuCase(pa, case)
    torch.cuda.synchronize()
    check_expand_append(g, oracle_case(case, tokens=[0]))


def test_expand_padding_and_errors(pa):
    spt = i32_dev(np.array([[5, 2, -1], [7, -1, -1]]))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tpt, kv, slot = pa.expand_ubatch(spt, i32_dev([0, -1, 1, 0, 3]), i32_dev([17, 0, 3, 40, 0]), 16,
                                     err=err)
    torch.cuda.synchronize()
    assert kv.cpu().tolist() == [18, 0, 4, 41, 0]
    assert slot.cpu().tolist() == [33, -1, 115, -1, -1]
    assert tpt[1].cpu().tolist() == [-1, -1, -1] and tpt[4].cpu().tolist() == [-1, -1, -1]
    assert int(err.item()) == pa.PA_ERR_SEQ_RANGE


def test_append_out_of_range_slot_is_skipped(pa):
    kp = torch.zeros((2, 1, 16, 64), dtype=torch.float16, device="cuda")
    vp = torch.zeros_like(kp)
    k = torch.ones((3, 1, 64), dtype=torch.float16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slot = torch.tensor([3, 32, -1], dtype=torch.int64, device="cuda")
    pa.kv_append(k, k * 2, slot, kp, vp, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == pa.PA_ERR_SLOT_RANGE
    assert float(kp.sum()) == 64.0 and float(vp.sum()) == 128.0
    assert float(kp[0, 0, 3].sum()) == 64.0


# ----------------------------------------------------------------- attention

def run_and_compare(pa, case, tokens=None, what=""):
    g = GpuCase(pa, case)
    out = g.forward(pa)
    assert pa.read_error(g.ws) == 0
    ref = oracle_case(case, tokens)
    check_expand_append(g, ref)
    got = out.float().cpu().numpy()
    if tokens is not None:
        got = got[np.asarray(tokens)]
    return assert_attn_close(got, ref[0], what or case.name)


@pytest.mark.parametrize("mode", ["default", "all_decode", "all_prefill"])
def test_tiny(pa, routing, mode):
    routing({"default": 16, "all_decode": ALL_DECODE, "all_prefill": 1}[mode])
    run_and_compare(pa, workloads.tiny(0))


@pytest.mark.parametrize("mode", ["default", "all_prefill"])
def test_decode_config(pa, routing, mode):
    routing({"default": 16, "all_prefill": 1}[mode])
    run_and_compare(pa, workloads.decode(0))


def test_longtail_config(pa):
    case = workloads.longtail(0)
    rng = np.random.default_rng(1)
    toks = sorted(set(rng.choice(case.T, 16, replace=False).tolist()) |
                  {int(np.argmax(case.seq_len)), int(np.argmin(case.seq_len))})
    run_and_compare(pa, case, tokens=toks)


def test_shared_prefix_config(pa):
    case = workloads.shared_prefix(0)
    decode_toks = list(range(12))
    rng = np.random.default_rng(2)
    pre = rng.choice(np.arange(12, case.T), 24, replace=False).tolist()
    run_and_compare(pa, case, tokens=decode_toks + sorted(pre) + [case.T - 1])


@pytest.mark.parametrize("P,d,Hq,Hkv", [(128, 128, 8, 2), (16, 64, 4, 2), (16, 128, 8, 1),
                                        (64, 128, 16, 2), (32, 64, 8, 8), (128, 64, 4, 4)])
@pytest.mark.parametrize("mode", ["default", "all_decode", "all_prefill"])
def test_small_mixed(pa, routing, P, d, Hq, Hkv, mode):
    routing({"default": 16, "all_decode": ALL_DECODE, "all_prefill": 1}[mode])
    case = workloads.small_prefill(3, P=P, d=d, Hq=Hq, Hkv=Hkv)
    run_and_compare(pa, case)


@pytest.mark.parametrize("gcase", _golden.load_cases(), ids=lambda c: c["name"])
@pytest.mark.parametrize("mode", ["all_decode", "all_prefill"])
def test_closed_form_on_gpu(pa, routing, gcase, mode):
    routing({"all_decode": ALL_DECODE, "all_prefill": 1}[mode])
    g = _golden.materialise(gcase)
    tpt, kv, slot = pa.expand_ubatch(i32_dev(g["seq_page_table"]), i32_dev(g["tok_seq"]),
                                     i32_dev(g["tok_pos"]), g["P"])
    out = pa.forward(f16_dev(g["q"]), f16_dev(g["k_pages"]), f16_dev(g["v_pages"]), tpt, kv,
                     g["scale"])
    torch.cuda.synchronize()
    assert_attn_close(out.float().cpu().numpy(), g["expected"], gcase["name"])


# ----------------------------------------------------------------- edge cases

def test_empty_ubatch_is_a_no_op(pa):
    q = torch.empty((0, 4, 64), dtype=torch.float16, device="cuda")
    kp = torch.zeros((2, 2, 16, 64), dtype=torch.float16, device="cuda")
    tpt = torch.empty((0, 3), dtype=torch.int32, device="cuda")
    kv = torch.empty((0,), dtype=torch.int32, device="cuda")
    out = pa.forward(q, kp, kp, tpt, kv, 0.125)
    assert out.shape == (0, 4, 64)


def test_zero_kv_len_rows_are_zero(pa):
    case = workloads.small_prefill(4, P=16, d=64, Hq=4, Hkv=2, chunks=((0, 0, 20),),
                                   extra_decode=2)
    g = GpuCase(pa, case)
    kv0 = g.kv.clone()
    kv0[3] = 0
    kv0[-1] = 0
    out = pa.forward(g.q, g.kp, g.vp, g.tpt, kv0, case.scale, workspace=g.ws)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    assert np.all(o[3] == 0) and np.all(o[-1] == 0)
    assert pa.read_error(g.ws) == 0


def test_max_length_sequence(pa, routing):
    """A 32768-token sequence (the long-tail clip) decoding and prefilling a tail."""
    L = 32768
    toks = [(0, L - 1)] + [(1, p) for p in range(L - 130, L)]
    case = workloads.build_case("maxlen", 12, [L, L], toks, 128, 8, 2, 128, free_frac=0.1)
    for mode in (16, ALL_DECODE):
        routing(mode)
        run_and_compare(pa, case, tokens=[0, 1, 64, 130], what=f"maxlen min_run={mode}")


def test_bad_page_id_sets_error_without_fault(pa):
    case = workloads.small_prefill(5, P=16, d=64, Hq=4, Hkv=2)
    g = GpuCase(pa, case)
    torch.cuda.synchronize()
    tpt = g.tpt.clone()
    tpt[0, 0] = case.num_pages + 5
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.validate(tpt, g.kv, case.P, case.num_pages, err)
    pa.forward(g.q, g.kp, g.vp, tpt, g.kv, case.scale, workspace=g.ws)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_ERR_PAGE_RANGE
    assert pa.read_error(g.ws) & pa.PA_ERR_PAGE_RANGE
    # the context is still usable
    out = g.forward(pa)
    assert pa.read_error(g.ws) == 0 and torch.isfinite(out.float()).all()


def test_repeat_is_bitwise_deterministic(pa):
    g = GpuCase(pa, workloads.decode(1))
    a = g.forward(pa).clone()
    b = g.forward(pa)
    assert torch.equal(a, b)


def test_plan_once_run_many(pa):
    """One plan, several runs (one per layer) on different pools."""
    case = workloads.small_prefill(8, P=128, d=128, Hq=8, Hkv=2)
    g = GpuCase(pa, case)
    pa.plan(g.tpt, g.kv, case.Hq, case.Hkv, case.P, case.d, g.ws)
    ref = oracle_case(case)[0]
    for _ in range(3):
        out = pa.run(g.q, g.kp, g.vp, g.tpt, g.kv, case.scale, workspace=g.ws)
        torch.cuda.synchronize()
        assert_attn_close(out.float().cpu().numpy(), ref, "plan once run many")
