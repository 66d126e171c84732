"""The no-allocation entry point, called through the C-ABI.

paged_attn_forward_noalloc serves callers that cannot allocate device memory
(a host framework owning all device memory, a fixed memory budget, or a
latency-critical path).  It must give the same output as paged_attn_forward
with an allocated workspace, and match the fp64 oracle, on two calls in a row
(the second call finds the first call's leftovers in the shared scratch); a
call with a bad page id must stay harmless (the bad access is skipped) and leave
the next call correct; and a ubatch too large for its fixed 64 MiB scratch is
rejected.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads
from tests._gpu import GpuCase, assert_attn_close, oracle_case

pytestmark = pytest.mark.gpu


def _noalloc(lib):
    fn = lib.paged_attn_forward_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, i, vp, i, i, i, i, i, i, ctypes.c_float, vp, vp]
    fn.restype = i
    return fn


def _call(fn, g, out, tpt=None):
    c = g.case
    tpt = g.tpt if tpt is None else tpt
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return fn(p(g.q), p(g.kp), p(g.vp), p(tpt), tpt.shape[1], p(g.kv), c.T, c.Hq, c.Hkv, c.P,
              c.d, c.num_pages, c.scale, p(out),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_forward_on_two_calls_in_a_row():
    import paged_kv_cache_pages_gb300 as pa
    fn = _noalloc(pa.lib())
    cases = [workloads.small_prefill(21, P=128, d=128, Hq=8, Hkv=2),
             workloads.decode(3)]
    for case in cases:
        g = GpuCase(pa, case)
        ref = g.forward(pa).float().cpu().numpy()
        assert pa.read_error(g.ws) == 0
        out = torch.full_like(g.q, float("nan"))
        assert _call(fn, g, out) == pa.PA_OK
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert_attn_close(got, ref, f"noalloc {case.name} vs forward")
        assert_attn_close(got, oracle_case(case)[0], f"noalloc {case.name} vs oracle")


def test_noalloc_bad_page_id_is_harmless_and_next_call_is_correct():
    import paged_kv_cache_pages_gb300 as pa
    fn = _noalloc(pa.lib())
    case = workloads.small_prefill(22, P=16, d=64, Hq=4, Hkv=2)
    g = GpuCase(pa, case)
    torch.cuda.synchronize()
    bad = g.tpt.clone()
    bad[0, 0] = case.num_pages + 5
    out = torch.zeros_like(g.q)
    assert _call(fn, g, out, tpt=bad) == pa.PA_OK    # host checks pass; the access is skipped
    torch.cuda.synchronize()
    out = torch.full_like(g.q, float("nan"))
    assert _call(fn, g, out) == pa.PA_OK
    torch.cuda.synchronize()
    assert_attn_close(out.float().cpu().numpy(), g.forward(pa).float().cpu().numpy(),
                      "noalloc after a bad call")


def test_noalloc_rejects_ubatch_beyond_its_scratch():
    import paged_kv_cache_pages_gb300 as pa
    fn = _noalloc(pa.lib())
    T, Hq, Hkv, d = 8192, 32, 8, 128
    assert pa.workspace_size(T, Hq, Hkv, d) > (64 << 20)
    q = torch.zeros((T, Hq, d), dtype=torch.float16, device="cuda")
    kp = torch.zeros((4, Hkv, 128, d), dtype=torch.float16, device="cuda")
    tpt = torch.zeros((T, 1), dtype=torch.int32, device="cuda")
    kv = torch.ones(T, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = fn(p(q), p(kp), p(kp), p(tpt), 1, p(kv), T, Hq, Hkv, 128, d, 4, 0.1, p(q), None)
    assert st == pa.PA_EWORKSPACE
