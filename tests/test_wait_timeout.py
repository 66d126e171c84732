"""The bounded-wait timeout path of the split-KV decode kernel, made to run on purpose
without faulting or hanging anything: a 1 us wait limit makes the combining warp's
wait for its first job (and other waits on another role's arrival) give up.  The call
must return, the workspace error word must carry PA_ERR_TIMEOUT, and the next plan +
decode at the default limit must match the oracle (the context stays usable).

The kernel's roles agree on where to stop: the consumers abandon only stages the
producer never issued, the producer lets its issued copies land before exiting, and
one thread decides for all consumers before each named barrier."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import workloads
from tests._gpu import GpuCase, assert_attn_close, oracle_case

pytestmark = pytest.mark.gpu


def test_decode_wait_timeout_is_reported_and_recoverable():
    import paged_kv_cache_pages_gb300 as pa
    case = workloads.decode(0)
    g = GpuCase(pa, case)
    ref = oracle_case(case)[0]
    out = torch.empty_like(g.q)

    def plan_and_decode():
        pa.plan_decode(g.tpt, g.kv, case.Hq, case.Hkv, case.P, case.d, g.ws)
        pa.decode(g.q, g.kp, g.vp, g.tpt, g.kv, case.scale, out, g.ws)
        torch.cuda.synchronize()

    old = pa.set_decode_wait_limit(1000)       # 1 us
    try:
        plan_and_decode()                       # returns; rows it did not finish are garbage
        err = pa.read_error(g.ws)
    finally:
        assert pa.set_decode_wait_limit(old) == 1000
    assert err & pa.PA_ERR_TIMEOUT, f"error word {err:#x}"
    assert err & ~pa.PA_ERR_TIMEOUT == 0
    # default limit again: a fresh plan, and the same call matches the oracle
    for _ in range(2):
        out.fill_(float("nan"))
        plan_and_decode()
        assert pa.read_error(g.ws) == 0
        assert_attn_close(out.float().cpu().numpy(), ref, "decode after a timed-out launch")
