"""Helpers of the GPU parity tests: run a workloads.Case through the C-ABI
(via the Python binding) and through the CPU oracle, and compare."""
import numpy as np
import torch

import oracle

ATOL, RTOL = 2e-3, 1e-2   # |gpu - ref| <= ATOL + RTOL * |ref|, elementwise


def f16_dev(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.float16)).to(dev)


def i32_dev(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def assert_attn_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                           f"max abs err {err.max():.3e}")
    return float(err.max())


class GpuCase:
    """A Case on the device after expand + append."""

    def __init__(self, pa, case, dev="cuda"):
        self.case = case
        self.spt = i32_dev(case.seq_page_table(), dev)
        self.tok_seq = i32_dev(case.tok_seq, dev)
        self.tok_pos = i32_dev(case.tok_pos, dev)
        self.kp = f16_dev(case.k_pool, dev)
        self.vp = f16_dev(case.v_pool, dev)
        self.q = f16_dev(case.q, dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.tpt, self.kv, self.slot = pa.expand_ubatch(self.spt, self.tok_seq, self.tok_pos,
                                                        case.P, err=self.err)
        pa.kv_append(f16_dev(case.k_new, dev), f16_dev(case.v_new, dev), self.slot, self.kp,
                     self.vp, err=self.err)
        self.ws = pa.new_workspace(case.T, case.Hq, case.Hkv, case.d, dev)

    def forward(self, pa):
        out = pa.forward(self.q, self.kp, self.vp, self.tpt, self.kv, self.case.scale,
                         workspace=self.ws)
        torch.cuda.synchronize()
        return out


def oracle_case(case, tokens=None):
    """Oracle expand + append + attention.  Returns (out, tpt, kv, slot, kp, vp)."""
    tpt, kv, slot = oracle.expand_ubatch(case.seq_page_table(), case.tok_seq, case.tok_pos,
                                         case.P)
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    oracle.kv_append(case.k_new, case.v_new, slot, kp, vp)
    out = oracle.paged_attention(case.q, kp, vp, tpt, kv, case.scale, tokens)
    return out, tpt, kv, slot, kp, vp
