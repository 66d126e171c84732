"""Python binding of libpagedattn.so: ubatch-aligned paged attention on GB300.

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are torch CUDA tensors (float16 for K/V/Q/out, int32 tables, int64
slot mapping); the current torch stream is passed to each call.  The library
must have been built (``paged_kv_cache_pages_gb300.build.build()`` or
``__graft_entry__.build()``); importing without it raises ImportError -- there
is no fallback.

Entry points mirror include/paged_attn.h:
  expand_ubatch   per-token page-table / kv_len expansion + slot mapping
  kv_append       reshape-and-cache into the paged pool
  copy_pages      page copy of a copy-on-write fork
  masked_decode / masked_prefill   the unified-span baseline (masked attention over a
                  shared span) on the split-KV and on the tcgen05 path
  kv_append_fp8 / decode_fp8 / prefill_fp8 / forward_fp8   FP8 (E4M3) KV pages with
                  per-row scales
  plan / prefill / decode / run / forward   the attention itself
  validate, read_error, set_prefill_min_run, workspace_size
  PagePool        host page allocator with reference-counted sharing
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpagedattn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python paged_kv_cache_pages_gb300/build.py` (needs nvcc)")

_lib = ctypes.CDLL(LIB_PATH)

PA_OK, PA_EINVAL, PA_EUNSUPPORTED, PA_EWORKSPACE = 0, -1, -2, -3
PA_ELAUNCH, PA_EDEVICE, PA_EALIGN, PA_ENOSPACE = -4, -5, -6, -7
PA_ERR_PAGE_RANGE, PA_ERR_KV_RANGE, PA_ERR_SLOT_RANGE = 0x1, 0x2, 0x4
PA_ERR_TIMEOUT, PA_ERR_SEQ_RANGE = 0x8, 0x10

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

_ATTN_ARGS = [_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp]
_SIGS = {
    "paged_attn_strerror": ([_i], ctypes.c_char_p),
    "paged_attn_version": ([], _i),
    "paged_expand_ubatch": ([_vp, _i, _i, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp], _i),
    "paged_kv_append": ([_vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _vp, _vp], _i),
    "paged_attn_workspace_size": ([_i, _i, _i, _i], _sz),
    "paged_attn_plan": ([_vp, _i, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp], _i),
    "paged_attn_prefill": (_ATTN_ARGS, _i),
    "paged_attn_decode": (_ATTN_ARGS, _i),
    "paged_attn_run": (_ATTN_ARGS, _i),
    "paged_attn_forward": (_ATTN_ARGS, _i),
    "paged_attn_validate": ([_vp, _i, _vp, _i, _i, _i, _vp, _vp], _i),
    "paged_attn_read_error": ([_vp, ctypes.POINTER(_i), _vp], _i),
    "paged_attn_set_prefill_min_run": ([_i], _i),
    "paged_attn_set_decode_wait_limit": ([ctypes.c_ulonglong], ctypes.c_ulonglong),
    "pa_pool_create": ([_i], _vp),
    "pa_pool_destroy": ([_vp], None),
    "pa_pool_num_free": ([_vp], _i),
    "pa_pool_alloc": ([_vp, _i, _vp], _i),
    "pa_pool_share": ([_vp, _vp, _i], _i),
    "pa_pool_release": ([_vp, _vp, _i], _i),
    "pa_pool_refcount": ([_vp, ctypes.c_int32], _i),
    "pa_pool_fork": ([_vp, _vp, _i, _i, _vp, _vp, _vp], _i),
    "paged_copy_pages": ([_vp, _vp, _i, _vp, _vp, _i, _i, _i, _i, _vp, _vp], _i),
    "paged_kv_append_fp8": ([_vp, _vp, _vp, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp],
                            _i),
    "paged_attn_decode_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                               ctypes.c_float, _vp, _vp, _sz, _vp], _i),
    "paged_attn_prefill_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                                ctypes.c_float, _vp, _vp, _sz, _vp], _i),
    "paged_attn_forward_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                                ctypes.c_float, _vp, _vp, _sz, _vp], _i),
    "paged_attn_plan_decode": ([_vp, _i, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp], _i),
    "paged_attn_masked_decode": ([_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                                  ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i),
    "paged_attn_decode_append": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i,
                                  _i, ctypes.c_float, _vp, _vp, _sz, _vp], _i),
    "paged_attn_plan_prefill": ([_vp, _i, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp], _i),
    "paged_attn_masked_prefill": ([_vp, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _i,
                                   ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp], _i),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded ctypes library (raw C-ABI access)."""
    return _lib


def strerror(status: int) -> str:
    return _lib.paged_attn_strerror(int(status)).decode()


def version() -> int:
    return int(_lib.paged_attn_version())


def _check(status: int, where: str):
    if status != PA_OK:
        raise PagedAttnError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _req(t, dtype, name):
    if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def workspace_size(T: int, Hq: int, Hkv: int, d: int) -> int:
    return int(_lib.paged_attn_workspace_size(T, Hq, Hkv, d))


def new_workspace(T: int, Hq: int, Hkv: int, d: int, device=None) -> torch.Tensor:
    n = workspace_size(T, Hq, Hkv, d)
    if n == 0:
        raise PagedAttnError(PA_EUNSUPPORTED, "workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def expand_ubatch(seq_page_table, tok_seq, tok_pos, P, out=None, err=None, stream=None):
    """Per-token expansion -> (tok_page_table, tok_kv_len, slot_mapping)."""
    _req(seq_page_table, torch.int32, "seq_page_table")
    _req(tok_seq, torch.int32, "tok_seq")
    _req(tok_pos, torch.int32, "tok_pos")
    n_seq, max_pages = seq_page_table.shape
    T = tok_seq.shape[0]
    dev = seq_page_table.device
    if out is None:
        out = (torch.empty((T, max_pages), dtype=torch.int32, device=dev),
               torch.empty(T, dtype=torch.int32, device=dev),
               torch.empty(T, dtype=torch.int64, device=dev))
    tpt, kv, slot = out
    _check(_lib.paged_expand_ubatch(_ptr(seq_page_table), n_seq, max_pages, _ptr(tok_seq),
                                    _ptr(tok_pos), T, P, _ptr(tpt), _ptr(kv), _ptr(slot),
                                    _ptr(err), _stream(stream)), "paged_expand_ubatch")
    return tpt, kv, slot


def kv_append(k, v, slot_mapping, k_pages, v_pages, err=None, stream=None):
    """reshape-and-cache: write k/v [T][Hkv][d] into the pool at slot_mapping."""
    for t, n in ((k, "k"), (v, "v"), (k_pages, "k_pages"), (v_pages, "v_pages")):
        _req(t, torch.float16, n)
    _req(slot_mapping, torch.int64, "slot_mapping")
    N, Hkv, P, d = k_pages.shape
    T = slot_mapping.shape[0]
    _check(_lib.paged_kv_append(_ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_pages),
                                _ptr(v_pages), N, Hkv, P, d, _ptr(err), _stream(stream)),
           "paged_kv_append")


def plan_decode(tok_page_table, tok_kv_len, Hq, Hkv, P, d, workspace, stream=None):
    """plan with every token on the split-KV path (for masked_decode / decode_fp8)."""
    _req(tok_page_table, torch.int32, "tok_page_table")
    _req(tok_kv_len, torch.int32, "tok_kv_len")
    T, max_pages = tok_page_table.shape
    _check(_lib.paged_attn_plan_decode(_ptr(tok_page_table), max_pages, _ptr(tok_kv_len), T, Hq,
                                       Hkv, P, d, _ptr(workspace), workspace.numel(),
                                       _stream(stream)), "paged_attn_plan_decode")


def plan_prefill(tok_page_table, tok_kv_len, Hq, Hkv, P, d, workspace, stream=None):
    """plan with every token in a tensor-core tile (for masked_prefill)."""
    _req(tok_page_table, torch.int32, "tok_page_table")
    _req(tok_kv_len, torch.int32, "tok_kv_len")
    T, max_pages = tok_page_table.shape
    _check(_lib.paged_attn_plan_prefill(_ptr(tok_page_table), max_pages, _ptr(tok_kv_len), T, Hq,
                                        Hkv, P, d, _ptr(workspace), workspace.numel(),
                                        _stream(stream)), "paged_attn_plan_prefill")


def masked_decode(q, k_pages, v_pages, tok_page_table, tok_kv_len, scale, cell_seq, cell_pos,
                  tok_seq, tok_pos, out, workspace, stream=None):
    """Unified-span baseline: split-KV attention of every token over its row, keeping
    only the slots whose cell belongs to the token's sequence at a position up to its
    own.  Runs on a plan from plan_decode."""
    return _masked("paged_attn_masked_decode", q, k_pages, v_pages, tok_page_table, tok_kv_len,
                   scale, cell_seq, cell_pos, tok_seq, tok_pos, out, workspace, stream)


def masked_prefill(q, k_pages, v_pages, tok_page_table, tok_kv_len, scale, cell_seq, cell_pos,
                   tok_seq, tok_pos, out, workspace, stream=None):
    """The same masked attention on the tcgen05 prefill tiles (the unified-span
    baseline of prefill).  Runs on a plan from plan_prefill."""
    return _masked("paged_attn_masked_prefill", q, k_pages, v_pages, tok_page_table, tok_kv_len,
                   scale, cell_seq, cell_pos, tok_seq, tok_pos, out, workspace, stream)


def _masked(fn_name, q, k_pages, v_pages, tok_page_table, tok_kv_len, scale, cell_seq, cell_pos,
            tok_seq, tok_pos, out, workspace, stream):
    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages"), (out, "out")):
        _req(t, torch.float16, n)
    for t, n in ((tok_page_table, "tok_page_table"), (tok_kv_len, "tok_kv_len"),
                 (cell_seq, "cell_seq"), (cell_pos, "cell_pos"), (tok_seq, "tok_seq"),
                 (tok_pos, "tok_pos")):
        _req(t, torch.int32, n)
    T, Hq, d = q.shape
    N, Hkv, P, _ = k_pages.shape
    max_pages = tok_page_table.shape[1]
    _check(getattr(_lib, fn_name)(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(tok_page_table), max_pages, _ptr(tok_kv_len),
        T, Hq, Hkv, P, d, N, float(scale), _ptr(cell_seq), _ptr(cell_pos), _ptr(tok_seq),
        _ptr(tok_pos), _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)), fn_name)
    return out


def new_fp8_pool(num_pages, Hkv, P, d, device=None):
    """Empty FP8 pool: (k8 [N][Hkv][P][d] uint8, v8t [N][Hkv][d][P] uint8,
    k_scale, v_scale [N][Hkv][P] float32)."""
    dev = device or "cuda"
    return (torch.zeros((num_pages, Hkv, P, d), dtype=torch.uint8, device=dev),
            torch.zeros((num_pages, Hkv, d, P), dtype=torch.uint8, device=dev),
            torch.ones((num_pages, Hkv, P), dtype=torch.float32, device=dev),
            torch.ones((num_pages, Hkv, P), dtype=torch.float32, device=dev))


def kv_append_fp8(k, v, slot_mapping, k8, v8t, k_scale, v_scale, err=None, stream=None):
    """Quantising reshape-and-cache into FP8 pages (E4M3 codes, one scale per row)."""
    _req(k, torch.float16, "k")
    _req(v, torch.float16, "v")
    _req(slot_mapping, torch.int64, "slot_mapping")
    for t, n in ((k8, "k8"), (v8t, "v8t")):
        _req(t, torch.uint8, n)
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _req(t, torch.float32, n)
    N, Hkv, P, d = k8.shape
    _check(_lib.paged_kv_append_fp8(_ptr(k), _ptr(v), _ptr(slot_mapping), slot_mapping.shape[0],
                                    _ptr(k8), _ptr(v8t), _ptr(k_scale), _ptr(v_scale), N, Hkv, P,
                                    d, _ptr(err), _stream(stream)), "paged_kv_append_fp8")


def _attn_fp8(name, q, k8, v8t, k_scale, v_scale, tok_page_table, tok_kv_len, scale, out,
              workspace, stream):
    _req(q, torch.float16, "q")
    _req(tok_page_table, torch.int32, "tok_page_table")
    _req(tok_kv_len, torch.int32, "tok_kv_len")
    T, Hq, d = q.shape
    N, Hkv, P, _ = k8.shape
    if out is None:
        out = torch.empty_like(q)
    _req(out, torch.float16, "out")
    if workspace is None:
        workspace = new_workspace(T, Hq, Hkv, d, q.device)
    _check(getattr(_lib, name)(
        _ptr(q), _ptr(k8), _ptr(v8t), _ptr(k_scale), _ptr(v_scale), _ptr(tok_page_table),
        tok_page_table.shape[1], _ptr(tok_kv_len), T, Hq, Hkv, P, d, N, float(scale), _ptr(out),
        _ptr(workspace), workspace.numel(), _stream(stream)), name)
    return out


def decode_fp8(q, k8, v8t, k_scale, v_scale, tok_page_table, tok_kv_len, scale, out, workspace,
               stream=None):
    """Split-KV decode attention over FP8 pages (on a plan from plan_decode or plan)."""
    return _attn_fp8("paged_attn_decode_fp8", q, k8, v8t, k_scale, v_scale, tok_page_table,
                     tok_kv_len, scale, out, workspace, stream)


def prefill_fp8(q, k8, v8t, k_scale, v_scale, tok_page_table, tok_kv_len, scale, out, workspace,
                stream=None):
    """Tensor-core prefill tiles over FP8 pages (on a plan from plan or plan_prefill)."""
    return _attn_fp8("paged_attn_prefill_fp8", q, k8, v8t, k_scale, v_scale, tok_page_table,
                     tok_kv_len, scale, out, workspace, stream)


def forward_fp8(q, k8, v8t, k_scale, v_scale, tok_page_table, tok_kv_len, scale, out=None,
                workspace=None, stream=None):
    """Plan + prefill + decode for one ubatch over FP8 pages; returns out [T][Hq][d]."""
    return _attn_fp8("paged_attn_forward_fp8", q, k8, v8t, k_scale, v_scale, tok_page_table,
                     tok_kv_len, scale, out, workspace, stream)


def copy_pages(src, dst, k_pages, v_pages, err=None, stream=None):
    """Page copy of a copy-on-write fork: page dst[i] <- page src[i] in both pools."""
    _req(src, torch.int32, "src")
    _req(dst, torch.int32, "dst")
    _req(k_pages, torch.float16, "k_pages")
    _req(v_pages, torch.float16, "v_pages")
    if src.shape != dst.shape:
        raise ValueError("src and dst must have the same length")
    N, Hkv, P, d = k_pages.shape
    _check(_lib.paged_copy_pages(_ptr(src), _ptr(dst), src.shape[0], _ptr(k_pages), _ptr(v_pages),
                                 N, Hkv, P, d, _ptr(err), _stream(stream)), "paged_copy_pages")


def plan(tok_page_table, tok_kv_len, Hq, Hkv, P, d, workspace, stream=None):
    _req(tok_page_table, torch.int32, "tok_page_table")
    _req(tok_kv_len, torch.int32, "tok_kv_len")
    T, max_pages = tok_page_table.shape
    _check(_lib.paged_attn_plan(_ptr(tok_page_table), max_pages, _ptr(tok_kv_len), T, Hq, Hkv, P,
                                d, _ptr(workspace), workspace.numel(), _stream(stream)),
           "paged_attn_plan")


def _attn(fn_name, q, k_pages, v_pages, tok_page_table, tok_kv_len, scale, out, workspace,
          stream):
    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages")):
        _req(t, torch.float16, n)
    _req(tok_page_table, torch.int32, "tok_page_table")
    _req(tok_kv_len, torch.int32, "tok_kv_len")
    T, Hq, d = q.shape
    N, Hkv, P, d2 = k_pages.shape
    if d2 != d:
        raise ValueError("head_dim of q and k_pages differ")
    max_pages = tok_page_table.shape[1]
    if out is None:
        out = torch.empty_like(q)
    _req(out, torch.float16, "out")
    if workspace is None:
        workspace = new_workspace(T, Hq, Hkv, d, q.device)
    st = getattr(_lib, fn_name)(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(tok_page_table),
                                max_pages, _ptr(tok_kv_len), T, Hq, Hkv, P, d, N, float(scale),
                                _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, fn_name)
    return out


def forward(q, k_pages, v_pages, tok_page_table, tok_kv_len, scale, out=None, workspace=None,
            stream=None):
    """Plan + prefill + decode for one ubatch; returns out [T][Hq][d] float16."""
    return _attn("paged_attn_forward", q, k_pages, v_pages, tok_page_table, tok_kv_len, scale,
                 out, workspace, stream)


def run(q, k_pages, v_pages, tok_page_table, tok_kv_len, scale, out=None, workspace=None,
        stream=None):
    """Prefill + decode of an already planned ubatch."""
    return _attn("paged_attn_run", q, k_pages, v_pages, tok_page_table, tok_kv_len, scale, out,
                 workspace, stream)


def prefill(q, k_pages, v_pages, tok_page_table, tok_kv_len, scale, out, workspace, stream=None):
    return _attn("paged_attn_prefill", q, k_pages, v_pages, tok_page_table, tok_kv_len, scale, out,
                 workspace, stream)


def decode(q, k_pages, v_pages, tok_page_table, tok_kv_len, scale, out, workspace, stream=None):
    return _attn("paged_attn_decode", q, k_pages, v_pages, tok_page_table, tok_kv_len, scale, out,
                 workspace, stream)


def decode_append(q, k_new, v_new, slot_mapping, k_pages, v_pages, tok_page_table, tok_kv_len,
                  scale, out, workspace, stream=None):
    """decode with the decode tokens' K/V append fused into the same launch (f16 pages):
    equals kv_append(k_new, v_new, slot_mapping, ...) then decode(...)."""
    for t, n in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (k_pages, "k_pages"),
                 (v_pages, "v_pages"), (out, "out")):
        _req(t, torch.float16, n)
    _req(slot_mapping, torch.int64, "slot_mapping")
    _req(tok_page_table, torch.int32, "tok_page_table")
    _req(tok_kv_len, torch.int32, "tok_kv_len")
    T, Hq, d = q.shape
    N, Hkv, P, _ = k_pages.shape
    _check(_lib.paged_attn_decode_append(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), _ptr(k_pages), _ptr(v_pages),
        _ptr(tok_page_table), tok_page_table.shape[1], _ptr(tok_kv_len), T, Hq, Hkv, P, d, N,
        float(scale), _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)),
        "paged_attn_decode_append")
    return out


def validate(tok_page_table, tok_kv_len, P, num_pages, err, stream=None):
    T, max_pages = tok_page_table.shape
    _check(_lib.paged_attn_validate(_ptr(tok_page_table), max_pages, _ptr(tok_kv_len), T, P,
                                    num_pages, _ptr(err), _stream(stream)), "paged_attn_validate")


def read_error(workspace, stream=None) -> int:
    """Synchronise and return the workspace's device error word (PA_ERR_* bits)."""
    v = ctypes.c_int(0)
    st = _lib.paged_attn_read_error(_ptr(workspace), ctypes.byref(v), _stream(stream))
    if st not in (PA_OK, PA_EDEVICE):
        raise PagedAttnError(st, "paged_attn_read_error")
    return int(v.value)


def set_decode_wait_limit(ns: int) -> int:
    """Limit (ns) of the split-KV decode kernel's bounded waits (0: the 2 s default).
    Returns the previous value."""
    return int(_lib.paged_attn_set_decode_wait_limit(int(ns)))


def set_prefill_min_run(n: int) -> int:
    """Shortest same-row run sent to the tensor-core prefill path; returns the old value."""
    return int(_lib.paged_attn_set_prefill_min_run(int(n)))


class PagePool:
    """Host page allocator (native): lowest-id-first free list, reference counts."""

    def __init__(self, num_pages: int):
        self._h = _lib.pa_pool_create(int(num_pages))
        if not self._h:
            raise PagedAttnError(PA_EINVAL, "pa_pool_create")
        self.num_pages = int(num_pages)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _lib.pa_pool_destroy(h)
            self._h = None

    @property
    def num_free(self) -> int:
        return int(_lib.pa_pool_num_free(self._h))

    def alloc(self, n: int):
        buf = (ctypes.c_int32 * max(n, 1))()
        st = _lib.pa_pool_alloc(self._h, int(n), buf)
        if st < 0:
            raise PagedAttnError(st, "pa_pool_alloc")
        return [int(buf[i]) for i in range(n)]

    def share(self, pages):
        buf = (ctypes.c_int32 * max(len(pages), 1))(*pages)
        _check(_lib.pa_pool_share(self._h, buf, len(pages)), "pa_pool_share")

    def release(self, pages):
        buf = (ctypes.c_int32 * max(len(pages), 1))(*pages)
        _check(_lib.pa_pool_release(self._h, buf, len(pages)), "pa_pool_release")

    def refcount(self, page: int) -> int:
        return int(_lib.pa_pool_refcount(self._h, int(page)))

    def fork(self, pages, n_tokens: int, P: int):
        """Copy-on-write fork of a sequence holding n_tokens tokens in `pages`.
        Returns (child pages, (src, dst) page pair to copy, or None)."""
        n = (int(n_tokens) + P - 1) // P
        buf = (ctypes.c_int32 * max(n, 1))(*pages[:n])
        out = (ctypes.c_int32 * max(n, 1))()
        cs, cd = ctypes.c_int32(-1), ctypes.c_int32(-1)
        st = _lib.pa_pool_fork(self._h, buf, int(n_tokens), int(P), out, ctypes.byref(cs),
                               ctypes.byref(cd))
        if st < 0:
            raise PagedAttnError(st, "pa_pool_fork")
        return [int(out[i]) for i in range(n)], ((int(cs.value), int(cd.value)) if st else None)
