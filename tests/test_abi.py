"""The C-ABI library without a GPU: it loads, exports every symbol the header
declares, and its host-side checks and host page pool behave."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pa():
    import __graft_entry__
    __graft_entry__.build()
    import paged_kv_cache_pages_gb300 as m
    return m


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names) - {"defined"})


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("paged_kv_append", "paged_attn_forward", "paged_expand_ubatch", "paged_attn_plan",
              "paged_attn_prefill", "paged_attn_decode", "paged_attn_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(pa):
    lib = ctypes.CDLL(pa.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_strerror_and_version(pa):
    assert pa.version() >= 100
    for st in (0, -1, -2, -3, -4, -5, -6, -7, -99):
        assert isinstance(pa.strerror(st), str) and pa.strerror(st)


def test_host_argument_checks(pa):
    L = pa.lib()
    nul = None
    # attention: null tables, bad shapes, unsupported head_dim / page size / group
    assert L.paged_attn_forward(nul, nul, nul, nul, 4, nul, 8, 4, 2, 16, 64, 32, 0.1, nul, nul, 0,
                                nul) == pa.PA_EINVAL
    assert L.paged_attn_forward(nul, nul, nul, nul, 4, nul, 8, 4, 2, 16, 80, 32, 0.1, nul, nul, 0,
                                nul) == pa.PA_EUNSUPPORTED
    assert L.paged_attn_forward(nul, nul, nul, nul, 4, nul, 8, 4, 2, 24, 64, 32, 0.1, nul, nul, 0,
                                nul) == pa.PA_EUNSUPPORTED
    assert L.paged_attn_forward(nul, nul, nul, nul, 4, nul, 8, 6, 4, 16, 64, 32, 0.1, nul, nul, 0,
                                nul) == pa.PA_EUNSUPPORTED
    assert L.paged_attn_forward(nul, nul, nul, nul, 4, nul, 8, 48, 2, 16, 64, 32, 0.1, nul, nul,
                                0, nul) == pa.PA_EUNSUPPORTED
    assert L.paged_attn_forward(nul, nul, nul, nul, 4, nul, -1, 4, 2, 16, 64, 32, 0.1, nul, nul,
                                0, nul) == pa.PA_EINVAL
    # T == 0 is a no-op that touches nothing
    assert L.paged_attn_forward(nul, nul, nul, nul, 4, nul, 0, 4, 2, 16, 64, 32, 0.1, nul, nul, 0,
                                nul) == pa.PA_OK
    # append / expand / validate null pointers
    assert L.paged_kv_append(nul, nul, nul, 4, nul, nul, 8, 2, 16, 64, nul, nul) == pa.PA_EINVAL
    assert L.paged_kv_append(nul, nul, nul, 0, nul, nul, 8, 2, 16, 64, nul, nul) == pa.PA_OK
    assert L.paged_expand_ubatch(nul, 2, 4, nul, nul, 3, 16, nul, nul, nul, nul, nul) == pa.PA_EINVAL
    assert L.paged_attn_validate(nul, 4, nul, 3, 16, 8, nul, nul) == pa.PA_EINVAL
    assert L.paged_attn_read_error(nul, nul, nul) == pa.PA_EINVAL


def test_workspace_size(pa):
    assert pa.workspace_size(8, 4, 2, 64) > 0
    assert pa.workspace_size(2048, 32, 8, 128) >= pa.workspace_size(8, 32, 8, 128)
    assert pa.workspace_size(8, 4, 2, 80) == 0
    assert pa.workspace_size(8, 6, 4, 64) == 0


def test_prefill_min_run_knob(pa):
    old = pa.set_prefill_min_run(5)
    assert pa.set_prefill_min_run(0) == 5      # clamps to 1
    assert pa.set_prefill_min_run(old) == 1


def test_page_pool(pa):
    pool = pa.PagePool(6)
    assert pool.num_free == 6
    a = pool.alloc(3)
    assert a == [0, 1, 2] and pool.num_free == 3
    b = pool.alloc(2)
    assert b == [3, 4]
    with pytest.raises(pa.PagedAttnError):
        pool.alloc(2)                          # only one left: nothing taken
    assert pool.num_free == 1
    pool.share(a[:2])                          # a shared prefix: two owners
    assert pool.refcount(0) == 2 and pool.refcount(2) == 1
    pool.release(a)                            # first owner leaves
    assert pool.refcount(0) == 1 and pool.refcount(2) == 0 and pool.num_free == 2
    with pytest.raises(pa.PagedAttnError):
        pool.release([2])                      # already free
    with pytest.raises(pa.PagedAttnError):
        pool.release([0, 0])                   # only one reference left
    pool.release(a[:2])
    assert pool.num_free == 4
    assert pool.alloc(2) == [0, 1]             # lowest ids first
    with pytest.raises(pa.PagedAttnError):
        pool.share([7])
    assert pool.refcount(99) == pa.PA_EINVAL


def test_noalloc_host_checks_match_forward(pa):
    """The no-allocation entry point returns, for every input its host checks
    reject, the status paged_attn_forward returns for the same input."""
    L = pa.lib()
    fwd, noa = L.paged_attn_forward, L.paged_attn_forward_noalloc
    noa.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_void_p] + [ctypes.c_int] * 6 + \
        [ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
    noa.restype = ctypes.c_int
    nul = None
    # (max_pages, T, Hq, Hkv, P, d, num_pages)
    cases = [(4, 8, 0, 2, 16, 64, 32),      # Hq <= 0
             (4, 8, 4, 0, 16, 64, 32),      # Hkv <= 0
             (4, 8, 4, 2, 16, 80, 32),      # unsupported d
             (4, 8, 4, 2, 24, 64, 32),      # unsupported P
             (4, 8, 6, 4, 16, 64, 32),      # Hq % Hkv != 0
             (4, -1, 4, 2, 16, 64, 32),     # T < 0
             (4, 0, 4, 2, 16, 80, 32),      # T == 0 with a bad shape
             (4, 0, 4, 0, 16, 64, 32),      # T == 0 with Hkv == 0
             (4, 0, 4, 2, 16, 64, 32),      # T == 0, good shape: a no-op
             (4, 8, 4, 2, 16, 64, 32),      # null tables
             (0, 8, 4, 2, 16, 64, 32)]      # max_pages == 0
    for mp, T, Hq, Hkv, P, d, npg in cases:
        want = fwd(nul, nul, nul, nul, mp, nul, T, Hq, Hkv, P, d, npg, 0.1, nul, nul, 0, nul)
        got = noa(nul, nul, nul, nul, mp, nul, T, Hq, Hkv, P, d, npg, 0.1, nul, nul)
        assert got == want, ((mp, T, Hq, Hkv, P, d, npg), got, want)


def test_decode_wait_limit_setter(pa):
    default = pa.set_decode_wait_limit(5000)
    assert default == 2_000_000_000
    assert pa.set_decode_wait_limit(10) == 5000          # clamps to 1 us
    assert pa.set_decode_wait_limit(0) == 1000           # 0 restores the default
    assert pa.set_decode_wait_limit(default) == 2_000_000_000
