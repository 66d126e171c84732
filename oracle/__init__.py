"""CPU fp64 oracle for paged attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it.

The arithmetic lives in ``paged_attention_ref.c`` (plain C, double precision,
OpenMP over (token, head)); this module compiles it with gcc on first use and
marshals numpy arrays through ctypes.  Each function follows the page
"面向多并发长上下文的 llama.cpp 分页式 KV Cache 与计算加速优化", section 作品简介
(per-sequence page mapping + true length, expanded per ubatch token; each query
reads only its own sequence's valid pages), and the CacheFlow page, section
核心架构 3 (reshape-and-cache).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attention_ref.c")
_LIB = os.path.join(_HERE, "libpaged_attention_ref.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP).  Returns the .so path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
            i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
            u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
            f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
            c_int, c_double = ctypes.c_int, ctypes.c_double
            lib.ref_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.ref_f16_to_f64.restype = c_double
            lib.ref_expand_ubatch.argtypes = [i32p, c_int, c_int, i32p, i32p, c_int, c_int,
                                              i32p, i32p, i64p]
            lib.ref_expand_ubatch.restype = c_int
            lib.ref_kv_append.argtypes = [u16p, u16p, i64p, c_int, u16p, u16p,
                                          c_int, c_int, c_int, c_int]
            lib.ref_kv_append.restype = c_int
            lib.ref_paged_attention.argtypes = [u16p, u16p, u16p, i32p, c_int, i32p,
                                                c_int, c_int, c_int, c_int, c_int, c_int,
                                                c_double, ctypes.c_void_p, c_int, f64p]
            lib.ref_paged_attention.restype = c_int
            lib.ref_copy_pages.argtypes = [i32p, i32p, c_int, u16p, u16p, c_int, c_int, c_int,
                                           c_int]
            lib.ref_copy_pages.restype = c_int
            lib.ref_masked_attention.argtypes = [u16p, u16p, u16p, i32p, c_int, i32p,
                                                 c_int, c_int, c_int, c_int, c_int, c_int,
                                                 c_double, i32p, i32p, i32p, i32p,
                                                 ctypes.c_void_p, c_int, f64p]
            lib.ref_masked_attention.restype = c_int
            u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
            f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
            lib.ref_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.ref_e4m3_to_f64.restype = c_double
            lib.ref_f32_to_e4m3.argtypes = [ctypes.c_float]
            lib.ref_f32_to_e4m3.restype = ctypes.c_uint8
            lib.ref_kv_append_fp8.argtypes = [u16p, u16p, i64p, c_int, u8p, u8p, f32p, f32p,
                                              c_int, c_int, c_int, c_int]
            lib.ref_kv_append_fp8.restype = c_int
            lib.ref_paged_attention_fp8.argtypes = [u16p, u8p, u8p, f32p, f32p, i32p, c_int, i32p,
                                                    c_int, c_int, c_int, c_int, c_int, c_int,
                                                    c_double, ctypes.c_void_p, c_int, f64p]
            lib.ref_paged_attention_fp8.restype = c_int
            lib.ref_num_threads.argtypes = []
            lib.ref_num_threads.restype = c_int
            _lib = lib
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def f16_to_f64(bits: int) -> float:
    """Exact binary16 -> double of one bit pattern."""
    return float(_load().ref_f16_to_f64(int(bits) & 0xFFFF))


def num_threads() -> int:
    """OpenMP threads the oracle runs on."""
    return int(_load().ref_num_threads())


def expand_ubatch(seq_page_table, tok_seq, tok_pos, P):
    """Per-token expansion: returns (tok_page_table, tok_kv_len, slot_mapping)."""
    spt = _c(seq_page_table, np.int32)
    n_seq, max_pages = spt.shape
    tok_seq = _c(tok_seq, np.int32)
    tok_pos = _c(tok_pos, np.int32)
    T = tok_seq.shape[0]
    tpt = np.empty((T, max_pages), np.int32)
    kv = np.empty(T, np.int32)
    slot = np.empty(T, np.int64)
    rc = _load().ref_expand_ubatch(spt, n_seq, max_pages, tok_seq, tok_pos, T, P, tpt, kv, slot)
    if rc != 0:
        raise ValueError("expand_ubatch: sequence index or position out of range")
    return tpt, kv, slot


def kv_append(k, v, slot_mapping, k_pages, v_pages):
    """reshape-and-cache on host arrays.  k_pages / v_pages ([N][Hkv][P][d] uint16)
    are updated in place (and returned)."""
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    slot = _c(slot_mapping, np.int64)
    assert k_pages.flags.c_contiguous and v_pages.flags.c_contiguous
    assert k_pages.dtype == np.uint16 and v_pages.dtype == np.uint16
    N, Hkv, P, d = k_pages.shape
    T = slot.shape[0]
    rc = _load().ref_kv_append(k, v, slot, T, k_pages, v_pages, N, Hkv, P, d)
    if rc != 0:
        raise ValueError("kv_append: slot beyond the pool")
    return k_pages, v_pages


def copy_pages(src, dst, k_pages, v_pages):
    """Page copy of a copy-on-write fork on host arrays: page dst[i] <- page src[i]
    in both pools ([N][Hkv][P][d] uint16, updated in place).  Returns the number of
    pairs skipped because an id is outside the pool."""
    src = _c(src, np.int32)
    dst = _c(dst, np.int32)
    assert k_pages.flags.c_contiguous and v_pages.flags.c_contiguous
    assert k_pages.dtype == np.uint16 and v_pages.dtype == np.uint16
    N, Hkv, P, d = k_pages.shape
    return int(_load().ref_copy_pages(src, dst, src.shape[0], k_pages, v_pages, N, Hkv, P, d))


def paged_attention(q, k_pages, v_pages, tok_page_table, tok_kv_len, scale, tokens=None):
    """fp64 paged attention by definition.  q: [T][Hq][d] uint16 (binary16 bits).
    Returns float64 [T or len(tokens)][Hq][d]."""
    q = _c(q, np.uint16)
    k_pages = _c(k_pages, np.uint16)
    v_pages = _c(v_pages, np.uint16)
    tpt = _c(tok_page_table, np.int32)
    kv = _c(tok_kv_len, np.int32)
    T, Hq, d = q.shape
    N, Hkv, P, d2 = k_pages.shape
    assert d2 == d and Hq % Hkv == 0
    max_pages = tpt.shape[1] if tpt.ndim == 2 else 0
    if tokens is None:
        sel, n = None, T
        tok_arr = None
    else:
        tok_arr = _c(tokens, np.int32)
        n = tok_arr.shape[0]
        sel = tok_arr.ctypes.data_as(ctypes.c_void_p)
    out = np.zeros((n, Hq, d), np.float64)
    if n == 0:
        return out
    rc = _load().ref_paged_attention(q, k_pages, v_pages, tpt, max_pages, kv, T, Hq, Hkv, P, d, N,
                                     float(scale), sel, n, out)
    if rc != 0:
        raise ValueError("paged_attention: page id or kv_len out of range")
    return out


def masked_attention(q, k_pages, v_pages, tok_page_table, tok_kv_len, scale, cell_seq, cell_pos,
                     tok_seq, tok_pos, tokens=None):
    """fp64 attention over each token's table row, keeping only the slots that hold a
    cell of the token's own sequence at a position up to its own (the unified-span
    baseline).  cell_seq / cell_pos: [num_pages * P] int32.  Returns float64
    [T or len(tokens)][Hq][d]."""
    q = _c(q, np.uint16)
    k_pages = _c(k_pages, np.uint16)
    v_pages = _c(v_pages, np.uint16)
    tpt = _c(tok_page_table, np.int32)
    kv = _c(tok_kv_len, np.int32)
    cs, cp = _c(cell_seq, np.int32), _c(cell_pos, np.int32)
    ts, tp = _c(tok_seq, np.int32), _c(tok_pos, np.int32)
    T, Hq, d = q.shape
    N, Hkv, P, d2 = k_pages.shape
    assert d2 == d and Hq % Hkv == 0 and cs.shape[0] >= N * P and cp.shape[0] >= N * P
    max_pages = tpt.shape[1]
    if tokens is None:
        sel, n = None, T
    else:
        tok_arr = _c(tokens, np.int32)
        n = tok_arr.shape[0]
        sel = tok_arr.ctypes.data_as(ctypes.c_void_p)
    out = np.zeros((n, Hq, d), np.float64)
    if n == 0:
        return out
    rc = _load().ref_masked_attention(q, k_pages, v_pages, tpt, max_pages, kv, T, Hq, Hkv, P, d,
                                      N, float(scale), cs, cp, ts, tp, sel, n, out)
    if rc != 0:
        raise ValueError("masked_attention: page id or kv_len out of range")
    return out


def e4m3_to_f64(code: int) -> float:
    """Value of one FP8 E4M3 code."""
    return float(_load().ref_e4m3_to_f64(int(code)))


def f32_to_e4m3(x: float) -> int:
    """E4M3 code of a binary32 value: nearest, ties to even, saturating at 448."""
    return int(_load().ref_f32_to_e4m3(float(np.float32(x))))


def kv_append_fp8(k, v, slot_mapping, k8, v8t, k_scale, v_scale):
    """Quantising reshape-and-cache on host arrays (updated in place):
    k8 [N][Hkv][P][d] uint8, v8t [N][Hkv][d][P] uint8, scales [N][Hkv][P] float32."""
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    slot = _c(slot_mapping, np.int64)
    for a, dt in ((k8, np.uint8), (v8t, np.uint8), (k_scale, np.float32), (v_scale, np.float32)):
        assert a.flags.c_contiguous and a.dtype == dt
    N, Hkv, P, d = k8.shape
    rc = _load().ref_kv_append_fp8(k, v, slot, slot.shape[0], k8, v8t, k_scale, v_scale, N, Hkv,
                                   P, d)
    if rc != 0:
        raise ValueError("kv_append_fp8: slot beyond the pool")


def paged_attention_fp8(q, k8, v8t, k_scale, v_scale, tok_page_table, tok_kv_len, scale,
                        tokens=None):
    """fp64 paged attention over FP8 pages (dequantised by definition)."""
    q = _c(q, np.uint16)
    k8, v8t = _c(k8, np.uint8), _c(v8t, np.uint8)
    ks, vs = _c(k_scale, np.float32), _c(v_scale, np.float32)
    tpt = _c(tok_page_table, np.int32)
    kv = _c(tok_kv_len, np.int32)
    T, Hq, d = q.shape
    N, Hkv, P, d2 = k8.shape
    assert d2 == d and Hq % Hkv == 0
    if tokens is None:
        sel, n = None, T
    else:
        tok_arr = _c(tokens, np.int32)
        n = tok_arr.shape[0]
        sel = tok_arr.ctypes.data_as(ctypes.c_void_p)
    out = np.zeros((n, Hq, d), np.float64)
    if n == 0:
        return out
    rc = _load().ref_paged_attention_fp8(q, k8, v8t, ks, vs, tpt, tpt.shape[1], kv, T, Hq, Hkv, P,
                                         d, N, float(scale), sel, n, out)
    if rc != 0:
        raise ValueError("paged_attention_fp8: page id or kv_len out of range")
    return out
