"""Seeded synthetic inputs for paged attention.

This module is shared by the oracle tests, the GPU parity tests and the
benchmark.  It holds none of the attention arithmetic: only random numbers,
which physical page holds which sequence's tokens (the page assignment a KV
manager would make), and which tokens form a ubatch.  Both the CUDA path and
the CPU oracle consume what it produces; neither is imported here.

Conventions
-----------
* binary16 data are carried as ``uint16`` bit patterns.
* KV pool layout: ``[num_pages][Hkv][P][d]`` for K and for V.
* A sequence owns an ordered list of physical page ids; position ``p`` of the
  sequence lives in page ``pages[p // P]`` at in-page offset ``p % P``.
* Free pages, tail cells past a sequence's length, and the cells of the
  ubatch's own tokens (not yet appended) hold NaN (``0x7E00``).
* Values are N(0, 1) drawn in float32 with numpy ``default_rng(seed)`` and
  rounded to binary16.

Workloads follow the Qwen3-8B attention shape (32 query heads, 8 KV heads,
head_dim 128, page size 128) used by the UA-PagedAttention page, section
快速开始 (``--page-size 128``, ``-np 4``), and its 16K-prompt x 8 concurrency
measurement (section 作品简介).  No public dataset is involved: these seeded
draws stand in for the real prompts.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F16_NAN = np.uint16(0x7E00)


def randn_f16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) float32 draws rounded to binary16, returned as uint16 bits."""
    return rng.standard_normal(shape, dtype=np.float32).astype(np.float16).view(np.uint16)


@dataclass
class Case:
    """One ubatch over a paged KV pool.

    ``k_pool``/``v_pool`` hold the pool *before* the ubatch's own K/V rows are
    appended; ``k_new``/``v_new`` are those rows.  ``k_ctx[s]``/``v_ctx[s]`` are
    sequence s's contiguous K/V ``[L_s][Hkv][d]`` (before paging), kept for the
    brute-force pins.
    """
    name: str
    P: int
    Hq: int
    Hkv: int
    d: int
    scale: float
    num_pages: int
    seq_pages: list            # list of int32 arrays (physical page ids, in order)
    seq_len: np.ndarray        # int32 [S]: length of each sequence after this ubatch
    tok_seq: np.ndarray        # int32 [T]: sequence of each ubatch token (-1 = padding)
    tok_pos: np.ndarray        # int32 [T]: position of each token in its sequence
    q: np.ndarray              # uint16 [T][Hq][d]
    k_new: np.ndarray          # uint16 [T][Hkv][d]
    v_new: np.ndarray          # uint16 [T][Hkv][d]
    k_pool: np.ndarray         # uint16 [N][Hkv][P][d]
    v_pool: np.ndarray
    k_ctx: list = field(default_factory=list)
    v_ctx: list = field(default_factory=list)
    max_pages: int = 0

    @property
    def T(self) -> int:
        return int(self.tok_seq.shape[0])

    def seq_page_table(self) -> np.ndarray:
        """int32 [S][max_pages], rows padded with -1."""
        S = len(self.seq_pages)
        spt = np.full((S, self.max_pages), -1, np.int32)
        for s, pg in enumerate(self.seq_pages):
            spt[s, :len(pg)] = pg
        return spt


def span_view(case: Case):
    """The same cache seen as one span of cells shared by all sequences (the layout
    paging replaces): every token's row names every page of the pool in order, its
    kv_len is the whole span (0 for padding tokens), and each slot carries the
    (sequence, position) of the cell it holds, -1 where free.  A page shared by two
    sequences has no single owner per cell, so cases with shared pages are refused.
    Returns (tok_page_table, tok_kv_len, cell_seq, cell_pos, tok_seq, tok_pos)."""
    N, P = case.num_pages, case.P
    cell_seq = np.full(N * P, -1, np.int32)
    cell_pos = np.full(N * P, -1, np.int32)
    for s, pages in enumerate(case.seq_pages):
        L = int(case.seq_len[s])
        pos = np.arange(L)
        slots = np.asarray(pages, np.int64)[pos // P] * P + pos % P
        if np.any(cell_seq[slots] != -1):
            raise ValueError("span_view: a cell belongs to two sequences")
        cell_seq[slots] = s
        cell_pos[slots] = pos
    T = case.T
    tpt = np.tile(np.arange(N, dtype=np.int32), (T, 1))
    kv = np.where(case.tok_seq >= 0, N * P, 0).astype(np.int32)
    return (tpt, kv, cell_seq, cell_pos, case.tok_seq.astype(np.int32),
            case.tok_pos.astype(np.int32))


def _fill_pool(pool: np.ndarray, pages: np.ndarray, rows: np.ndarray, P: int, n_pos: int,
               skip_pos=None):
    """Lay rows [n_pos][Hkv][d] of one sequence into its pages (layout only)."""
    Hkv, d = rows.shape[1], rows.shape[2]
    npg = -(-n_pos // P)
    buf = np.full((npg * P, Hkv, d), F16_NAN, np.uint16)
    buf[:n_pos] = rows[:n_pos]
    if skip_pos is not None and len(skip_pos):
        buf[np.asarray(skip_pos)] = F16_NAN
    pool[pages[:npg]] = buf.reshape(npg, P, Hkv, d).transpose(0, 2, 1, 3)


def build_case(name, seed, seq_lens, tokens, P, Hq, Hkv, d, *, num_pages=None,
               free_frac=0.25, shared_prefix_tokens=0, extra_pages=0, scale=None,
               max_pages=None) -> Case:
    """Generic ubatch builder.

    seq_lens: length of each sequence after the ubatch (its tokens included).
    tokens:   list of (seq, pos) for the ubatch, in ubatch order; seq -1 = padding.
    shared_prefix_tokens: the first ``shared_prefix_tokens`` positions (a multiple
        of P) of every sequence live in the same physical pages with the same K/V.
    num_pages: pool size; default ceil(used / (1 - free_frac)).
    """
    rng = np.random.default_rng(seed)
    seq_lens = [int(x) for x in seq_lens]
    S = len(seq_lens)
    assert shared_prefix_tokens % P == 0
    n_pref = shared_prefix_tokens // P
    priv = [max(0, -(-(L - shared_prefix_tokens) // P)) for L in seq_lens]
    used = n_pref + sum(priv) + extra_pages * S
    if num_pages is None:
        num_pages = max(used, int(math.ceil(used / (1.0 - free_frac))))
    assert num_pages >= used
    perm = rng.permutation(num_pages).astype(np.int32)
    pref_pages = perm[:n_pref]
    cur = n_pref
    seq_pages = []
    for s in range(S):
        n = priv[s] + extra_pages
        pg = np.concatenate([pref_pages, perm[cur:cur + n]]).astype(np.int32)
        cur += n
        seq_pages.append(pg)
    if max_pages is None:
        max_pages = max(len(p) for p in seq_pages) if S else 1
    # contiguous K/V per sequence; the shared prefix is drawn once
    k_pref = randn_f16(rng, (shared_prefix_tokens, Hkv, d))
    v_pref = randn_f16(rng, (shared_prefix_tokens, Hkv, d))
    k_ctx, v_ctx = [], []
    for s, L in enumerate(seq_lens):
        n_own = max(0, L - shared_prefix_tokens)
        k_ctx.append(np.concatenate([k_pref[:min(L, shared_prefix_tokens)],
                                     randn_f16(rng, (n_own, Hkv, d))]))
        v_ctx.append(np.concatenate([v_pref[:min(L, shared_prefix_tokens)],
                                     randn_f16(rng, (n_own, Hkv, d))]))
    tok_seq = np.array([t[0] for t in tokens], np.int32).reshape(-1)
    tok_pos = np.array([t[1] for t in tokens], np.int32).reshape(-1)
    T = tok_seq.shape[0]
    q = randn_f16(rng, (T, Hq, d))
    k_new = np.full((T, Hkv, d), F16_NAN, np.uint16)
    v_new = np.full((T, Hkv, d), F16_NAN, np.uint16)
    for i in range(T):
        s, p = int(tok_seq[i]), int(tok_pos[i])
        if s >= 0:
            k_new[i] = k_ctx[s][p]
            v_new[i] = v_ctx[s][p]
    k_pool = np.full((num_pages, Hkv, P, d), F16_NAN, np.uint16)
    v_pool = np.full((num_pages, Hkv, P, d), F16_NAN, np.uint16)
    for s, L in enumerate(seq_lens):
        mine = [int(p) for (ss, p) in tokens if ss == s]
        # the shared prefix is never part of a ubatch, so writing it again is harmless
        _fill_pool(k_pool, seq_pages[s], k_ctx[s], P, L, mine)
        _fill_pool(v_pool, seq_pages[s], v_ctx[s], P, L, mine)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return Case(name, P, Hq, Hkv, d, float(scale), num_pages, seq_pages,
                np.array(seq_lens, np.int32), tok_seq, tok_pos, q, k_new, v_new,
                k_pool, v_pool, k_ctx, v_ctx, max_pages)


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

def tiny(seed: int = 0) -> Case:
    """2 sequences (lengths 37 and 100), page size 16, pool of 32 permuted pages,
    4 query / 2 KV heads, d = 64; 8 ubatch tokens (seq0 positions 32..36, seq1
    positions 97..99), scale 1/sqrt(64)."""
    tokens = [(0, p) for p in range(32, 37)] + [(1, p) for p in range(97, 100)]
    return build_case("tiny", seed, [37, 100], tokens, P=16, Hq=4, Hkv=2, d=64,
                      num_pages=32, scale=1.0 / 8.0)


def decode(seed: int = 0, n_seq: int = 8) -> Case:
    """Qwen3-8B-shaped decode: n_seq sequences with KV length uniform in
    [1024, 4096], one query token each (the newest position), 32/8 heads,
    d = 128, page size 128, pool with 25% free pages, pages shuffled."""
    rng = np.random.default_rng(seed + 1000)
    lens = rng.integers(1024, 4096, size=n_seq, endpoint=True)
    tokens = [(s, int(L) - 1) for s, L in enumerate(lens)]
    return build_case("decode", seed, lens, tokens, P=128, Hq=32, Hkv=8, d=128,
                      free_frac=0.25)


def longtail(seed: int = 0, n_seq: int = 64) -> Case:
    """Long-tail decode: 64 sequences, KV length lognormal (median 2048,
    sigma 1.0) clipped to [256, 32768]; 30% free pages."""
    rng = np.random.default_rng(seed + 2000)
    lens = np.clip(np.round(rng.lognormal(math.log(2048.0), 1.0, size=n_seq)), 256, 32768)
    lens = lens.astype(np.int64)
    tokens = [(s, int(L) - 1) for s, L in enumerate(lens)]
    return build_case("longtail", seed, lens, tokens, P=128, Hq=32, Hkv=8, d=128,
                      free_frac=0.30)


def shared_prefix(seed: int = 0) -> Case:
    """16 sequences whose tables point at the same 64 physical prefix pages
    (8192 tokens), with private suffixes uniform in [512, 2048].  Sequences
    0..11 are decoding (suffix done, then 1..256 generated tokens; one query
    token each); sequences 12..15 are prefilling their suffix: the ubatch takes
    a 256-token chunk from each at a random offset inside the suffix.  Ubatch =
    12 decode tokens + 1024 prefill tokens."""
    rng = np.random.default_rng(seed + 3000)
    pref = 8192
    suffix = rng.integers(512, 2048, size=16, endpoint=True)
    gen = rng.integers(1, 256, size=12, endpoint=True)
    lens, tokens = [], []
    for s in range(12):
        L = pref + int(suffix[s]) + int(gen[s])
        lens.append(L)
        tokens.append((s, L - 1))
    for s in range(12, 16):
        off = int(rng.integers(0, int(suffix[s]) - 256, endpoint=True))
        start = pref + off
        lens.append(start + 256)
        tokens += [(s, p) for p in range(start, start + 256)]
    return build_case("shared_prefix", seed, lens, tokens, P=128, Hq=32, Hkv=8, d=128,
                      free_frac=0.25, shared_prefix_tokens=pref)


def small_prefill(seed: int = 0, P: int = 128, d: int = 128, Hq: int = 8, Hkv: int = 2,
                  chunks=((0, 300, 181), (1, 0, 130), (2, 700, 1)), extra_decode=2) -> Case:
    """A small mixed ubatch for parity: each chunk (seq, start, n) is n causal
    tokens of one sequence from position start, plus extra_decode single-token
    sequences.  Spans several 128-token tiles and a ragged tail."""
    rng = np.random.default_rng(seed + 4000)
    lens, tokens = {}, []
    for (s, start, n) in chunks:
        tokens += [(s, p) for p in range(start, start + n)]
        lens[s] = max(lens.get(s, 0), start + n)
    S0 = max(lens) + 1 if lens else 0
    for i in range(extra_decode):
        L = int(rng.integers(1, 600, endpoint=True))
        lens[S0 + i] = L
        tokens.append((S0 + i, L - 1))
    S = max(lens) + 1
    seq_lens = [lens.get(s, 1) for s in range(S)]
    return build_case(f"small_prefill_P{P}_d{d}", seed, seq_lens, tokens, P=P, Hq=Hq, Hkv=Hkv,
                      d=d, free_frac=0.3)


# ---------------------------------------------------------------------------
# 8 x 16K prefill, chunked into ubatches
# ---------------------------------------------------------------------------

class Prefill8x16K:
    """8 sequences x 16384-token prompts prefilled in ubatches of <= 2048 tokens.

    Schedule (the page gives 4 server slots, ``-np 4``, and 16K prompts x 8):
    slot k (0..3) serves sequence k then sequence k+4 as one 32768-token stream;
    ubatch u takes from slot k the stream range
    ``[512u - 128k, 512(u+1) - 128k) & [0, 32768)``.  Chunks from the 4 slots sit
    at prefix offsets that differ by 128 tokens; chunks that straddle the switch
    from sequence k to k+4 give two runs.  65 ubatches in total.

    K/V of every (sequence, position) is drawn once from ``seed``; q of ubatch u
    from ``seed`` and u.  ``pool_final()`` is the pool after all appends.
    """

    def __init__(self, seed: int = 0, n_seq: int = 8, seq_len: int = 16384, slots: int = 4,
                 chunk: int = 512, stagger: int = 128, P: int = 128, Hq: int = 32, Hkv: int = 8,
                 d: int = 128, free_frac: float = 0.2):
        assert n_seq % slots == 0
        self.seed, self.n_seq, self.seq_len = seed, n_seq, seq_len
        self.slots, self.chunk, self.stagger = slots, chunk, stagger
        self.P, self.Hq, self.Hkv, self.d = P, Hq, Hkv, d
        self.scale = 1.0 / math.sqrt(d)
        rng = np.random.default_rng(seed + 5000)
        self.pages_per_seq = seq_len // P
        used = n_seq * self.pages_per_seq
        self.num_pages = int(math.ceil(used / (1.0 - free_frac)))
        perm = rng.permutation(self.num_pages).astype(np.int32)
        self.max_pages = self.pages_per_seq
        self.seq_page_table = perm[:used].reshape(n_seq, self.pages_per_seq).copy()
        self._kv_rng_seed = seed + 5001
        self._k = None
        self._v = None
        self.ubatches = self._schedule()

    def _schedule(self):
        per_slot = self.n_seq // self.slots
        stream_len = per_slot * self.seq_len
        ubs = []
        u = 0
        # stop once every slot's range starts past the end of its stream
        while self.chunk * u - self.stagger * (self.slots - 1) < stream_len:
            toks_seq, toks_pos = [], []
            for k in range(self.slots):
                lo = max(0, self.chunk * u - self.stagger * k)
                hi = min(stream_len, self.chunk * (u + 1) - self.stagger * k)
                if hi <= lo:
                    continue
                pos = np.arange(lo, hi)
                seq = k + self.slots * (pos // self.seq_len)
                toks_seq.append(seq.astype(np.int32))
                toks_pos.append((pos % self.seq_len).astype(np.int32))
            ubs.append((np.concatenate(toks_seq), np.concatenate(toks_pos)))
            u += 1
        return ubs

    def _draw_kv(self):
        if self._k is None:
            rng = np.random.default_rng(self._kv_rng_seed)
            shape = (self.n_seq, self.seq_len, self.Hkv, self.d)
            self._k = randn_f16(rng, shape)
            self._v = randn_f16(rng, shape)
        return self._k, self._v

    def ubatch(self, u: int):
        """(tok_seq, tok_pos, q, k_new, v_new) of ubatch u."""
        tok_seq, tok_pos = self.ubatches[u]
        rng = np.random.default_rng([self.seed + 5002, u])
        q = randn_f16(rng, (tok_seq.shape[0], self.Hq, self.d))
        K, V = self._draw_kv()
        return tok_seq, tok_pos, q, K[tok_seq, tok_pos], V[tok_seq, tok_pos]

    def pool_final(self):
        """Pool after every ubatch has been appended; free pages hold NaN."""
        K, V = self._draw_kv()
        kp = np.full((self.num_pages, self.Hkv, self.P, self.d), F16_NAN, np.uint16)
        vp = np.full_like(kp, F16_NAN)
        for s in range(self.n_seq):
            _fill_pool(kp, self.seq_page_table[s], K[s], self.P, self.seq_len)
            _fill_pool(vp, self.seq_page_table[s], V[s], self.P, self.seq_len)
        return kp, vp

    def flops(self) -> float:
        """Causal attention FLOPs of the whole prefill: 4 d Hq sum_t kv_len_t."""
        per_seq = self.seq_len * (self.seq_len + 1) // 2
        return 4.0 * self.d * self.Hq * self.n_seq * per_seq
