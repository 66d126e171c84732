// Prefill attention on tcgen05 tensor cores with TMEM accumulators (sm_103a).
//
// Work item = (tile of <= 128 consecutive ubatch tokens whose page-table rows
// are identical, KV head g, pair of query heads of that group).  The two query
// heads share every K/V tile the CTA loads (GQA grouping), so one 128-key block
// of K and of V is fetched once for 2 x 128 query rows.
//
// Scheduling is stream-K: the (item, 128-key block) units of the ubatch are
// laid end to end and cut into C equal contiguous ranges, one per CTA, so
// every SM gets the same tensor work whatever the item count.  An item cut by
// a range boundary is computed in parts; each part leaves (m, l, unnormalised
// O) per row, and the CTA that finishes the item's last part combines them
// (an arrival counter decides who is last; nobody waits).
//
// Warp roles (384 threads = 3 warpgroups, one CTA per SM, persistent over items):
//   warps 0-3  softmax of query tile 0 (thread = query row = TMEM lane)
//   warps 4-7  softmax of query tile 1
//   warp 8     TMA producer: Q tiles (3-D map over [T][Hq][d]) and, for each
//              128-key block, the K and V boxes of the tile's pages (2-D map
//              over the pool rows), 128-byte swizzled, 2-stage ring
//   warps 9-10 MMA issuers, one thread each, one per query tile i:
//              S_i = Q_i K^T (SS, f16 -> f32 in TMEM), then O_i += P_i V with P_i
//              read from TMEM (TS), V MN-major in smem.  A thread's barrier waits cost
//              ~100 cycles each even when the phase has completed; with one issuer per
//              tile, taking turns block by block, the other tile's MMAs keep the tensor
//              pipe busy meanwhile.
//   warp 11    idle
// The softmax warpgroups raise their register budget with setmaxnreg so that a
// softmax thread holds its whole 128-column score row in registers (one TMEM round
// trip per block); the third warpgroup lowers its own.
// TMEM (512 columns): S0 | S1 | O0 | O1.  P_i (f16) overwrites the first 64
// columns of S_i.  Tile i's issuer runs PV_i(kb) then S_i(kb+1) (in order on the
// tensor core, so S_i(kb+1) overwrites P_i only after PV_i read it); the softmax of
// one tile runs while the tensor core works on the other.
//
// Masking: key j of a block is valid for query row t iff j < tok_kv_len[t]
// (causal per token).  Scores of invalid keys are replaced by -inf (select, so
// NaN cells never leak); V rows past the tile's longest kv_len are zeroed in
// shared memory before the PV product (0 * NaN would poison it).  The softmax
// is online in base 2 with a lazy rescale: O is rescaled only when a row's max
// grows by more than 2^8.
#include "tc.cuh"
#include "tmap.cuh"

namespace pa {

constexpr int kPfThreads = 384;
constexpr int kRegsSoftmax = 208;   // per thread, warpgroups 0 and 1
constexpr int kRegsOther = 88;      // per thread, warpgroup 2
// registers the split needs from the launch (168 x 384); checked on the host before launching
constexpr int kRegsSplitTotal = 2 * 128 * kRegsSoftmax + 128 * kRegsOther;
constexpr int kPfStages = 2;
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr int kBoxBytes = 128 * 128;  // 128 rows x 64 halves
constexpr float kRescaleThreshold = 8.0f;

template <int D, bool KV8 = false>
struct PfCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kTile = kHalves * kBoxBytes;  // 128 rows x D halves
  static constexpr int kQ0 = 0;
  static constexpr int kQ1 = kTile;
  static constexpr int kK = 2 * kTile;
  static constexpr int kV = kK + kPfStages * kTile;
  // FP8 pages: the codes of the next K block and of the next V block wait here
  static constexpr int kStgK = kV + kPfStages * kTile;
  static constexpr int kStgV = kStgK + (KV8 ? kBoxBytes : 0);
  static constexpr int kBarOff = kStgV + (KV8 ? kBoxBytes : 0);
  // masked variant: (sequence, position) of each key of the block, per softmax
  // warpgroup, two buffers; FP8 pages: the V scales of each stage's block (binary32),
  // then the K widening's scale table (binary16 hi and lo of each row)
  static constexpr int kCinfo = kBarOff + 256;
  static constexpr int kKtab = kCinfo + kPfStages * 128 * 4;
  static constexpr int kUsed = KV8 ? kKtab + 128 * 4 : kCinfo + 2 * 2 * 128 * 8;
  // at least ~120 KB so that a second CTA never shares the SM (and its TMEM)
  static constexpr int kSmem = (kUsed < 120 * 1024 ? 120 * 1024 : kUsed) + 1024;
  static_assert(kSmem <= 227 * 1024, "shared memory of one CTA");
};

struct PfBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[kPfStages], k_empty[kPfStages], v_full[kPfStages], v_empty[kPfStages];
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
  uint64_t turn[2];  // issuer turns: tile 1's issuer -> tile 0's, tile 0's -> tile 1's
  // FP8 pages: a block's codes have landed (K, V); the V scales of the stage's block are in
  uint64_t kc_full, vc_full;
  uint64_t vs_full[kPfStages];
  uint32_t tmem_base;
  int abort;
};

// Bounded wait that also gives up as soon as another role of the CTA gave up.
__device__ __forceinline__ bool pf_wait(uint64_t *bar, uint32_t parity, int *err,
                                        volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if ((it & 127u) == 127u && globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, PA_ERR_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

// ---- FP8 pages: E4M3 codes widened to binary16 in shared memory -----------------
// A block's codes (128 rows x 128 bytes, the 128-byte swizzle) land in a staging buffer
// one block ahead and are widened into the stage's binary16 tile once the stage is free.
// K: each element becomes binary16(code * scale of its key): the exact E4M3 value (cvt),
// times the scale split in two binary16 parts (hi = rn(s), lo = rn(s - hi)),
// x * hi + x * lo, so the result is the binary16 rounding of code * scale up to the
// rounding of the small x * lo term.  V: the exact E4M3 values; each key's scale goes
// into P instead (the softmax stores binary16(p * scale)), as in the split-KV decode.

// (hi, lo) of the scale s packed in one word: hi = rn(s), lo = rn(s - hi), binary16
__device__ __forceinline__ uint32_t scale_hl(float s) {
  const __half hi = __float2half_rn(s);
  const __half lo = __float2half_rn(s - __half2float(hi));
  const __half2 h = __halves2half2(hi, lo);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// (hi, hi) and (lo, lo) from a packed (hi, lo)
__device__ __forceinline__ uint2 hl_pairs(uint32_t hl) {
  return make_uint2(__byte_perm(hl, 0, 0x1010), __byte_perm(hl, 0, 0x3232));
}

// four E4M3 codes (byte i = element i) -> two binary16 pairs, exact
__device__ __forceinline__ void e4m3x4_widen(uint32_t w, uint32_t &p01, uint32_t &p23) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(p01), "=r"(p23) : "r"(w));
}

// x * hi + x * lo on binary16 pairs
__device__ __forceinline__ uint32_t h2_scale(uint32_t x, uint32_t hi, uint32_t lo) {
  uint32_t t, r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(t) : "r"(x), "r"(lo));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(hi), "r"(t));
  return r;
}

// 16 codes (one 16-byte chunk) -> 16 binary16 values in two 16-byte chunks, scaled by
// rs = (hi2, lo2) if SCALE; with CLR the codes are first masked by cmask.
template <bool SCALE, bool CLR>
__device__ __forceinline__ void widen_chunk(uint4 x, uint2 rs, const uint32_t (&cmask)[4],
                                            uint4 &o0, uint4 &o1) {
  const uint32_t wd[4] = {CLR ? x.x & cmask[0] : x.x, CLR ? x.y & cmask[1] : x.y,
                          CLR ? x.z & cmask[2] : x.z, CLR ? x.w & cmask[3] : x.w};
  uint32_t h[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    uint32_t p01, p23;
    e4m3x4_widen(wd[e], p01, p23);
    h[2 * e] = SCALE ? h2_scale(p01, rs.x, rs.y) : p01;
    h[2 * e + 1] = SCALE ? h2_scale(p23, rs.x, rs.y) : p23;
  }
  o0 = make_uint4(h[0], h[1], h[2], h[3]);
  o1 = make_uint4(h[4], h[5], h[6], h[7]);
}

// Widen rows [4 i0, 4 i1) of the 128 x 128 codes at stg (rows of 128 bytes, the 128-byte
// swizzle) into the binary16 tile (two boxes of 128 rows x 64 columns, the same swizzle).
// K (SCALE): one scale per row, packed (hi, lo) in rtab[row].  V (no SCALE): with CLR the
// codes of columns past the valid keys are cleared by cmask (they may be NaN codes).
// Iteration i covers rows 4i..4i+3 as two row pairs {R, R + 1}; lane (quarter-warp q,
// j = lane % 8) converts code chunk j of row R + ((q & 1) ^ (j / 4)) of pair q / 2, so a
// quarter-warp reads chunks 0-3 of one row of its pair and 4-7 of the other, and stores
// the even output chunk of each first: every 16-byte access of a quarter-warp lands in a
// distinct bank group, and no lane needs a select.
template <bool SCALE, bool CLR>
__device__ __forceinline__ void widen_tile(const unsigned char *stg, unsigned char *tile,
                                           const uint32_t *rtab, const uint32_t (&cmask)[4],
                                           int lane, int i0, int i1) {
  const int q = lane >> 3, j = lane & 7;
  const int r0 = 2 * (q >> 1) + ((q & 1) ^ (j >> 2));  // row in iterations' first group
  // row & 7 = r0 + 4 (i & 1): the swizzle phase of even and odd iterations
  const int ch = 2 * (j & 3);  // output chunks ch, ch + 1 of box j / 4
  const uint32_t ld_e = r0 * 128 + ((j ^ r0) << 4), ld_o = r0 * 128 + ((j ^ r0 ^ 4) << 4) + 512;
  const uint32_t s0_e = r0 * 128 + ((ch ^ r0) << 4), s1_e = r0 * 128 + (((ch + 1) ^ r0) << 4);
  const uint32_t s0_o = r0 * 128 + ((ch ^ r0 ^ 4) << 4) + 512,
                 s1_o = r0 * 128 + (((ch + 1) ^ r0 ^ 4) << 4) + 512;
  unsigned char *box = tile + (j >> 2) * kBoxBytes;
#pragma unroll 2
  for (int i = i0; i < i1; i += 2) {
    const uint32_t base = (uint32_t)i * 512;
    const uint4 xe = *reinterpret_cast<const uint4 *>(stg + base + ld_e);
    const uint4 xo = *reinterpret_cast<const uint4 *>(stg + base + ld_o);
    uint2 re = make_uint2(0, 0), ro = re;
    if (SCALE) {  // rows 4i + r0 and 4i + 4 + r0
      re = hl_pairs(rtab[4 * i + r0]);
      ro = hl_pairs(rtab[4 * i + 4 + r0]);
    }
    uint4 a0, a1, b0, b1;
    widen_chunk<SCALE, CLR>(xe, re, cmask, a0, a1);
    widen_chunk<SCALE, CLR>(xo, ro, cmask, b0, b1);
    *reinterpret_cast<uint4 *>(box + base + s0_e) = a0;
    *reinterpret_cast<uint4 *>(box + base + s1_e) = a1;
    *reinterpret_cast<uint4 *>(box + base + s0_o) = b0;
    *reinterpret_cast<uint4 *>(box + base + s1_o) = b1;
  }
}

// One contiguous piece of work of a CTA: key blocks [kb_b, kb_e) of one item.
// A CTA runs its unit range [w0, w1) as [ws, w1) then [w0, ws), ws the first unit of
// the item holding w1 - 1: the parts of the items it shares with its neighbours then
// both come early, and so does their combine, instead of at the end of the launch.
struct Seg {
  int tile, j;              // tile index, item within the tile
  int kb_b, kb_e;           // key-block range of this piece
  int nkb, max_kv;          // whole item: key blocks, longest kv_len of the tile
  int tile_start, n_tok;    // tokens of the tile
  int g, h0, h1;            // KV head, query heads of the pair
  long long w, w_end;       // unit position of this piece, end of the current run
  long long item_start;     // unit index of the item's key block 0
  int4 rest;                // start (tile, item, kb) of the second run; rest.x < 0: none
  long long rest_w0, rest_w1;
};

struct SegCtx {
  const int4 *tiles;
  const int *tile_off;
  int Hkv, NP, G, items_per_tile;
};

__device__ __forceinline__ void seg_load(Seg &s, const SegCtx &x) {
  int4 tl = x.tiles[s.tile];
  s.tile_start = tl.x;
  s.n_tok = tl.y;
  s.nkb = tl.z;
  s.max_kv = tl.w;
  s.g = s.j / x.NP;
  const int pair = s.j - s.g * x.NP;
  s.h0 = x.G >= 2 ? s.g * x.G + 2 * pair : s.g;
  s.h1 = s.h0 + 1;
  // an item spans pf_item_units(nkb) units: its key blocks, then virtual ones (no work)
  s.item_start = (long long)x.tile_off[s.tile] + (long long)s.j * pf_item_units(s.nkb);
}

// The next item, in the next tile that has keys when this tile's items are done (there
// is one: the caller checked that units are left before the end of the run).
__device__ __forceinline__ void seg_next_item(Seg &s, const SegCtx &x) {
  if (++s.j == x.items_per_tile) {
    s.j = 0;
    do { ++s.tile; } while (x.tiles[s.tile].z == 0);
  }
  seg_load(s, x);
}

// Settle at unit position s.w of the current item: the piece is the item's key blocks
// from there to the run's end; a position in an item's virtual units moves on to the
// next item.  False when no key block is left before the run's end.
__device__ __forceinline__ bool seg_settle(Seg &s, const SegCtx &x) {
  for (;;) {
    if (s.w >= s.w_end) return false;
    const long long kb = s.w - s.item_start;
    if (kb < s.nkb) {
      s.kb_b = (int)kb;
      s.kb_e = (int)min((long long)s.nkb, s.w_end - s.item_start);
      return true;
    }
    s.w = s.item_start + pf_item_units(s.nkb);
    if (s.w >= s.w_end) return false;
    seg_next_item(s, x);
  }
}

// Start a run of units [w0, w1) in the item start = (tile, item, -) that holds w0.
__device__ __forceinline__ bool seg_begin(Seg &s, const SegCtx &x, int4 start, long long w0,
                                          long long w1) {
  if (w0 >= w1) return false;
  s.tile = start.x;
  s.j = start.y;
  seg_load(s, x);
  s.w = w0;
  s.w_end = w1;
  return seg_settle(s, x);
}

__device__ __forceinline__ bool seg_next(Seg &s, const SegCtx &x) {
  // past the piece just done: the run ended inside the item, or the next item starts
  // after the item's virtual units
  if (s.kb_e == s.nkb) {
    s.w = s.item_start + pf_item_units(s.nkb);
    if (s.w < s.w_end) {
      seg_next_item(s, x);
      if (seg_settle(s, x)) return true;
    }
  }
  if (s.rest.x < 0) return false;
  const int4 r = s.rest;
  s.rest.x = -1;
  return seg_begin(s, x, r, s.rest_w0, s.rest_w1);
}

// The CTA's share of the prefill work, read from the plan.  Each warp role reads it
// afresh (through an opaque workspace pointer) instead of keeping values from the
// common prologue live into every role: registers live across the role split must fit
// the smallest setmaxnreg budget of the roles.
struct PfWork {
  SegCtx sx;
  int4 start;           // first (tile, item, key block) of this CTA
  long long W, w0, w1;  // total work units; this CTA's range [w0, w1)
  int C;                // CTAs the plan was cut for
};

__device__ __forceinline__ PfWork pf_work(const AttnArgs &a, int NP, int G) {
  uint64_t wsp = reinterpret_cast<uint64_t>(a.ws);
  asm volatile("" : "+l"(wsp));
  const unsigned char *ws = reinterpret_cast<const unsigned char *>(wsp);
  const WsHeader *hdr = reinterpret_cast<const WsHeader *>(ws);
  PfWork r;
  r.C = hdr->C;
  r.W = hdr->pf_work;
  const int c = blockIdx.x;
  r.w0 = (long long)c * r.W / r.C;
  r.w1 = (long long)(c + 1) * r.W / r.C;
  r.sx.tiles = reinterpret_cast<const int4 *>(ws + a.lay.tiles);
  r.sx.tile_off = reinterpret_cast<const int *>(ws + a.lay.tile_off);
  r.sx.Hkv = a.Hkv;
  r.sx.NP = NP;
  r.sx.G = G;
  r.sx.items_per_tile = a.Hkv * NP;
  r.start = reinterpret_cast<const int4 *>(ws + a.lay.pf_start)[c];
  return r;
}

// First piece of the CTA's work (see Seg for the order of its two runs).
__device__ __forceinline__ bool seg_first(Seg &s, const SegCtx &x, const PfWork &pw) {
  if (pw.w0 >= pw.w1) return false;
  const int tl = pw.start.w / x.items_per_tile, jl = pw.start.w - tl * x.items_per_tile;
  const long long ws = (long long)x.tile_off[tl] + (long long)jl * pf_item_units(x.tiles[tl].z);
  if (ws > pw.w0 && ws < pw.w1) {
    s.rest = pw.start;
    s.rest_w0 = pw.w0;
    s.rest_w1 = ws;
    return seg_begin(s, x, make_int4(tl, jl, 0, 0), ws, pw.w1);
  }
  s.rest.x = -1;
  return seg_begin(s, x, pw.start, pw.w0, pw.w1);
}

// FP8 pages: the staging and widening of one tensor's codes, whole warp (ISK: K, warp
// 8, which also loads the Q tiles; else V, warp 11).  Each warp stages its tensor's
// codes one block ahead: block n + 1 is copied (one TMA box into the staging buffer) as
// soon as block n has been widened out of it, and the block after that is asked into
// L2.  K rows are widened with their scales; V rows keep the exact E4M3 values and the
// warp hands the block's V scales to the softmax, which folds them into P.
template <bool ISK>
__device__ __forceinline__ void kv8_widen_role(const AttnArgs &a, const AttnMaps &maps,
                                               PfBars *bars, unsigned char *smem, int *err,
                                               volatile int *abort, int lane, int NQ, int NP,
                                               int G) {
  using Cfg = PfCfg<128, true>;
  const PfWork pw = pf_work(a, NP, G);
  const SegCtx &sx = pw.sx;
  const float *scales = ISK ? a.k_scale : a.v_scale;
  const CUtensorMap *map = ISK ? &maps.k : &maps.v;
  uint64_t *cfull = ISK ? &bars->kc_full : &bars->vc_full;
  uint64_t *tfull = ISK ? bars->k_full : bars->v_full;
  uint64_t *tempty = ISK ? bars->k_empty : bars->v_empty;
  unsigned char *stg = smem + (ISK ? Cfg::kStgK : Cfg::kStgV);
  unsigned char *tiles = smem + (ISK ? Cfg::kK : Cfg::kV);
  float *vsc = reinterpret_cast<float *>(smem + Cfg::kCinfo);  // V scales, per stage
  uint32_t *ktab = reinterpret_cast<uint32_t *>(smem + Cfg::kKtab);  // K rows' (hi, lo)
  const int c8 = lane & 7;
  // rows of one (page, head) block in the code maps (K keys, V dims: both 128); the
  // first row past the pool reads zeros
  const int oob_row = a.num_pages * a.Hkv * KB;
  Seg w{};
  bool more = seg_first(w, sx, pw);
  int kb = more ? w.kb_b : 0;
  // (page, head) index of block x of the current item's rows, -1 for a missing page
  auto block_of = [&](int x) -> int {
    const int page = a.tpt[(size_t)w.tile_start * a.max_pages + x];
    return page >= 0 && page < a.num_pages ? page * a.Hkv + w.g : -1;
  };
  // stage the codes of block (w, kb), (page, head) hp
  auto stage = [&](int hp) {
    if (lane != 0) return;
    if (ISK && hp < 0) atomicOr(err, PA_ERR_PAGE_RANGE);
    mbar_arrive_expect_tx(cfull, kBoxBytes);
    tc::tma_load_2d(stg, map, 0, hp >= 0 ? hp * KB : oob_row, cfull);
    if (kb + 1 < w.kb_e) {
      const int hn = block_of(kb + 1);
      if (hn >= 0) tc::tma_prefetch_2d(map, 0, hn * KB);
    }
    if (ISK && kb == w.kb_b)  // the item's Q tiles into L2 ahead of their load
      for (int hf = 0; hf < Cfg::kHalves; ++hf) {
        tc::tma_prefetch_3d(&maps.q, hf * 64, w.h0, w.tile_start);
        if (NQ == 2) tc::tma_prefetch_3d(&maps.q, hf * 64, w.h1, w.tile_start);
      }
  };
  // scales of keys 4 lane .. 4 lane + 3 of (page, head) hp; a missing page: zero scales
  // (and zero codes: the box is past the pool)
  auto load_scales = [&](int hp) -> float4 {
    return hp >= 0 ? __ldg(reinterpret_cast<const float4 *>(scales + (size_t)hp * KB) + lane)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  auto load_q = [&](int ts, int h0, int h1) {
    mbar_arrive_expect_tx(&bars->q_full, NQ * Cfg::kTile);
    for (int hf = 0; hf < Cfg::kHalves; ++hf) {
      tc::tma_load_3d(smem + Cfg::kQ0 + hf * kBoxBytes, &maps.q, hf * 64, h0, ts, &bars->q_full);
      if (NQ == 2)
        tc::tma_load_3d(smem + Cfg::kQ1 + hf * kBoxBytes, &maps.q, hf * 64, h1, ts, &bars->q_full);
    }
  };
  if (!more) return;
  // the current block: item, key count, scales
  int first, ts, h0, h1, nvalid;
  float4 s4;
  auto take = [&]() {  // (w, kb) becomes the current block; step (w, kb) to the next
    first = kb == w.kb_b;
    ts = w.tile_start;
    h0 = w.h0;
    h1 = w.h1;
    nvalid = min(KB, w.max_kv - kb * KB);
    if (++kb >= w.kb_e) {
      more = seg_next(w, sx);
      kb = more ? w.kb_b : 0;
    }
  };
  {
    const int hp = block_of(kb);
    s4 = load_scales(hp);
    if (ISK && lane == 0) load_q(w.tile_start, w.h0, w.h1);
    stage(hp);
    take();
  }
  uint32_t it = 0;
  int nitem = 0;
  for (;;) {
    const int st = it % kPfStages;
    const uint32_t ph = (it / kPfStages) & 1u;
    // the next block's (page, head) and scales, in flight during this block's widening
    const int nhp = more ? block_of(kb) : -1;
    const float4 s4n = more ? load_scales(nhp) : make_float4(0.f, 0.f, 0.f, 0.f);
    uint32_t cmask[4] = {~0u, ~0u, ~0u, ~0u};
    if (ISK) {
      __syncwarp();  // the previous block's table reads are done
      reinterpret_cast<uint4 *>(ktab)[lane] =
          make_uint4(scale_hl(s4.x), scale_hl(s4.y), scale_hl(s4.z), scale_hl(s4.w));
      __syncwarp();
    } else {
      // keys past the tile's longest kv_len: cleared codes (they may be NaN codes: P is 0
      // there, but 0 * NaN is NaN) and a zero scale
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int nb = min(max(nvalid - (16 * c8 + 4 * q), 0), 4);  // valid codes of the word
        cmask[q] = nb >= 4 ? ~0u : (1u << (8 * nb)) - 1u;
      }
    }
    if (!__all_sync(~0u, pf_wait(cfull, it & 1u, err, abort))) break;
    if (!__all_sync(~0u, pf_wait(&tempty[st], ph ^ 1u, err, abort))) break;
    unsigned char *tile = tiles + st * Cfg::kTile;
    if (ISK) {
      widen_tile<true, false>(stg, tile, ktab, cmask, lane, 0, 32);
    } else {
      // the block's V scales for the softmax (the stage's previous block is done with them)
      float4 sc = s4;
      if (4 * lane + 0 >= nvalid) sc.x = 0.f;
      if (4 * lane + 1 >= nvalid) sc.y = 0.f;
      if (4 * lane + 2 >= nvalid) sc.z = 0.f;
      if (4 * lane + 3 >= nvalid) sc.w = 0.f;
      reinterpret_cast<float4 *>(vsc + st * KB)[lane] = sc;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->vs_full[st]);
      if (nvalid < KB)
        widen_tile<false, true>(stg, tile, nullptr, cmask, lane, 0, 32);
      else
        widen_tile<false, false>(stg, tile, nullptr, cmask, lane, 0, 32);
    }
    // generic-proxy writes -> the tensor core's reads; the staging reads before the next
    // block's copy overwrites it
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) mbar_arrive(&tfull[st]);
    ++it;
    if (more) stage(nhp);
    if (ISK && first) {
      // a new item: its Q tiles once the previous item's MMAs have released them
      if (nitem > 0) {
        if (!__all_sync(~0u, lane != 0 || pf_wait(&bars->q_empty, (nitem - 1) & 1, err, abort)))
          break;
        if (lane == 0) load_q(ts, h0, h1);
      }
      ++nitem;
    }
    if (!more) break;
    s4 = s4n;
    take();
  }
}

// MASK: the unified-span baseline.  Every tile token's row names the same span of
// cells; key j is kept only if its cell belongs to the token's sequence at a position
// up to the token's own (cell_seq[slot] == tok_seq[t] && cell_pos[slot] <= tok_pos[t]),
// and the V rows of free cells (cell_seq < 0, which may hold NaN) are zeroed.
//
// KV8: FP8 pages (page size 128 = one key block, d = 128).  Warp 8 loads Q and the K
// codes and widens them; warp 11 loads and widens the V codes, stored transposed
// ([d][key]), so the binary16 V tile is K-major for the PV product.  Both widen into
// the stage's binary16 tile (see widen_tile); the MMA issuers and the softmax then run
// exactly as for binary16 pages.
template <int D, bool MASK, bool KV8>
__global__ void __launch_bounds__(kPfThreads, 1)
k_prefill(AttnArgs a, const __grid_constant__ AttnMaps maps) {
  static_assert(!(MASK && KV8), "one variant at a time");
  static_assert(!KV8 || D == 128, "FP8 pages: d 128");
  using Cfg = PfCfg<D, KV8>;
  // rows of a split part's record: O[D] | m | l | 2 unused (D + 4 rows of 128 floats)
  constexpr int kPartStride = D + 4;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  unsigned char *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  PfBars *bars = reinterpret_cast<PfBars *>(smem + Cfg::kBarOff);

  WsHeader *hdr = reinterpret_cast<WsHeader *>(a.ws);
  int *err = &hdr->err;
  const int4 *tiles = reinterpret_cast<const int4 *>(a.ws + a.lay.tiles);
  const int G = a.Hq / a.Hkv;
  const int NQ = G >= 2 ? 2 : 1;
  const int NP = G >= 2 ? G / 2 : 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = hdr->C;
  const int c = blockIdx.x;
  if (c >= C) return;
  // tiles whose tokens all have kv_len 0 own no work unit: their rows are zero
  for (int t = c; t < hdr->n_tiles; t += C) {
    const int4 tl = tiles[t];
    if (tl.z != 0) continue;
    for (int x = tid; x < tl.y * a.Hq * (D / 8); x += blockDim.x)
      reinterpret_cast<uint4 *>(a.out + (size_t)tl.x * a.Hq * D)[x] = make_uint4(0, 0, 0, 0);
  }
  {
    const PfWork pw = pf_work(a, NP, G);
    if (pw.w0 >= pw.w1) return;
  }
  if (tid == 0) {
    // stages and Q tiles are released by both MMA-issuing threads (one per query tile)
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, NQ);
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], NQ);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], NQ);
    }
    mbar_init(&bars->turn[0], 1);
    mbar_init(&bars->turn[1], 1);
    mbar_init(&bars->kc_full, 1);
    mbar_init(&bars->vc_full, 1);
    for (int s = 0; s < kPfStages; ++s) mbar_init(&bars->vs_full[s], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 128);
      mbar_init(&bars->o_full[i], 1);
      mbar_init(&bars->o_empty[i], 128);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&bars->tmem_base, 512);
    tc::tmem_relinquish();
  }
  if (warp == kWarpTma && lane == 0) {
    tc::prefetch_tmap(&maps.q);
    tc::prefetch_tmap(&maps.k);
    tc::prefetch_tmap(&maps.v);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  volatile int *abort = &bars->abort;
  const int cap = a.max_pages * a.P;

  if (warp >= 8) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
   if (KV8 && warp == kWarpTma) {
    kv8_widen_role<true>(a, maps, bars, smem, err, abort, lane, NQ, NP, G);
   } else if (KV8 && warp == kWarpTma + 3) {
    kv8_widen_role<false>(a, maps, bars, smem, err, abort, lane, NQ, NP, G);
   } else if (!KV8 && warp == kWarpTma && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    {
      const PfWork pw = pf_work(a, NP, G);
      const SegCtx &sx = pw.sx;
      uint32_t it = 0;
      int nitem = 0;
      const int pages_per_block = KB / a.P;
      const int oob_row = a.num_pages * a.Hkv * a.P;  // first row past the pool: zero fill
      Seg w{};
      const int32_t *row = nullptr;
      // row coordinate of page j of key block kb in the pool map (past the end when
      // invalid: the box is zero-filled and nothing outside the pool is touched)
      auto ycoord = [&](int kb, int j) {
        int page = row[kb * pages_per_block + j];
        if (page < 0 || page >= a.num_pages) {
          atomicOr(err, PA_ERR_PAGE_RANGE);
          return oob_row;
        }
        return (page * a.Hkv + w.g) * a.P;
      };
      // K and V boxes of key block kb into ring stage it % kPfStages
      auto load_kv = [&](int kb) -> bool {
        const int st = it % kPfStages;
        const uint32_t ph = (it / kPfStages) & 1u;
        const int keys = min(KB, w.max_kv - kb * KB);
        const int npg = (keys + a.P - 1) / a.P;
        const uint32_t bytes = (uint32_t)npg * a.P * 128u * Cfg::kHalves;
        if (!pf_wait(&bars->k_empty[st], ph ^ 1u, err, abort)) return false;
        mbar_arrive_expect_tx(&bars->k_full[st], bytes);
        for (int j = 0; j < npg; ++j)
          for (int hf = 0; hf < Cfg::kHalves; ++hf)
            tc::tma_load_2d(smem + Cfg::kK + st * Cfg::kTile + hf * kBoxBytes + j * a.P * 128,
                            &maps.k, hf * 64, ycoord(kb, j), &bars->k_full[st]);
        if (!pf_wait(&bars->v_empty[st], ph ^ 1u, err, abort)) return false;
        mbar_arrive_expect_tx(&bars->v_full[st], bytes);
        for (int j = 0; j < npg; ++j)
          for (int hf = 0; hf < Cfg::kHalves; ++hf)
            tc::tma_load_2d(smem + Cfg::kV + st * Cfg::kTile + hf * kBoxBytes + j * a.P * 128,
                            &maps.v, hf * 64, ycoord(kb, j), &bars->v_full[st]);
        ++it;
        return true;
      };
      for (bool more = seg_first(w, sx, pw); more; more = seg_next(w, sx)) {
        row = a.tpt + (size_t)w.tile_start * a.max_pages;
        int kb = w.kb_b;
        if (nitem > 0) {
          // the first key block of this item goes into the ring before the Q tiles wait for
          // the previous item to release them
          if (!load_kv(kb++)) break;
          if (!pf_wait(&bars->q_empty, (nitem - 1) & 1, err, abort)) break;
        }
        mbar_arrive_expect_tx(&bars->q_full, NQ * Cfg::kTile);
        for (int hf = 0; hf < Cfg::kHalves; ++hf) {
          tc::tma_load_3d(smem + Cfg::kQ0 + hf * kBoxBytes, &maps.q, hf * 64, w.h0, w.tile_start,
                          &bars->q_full);
          if (NQ == 2)
            tc::tma_load_3d(smem + Cfg::kQ1 + hf * kBoxBytes, &maps.q, hf * 64, w.h1,
                            w.tile_start, &bars->q_full);
        }
        {  // the next item's Q tiles into L2, so that its load at the switch is short
          Seg nx = w;
          if (seg_next(nx, sx))
            for (int hf = 0; hf < Cfg::kHalves; ++hf) {
              tc::tma_prefetch_3d(&maps.q, hf * 64, nx.h0, nx.tile_start);
              if (NQ == 2) tc::tma_prefetch_3d(&maps.q, hf * 64, nx.h1, nx.tile_start);
            }
        }
        bool ok = true;
        for (; kb < w.kb_e && ok; ++kb) ok = load_kv(kb);
        if (!ok) break;
        ++nitem;
      }
    }
   } else if ((warp == kWarpMma || warp == kWarpMma + 1) && lane == 0 &&
              warp - kWarpMma < NQ) {
    // ------------------------------------------------------------ MMA issuers
    // One thread per query tile: warp 9 issues tile 0's MMAs, warp 10 tile 1's.  Each
    // thread's waits then leave the tensor pipe to the other thread's MMAs.
    const int qi = warp - kWarpMma;
    const PfWork pw = pf_work(a, NP, G);
    const SegCtx &sx = pw.sx;
    constexpr uint32_t idS = tc::idesc_f16(128, 128, false);
    // V: MN-major ([key][d] rows) for binary16 pages; K-major ([d][key] rows) for FP8
    // pages, whose V codes are stored transposed
    constexpr uint32_t idPV = tc::idesc_f16(128, D, !KV8);
    const uint32_t sQ0 = smem_u32(smem + Cfg::kQ0), sQ1 = smem_u32(smem + Cfg::kQ1);
    const uint32_t sK = smem_u32(smem + Cfg::kK), sV = smem_u32(smem + Cfg::kV);
    // Operand descriptors by their low words (the high word is one constant): a k-step
    // moves the start address (bits 0-13, in 16-byte units) by a constant, and every
    // shared-memory address here is below 256 KB, so the add never carries out of the
    // field.  Each group's base goes through opaque() so that its eight descriptors are
    // formed at issue time, one add each, rather than held in registers.
    static_assert(kPfStages == 2, "two K/V stages");
    const uint32_t lQ0 = tc::sdesc_lo(sQ0, 16), lQ1 = tc::sdesc_lo(sQ1, 16);
    const uint32_t lK0 = tc::sdesc_lo(sK, 16), lK1 = tc::sdesc_lo(sK + Cfg::kTile, 16);
    const uint32_t lV0 = tc::sdesc_lo(sV, KV8 ? 16 : kBoxBytes),
                   lV1 = tc::sdesc_lo(sV + Cfg::kTile, KV8 ? 16 : kBoxBytes);
    auto issue_S = [&](int i, int st) {
      const uint32_t d = tmem + i * 128;
      const uint32_t a0 = tc::opaque(i ? lQ1 : lQ0), b0 = tc::opaque(st ? lK1 : lK0);
      tc::mma_ss_lo<0>(d, a0, b0, idS);
#pragma unroll
      for (int kk = 1; kk < D / 16; ++kk) {
        const uint32_t off16 = ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4;
        tc::mma_ss_lo<1>(d, a0 + off16, b0 + off16, idS);
      }
    };
    // O_i (+)= P_i V over the first nk 16-key steps of the block
    auto issue_PV = [&](int i, int st, bool acc, int nk) {
      const uint32_t d = tmem + 256 + i * D;
      const uint32_t p = tmem + i * 128;
      const uint32_t b0 = tc::opaque(st ? lV1 : lV0);
      tc::mma_ts_lo_pred(d, p, b0, idPV, acc ? 1u : 0u);
#pragma unroll
      for (int kk = 1; kk < KB / 16; ++kk) {
        // a 16-key step: 16 rows of the MN-major tile, or 32 bytes along the K-major rows
        const uint32_t off16 = KV8 ? ((kk / 4) * kBoxBytes + (kk % 4) * 32) >> 4
                                   : (uint32_t)((kk * 2048) >> 4);
        if (kk < nk) tc::mma_ts_lo<1>(d, p + kk * 8, b0 + off16, idPV);
      }
    };
    uint32_t it = 0, sc = 0;
    int nitem = 0;
    Seg w;
    for (bool more = seg_first(w, sx, pw); more; more = seg_next(w, sx)) {
      const int nseg = w.kb_e - w.kb_b;
      bool ok = pf_wait(&bars->q_full, nitem & 1, err, abort);
      const int st0 = it % kPfStages;
      ok = ok && pf_wait(&bars->k_full[st0], (it / kPfStages) & 1u, err, abort);
      if (!ok) break;
      tc::fence_after_sync();
      issue_S(qi, st0);
      tc::commit(&bars->s_full[qi]);
      tc::commit(&bars->k_empty[st0]);
      for (int kk = 0; kk < nseg; ++kk) {
        const int kb = w.kb_b + kk;  // absolute key block
        const uint32_t cur = it + kk;
        const int st = cur % kPfStages;
        const bool last = kk + 1 == nseg;
        if (!pf_wait(&bars->v_full[st], (cur / kPfStages) & 1u, err, abort)) { ok = false; break; }
        // the item's last block may hold fewer than 128 valid keys: the PV product then
        // runs only over the 16-key steps that hold valid keys, and the rows of the last
        // such step past the valid ones are zeroed (P is 0 there, but 0 * NaN is NaN).
        // Rows are 128 B, so whole rows are zeroed and the swizzle inside a row does not
        // matter.  Tile 0's issuer zeroes before its PV; tile 1's issues its PV only after
        // tile 0's turn, which ends after the zeroing.
        int nk = KB / 16;
        const int nvalid = w.max_kv - kb * KB;
        if (kb + 1 == w.nkb && nvalid < KB) {
          nk = (nvalid + 15) / 16;
          const int n16 = (nk * 16 - nvalid) * 8;
          if (!KV8 && qi == 0 && n16 > 0) {  // FP8 pages: cleared when widened
            for (int hf = 0; hf < Cfg::kHalves; ++hf) {
              uint4 *base = reinterpret_cast<uint4 *>(smem + Cfg::kV + st * Cfg::kTile +
                                                      hf * kBoxBytes + nvalid * 128);
              for (int x = 0; x < n16; ++x) base[x] = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async();
          }
        }
        if (!pf_wait(&bars->p_full[qi], (sc + kk) & 1u, err, abort)) { ok = false; break; }
        if (kk == 0 && nitem > 0 && !pf_wait(&bars->o_empty[qi], (nitem - 1) & 1, err, abort)) {
          ok = false;
          break;
        }
        // every wait of the block comes before its MMAs, so that PV_i(kb) and S_i(kb+1)
        // go to the tensor pipe as one burst of 16 (a wait between them would leave the
        // pipe idle: each costs ~100 cycles even when the phase has completed)
        const uint32_t nxt = cur + 1;
        const int st2 = nxt % kPfStages;
        if (!last && !pf_wait(&bars->k_full[st2], (nxt / kPfStages) & 1u, err, abort)) {
          ok = false;
          break;
        }
        // strict alternation of the two issuers, block by block: tile 0's PV(kb), S(kb+1),
        // then tile 1's, then tile 0's PV(kb+1) ...  A thread waits for its turn while the
        // other's MMAs run, and the two softmax warpgroups stay half a period apart.
        if (NQ == 2 && (qi == 1 || cur > 0) &&
            !pf_wait(&bars->turn[qi], (qi ? cur : cur - 1) & 1u, err, abort)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        issue_PV(qi, st, kk > 0, nk);
        if (last) tc::commit(&bars->o_full[qi]);
        tc::commit(&bars->v_empty[st]);
        if (!last) {
          issue_S(qi, st2);
          tc::commit(&bars->s_full[qi]);
          tc::commit(&bars->k_empty[st2]);
        }
        if (NQ == 2) mbar_arrive(&bars->turn[qi ^ 1]);
      }
      if (!ok) break;
      tc::commit(&bars->q_empty);
      it += nseg;
      sc += nseg;
      ++nitem;
    }
   }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    const int wg = warp >> 2;
    const int wl = warp & 3;
    const int row = wl * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wl * 32) << 16;
    const uint32_t tS = tmem + wg * 128 + lane_off;
    const uint32_t tO = tmem + 256 + wg * D + lane_off;
    if (wg < NQ) {
      const PfWork pw = pf_work(a, NP, G);
      const SegCtx &sx = pw.sx;
      const long long W = pw.W, w0 = pw.w0;
      const int C = pw.C;
      uint32_t sc = 0;
      int nitem = 0;
      float *parts = reinterpret_cast<float *>(a.ws + a.lay.partials);
      int *cnt = reinterpret_cast<int *>(a.ws + a.lay.pf_cnt);
      Seg w;
      for (bool more = seg_first(w, sx, pw); more; more = seg_next(w, sx)) {
        const int h = wg ? w.h1 : w.h0;
        const int tok = w.tile_start + row;
        const bool valid = row < w.n_tok;
        const int L = valid ? min(max(a.kv[tok], 0), cap) : 0;
        // masked variant: this row's (sequence, position); -2 matches no cell
        const int my_seq = MASK && valid ? a.tok_seq[tok] : -2;
        const int my_pos = MASK && valid ? a.tok_pos[tok] : -1;
        // (sequence, position) of key `row` of block kb of this item; -1 past the keys
        auto cell_of = [&](int kb) -> int2 {
          const int key = kb * KB + row;
          if (!MASK || kb >= w.nkb || key >= w.max_kv) return make_int2(-1, 0);
          const int page = a.tpt[(size_t)w.tile_start * a.max_pages + key / a.P];
          if (page < 0 || page >= a.num_pages) return make_int2(-1, 0);
          const size_t slot = (size_t)page * a.P + key % a.P;
          return make_int2(a.cell_seq[slot], a.cell_pos[slot]);
        };
        int2 nxt_cell = cell_of(w.kb_b);
        uint4 *orow = reinterpret_cast<uint4 *>(a.out + ((size_t)tok * a.Hq + h) * D);
        const int nseg = w.kb_e - w.kb_b;
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        const bool split = w.kb_b != 0 || w.kb_e != w.nkb;
        for (int kk = 0; kk < nseg; ++kk) {
          const int kb = w.kb_b + kk;
          if (split && kk + 1 == nseg && wl == 0 && lane == 0) {
            // the records of the item's other parts, which this warpgroup may combine
            // after this block: into L2 now (one written long ago may have left it)
            const long long ie = w.item_start + w.nkb;
            for (int cc = cta_of_unit(w.item_start, W, C); cc <= cta_of_unit(ie - 1, W, C); ++cc)
              if (cc != c && cta_has_units(cc, W, C))
                bulk_prefetch_l2(parts + ((size_t)(2 * cc + (w.item_start <= (long long)cc * W / C
                                                                  ? 0 : 1)) * 2 + wg) *
                                             (size_t)kPartStride * 128,
                                 kPartStride * 128 * 4);
          }
          const int2 my_cell = nxt_cell;
          if (MASK && kk + 1 < nseg) nxt_cell = cell_of(kb + 1);  // loads in flight meanwhile
          if (!pf_wait(&bars->s_full[wg], (sc + kk) & 1u, err, abort)) { ok = false; break; }
          tc::fence_after_sync();
          const int nv = min(max(L - kb * KB, 0), KB);  // valid keys of this row here
          const bool wfull = !MASK && __all_sync(0xffffffffu, nv == KB);
          const int2 *cb = reinterpret_cast<const int2 *>(smem + Cfg::kCinfo) +
                           (wg * 2 + ((sc + kk) & 1u)) * 128;
          if (MASK) {
            // every thread of the warpgroup publishes its key's cell, then reads all 128
            // (two buffers: a buffer is rewritten two blocks later, after the next sync)
            const_cast<int2 *>(cb)[row] = my_cell;
            asm volatile("bar.sync %0, 128;" ::"r"(1 + wg) : "memory");
          }
          // The whole 128-column score row in one TMEM round trip (the tensor core keeps
          // TMEM busy, so each round trip costs hundreds of cycles).  Row max of the raw
          // scores over the valid keys (scale > 0 commutes with max); masked scores become
          // -inf by select, so NaN cells never propagate.
          uint32_t t[128];
          tc::ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(t));
          tc::ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(t + 32));
          tc::ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(t + 64));
          tc::ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(t + 96));
          tc::wait_ld();
          if (MASK) {
            // the kept keys as a 128-bit mask first (a rolled loop over the cells keeps
            // few registers live beside the score row), then applied to the scores
            uint32_t mw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t m = 0;
#pragma unroll 4
              for (int b = 0; b < 32; ++b) {
                const int2 ce = cb[q * 32 + b];
                m |= (q * 32 + b < nv && ce.x == my_seq && ce.y <= my_pos) ? 1u << b : 0u;
              }
              mw[q] = m;
            }
#pragma unroll
            for (int j = 0; j < 128; ++j)
              t[j] = (mw[j >> 5] >> (j & 31)) & 1u ? t[j] : 0xff800000u;
          } else if (!wfull) {
#pragma unroll
            for (int j = 0; j < 128; ++j) t[j] = j < nv ? t[j] : 0xff800000u;  // -inf
          }
          float mx = -INFINITY;
#pragma unroll
          for (int j = 0; j < 128; j += 2)
            mx = fmax3(mx, __uint_as_float(t[j]), __uint_as_float(t[j + 1]));
          const float m_new = fmaxf(m_run, mx * a.scale_log2);
          const bool need = m_new > m_run + kRescaleThreshold;
          float alpha = 1.f;
          if (need) {
            alpha = exp2_approx(m_run - m_new);
            m_run = m_new;
          }
          // p = 2^(s * scale_log2 - m), one packed FMA per pair, then ex2; a row with no
          // valid key yet uses m = 0 so that its -inf scores give exactly 0.  P (f16) goes
          // to the first 64 columns of S (already in registers): half hh lands in columns
          // [32hh, 32hh+32).
          const float m_use = m_run == -INFINITY ? 0.f : m_run;
          const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
          const float2 nm2 = make_float2(-m_use, -m_use);
          float2 rs2 = make_float2(0.f, 0.f);
          // FP8 pages: P carries each key's V scale (binary16(p * scale); the row sum l
          // does not), so the V tile holds the exact E4M3 values
          const float2 *vs2 = nullptr;
          if (KV8) {
            const uint32_t cur = sc + kk;
            const int st = cur % kPfStages;
            if (!pf_wait(&bars->vs_full[st], (cur / kPfStages) & 1u, err, abort)) { ok = false; break; }
            vs2 = reinterpret_cast<const float2 *>(smem + Cfg::kCinfo) + st * (KB / 2);
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const int c = 32 * q4 + j;
              const float2 x =
                  ffma2(make_float2(__uint_as_float(t[c]), __uint_as_float(t[c + 1])), sc2, nm2);
              float2 p = make_float2(exp2_approx(x.x), exp2_approx(x.y));
              rs2 = fadd2(rs2, p);
              if (KV8) p = fmul2(p, vs2[c >> 1]);
              __half2 hp = __floats2half2_rn(p.x, p.y);
              pk[j >> 1] = *reinterpret_cast<uint32_t *>(&hp);
            }
            tc::st16(tS + 16 * q4, pk);
          }
          const float rs = rs2.x + rs2.y;
          l_run = l_run * alpha + rs;
          if (kk > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tc::ld32(tO + c * 32, o);
              tc::wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
              tc::st32(tO + c * 32, o);
            }
          }
          if (MASK && wg == 0) {
            // free cells may hold NaN: their V rows are zeroed before this block's PV
            // products (the other tile's issuer runs its PV only after tile 0's turn)
            const uint32_t cur = sc + kk;
            const int st = cur % kPfStages;
            if (!pf_wait(&bars->v_full[st], (cur / kPfStages) & 1u, err, abort)) { ok = false; break; }
            if (my_cell.x < 0) {
              for (int hf = 0; hf < Cfg::kHalves; ++hf) {
                uint4 *vrow = reinterpret_cast<uint4 *>(smem + Cfg::kV + st * Cfg::kTile +
                                                        hf * kBoxBytes + row * 128);
#pragma unroll
                for (int x = 0; x < 8; ++x) vrow[x] = make_uint4(0, 0, 0, 0);
              }
            }
            fence_proxy_async();
          }
          tc::wait_st();
          tc::fence_before_sync();
          mbar_arrive(&bars->p_full[wg]);
        }
        if (!ok) break;
        if (!pf_wait(&bars->o_full[wg], nitem & 1, err, abort)) break;
        tc::fence_after_sync();
        if (w.kb_b == 0 && w.kb_e == w.nkb) {
          // the whole item: normalise and store f16
          const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
          uint32_t o[D];  // the whole O row in one TMEM round trip
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch)
            tc::ld32(tO + ch * 32, *reinterpret_cast<uint32_t(*)[32]>(o + ch * 32));
          tc::wait_ld();
          if (valid) {
#pragma unroll
            for (int q = 0; q < D / 8; ++q) {
              uint32_t hw[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                __half2 hv = __floats2half2_rn(__uint_as_float(o[q * 8 + 2 * e]) * inv,
                                               __uint_as_float(o[q * 8 + 2 * e + 1]) * inv);
                hw[e] = *reinterpret_cast<uint32_t *>(&hv);
              }
              orow[q] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            }
          }
          tc::fence_before_sync();
          mbar_arrive(&bars->o_empty[wg]);
        } else {
          // one part of a split item: leave (O unnormalised, m, l) in this CTA's slot.  A
          // slot holds D + 2 rows of 128 floats (element-major: element e of query row r
          // at [e][r]), so that a warp's accesses to one element are one 128-byte line.
          const bool first_seg = w.item_start <= w0;
          const int my_slot = 2 * c + (first_seg ? 0 : 1);
          auto slot_base = [&](int sl) {
            return parts + ((size_t)sl * 2 + wg) * (size_t)kPartStride * 128 + row;
          };
          float *rec = slot_base(my_slot);
          uint32_t o[D];
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch)
            tc::ld32(tO + ch * 32, *reinterpret_cast<uint32_t(*)[32]>(o + ch * 32));
          tc::wait_ld();
#pragma unroll
          for (int e = 0; e < D; ++e) rec[e * 128] = __uint_as_float(o[e]);
          rec[D * 128] = m_run;
          rec[(D + 1) * 128] = l_run;
          tc::fence_before_sync();
          mbar_arrive(&bars->o_empty[wg]);
          // count the parts that have landed; the last one combines (no waiting)
          const long long item_end = w.item_start + w.nkb;
          const int c1 = cta_of_unit(w.item_start, W, C), c2 = cta_of_unit(item_end - 1, W, C);
          int n_parts = 0;
          for (int cc = c1; cc <= c2; ++cc) n_parts += cta_has_units(cc, W, C) ? 1 : 0;
          // one counter per (item, warpgroup, warp): a warp's 32 rows only need the same
          // 32 rows of the other parts, so warps decide independently (no cross-warp wait)
          int *my_cnt = &cnt[((w.tile * sx.items_per_tile + w.j) * 2 + wg) * 4 + wl];
          __threadfence();
          __syncwarp();
          int old = 0;
          if (lane == 0) old = atomicAdd(my_cnt, 1);
          old = __shfl_sync(0xffffffffu, old, 0);
          if (old == n_parts - 1) {
            __threadfence();
            // Parts are folded in CTA order with the same arithmetic whichever CTA
            // combines, so results are reproducible.  The other parts were written by
            // other SMs: read them past L1 (ld.global.cg).
            auto slot_of = [&](int cc) {
              return 2 * cc + (w.item_start <= (long long)cc * W / C ? 0 : 1);
            };
            auto store_chunk = [&](int ch, const float (&acc)[16], float inv) {
              if (!valid) return;
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                uint32_t hw[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  __half2 hv = __floats2half2_rn(acc[q * 8 + 2 * e] * inv,
                                                 acc[q * 8 + 2 * e + 1] * inv);
                  hw[e] = *reinterpret_cast<uint32_t *>(&hv);
                }
                orow[ch * 2 + q] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
              }
            };
            constexpr int kFastParts = 3;
            if (!MASK && W >= C && c2 - c1 < kFastParts) {
              // Every CTA of [c1, c2] holds a part (W >= C: no CTA is empty), at most
              // three.  All parts, this CTA's included, are read back from their records,
              // and every load of a step is issued before any of its values is used: the
              // (m, l) of all parts in one round trip, then the 16-element chunks with the
              // next chunk's loads in flight while the current one is folded and stored.
              const int np = c2 - c1 + 1;
              const float *rp[kFastParts];
              float mk[kFastParts], lk[kFastParts], fk[kFastParts];
#pragma unroll
              for (int k = 0; k < kFastParts; ++k) {
                rp[k] = slot_base(slot_of(k < np ? c1 + k : c1));
                mk[k] = k < np ? __ldcg(rp[k] + D * 128) : -INFINITY;
                lk[k] = k < np ? __ldcg(rp[k] + (D + 1) * 128) : 0.f;
              }
              float M = -INFINITY;
#pragma unroll
              for (int k = 0; k < kFastParts; ++k) M = fmaxf(M, mk[k]);
              float Ls = 0.f;
#pragma unroll
              for (int k = 0; k < kFastParts; ++k) {
                fk[k] = (mk[k] == -INFINITY) ? 0.f : exp2_approx(mk[k] - M);
                if (k < np) Ls += (mk[k] == -INFINITY) ? 0.f : lk[k] * fk[k];
              }
              const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
              float vb[2][kFastParts][16];
              auto load_chunk = [&](int ch, float (&v)[kFastParts][16]) {
#pragma unroll
                for (int k = 0; k < kFastParts; ++k)
#pragma unroll
                  for (int e = 0; e < 16; ++e)
                    v[k][e] = k < np ? __ldcg(rp[k] + (ch * 16 + e) * 128) : 0.f;
              };
              load_chunk(0, vb[0]);
#pragma unroll
              for (int ch = 0; ch < D / 16; ++ch) {
                if (ch + 1 < D / 16) load_chunk(ch + 1, vb[(ch + 1) & 1]);
                float acc[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[e] = 0.f;
#pragma unroll
                for (int k = 0; k < kFastParts; ++k) {
                  if (k >= np) continue;
#pragma unroll
                  for (int e = 0; e < 16; ++e) acc[e] += fk[k] * vb[ch & 1][k][e];
                }
                store_chunk(ch, acc, inv);
              }
            } else {
              // any number of parts: this CTA's own part from registers, the others one
              // chunk at a time
              float M = -INFINITY;
              for (int cc = c1; cc <= c2; ++cc) {
                if (!cta_has_units(cc, W, C)) continue;
                M = fmaxf(M, cc == c ? m_run : __ldcg(slot_base(slot_of(cc)) + D * 128));
              }
              float Ls = 0.f;
              for (int cc = c1; cc <= c2; ++cc) {
                if (!cta_has_units(cc, W, C)) continue;
                const float *r = slot_base(slot_of(cc));
                const float m_p = cc == c ? m_run : __ldcg(r + D * 128);
                const float l_p = cc == c ? l_run : __ldcg(r + (D + 1) * 128);
                Ls += (m_p == -INFINITY) ? 0.f : l_p * exp2_approx(m_p - M);
              }
              const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
              for (int ch = 0; ch < D / 16; ++ch) {
                float acc[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[e] = 0.f;
                for (int cc = c1; cc <= c2; ++cc) {
                  if (!cta_has_units(cc, W, C)) continue;
                  if (cc == c) {
                    const float f = (m_run == -INFINITY) ? 0.f : exp2_approx(m_run - M);
#pragma unroll
                    for (int e = 0; e < 16; ++e) acc[e] += f * __uint_as_float(o[ch * 16 + e]);
                  } else {
                    const float *r = slot_base(slot_of(cc));
                    float v[16];
                    const float m_p = __ldcg(r + D * 128);
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = __ldcg(r + (ch * 16 + e) * 128);
                    const float f = (m_p == -INFINITY) ? 0.f : exp2_approx(m_p - M);
#pragma unroll
                    for (int e = 0; e < 16; ++e) acc[e] += f * v[e];
                  }
                }
                store_chunk(ch, acc, inv);
              }
            }
            if (lane == 0) *my_cnt = 0;  // ready for the next run of this plan
          }
        }
        sc += nseg;
        ++nitem;
      }
    }
  }

  __syncthreads();
  if (*abort && (warp == kWarpMma || warp == kWarpMma + 1) && lane == 0) {
    // a role gave up: let the tensor pipe drain (bounded) before TMEM is freed
    uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) {
    }
  }
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <int D, bool MASK, bool KV8>
static cudaError_t launch_prefill_t(const AttnArgs &a, int num_sms, const AttnMaps *maps,
                                    cudaStream_t s) {
  using Cfg = PfCfg<D, KV8>;
  static PerDeviceOnce setup;
  if (setup.first()) {
    // setmaxnreg.inc can only draw on registers the block was launched with: refuse to
    // launch (rather than wait forever) if the compiled allocation does not cover the split
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, k_prefill<D, MASK, KV8>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * kPfThreads < kRegsSplitTotal) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(k_prefill<D, MASK, KV8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::kSmem);
    if (e != cudaSuccess) return e;
    setup.mark();
  }
  k_prefill<D, MASK, KV8><<<num_sms, kPfThreads, Cfg::kSmem, s>>>(a, *maps);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const AttnArgs &a, int num_sms, const void *tmaps, cudaStream_t s) {
  const AttnMaps *maps = static_cast<const AttnMaps *>(tmaps);
  const bool mask = a.cell_seq != nullptr;
  if (a.k_scale) {  // FP8 pages: page size 128, d 128
    if (a.D != 128 || a.P != KB || mask) return cudaErrorInvalidValue;
    return launch_prefill_t<128, false, true>(a, num_sms, maps, s);
  }
  if (a.D == 128) return mask ? launch_prefill_t<128, true, false>(a, num_sms, maps, s)
                              : launch_prefill_t<128, false, false>(a, num_sms, maps, s);
  if (a.D == 64) return mask ? launch_prefill_t<64, true, false>(a, num_sms, maps, s)
                             : launch_prefill_t<64, false, false>(a, num_sms, maps, s);
  return cudaErrorInvalidValue;
}

}  // namespace pa
