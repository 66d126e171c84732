// Split-KV decode attention with a fused log-sum-exp reduce (sm_103a).
//
// The work is the planned decode tokens.  Each (token i, KV head g) owns
// ceil(kv_len / 128) key blocks ("units"); all units of all (i, g) are laid end
// to end and cut into C = min(gridDim.x, units) equal contiguous ranges, one per
// CTA (one CTA per SM), so every SM streams the same number of KV bytes whatever
// the length mix.  A (i, g) whose units fall in one CTA is finished there; one
// that spans CTAs leaves one partial (m, l, acc) per CTA and the CTA whose part
// arrives last combines them (the partition + reduce scheme of the CacheFlow page,
// section 核心架构 3, "Paged Attention V2", fused into one launch: an
// acquire/release arrival counter decides who combines, nobody waits).
//
// CTA = 12 warps.  One producer thread streams, for every unit, the 128 K rows
// and 128 V rows of the block as 128-byte-swizzled TMA boxes (one per page and
// 64-dim half) and, at the start of each (i, g), the G query rows, into a ring
// of stages; it runs up to NS units ahead.  Eight consumer warps each take 16
// of the block's keys.  The G query heads of the group are the rows of a
// 16-row tile (GQA grouping: every K/V byte is read from HBM once per KV head),
// and both contractions run on the warp-level tensor path (mma.sync m16n8k16,
// f16 inputs, f32 accumulation): S = Q K^T for the warp's 16 keys, then
// O += P V with P taken straight from the S registers.  The softmax is online
// with quad shuffles and a lazy running max; warps merge at segment ends.  A
// combining warp folds the splits that end inside the CTA's range and, for the
// split that ends it, fetches the other CTAs' parts into shared memory as soon as
// they are published.  Scalar FP32 FMAs plus f16 -> f32 conversions could not
// keep up with HBM on this part (about 3200 issue cycles of math per 128-key
// block against about 3000 cycles of HBM time), which is why the two small
// contractions use the tensor path; tcgen05 and TMEM stay with the prefill tiles.
//
// The launch is a programmatic dependent of the kernel before it: before waiting
// for it, the producer asks L2 for the CTA's first blocks, and right after the
// wait the grid releases the next launch, whose CTAs then take SMs as this grid's
// CTAs leave them.  Two variants share the engine: MASK (per-slot sequence and
// position mask: the unified-span baseline) and KV8 (FP8 E4M3 pages).
#include "kernels.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace pa {

constexpr int kDecWarps = 8;                       // consumer warps (warpgroups 0, 1)
constexpr int kDecThreads = 12 * 32;               // warpgroup 2: producer, combiner, 2 idle
constexpr int kDecRegsConsumer = 216;              // setmaxnreg split (per thread)
constexpr int kDecRegsOther = 72;
// registers the split needs from the launch; checked on the host before launching
constexpr int kDecRegsSplitTotal = 256 * kDecRegsConsumer + 128 * kDecRegsOther;
constexpr int kKeysPerWarp = KB / kDecWarps;       // 16
constexpr float kDecRescale = 8.0f;                // lazy max: rescale when it grows by > 2^8
constexpr int kBox = KB * 128;                     // one 128-row x 64-dim swizzled box (16 KB)
static_assert(kKeysPerWarp == 16, "warp key slice is 16 rows");

constexpr int kBarBytes = 1024;  // barriers, stage metadata, jobs, flags

template <int D, int G, bool MASK, bool KV8>
struct DecCfg {
  static_assert(!(MASK && KV8), "one variant at a time");
  static_assert(!KV8 || D == 128, "FP8 pages: 128-byte rows");
  static constexpr int kHalves = KV8 ? 1 : D / 64;
  static constexpr int kBlk = KV8 ? KB * D : kHalves * kBox;  // one block of K (or V)
  static constexpr int kQ = ((G * D * 2) + 1023) / 1024 * 1024;  // the group's query rows
  static constexpr int kCells = MASK ? 2 * KB * 4 : 0;        // (sequence, position) of each key
  static constexpr int kScales = KV8 ? 2 * KB * 4 : 0;        // K and V scale of each key
  static constexpr int kStage = 2 * kBlk + kQ + kCells + kScales;  // multiple of 1024
  static constexpr int kMergeDims = 64;                       // the warps merge 64 dims at a time
  static constexpr int kMerge = kDecWarps * G * (kMergeDims + 2) * 4;
  static constexpr int kPart = G * (D + 2) * 4;               // one split partial (m, l, acc)
  static constexpr int kBase = kMerge + kPart + kBarBytes;    // + own partial, barriers, jobs
  static constexpr int kBudget = 227 * 1024 - 2048;           // minus alignment slack
  static constexpr int NS0 = (kBudget - kBase) / kStage;
  static constexpr int NS = NS0 > 6 ? 6 : NS0;
  static_assert(NS >= 2, "at least two stages");
  // what the stages leave holds the other CTAs' partials of the final segment
  static constexpr int kPref0 = (kBudget - kBase - NS * kStage) / kPart;
  static constexpr int kPref = kPref0 > 7 ? 7 : kPref0;
  static constexpr int kFixed = kBase + kPref * kPart;
  static constexpr int kSmem = NS * kStage + kFixed + 1024;
};

constexpr int kJobs = 4;  // hand-off ring from the consumers to the combining warp

struct DecJob {
  int ig, tok, g;  // ig < 0: no more jobs
  int c_first, n_parts;  // the segment's parts (SegParts)
  int fetch;             // 1: fetch the other parts of the final segment
  int pad[2];
};

// What the producer tells the consumers about the unit a stage holds.
struct StageMeta {
  int rows;       // valid keys of the block (0: skip the block)
  int i, g, kb;   // decode token index, KV head, key block
  int units;      // key blocks of token i
  int tok;        // ubatch token
  int seg_begin;  // global unit index of the first block of (i, g)
  int seq, pos;   // masked variant: the token's sequence and position
  int pad;
};

struct DecBars {
  uint64_t full[6], empty[6];
  uint64_t job_full[kJobs], job_empty[kJobs];
  DecJob jobs[kJobs];
  uint64_t fetched;  // the combining warp answered the fetch of the final segment's parts
  int append_upto;   // fused append: the new rows of this CTA's units < append_upto are in the pool
  StageMeta meta[6];
  int abort;
  int issued;     // stages the producer has issued (consumers' view after an abort)
  int prod_done;  // 1: the producer issues no more stages
  int fetch_go;   // the outcome of the consumers' wait for the fetch, one for all
  int last;     // the consumers complete the split of the CTA's final segment
  int fetch_ok; // 1: every other part of the final segment sits in the fetch area
  int tail;     // the consumers reached the end of the final segment
};

static_assert(sizeof(DecBars) <= kBarBytes, "barrier area");

// Position in the unit sequence of this CTA.
struct UnitIt {
  int i;      // decode token index (into dec_tok)
  int g;      // KV head
  int kb;     // key block within the token
  int units;  // key blocks of token i
  int tok;    // ubatch token
  int L;      // kv_len of the token (clamped to the row capacity)
  int uoff;   // first key block of token i among the decode tokens' blocks
  int seq, pos;  // masked variant: the token's sequence and position (else 0)
};

struct DecView {
  const int *dec_tok;
  const int *tok_unit_off;
  int n_dec;
  int Hkv;
  int cap;
  const int32_t *kv;
  const int32_t *tok_seq, *tok_pos;  // masked variant only, else null
};

__device__ __forceinline__ void it_token(UnitIt &it, int i, const DecView &v) {
  it.i = i;
  it.uoff = v.tok_unit_off[i];
  it.units = v.tok_unit_off[i + 1] - it.uoff;
  it.tok = v.dec_tok[i];
  int L = v.kv[it.tok];
  it.L = min(max(L, 0), v.cap);
  it.seq = v.tok_seq ? v.tok_seq[it.tok] : 0;
  it.pos = v.tok_pos ? v.tok_pos[it.tok] : 0;
}

// Iterator at the CTA's first unit, as placed by the planner: (i, g, kb, token) and
// (units, kv_len) -- no dependent loads before the first copy.
__device__ __forceinline__ void it_start(UnitIt &it, int4 s0, int4 s1, const DecView &v) {
  it.i = s0.x;
  it.g = s0.y;
  it.kb = s0.z;
  it.tok = s0.w;
  it.units = s1.x;
  it.L = s1.y;
  it.uoff = s1.z;
  it.seq = v.tok_seq ? v.tok_seq[it.tok] : 0;
  it.pos = v.tok_pos ? v.tok_pos[it.tok] : 0;
}

__device__ __forceinline__ void it_next(UnitIt &it, const DecView &v) {
  if (++it.kb < it.units) return;
  it.kb = 0;
  if (++it.g < v.Hkv) return;
  it.g = 0;
  int i = it.i + 1;
  while (i < v.n_dec) {
    it_token(it, i, v);
    if (it.units > 0) return;
    ++i;
  }
  it.i = v.n_dec;  // past the end (never consumed)
}

// Bounded wait (limit in ns) that also gives up as soon as another thread of the CTA
// gave up.
__device__ __forceinline__ bool dec_wait(uint64_t *bar, uint32_t parity, int *err,
                                         volatile int *abort, uint64_t limit) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    // each try_wait may suspend the thread for a while: the clock is read every time
    if (globaltimer_ns() - t0 > limit) {
      atomicOr(err, PA_ERR_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

// The consumers' wait for stage k.  Every consumer warp must reach the same decision,
// since they meet at named barriers afterwards: once the CTA gives up, stage k is still
// consumed if the producer had issued it (its copies land; wait for them), and
// abandoned only when the producer has stopped short of it.  The last-resort bound,
// twice the drain bound, is never reached while the producer's own waits are bounded.
__device__ __forceinline__ bool dec_wait_stage(uint64_t *bar, uint32_t parity, int k, int *err,
                                               volatile int *abort, volatile int *issued,
                                               volatile int *prod_done, uint64_t limit) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) {
      if (*prod_done) {
        __threadfence_block();
        if (k >= *issued) return false;
      }
      if (globaltimer_ns() - t0 > 2 * kDrainLimitNs) return false;
      continue;
    }
    if (globaltimer_ns() - t0 > limit) {
      atomicOr(err, PA_ERR_TIMEOUT);
      *abort = 1;
    }
  }
}

// Barrier of the consumer warps only (the producer warpgroup never joins).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
}

// Loads of the plan issued in program order at the point where they stand (volatile:
// the compiler neither sinks them into the branch that uses them nor merges them with
// the speculative reads made before the dependency wait), served by L2 (.cg), so a
// line the speculative reads left in L1 is never used.
__device__ __forceinline__ int2 ld_v2_early(const int *p) {
  int2 r;
  asm volatile("ld.global.cg.v2.s32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
__device__ __forceinline__ int4 ld_v4_early(const int4 *p) {
  int4 r;
  asm volatile("ld.global.cg.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Arrival counters of split segments: a part is published by a release increment
// after its partial is written; whoever sees every other part published reads them.
__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// CTA-scope release/acquire on a shared-memory flag
__device__ __forceinline__ void st_release_cta(int *p, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_cta(const int *p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ int atom_add_acq_rel(int *p, int x) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(x)
               : "memory");
  return old;
}

// Fold one partial (mp, lp, op) into the running (M, L, O) of two output dims of one
// head.  Every combine path applies this arithmetic to the parts in CTA order, so the
// result does not depend on which CTA or warp happens to do the combine.
__device__ __forceinline__ void fold_pair(float &M, float &L, float2 &O, float mp, float lp,
                                          float2 op) {
  const float Mn = fmaxf(M, mp);
  const float fo = M == -INFINITY ? 0.f : exp2_approx(M - Mn);
  const float fp = mp == -INFINITY ? 0.f : exp2_approx(mp - Mn);
  L = __fmaf_rn(lp, fp, __fmul_rn(L, fo));
  O.x = __fmaf_rn(op.x, fp, __fmul_rn(O.x, fo));
  O.y = __fmaf_rn(op.y, fp, __fmul_rn(O.y, fo));
  M = Mn;
}

// The parts of a split segment (global units [ub, ue)) in CTA order: every CTA owns
// at least one unit, so they are CTAs c_first, c_first + 1, ..., c_first + n - 1.
struct SegParts {
  int c_first;  // CTA of the segment's first unit
  int n;        // number of parts
};
__device__ __forceinline__ SegParts seg_parts(int ub, int ue, int U, int C) {
  SegParts sp;
  sp.c_first = cta_of_unit(ub, U, C);
  sp.n = cta_of_unit(ue - 1, U, C) - sp.c_first + 1;
  return sp;
}

// ---- warp-level tensor path helpers ---------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A(16x16, f16, row) * B(16x8, f16, col) + D, f32 accumulators
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Byte offset of (row r, 16-byte chunk c) inside a 128-byte-swizzled box of 128-byte rows.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}
// Two FP8 E4M3 codes (the low byte is the element of the lower index) widened to f16x2
// (exact: every E4M3 value is a binary16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint16_t c) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(c));
  return r;
}
__device__ __forceinline__ uint16_t lds_u16(const unsigned char *p) {
  return *reinterpret_cast<const uint16_t *>(p);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// MASK: per-slot masked variant (the unified-span baseline): key j of a token is used
// only if its slot holds a cell of the token's own sequence at a position up to the
// token's own (cell_seq / cell_pos, copied into the stage with the block).
// KV8: FP8 pages (E4M3 codes, one scale per cached row; V transposed inside each
// (page, head) block; page size 128, d 128): the consumers widen the codes to f16
// for the same tensor-path contractions, apply the K scales to the scores and fold
// the V scales into P.
template <int D, int G, bool MASK, bool KV8>
__global__ void __launch_bounds__(kDecThreads, 1)
k_decode(AttnArgs a, const __grid_constant__ AttnMaps maps) {
  using Cfg = DecCfg<D, G, MASK, KV8>;
  constexpr int NS = Cfg::NS;
  // units asked of L2 before the dependency wait, so that the first blocks stream in
  // while the launch before drains (the depth of each variant is the measured best)
  constexpr int kPre = KV8 ? 6 : MASK ? 3 : 6;
  constexpr int KSTEPS = D / 16;  // k-steps of the QK contraction
  constexpr int NT = D / 8;       // 8-dim tiles of the PV product
  static_assert(G <= 8, "the group fits in rows 0..7 of the 16-row tile");

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  unsigned char *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  unsigned char *ring = smem;
  float *merge = reinterpret_cast<float *>(smem + NS * Cfg::kStage);
  DecBars *bars = reinterpret_cast<DecBars *>(smem + NS * Cfg::kStage + Cfg::kMerge);
  // this CTA's partial of its final segment, then the other CTAs' partials of it
  float *own = reinterpret_cast<float *>(smem + NS * Cfg::kStage + Cfg::kMerge + kBarBytes);
  float *pref = own + G * (D + 2);

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], kDecWarps);
    }
    for (int j = 0; j < kJobs; ++j) {
      mbar_init(&bars->job_full[j], 1);
      mbar_init(&bars->job_empty[j], 1);
    }
    mbar_init(&bars->fetched, 1);
    bars->append_upto = 0;
    bars->abort = 0;
    bars->issued = 0;
    bars->prod_done = 0;
    bars->fetch_ok = 0;
    bars->tail = 0;
    fence_mbar_init();
  }
  if (w == kDecWarps && lane == 0) {
    tc::prefetch_tmap(&maps.k);
    tc::prefetch_tmap(&maps.v);
  }
  // Launched as a programmatic dependent of the append kernel: the launch and the
  // setup above overlap its tail.  Before waiting for it, the producer thread asks L2
  // for the CTA's first key blocks: the plan's start record and the page table were
  // written by kernels that finished before the append began, and a prefetch changes
  // no result (if the append writes into a block, L2 holds the new rows; if a record
  // is stale, the prefetch is merely wasted).
  if (w == kDecWarps && lane == 0) {
    // reads past L1 (.cg): they precede the wait and must leave no line there
    const int4 *srec = reinterpret_cast<const int4 *>(a.ws + a.lay.dec_start) + 4 * blockIdx.x;
    const int4 s0 = __ldcg(srec), s1 = __ldcg(srec + 1), p0 = __ldcg(srec + 2),
               p1 = __ldcg(srec + 3);
    const int2 cnt0 =
        KV8 ? make_int2(0, 0) : ld_v2_early(&reinterpret_cast<const WsHeader *>(a.ws)->n_dec);
    const int g = s0.y, kb = s0.z, tok = s0.w, units = s1.x;
    const int ppb = KB / a.P;  // pages per key block
    // the length of the CTA's range, as the plan cuts it
    const int U0 = cnt0.y, C0 = min((int)gridDim.x, U0);
    const int n0 = (int)blockIdx.x < C0 ? (int)((int64_t)(blockIdx.x + 1) * U0 / C0 -
                                               (int64_t)blockIdx.x * U0 / C0)
                                        : 0;
    // a CTA without units has no record: only in-range rows are looked up
    const bool sane = tok >= 0 && tok < a.T && kb >= 0 && g >= 0 && g < a.Hkv && units > 0 &&
                      kb < units;
    // The first kPre units of the range, continuing into the token's next heads (which
    // use the same page ids; FP8 pages: the first head's units only); all page ids are
    // requested as soon as the record is in, before the first is used, and the range
    // length bounds only the prefetches.  Single-page blocks, the usual case; wider
    // blocks prefetch their first unit only.
    const int nld = !sane ? 0 : ppb != 1 ? 1 : KV8 ? min(kPre, units - kb) : kPre;
    int pid[kPre], gid[kPre];
    int ku = kb, gu = sane ? g : a.Hkv;  // (block, head) of unit u, stepped without division
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      gid[u] = gu;
      pid[u] = u == 0 ? p0.x
                      : (u < nld && gu < a.Hkv ? __ldcg(a.tpt + (size_t)tok * a.max_pages + ku) : -1);
      if (++ku >= units) {
        ku = 0;
        ++gu;
      }
    }
    const int nu = KV8 ? nld : min(nld, n0);
    const int pg0[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
    for (int u = 0; u < nu; ++u) {
      int pu = pid[0], gu = gid[0];
#pragma unroll
      for (int x = 1; x < kPre; ++x)
        if (u == x) {
          pu = pid[x];
          gu = gid[x];
        }
      if (gu >= a.Hkv) break;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j >= ppb) break;
        const int page = ppb == 1 ? pu : pg0[j];
        if (page < 0 || page >= a.num_pages) continue;
        const int y = (page * a.Hkv + gu) * a.P;
        const int yv = KV8 ? (page * a.Hkv + gu) * D : y;  // FP8 V: [page][h][d][P]
        for (int hf = 0; hf < Cfg::kHalves; ++hf) {
          tc::tma_prefetch_2d(&maps.k, hf * 64, y);
          tc::tma_prefetch_2d(&maps.v, hf * 64, yv);
        }
      }
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the next kernel in the stream may be scheduled onto SMs as this grid's CTAs leave
  // them (a programmatically launched successor still waits for this grid to complete)
  asm volatile("griddepcontrol.launch_dependents;");
  WsHeader *hdr = reinterpret_cast<WsHeader *>(a.ws);
  const int c = blockIdx.x;
  // Everything the first copy needs is loaded here, at once, so that it costs one L2
  // round trip after the wait rather than a chain of dependent ones: the header's
  // counts (every thread) and the CTA's start record with its first page ids (the
  // producer warp).
  const int2 counts = ld_v2_early(&hdr->n_dec);  // (n_dec, n_units)
  const int4 *start = reinterpret_cast<const int4 *>(a.ws + a.lay.dec_start) + 4 * c;
  int4 start0 = make_int4(0, 0, 0, 0), start1 = start0, start2 = start0, start3 = start0;
  if (w == kDecWarps) {
    start0 = ld_v4_early(start);
    start1 = ld_v4_early(start + 1);
    start2 = ld_v4_early(start + 2);
    start3 = ld_v4_early(start + 3);
  }
  __syncthreads();
  int *err = &hdr->err;
  DecView v;
  v.dec_tok = reinterpret_cast<const int *>(a.ws + a.lay.dec_tok);
  v.tok_unit_off = reinterpret_cast<const int *>(a.ws + a.lay.tok_unit_off);
  v.n_dec = counts.x;
  v.Hkv = a.Hkv;
  v.cap = a.max_pages * a.P;
  v.kv = a.kv;
  v.tok_seq = MASK ? a.tok_seq : nullptr;
  v.tok_pos = MASK ? a.tok_pos : nullptr;
  float *partials = reinterpret_cast<float *>(a.ws + a.lay.partials);
  int *dec_cnt = reinterpret_cast<int *>(a.ws + a.lay.dec_cnt);

  const int U = counts.y;
  // decode tokens with no key (kv_len 0) own no unit: their rows are zero (written by
  // a warp that has no other work, off the path of the first copy)
  if (w == kDecWarps + 2) {
    for (int i = c; i < v.n_dec; i += gridDim.x) {
      if (v.tok_unit_off[i + 1] != v.tok_unit_off[i]) continue;
      uint16_t *orow = a.out + (size_t)v.dec_tok[i] * a.Hq * D;
      for (int x = lane; x < a.Hq * D; x += 32) orow[x] = 0;
    }
  }
  // the units go to C = min(gridDim.x, U) CTAs, each of which owns at least one
  const int C = min((int)gridDim.x, U);
  if (c >= C) return;
  const int u0 = (int)((int64_t)c * U / C), u1 = (int)((int64_t)(c + 1) * U / C);
  if (u0 >= u1) return;
  const int n = u1 - u0;

  volatile int *abort = &bars->abort;
  const bool appending = !KV8 && !MASK && a.k_new != nullptr;

  if (w >= kDecWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kDecRegsOther));
    if (w == kDecWarps && lane == 0) {
      // ---------------------------------------------------------------- producer
      const int pages_per_block = KB / a.P;
      const int oob_row = a.num_pages * a.Hkv * a.P;  // first row past the pool: zero fill
      UnitIt pit;
      it_start(pit, start0, start1, v);
      int issued = 0;
      // page ids of the unit about to be issued, loaded one unit ahead (while the
      // producer waits for a free stage) so no global load sits on the issue path
      int pgs[8];
      int npg = 0;
      auto fetch_pages = [&](const UnitIt &u) {
        const int key0 = u.kb * KB;
        const int rows = min(KB, u.L - key0);
        npg = (rows + a.P - 1) / a.P;
        const int32_t *row = a.tpt + (size_t)u.tok * a.max_pages + key0 / a.P;
#pragma unroll
        for (int j = 0; j < 8; ++j) pgs[j] = j < npg ? row[j] : -1;
      };
      {  // the first unit's page ids come with its start record
        const int4 p0 = start2, p1 = start3;
        npg = (min(KB, pit.L - pit.kb * KB) + a.P - 1) / a.P;
        pgs[0] = p0.x; pgs[1] = p0.y; pgs[2] = p0.z; pgs[3] = p0.w;
        pgs[4] = p1.x; pgs[5] = p1.y; pgs[6] = p1.z; pgs[7] = p1.w;
      }
      int appended = appending ? 0 : n;  // units whose new rows are known to be written
      for (int k = 0; k < n; ++k) {
        const int st = k % NS;
        if (!dec_wait(&bars->empty[st], ((k / NS) & 1) ^ 1, err, abort, a.wait_ns)) break;
        // fused append: a token's last key block holds its new row, which this CTA's
        // append warp writes (in unit order, publishing how far it got); read the block
        // only once its row is written
        if (appended <= k && pit.kb + 1 == pit.units) {
          uint64_t t0 = 0;
          while ((appended = ld_acquire_cta(&bars->append_upto)) <= k) {
            if (*abort) break;
            if (t0 == 0) {
              t0 = globaltimer_ns();
            } else if (globaltimer_ns() - t0 > a.wait_ns) {
              atomicOr(err, PA_ERR_TIMEOUT);
              *abort = 1;
              break;
            }
          }
          if (appended <= k) break;
        }
        unsigned char *stage = ring + st * Cfg::kStage;
        int rows = min(KB, pit.L - pit.kb * KB);
        // every page of the block must exist, else the block is skipped (and flagged)
        int ys[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int page = pgs[j];
          const bool bad = j < npg && (page < 0 || page >= a.num_pages);
          if (bad) {
            atomicOr(err, PA_ERR_PAGE_RANGE);
            rows = 0;
          }
          ys[j] = (j < npg && !bad) ? (page * a.Hkv + pit.g) * a.P : oob_row;
        }
        const bool seg_first = (k == 0) || pit.kb == 0;
        {
          StageMeta &m = bars->meta[st];
          m.rows = rows;
          m.i = pit.i;
          m.g = pit.g;
          m.kb = pit.kb;
          m.units = pit.units;
          m.tok = pit.tok;
          m.seg_begin = a.Hkv * pit.uoff + pit.g * pit.units;
          m.seq = pit.seq;
          m.pos = pit.pos;
        }
        const uint32_t qbytes = seg_first ? (uint32_t)(G * D * 2) : 0u;
        // masked variant: the (sequence, position) of each slot of the block's pages
        const uint32_t cbytes = (MASK && rows > 0) ? (uint32_t)(2 * npg * a.P * 4) : 0u;
        // FP8 pages: the K and V scales of the block's rows
        const uint32_t sbytes = (KV8 && rows > 0) ? (uint32_t)(2 * KB * 4) : 0u;
        mbar_arrive_expect_tx(&bars->full[st], 2u * Cfg::kBlk + qbytes + cbytes + sbytes);
        if (KV8 && rows > 0) {
          unsigned char *sc = stage + 2 * Cfg::kBlk + Cfg::kQ;
          const size_t r0 = ((size_t)pgs[0] * a.Hkv + pit.g) * KB;
          bulk_g2s(sc, a.k_scale + r0, KB * 4, &bars->full[st]);
          bulk_g2s(sc + KB * 4, a.v_scale + r0, KB * 4, &bars->full[st]);
        }
        if (MASK && rows > 0) {
          unsigned char *cells = stage + 2 * Cfg::kBlk + Cfg::kQ;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (j >= npg) break;
            const size_t slot0 = (size_t)pgs[j] * a.P;
            bulk_g2s(cells + j * a.P * 4, a.cell_seq + slot0, a.P * 4, &bars->full[st]);
            bulk_g2s(cells + KB * 4 + j * a.P * 4, a.cell_pos + slot0, a.P * 4, &bars->full[st]);
          }
        }
        if (KV8) {
          // one page per block: K rows [128][128 B], V transposed [128 dims][128 B]
          const int yk = rows > 0 ? ys[0] : oob_row;
          const int yv = rows > 0 ? (pgs[0] * a.Hkv + pit.g) * D : a.num_pages * a.Hkv * D;
          tc::tma_load_2d(stage, &maps.k, 0, yk, &bars->full[st]);
          tc::tma_load_2d(stage + Cfg::kBlk, &maps.v, 0, yv, &bars->full[st]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (KV8 || j >= pages_per_block) break;
          // pages past the sequence (or a skipped block) load the zero-filled tail of the map
          const int y = rows > 0 ? ys[j] : oob_row;
          for (int hf = 0; hf < Cfg::kHalves; ++hf) {
            tc::tma_load_2d(stage + hf * kBox + j * a.P * 128, &maps.k, hf * 64, y,
                            &bars->full[st]);
            tc::tma_load_2d(stage + Cfg::kBlk + hf * kBox + j * a.P * 128, &maps.v, hf * 64, y,
                            &bars->full[st]);
          }
        }
        if (seg_first)
          bulk_g2s(stage + 2 * Cfg::kBlk, a.q + ((size_t)pit.tok * a.Hq + pit.g * G) * D, qbytes,
                   &bars->full[st]);
        ++issued;
        *reinterpret_cast<volatile int *>(&bars->issued) = issued;
        it_next(pit, v);
        if (k + 1 < n) fetch_pages(pit);
      }
      // no more stages: the consumers may stop waiting for any stage past `issued`
      __threadfence_block();
      *reinterpret_cast<volatile int *>(&bars->prod_done) = 1;
      // after giving up, let copies already in flight land before the CTA exits
      if (*abort) {
        for (int k = issued - NS > 0 ? issued - NS : 0; k < issued; ++k) {
          uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&bars->full[k % NS], (k / NS) & 1) &&
                 globaltimer_ns() - t0 < kDrainLimitNs) {
          }
        }
      }
    } else if (w == kDecWarps + 2 && appending) {
      // -------------------------------------------------------------- fused append
      // The new K/V row of each decode token is its last key (position kv_len - 1),
      // in the last key block of each (token, head), and only the CTA owning that unit
      // reads it: this warp writes the rows of this CTA's such units (a row of one
      // head is D / 8 16-byte chunks of K, then as many of V, one lane each), then
      // releases the producer.  A slot other than the last key's is flagged, not
      // written.
      // (token, head) segments are visited in unit order from the CTA's first; a
      // segment's last unit is in this CTA's range [u0, u1) or not, without walking
      // the units one by one.  The lanes load 32 tokens' records at once (a range of
      // short sequences covers many tokens), then the warp walks them in order.
      const int4 rec0 = reinterpret_cast<const int4 *>(a.ws + a.lay.dec_start)[4 * c];
      uint16_t *kpw = const_cast<uint16_t *>(a.k_pages);
      uint16_t *vpw = const_cast<uint16_t *>(a.v_pages);
      constexpr int kCh = D / 8;
      bool done = false;
      for (int base = rec0.x; base < v.n_dec && !done; base += 32) {
        // this lane's token: its units, slot and the slot of its last key
        const int il = base + lane;
        int uoff = 0, units = 0, tok = 0, page = -1, off = 0;
        int64_t slot = -1;
        if (il < v.n_dec) {
          uoff = v.tok_unit_off[il];
          units = v.tok_unit_off[il + 1] - uoff;
          tok = v.dec_tok[il];
          slot = a.slot[tok];
          const int L = min(max(v.kv[tok], 0), v.cap);
          if (units > 0) {
            page = a.tpt[(size_t)tok * a.max_pages + (L - 1) / a.P];
            off = (L - 1) % a.P;
          }
        }
        for (int j = 0; j < 32 && base + j < v.n_dec; ++j) {
          const int uo = __shfl_sync(0xffffffffu, uoff, j);
          const int un = __shfl_sync(0xffffffffu, units, j);
          const int tk = __shfl_sync(0xffffffffu, tok, j);
          const int pg = __shfl_sync(0xffffffffu, page, j);
          const int of = __shfl_sync(0xffffffffu, off, j);
          const int64_t sl = __shfl_sync(0xffffffffu, slot, j);
          int g = base + j == rec0.x ? rec0.y : 0;
          if (a.Hkv * uo + g * un >= u1) {
            done = true;
            break;
          }
          if (un == 0 || sl < 0) continue;
          const bool ok = pg >= 0 && pg < a.num_pages && sl == (int64_t)pg * a.P + of;
          for (; g < a.Hkv; ++g) {
            const int last = a.Hkv * uo + g * un + un - 1;
            if (last - un + 1 >= u1) break;
            if (last < u0 || last >= u1) continue;  // another CTA reads this segment's end
            if (!ok) {
              if (lane == 0) atomicOr(err, PA_ERR_SLOT_RANGE);
              __syncwarp();
              if (lane == 0) st_release_cta(&bars->append_upto, last - u0 + 1);
              continue;
            }
            const size_t dst = (((size_t)pg * a.Hkv + g) * a.P + of) * D;
            const size_t src = ((size_t)tk * a.Hkv + g) * D;
            if (lane < kCh)
              reinterpret_cast<uint4 *>(kpw + dst)[lane] =
                  reinterpret_cast<const uint4 *>(a.k_new + src)[lane];
            else if (lane < 2 * kCh)
              reinterpret_cast<uint4 *>(vpw + dst)[lane - kCh] =
                  reinterpret_cast<const uint4 *>(a.v_new + src)[lane - kCh];
            // generic-proxy writes, read next by the producer's TMA (async proxy)
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __syncwarp();
            if (lane == 0) st_release_cta(&bars->append_upto, last - u0 + 1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) st_release_cta(&bars->append_upto, n);  // no more rows
    } else if (w == kDecWarps + 1) {
      // -------------------------------------------------------------- combining warp
      // Jobs from the consumers, in order: (a) a split segment that ended inside the
      // range: publish this CTA's part; if it was the last part to arrive, combine all
      // parts and write the row.  Runs beside the consumers, so their next segment
      // never waits on it.  (b) the final segment, when it is split: as soon as every
      // other part is published, copy them into shared memory, so the consumers can
      // finish the row at the end of the range with no global round trip.
      volatile int *tail = &bars->tail;
      for (int j = 0;; ++j) {
        const int q = j % kJobs;
        if (!dec_wait(&bars->job_full[q], (j / kJobs) & 1, err, abort, a.wait_ns)) break;
        const DecJob job = bars->jobs[q];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->job_empty[q]);
        if (job.ig < 0) break;
        SegParts sp;
        sp.c_first = job.c_first;
        sp.n = job.n_parts;
        const int n_parts = sp.n;
        if (job.fetch) {
          int ok = 0;
          if (n_parts - 1 <= Cfg::kPref) {
            // poll until the other parts are published or the consumers get there first
            const uint64_t t0 = globaltimer_ns();
            for (;;) {
              int cnt = 0;
              if (lane == 0) cnt = ld_acquire(&dec_cnt[job.ig]);
              cnt = __shfl_sync(0xffffffffu, cnt, 0);
              if (cnt == n_parts - 1) {
                ok = 1;
                break;
              }
              if (*tail || *abort || globaltimer_ns() - t0 > a.wait_ns) break;
              __nanosleep(128);
            }
          }
          if (ok) {
            __syncwarp();  // lane 0's acquire orders every lane's reads below
            // copy in float2 steps, a batch of loads in flight per part
            constexpr int N2 = G * (D + 2) / 2;
            constexpr int PER = (N2 + 31) / 32;
            int slot = 0;
            for (int jp = 0; jp < n_parts; ++jp) {
              const int cc = sp.c_first + jp;
              if (cc == c) continue;
              const float2 *src =
                  reinterpret_cast<const float2 *>(partials + (size_t)(job.ig + cc) * G * (D + 2));
              float2 *dst = reinterpret_cast<float2 *>(pref + slot * G * (D + 2));
              float2 t[PER];
#pragma unroll
              for (int r = 0; r < PER; ++r) {
                const int x = lane + 32 * r;
                t[r] = x < N2 ? __ldcg(src + x) : make_float2(0.f, 0.f);
              }
#pragma unroll
              for (int r = 0; r < PER; ++r) {
                const int x = lane + 32 * r;
                if (x < N2) dst[x] = t[r];
              }
              ++slot;
            }
          }
          __syncwarp();
          if (lane == 0) {
            bars->fetch_ok = ok;
            mbar_arrive(&bars->fetched);
          }
          continue;
        }
        int old = 0;
        if (lane == 0) old = atom_add_acq_rel(&dec_cnt[job.ig], 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old != n_parts - 1) continue;
        __syncwarp();  // lane 0's acquire orders every lane's reads below
        // Online fold over the parts in CTA order.  Lane owns outputs idx = lane + 32 t;
        // per part, lanes < G fetch (m, l) of head `lane` and broadcast the factors, and
        // every lane issues all its accumulator loads before using any (one L2 round
        // trip per part).  The parts were written by other SMs: read them past L1.
        constexpr int NOUT = G * D / 32;
        float O[NOUT];
#pragma unroll
        for (int t = 0; t < NOUT; ++t) O[t] = 0.f;
        float Mh = -INFINITY, Lh = 0.f;  // lane h < G: running max / sum of head h
        for (int jp = 0; jp < n_parts; ++jp) {
          const int cc = sp.c_first + jp;
          const float *base = partials + (size_t)(job.ig + cc) * G * (D + 2);
          float Op[NOUT];
#pragma unroll
          for (int t = 0; t < NOUT; ++t) {
            const int idx = lane + 32 * t, h = idx / D, dd = idx - h * D;
            Op[t] = __ldcg(base + h * (D + 2) + 2 + dd);
          }
          float mp = -INFINITY, lp = 0.f;
          if (lane < G) {
            mp = __ldcg(base + lane * (D + 2));
            lp = __ldcg(base + lane * (D + 2) + 1);
          }
          // the same arithmetic as fold_pair, with the factors shared across a head
          const float Mn = fmaxf(Mh, mp);
          const float fo = Mh == -INFINITY ? 0.f : exp2_approx(Mh - Mn);
          const float fp = mp == -INFINITY ? 0.f : exp2_approx(mp - Mn);
          Lh = __fmaf_rn(lp, fp, __fmul_rn(Lh, fo));
          Mh = Mn;
#pragma unroll
          for (int t = 0; t < NOUT; ++t) {
            const int h = (lane + 32 * t) / D;
            const float a_o = __shfl_sync(0xffffffffu, fo, h);
            const float a_p = __shfl_sync(0xffffffffu, fp, h);
            O[t] = __fmaf_rn(Op[t], a_p, __fmul_rn(O[t], a_o));
          }
        }
#pragma unroll
        for (int t = 0; t < NOUT; ++t) {
          const int idx = lane + 32 * t, h = idx / D, dd = idx - h * D;
          const float L = __shfl_sync(0xffffffffu, Lh, h);
          a.out[((size_t)job.tok * a.Hq + job.g * G + h) * D + dd] =
              __half_as_ushort(__float2half_rn(L > 0.f ? O[t] / L : 0.f));
        }
        if (lane == 0) dec_cnt[job.ig] = 0;  // ready for the next run of this plan
      }
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kDecRegsConsumer));
  // fragment coordinates: this lane holds rows (heads) r = lane/4 and r + 8 (padding),
  // and columns 2*(lane%4) + {0, 1} of each 8-column tile
  const int hr = lane >> 2, cq = lane & 3;
  const bool head_lane = hr < G;
  const int key_base = w * kKeysPerWarp;

  int seg_begin = 0;
  uint32_t qa[KSTEPS][2];  // A fragments of Q: columns 2cq.. and 8+2cq.. of each k-step
  float o[NT][4];          // O accumulators (rows hr and hr + 8)
  float m_run = -INFINITY; // running max of head hr (log2 domain)
  float l_part = 0.f;      // this lane's share of the row sum of head hr
  int n_jobs = 0;          // jobs handed to the combining warp
  SegParts fin = {0, 0};  // parts of a split final segment

  for (int k = 0; k < n; ++k) {
    const int st = k % NS;
    unsigned char *stage = ring + st * Cfg::kStage;
    const uint32_t sK = smem_u32(stage), sV = smem_u32(stage + Cfg::kBlk);
    // every consumer warp sees the same outcome of this wait, so all leave together
    if (!dec_wait_stage(&bars->full[st], (k / NS) & 1, k, err, abort, &bars->issued,
                        &bars->prod_done, a.wait_ns))
      break;
    const StageMeta cit = bars->meta[st];  // the unit this stage holds
    const int rows = cit.rows;
    const bool seg_first = (k == 0) || cit.kb == 0;
    const bool seg_last = (k == n - 1) || cit.kb + 1 == cit.units;

    if (seg_first) {
      seg_begin = cit.seg_begin;
      const int seg_end = seg_begin + cit.units;
      if (seg_end >= u1 && !(seg_begin >= u0 && seg_end <= u1)) {
        // the range ends inside a segment split over CTAs: have the combining warp
        // fetch the other parts while this one streams
        fin = seg_parts(seg_begin, seg_end, U, C);
        if (tid == 0) {
          const int q = n_jobs % kJobs;
          if (dec_wait(&bars->job_empty[q], ((n_jobs / kJobs) & 1) ^ 1, err, abort, a.wait_ns)) {
            DecJob job;
            job.ig = cit.i * a.Hkv + cit.g;
            job.tok = cit.tok;
            job.g = cit.g;
            job.c_first = fin.c_first;
            job.n_parts = fin.n;
            job.fetch = 1;
            bars->jobs[q] = job;
            mbar_arrive(&bars->job_full[q]);
          }
        }
        ++n_jobs;
      }
      const uint16_t *qs = reinterpret_cast<const uint16_t *>(stage + 2 * Cfg::kBlk);
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        qa[ks][0] = head_lane
                        ? *reinterpret_cast<const uint32_t *>(qs + hr * D + ks * 16 + 2 * cq)
                        : 0u;
        qa[ks][1] = head_lane
                        ? *reinterpret_cast<const uint32_t *>(qs + hr * D + ks * 16 + 8 + 2 * cq)
                        : 0u;
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
      m_run = -INFINITY;
      l_part = 0.f;
    }

    const int nr = min(max(rows - key_base, 0), kKeysPerWarp);
    bool zeroed = false;
    // masked variant: a slice whose 16 cells all fail the mask adds exactly nothing
    // (every probability is 0), so the warp skips it (the block is still read whole)
    bool any_kept = true;
    if (MASK && nr > 0) {
      const int *cs = reinterpret_cast<const int *>(stage + 2 * Cfg::kBlk + Cfg::kQ);
      const int kr = lane & 15;
      const bool keep = lane < 16 && kr < nr && cs[key_base + kr] == cit.seq &&
                        cs[KB + key_base + kr] <= cit.pos;
      any_kept = __ballot_sync(0xffffffffu, keep) != 0u;
    }
    if (nr > 0 && any_kept) {
      // ---- S = Q K^T for the warp's 16 keys (two 8-key tiles), f32 accumulators
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      // ldmatrix x4 row addresses: matrix = lane / 8 -> (key half, dim half)
      const int lm_key = key_base + ((lane >> 4) << 3) + (lane & 7);
      const int lm_chunk = (lane >> 3) & 1;
      if (KV8) {
        // K codes [key][128 B], 128-byte swizzle: this lane's key of each 8-key tile,
        // dims 16ks + 2cq (+1) and 16ks + 8 + 2cq (+1) -- the B fragment, widened
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int key = key_base + t * 8 + hr;
            const unsigned char *row = stage + key * 128 + ((ks ^ (key & 7)) << 4);
            mma16816(s[t], qa[ks][0], 0u, qa[ks][1], 0u, e4m3x2_to_h2(lds_u16(row + 2 * cq)),
                     e4m3x2_to_h2(lds_u16(row + 8 + 2 * cq)));
          }
      } else {
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
          const int box = ks >> 2, chunk = (ks & 3) * 2 + lm_chunk;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(sK + box * kBox + sw128(lm_key, chunk), b0, b1, b2, b3);
          mma16816(s[0], qa[ks][0], 0u, qa[ks][1], 0u, b0, b1);
          mma16816(s[1], qa[ks][0], 0u, qa[ks][1], 0u, b2, b3);
        }
      }
      // ---- online softmax on the fragment: this lane has keys 2cq, 2cq+1 (+8) of head hr
      float x[4];
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kk = t * 8 + 2 * cq + e;
          bool ok = kk < nr;
          if (MASK) {
            const int *cs = reinterpret_cast<const int *>(stage + 2 * Cfg::kBlk + Cfg::kQ);
            ok = ok && cs[key_base + kk] == cit.seq && cs[KB + key_base + kk] <= cit.pos;
          }
          float sv = s[t][e];
          if (KV8) sv *= reinterpret_cast<const float *>(stage + 2 * Cfg::kBlk + Cfg::kQ)[key_base + kk];
          x[t * 2 + e] = ok ? sv * a.scale_log2 : -INFINITY;
        }
      const float xm = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
      if (__any_sync(0xffffffffu, xm > m_run + kDecRescale)) {
        // the running max moves: exact block max of the row (its quad), rescale
        float bm = fmaxf(xm, __shfl_xor_sync(0xffffffffu, xm, 1));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
        const float m_new = fmaxf(m_run, bm);
        const float alpha = (m_run == -INFINITY) ? 0.f : exp2_approx(m_run - m_new);
        m_run = m_new;
        l_part *= alpha;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          o[t][0] *= alpha;
          o[t][1] *= alpha;
        }
      }
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      float p[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) p[j] = exp2_approx(x[j] - m_use);  // -inf -> 0
      l_part += (p[0] + p[1]) + (p[2] + p[3]);
      // P as the A fragment of the PV product (k = the warp's 16 keys; rows 8..15 zero)
      uint32_t pa0, pa2;
      if (KV8) {
        // fold each key's V scale into P (a key past the valid ones contributes 0)
        const float *vsc = reinterpret_cast<const float *>(stage + 2 * Cfg::kBlk + Cfg::kQ) + KB;
        float pv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int kk = (j >> 1) * 8 + 2 * cq + (j & 1);
          pv[j] = kk < nr ? p[j] * vsc[key_base + kk] : 0.f;
        }
        pa0 = pack_h2(pv[0], pv[1]);
        pa2 = pack_h2(pv[2], pv[3]);
      } else {
        pa0 = pack_h2(p[0], p[1]);
        pa2 = pack_h2(p[2], p[3]);
      }
      // V rows past the valid keys may hold stale data or NaN: zero them (0 * NaN)
      if (nr < kKeysPerWarp) {
        if (KV8) {
          // V transposed: the warp's 16 keys are one 16-byte chunk of every dim row
          for (int r = lane; r < D; r += 32) {
            uint4 *c = reinterpret_cast<uint4 *>(stage + Cfg::kBlk + r * 128 +
                                                 (((key_base >> 4) ^ (r & 7)) << 4));
            uint4 x4 = *c;
            unsigned char *b = reinterpret_cast<unsigned char *>(&x4);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (j >= nr) b[j] = 0;
            *c = x4;
          }
        } else {
          for (int r = key_base + nr + (lane >> 3); r < key_base + kKeysPerWarp; r += 4)
            for (int hf = 0; hf < Cfg::kHalves; ++hf)
              reinterpret_cast<uint4 *>(stage + Cfg::kBlk + hf * kBox + r * 128)[lane & 7] =
                  make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
        zeroed = true;
      }
      if (MASK) {
        // so may the V rows of masked slots (free cells, other sequences' cells)
        const int *cs = reinterpret_cast<const int *>(stage + 2 * Cfg::kBlk + Cfg::kQ);
        const int kr = lane & 15;
        const bool masked = kr < nr && !(cs[key_base + kr] == cit.seq &&
                                         cs[KB + key_base + kr] <= cit.pos);
        uint32_t bits = __ballot_sync(0xffffffffu, masked && lane < 16);
        while (bits) {
          const int r = key_base + __ffs(bits) - 1;
          bits &= bits - 1;
          // one row: Cfg::kHalves boxes x 8 chunks of 16 bytes
          if (lane < Cfg::kHalves * 8)
            reinterpret_cast<uint4 *>(stage + Cfg::kBlk + (lane >> 3) * kBox + r * 128)[lane & 7] =
                make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
        zeroed = true;
      }
      // ---- O += P V, 8 dims per tile; ldmatrix.trans gives the V fragments
      const int lt_key = key_base + (((lane >> 3) & 1) << 3) + (lane & 7);
      const int lt_tile = lane >> 4;
      if (KV8) {
        // V codes transposed [dim][128 B of keys]: this lane's dim of each 8-dim tile,
        // keys 2cq (+1) and 8 + 2cq (+1) of the warp's 16 -- the B fragment, widened
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int dim = t * 8 + hr;
          const unsigned char *row =
              stage + Cfg::kBlk + dim * 128 + (((key_base >> 4) ^ (dim & 7)) << 4);
          mma16816(o[t], pa0, 0u, pa2, 0u, e4m3x2_to_h2(lds_u16(row + 2 * cq)),
                   e4m3x2_to_h2(lds_u16(row + 8 + 2 * cq)));
        }
      } else {
#pragma unroll
        for (int t = 0; t < NT; t += 2) {
          const int dchunk = t + lt_tile;  // 16-byte chunk = 8-dim tile
          const int box = dchunk >> 3, chunk = dchunk & 7;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sV + box * kBox + sw128(lt_key, chunk), b0, b1, b2, b3);
          mma16816(o[t], pa0, 0u, pa2, 0u, b0, b1);
          mma16816(o[t + 1], pa0, 0u, pa2, 0u, b2, b3);
        }
      }
    }
    if (zeroed) fence_proxy_async();  // generic writes before async copies refill the stage
    __syncwarp();
    // the stage's K/V are consumed: release it now, so the producer keeps streaming
    // while the warps merge below
    if (lane == 0) mbar_arrive(&bars->empty[st]);

    if (seg_last) {
      // ---- merge the warps 64 dims at a time in the merge area; write the row out,
      // or a partial: in global memory for the combining warp (a segment that ends
      // inside the range), in shared memory for the final segment
      constexpr int MD = Cfg::kMergeDims < D ? Cfg::kMergeDims : D;
      float *mw = merge;                  // [warps][G]
      float *lw = mw + kDecWarps * G;     // [warps][G]
      float *aw = lw + kDecWarps * G;     // [warps][G][MD]
      float ls = l_part;
      ls += __shfl_xor_sync(0xffffffffu, ls, 1);
      ls += __shfl_xor_sync(0xffffffffu, ls, 2);
      if (head_lane && cq == 0) {
        mw[w * G + hr] = m_run;
        lw[w * G + hr] = ls;
      }
      const int seg_units = cit.units;
      const bool direct = seg_begin >= u0 && seg_begin + seg_units <= u1;
      const bool final_split = !direct && k == n - 1;
      const int ig = cit.i * a.Hkv + cit.g;
      const int slot = ig + c;
      float *part = final_split ? own : partials + (size_t)slot * G * (D + 2);
#pragma unroll
      for (int d0 = 0; d0 < D; d0 += MD) {
        if (head_lane) {
#pragma unroll
          for (int t = d0 / 8; t < (d0 + MD) / 8; ++t) {
            aw[(w * G + hr) * MD + t * 8 - d0 + 2 * cq] = o[t][0];
            aw[(w * G + hr) * MD + t * 8 - d0 + 2 * cq + 1] = o[t][1];
          }
        }
        consumers_sync();
        for (int idx = tid; idx < G * MD; idx += kDecWarps * 32) {
          const int h = idx / MD, dd = d0 + (idx - h * MD);
          float M = -INFINITY;
#pragma unroll
          for (int xw = 0; xw < kDecWarps; ++xw) M = fmaxf(M, mw[xw * G + h]);
          float oo = 0.f, Ls = 0.f;
          if (M != -INFINITY) {
#pragma unroll
            for (int xw = 0; xw < kDecWarps; ++xw) {
              const float mx = mw[xw * G + h];
              const float f = mx == -INFINITY ? 0.f : exp2_approx(mx - M);
              oo += f * aw[(xw * G + h) * MD + dd - d0];
              Ls += f * lw[xw * G + h];
            }
          }
          if (direct) {
            const float r = Ls > 0.f ? oo / Ls : 0.f;
            a.out[((size_t)cit.tok * a.Hq + cit.g * G + h) * D + dd] =
                __half_as_ushort(__float2half_rn(r));
          } else {
            float *pp = part + h * (D + 2);
            pp[2 + dd] = oo;
            if (dd == 0) { pp[0] = M; pp[1] = Ls; }
          }
        }
        consumers_sync();  // the merge area may be rewritten
      }
      if (final_split) {
        // The CTA's final segment is split over CTAs.  The others usually finished
        // their parts long ago (the next CTA starts its range with it) and the combining
        // warp has already copied them here; then the row is finished from shared
        // memory.  Otherwise publish this part; the last to arrive combines.
        if (tid == 0) {
          *reinterpret_cast<volatile int *>(&bars->tail) = 1;
          // one waiter decides for all the consumers, which meet at named barriers below
          bars->fetch_go = dec_wait(&bars->fetched, 0, err, abort, a.wait_ns) ? 1 : 0;
        }
        consumers_sync();
        if (*reinterpret_cast<volatile int *>(&bars->fetch_go)) {
          const bool fetched = *reinterpret_cast<volatile int *>(&bars->fetch_ok) != 0;
          bool combine = fetched;
          if (!fetched) {
            float *dst = partials + (size_t)slot * G * (D + 2);
            for (int x = tid; x < G * (D + 2); x += kDecWarps * 32) dst[x] = own[x];
            consumers_sync();
            if (tid == 0) bars->last = atom_add_acq_rel(&dec_cnt[ig], 1) == fin.n - 1;
            consumers_sync();
            combine = bars->last != 0;
          }
          if (combine) {
            // thread -> pairs of output dims (one head); every load of a batch of 8
            // parts, for all of the thread's pairs, is in flight before the first fold
            constexpr int NPAIR = G * D / 2;
            constexpr int ITERS = (NPAIR + kDecWarps * 32 - 1) / (kDecWarps * 32);
            const int own_j = c - fin.c_first;
            float M[ITERS], Ls[ITERS];
            float2 oo[ITERS];
#pragma unroll
            for (int r = 0; r < ITERS; ++r) {
              M[r] = -INFINITY;
              Ls[r] = 0.f;
              oo[r] = make_float2(0.f, 0.f);
            }
            for (int j0 = 0; j0 < fin.n; j0 += 8) {
              const int nb = min(8, fin.n - j0);
              const float *src[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int jp = j0 + j;
                if (jp == own_j || j >= nb) src[j] = own;
                else if (fetched) src[j] = pref + (jp < own_j ? jp : jp - 1) * G * (D + 2);
                else src[j] = partials + (size_t)(ig + fin.c_first + jp) * G * (D + 2);
              }
              float mp[ITERS][8], lp[ITERS][8];
              float2 op[ITERS][8];
#pragma unroll
              for (int r = 0; r < ITERS; ++r) {
                const int pair = tid + r * kDecWarps * 32;
                const int pr = pair < NPAIR ? pair : 0;
                const int h = (2 * pr) / D, dd = 2 * pr - h * D;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const bool local = fetched || j0 + j == own_j || j >= nb;
                  const float *pp = src[j] + h * (D + 2);
                  const float2 *p2 = reinterpret_cast<const float2 *>(pp + 2 + dd);
                  mp[r][j] = local ? pp[0] : __ldcg(pp);
                  lp[r][j] = local ? pp[1] : __ldcg(pp + 1);
                  op[r][j] = local ? *p2 : __ldcg(p2);
                }
              }
#pragma unroll
              for (int r = 0; r < ITERS; ++r)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  if (j < nb) fold_pair(M[r], Ls[r], oo[r], mp[r][j], lp[r][j], op[r][j]);
            }
#pragma unroll
            for (int r = 0; r < ITERS; ++r) {
              const int pair = tid + r * kDecWarps * 32;
              if (pair < NPAIR) {
                const int h = (2 * pair) / D, dd = 2 * pair - h * D;
                const float r0 = Ls[r] > 0.f ? oo[r].x / Ls[r] : 0.f;
                const float r1 = Ls[r] > 0.f ? oo[r].y / Ls[r] : 0.f;
                *reinterpret_cast<__half2 *>(a.out + ((size_t)cit.tok * a.Hq + cit.g * G + h) * D +
                                             dd) = __floats2half2_rn(r0, r1);
              }
            }
            if (tid == 0) dec_cnt[ig] = 0;  // ready for the next run of this plan
          }
        }
      } else if (!direct && tid == 0) {
        // hand the cross-CTA combine to the combining warp
        const int q = n_jobs % kJobs;
        if (dec_wait(&bars->job_empty[q], ((n_jobs / kJobs) & 1) ^ 1, err, abort, a.wait_ns)) {
          const SegParts sp = seg_parts(seg_begin, seg_begin + seg_units, U, C);
          DecJob job;
          job.ig = ig;
          job.tok = cit.tok;
          job.g = cit.g;
          job.c_first = sp.c_first;
          job.n_parts = sp.n;
          job.fetch = 0;
          bars->jobs[q] = job;
          mbar_arrive(&bars->job_full[q]);
        }
      }
      if (!direct && !final_split) ++n_jobs;
    }
  }
  if (tid == 0) {  // no more jobs
    const int q = n_jobs % kJobs;
    if (dec_wait(&bars->job_empty[q], ((n_jobs / kJobs) & 1) ^ 1, err, abort, a.wait_ns)) {
      bars->jobs[q].ig = -1;
      mbar_arrive(&bars->job_full[q]);
    }
  }
}

template <int D, int G, bool MASK, bool KV8>
static cudaError_t launch_decode_t(const AttnArgs &a, int num_sms, const AttnMaps *maps,
                                   cudaStream_t s) {
  using Cfg = DecCfg<D, G, MASK, KV8>;
  static PerDeviceOnce setup;
  if (setup.first()) {
    // setmaxnreg.inc can only draw on registers the block was launched with: refuse to
    // launch (rather than wait forever) if the compiled allocation does not cover the split
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, k_decode<D, G, MASK, KV8>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * kDecThreads < kDecRegsSplitTotal) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(k_decode<D, G, MASK, KV8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::kSmem);
    if (e != cudaSuccess) return e;
    setup.mark();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode<D, G, MASK, KV8>, a, *maps);
}

cudaError_t launch_decode(const AttnArgs &a, int num_sms, const void *tmaps, cudaStream_t s) {
  const AttnMaps *maps = static_cast<const AttnMaps *>(tmaps);
  const int G = a.Hq / a.Hkv;
  const bool masked = a.cell_seq != nullptr;
  if (a.k_scale) {  // FP8 pages: page size 128, d 128
    if (a.D != 128 || a.P != 128) return cudaErrorInvalidValue;
    if (G == 1) return launch_decode_t<128, 1, false, true>(a, num_sms, maps, s);
    if (G == 2) return launch_decode_t<128, 2, false, true>(a, num_sms, maps, s);
    if (G == 4) return launch_decode_t<128, 4, false, true>(a, num_sms, maps, s);
    if (G == 8) return launch_decode_t<128, 8, false, true>(a, num_sms, maps, s);
    return cudaErrorInvalidValue;
  }
#define PA_DEC_CASE(DD, GG)                                                           \
  if (a.D == DD && G == GG)                                                           \
    return masked ? launch_decode_t<DD, GG, true, false>(a, num_sms, maps, s)         \
                  : launch_decode_t<DD, GG, false, false>(a, num_sms, maps, s);
  PA_DEC_CASE(128, 1) PA_DEC_CASE(128, 2) PA_DEC_CASE(128, 4) PA_DEC_CASE(128, 8)
  PA_DEC_CASE(64, 1) PA_DEC_CASE(64, 2) PA_DEC_CASE(64, 4) PA_DEC_CASE(64, 8)
#undef PA_DEC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pa
