// Split-KV decode attention with a fused log-sum-exp reduce (sm_103a).
//
// The work is the planned decode tokens.  Each (token i, KV head g) owns
// ceil(kv_len / 128) key blocks ("units"); all units of all (i, g) are laid end
// to end and cut into gridDim.x equal contiguous ranges, one per CTA (one CTA
// per SM), so every SM streams the same number of KV bytes whatever the length
// mix.  A (i, g) whose units fall in one CTA is finished there; one that spans
// CTAs leaves one partial (m, l, acc) per CTA and the CTA that finishes last
// combines them (the partition + reduce scheme of the CacheFlow page, section
// 核心架构 3, "Paged Attention V2", fused into one launch: an arrival counter
// decides who combines, nobody waits).
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
// combining warp folds the splits of other CTAs.  Scalar FP32 FMAs plus f16 ->
// f32 conversions could not keep up with HBM on this part (about 3200 issue
// cycles of math per 128-key block against about 3000 cycles of HBM time),
// which is why the two small contractions use the tensor path; tcgen05 and
// TMEM stay with the prefill tiles.
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

template <int D, int G>
struct DecCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kBlk = kHalves * kBox;                 // one block of K (or V)
  static constexpr int kQ = ((G * D * 2) + 1023) / 1024 * 1024;  // the group's query rows
  static constexpr int kStage = 2 * kBlk + kQ;                // multiple of 1024
  static constexpr int kMergeDims = 64;                       // the warps merge 64 dims at a time
  static constexpr int kMerge = kDecWarps * G * (kMergeDims + 2) * 4;
  static constexpr int kFixed = kMerge + 512;                 // + barriers, jobs, flags
  static constexpr int kBudget = 227 * 1024 - 2048;           // minus alignment slack
  static constexpr int NS0 = (kBudget - kFixed) / kStage;
  static constexpr int NS = NS0 > 6 ? 6 : NS0;
  static_assert(NS >= 2, "at least two stages");
  static constexpr int kSmem = NS * kStage + kFixed + 1024;
};

constexpr int kJobs = 4;  // hand-off ring from the consumers to the combining warp

struct DecJob {
  int ig, tok, g, c_first, c_last;  // ig < 0: no more jobs
  int pad[3];
};

struct DecBars {
  uint64_t full[6], empty[6];
  uint64_t job_full[kJobs], job_empty[kJobs];
  DecJob jobs[kJobs];
  int rows[6];  // valid keys of the block held by each stage (0: skip the block)
  int abort;
  int last;     // the consumers complete the split of the CTA's final segment
};

// Position in the unit sequence of this CTA.
struct UnitIt {
  int i;      // decode token index (into dec_tok)
  int g;      // KV head
  int kb;     // key block within the token
  int units;  // key blocks of token i
  int tok;    // ubatch token
  int L;      // kv_len of the token (clamped to the row capacity)
};

struct DecView {
  const int *dec_tok;
  const int *tok_unit_off;
  int n_dec;
  int Hkv;
  int cap;
  const int32_t *kv;
};

__device__ __forceinline__ void it_token(UnitIt &it, int i, const DecView &v) {
  it.i = i;
  it.units = v.tok_unit_off[i + 1] - v.tok_unit_off[i];
  it.tok = v.dec_tok[i];
  int L = v.kv[it.tok];
  it.L = min(max(L, 0), v.cap);
}

// Iterator at the CTA's first unit, as placed by the planner: (i, g, kb, token) and
// (units, kv_len) -- no dependent loads before the first copy.
__device__ __forceinline__ void it_start(UnitIt &it, int4 s0, int4 s1) {
  it.i = s0.x;
  it.g = s0.y;
  it.kb = s0.z;
  it.tok = s0.w;
  it.units = s1.x;
  it.L = s1.y;
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

// Bounded wait that also gives up as soon as another thread of the CTA gave up.
__device__ __forceinline__ bool dec_wait(uint64_t *bar, uint32_t parity, int *err,
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

// Barrier of the consumer warps only (the producer warpgroup never joins).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
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
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

template <int D, int G>
__global__ void __launch_bounds__(kDecThreads, 1)
k_decode(AttnArgs a, const __grid_constant__ AttnMaps maps) {
  using Cfg = DecCfg<D, G>;
  constexpr int NS = Cfg::NS;
  constexpr int KSTEPS = D / 16;  // k-steps of the QK contraction
  constexpr int NT = D / 8;       // 8-dim tiles of the PV product
  static_assert(G <= 8, "the group fits in rows 0..7 of the 16-row tile");

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  unsigned char *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  unsigned char *ring = smem;
  float *merge = reinterpret_cast<float *>(smem + NS * Cfg::kStage);
  DecBars *bars = reinterpret_cast<DecBars *>(smem + NS * Cfg::kStage + Cfg::kMerge);

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
    bars->abort = 0;
    fence_mbar_init();
  }
  if (w == kDecWarps && lane == 0) {
    tc::prefetch_tmap(&maps.k);
    tc::prefetch_tmap(&maps.v);
  }
  // Launched as a programmatic dependent of the append kernel: the launch and the
  // setup above overlap its tail; nothing written by earlier kernels is read before here.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();
  WsHeader *hdr = reinterpret_cast<WsHeader *>(a.ws);
  int *err = &hdr->err;
  DecView v;
  v.dec_tok = reinterpret_cast<const int *>(a.ws + a.lay.dec_tok);
  v.tok_unit_off = reinterpret_cast<const int *>(a.ws + a.lay.tok_unit_off);
  v.n_dec = hdr->n_dec;
  v.Hkv = a.Hkv;
  v.cap = a.max_pages * a.P;
  v.kv = a.kv;
  float *partials = reinterpret_cast<float *>(a.ws + a.lay.partials);
  int *dec_cnt = reinterpret_cast<int *>(a.ws + a.lay.dec_cnt);

  const int U = hdr->n_units;
  const int C = gridDim.x, c = blockIdx.x;
  // decode tokens with no key (kv_len 0) own no unit: their rows are zero
  for (int i = c; i < v.n_dec; i += C) {
    if (v.tok_unit_off[i + 1] != v.tok_unit_off[i]) continue;
    uint16_t *orow = a.out + (size_t)v.dec_tok[i] * a.Hq * D;
    for (int x = threadIdx.x; x < a.Hq * D; x += blockDim.x) orow[x] = 0;
  }
  const int u0 = (int)((int64_t)c * U / C), u1 = (int)((int64_t)(c + 1) * U / C);
  if (u0 >= u1) return;
  const int n = u1 - u0;
  const int4 *start = reinterpret_cast<const int4 *>(a.ws + a.lay.dec_start) + 4 * c;
  const int4 start0 = start[0], start1 = start[1];

  volatile int *abort = &bars->abort;

  if (w >= kDecWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kDecRegsOther));
    if (w == kDecWarps && lane == 0) {
      // ---------------------------------------------------------------- producer
      const int pages_per_block = KB / a.P;
      const int oob_row = a.num_pages * a.Hkv * a.P;  // first row past the pool: zero fill
      UnitIt pit;
      it_start(pit, start0, start1);
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
        const int4 p0 = start[2], p1 = start[3];
        npg = (min(KB, pit.L - pit.kb * KB) + a.P - 1) / a.P;
        pgs[0] = p0.x; pgs[1] = p0.y; pgs[2] = p0.z; pgs[3] = p0.w;
        pgs[4] = p1.x; pgs[5] = p1.y; pgs[6] = p1.z; pgs[7] = p1.w;
      }
      for (int k = 0; k < n; ++k) {
        const int st = k % NS;
        if (!dec_wait(&bars->empty[st], ((k / NS) & 1) ^ 1, err, abort)) break;
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
        bars->rows[st] = rows;
        const uint32_t qbytes = seg_first ? (uint32_t)(G * D * 2) : 0u;
        mbar_arrive_expect_tx(&bars->full[st], 2u * Cfg::kBlk + qbytes);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j >= pages_per_block) break;
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
        it_next(pit, v);
        if (k + 1 < n) fetch_pages(pit);
      }
      // after giving up, let copies already in flight land before the CTA exits
      if (*abort) {
        for (int k = issued - NS > 0 ? issued - NS : 0; k < issued; ++k) {
          uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(&bars->full[k % NS], (k / NS) & 1) &&
                 globaltimer_ns() - t0 < kWaitLimitNs) {
          }
        }
      }
    } else if (w == kDecWarps + 1) {
      // -------------------------------------------------------------- combining warp
      // For each (i, g) this CTA left a partial of: count the arrival; the CTA whose
      // part lands last combines all parts and writes the row.  Runs beside the
      // consumers, so their next segment never waits on this.
      for (int j = 0;; ++j) {
        const int q = j % kJobs;
        if (!dec_wait(&bars->job_full[q], (j / kJobs) & 1, err, abort)) break;
        const DecJob job = bars->jobs[q];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->job_empty[q]);
        if (job.ig < 0) break;
        int n_parts = 0;
        for (int cc = job.c_first; cc <= job.c_last; ++cc)
          n_parts += cta_has_units(cc, U, C) ? 1 : 0;
        int old = 0;
        if (lane == 0) {
          __threadfence();  // the consumers' partial is visible before the count
          old = atomicAdd(&dec_cnt[job.ig], 1);
        }
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old != n_parts - 1) continue;
        __threadfence();
        // Online merge over the parts.  Lane owns outputs idx = lane + 32 t; per part,
        // lanes < G fetch (m, l) of head `lane` and broadcast them, and every lane
        // issues all its accumulator loads before using any (one L2 round trip per
        // part).  The parts were written by other SMs: read them past L1.
        constexpr int NOUT = G * D / 32;
        float O[NOUT];
#pragma unroll
        for (int t = 0; t < NOUT; ++t) O[t] = 0.f;
        float Mh = -INFINITY, Lh = 0.f;  // lane h < G: running max / sum of head h
        for (int cc = job.c_first; cc <= job.c_last; ++cc) {
          if (!cta_has_units(cc, U, C)) continue;
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
          const float Mn = fmaxf(Mh, mp);
          const float fo = Mh == -INFINITY ? 0.f : exp2_approx(Mh - Mn);
          const float fp = mp == -INFINITY ? 0.f : exp2_approx(mp - Mn);
          Lh = Lh * fo + lp * fp;
          Mh = Mn;
#pragma unroll
          for (int t = 0; t < NOUT; ++t) {
            const int h = (lane + 32 * t) / D;
            const float a_o = __shfl_sync(0xffffffffu, fo, h);
            const float a_p = __shfl_sync(0xffffffffu, fp, h);
            O[t] = O[t] * a_o + Op[t] * a_p;
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

  UnitIt cit;
  it_start(cit, start0, start1);
  int seg_begin = 0;
  uint32_t qa[KSTEPS][2];  // A fragments of Q: columns 2cq.. and 8+2cq.. of each k-step
  float o[NT][4];          // O accumulators (rows hr and hr + 8)
  float m_run = -INFINITY; // running max of head hr (log2 domain)
  float l_part = 0.f;      // this lane's share of the row sum of head hr
  bool dead = false;
  int n_jobs = 0;          // partials handed to the combining warp

  for (int k = 0; k < n; ++k) {
    const int st = k % NS;
    unsigned char *stage = ring + st * Cfg::kStage;
    const uint32_t sK = smem_u32(stage), sV = smem_u32(stage + Cfg::kBlk);
    const bool seg_first = (k == 0) || cit.kb == 0;
    const bool seg_last = (k == n - 1) || cit.kb + 1 == cit.units;
    if (!dead) dead = !dec_wait(&bars->full[st], (k / NS) & 1, err, abort);
    const int rows = dead ? 0 : bars->rows[st];

    if (seg_first) {
      seg_begin = a.Hkv * v.tok_unit_off[cit.i] + cit.g * cit.units;
      const uint16_t *qs = reinterpret_cast<const uint16_t *>(stage + 2 * Cfg::kBlk);
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        qa[ks][0] = (head_lane && !dead)
                        ? *reinterpret_cast<const uint32_t *>(qs + hr * D + ks * 16 + 2 * cq)
                        : 0u;
        qa[ks][1] = (head_lane && !dead)
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
    if (nr > 0) {
      // ---- S = Q K^T for the warp's 16 keys (two 8-key tiles), f32 accumulators
      float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      // ldmatrix x4 row addresses: matrix = lane / 8 -> (key half, dim half)
      const int lm_key = key_base + ((lane >> 4) << 3) + (lane & 7);
      const int lm_chunk = (lane >> 3) & 1;
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        const int box = ks >> 2, chunk = (ks & 3) * 2 + lm_chunk;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sK + box * kBox + sw128(lm_key, chunk), b0, b1, b2, b3);
        mma16816(s[0], qa[ks][0], 0u, qa[ks][1], 0u, b0, b1);
        mma16816(s[1], qa[ks][0], 0u, qa[ks][1], 0u, b2, b3);
      }
      // ---- online softmax on the fragment: this lane has keys 2cq, 2cq+1 (+8) of head hr
      float x[4];
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kk = t * 8 + 2 * cq + e;
          x[t * 2 + e] = (kk < nr) ? s[t][e] * a.scale_log2 : -INFINITY;
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
      const uint32_t pa0 = pack_h2(p[0], p[1]), pa2 = pack_h2(p[2], p[3]);
      // V rows past the valid keys may hold stale data or NaN: zero them (0 * NaN)
      if (nr < kKeysPerWarp) {
        for (int r = key_base + nr + (lane >> 3); r < key_base + kKeysPerWarp; r += 4)
          for (int hf = 0; hf < Cfg::kHalves; ++hf)
            reinterpret_cast<uint4 *>(stage + Cfg::kBlk + hf * kBox + r * 128)[lane & 7] =
                make_uint4(0, 0, 0, 0);
        __syncwarp();
        zeroed = true;
      }
      // ---- O += P V, 8 dims per tile; ldmatrix.trans gives the V fragments
      const int lt_key = key_base + (((lane >> 3) & 1) << 3) + (lane & 7);
      const int lt_tile = lane >> 4;
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
    if (zeroed) fence_proxy_async();  // generic writes before async copies refill the stage
    __syncwarp();
    // the stage's K/V are consumed: release it now, so the producer keeps streaming
    // while the warps merge below
    if (lane == 0) mbar_arrive(&bars->empty[st]);

    if (seg_last) {
      // ---- merge the warps 64 dims at a time in the merge area; write the row out,
      // or a partial that the combining warp will fold across CTAs
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
      const int ig = cit.i * a.Hkv + cit.g;
      const int slot = ig + c;
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
            float *pp = partials + ((size_t)slot * G + h) * (D + 2);
            pp[2 + dd] = oo;
            if (dd == 0) { pp[0] = M; pp[1] = Ls; }
          }
        }
        consumers_sync();  // the merge area may be rewritten
      }
      if (!direct && k == n - 1) {
        // The CTA's final segment continues into the next CTA, which handled its part
        // first, so this CTA is almost always the last to arrive; everyone else is
        // done too, so the consumers fold the parts right here, all loads at once.
        const int64_t ub = seg_begin, ue = ub + seg_units;
        const int c_first = cta_of_unit(ub, U, C), c_last = cta_of_unit(ue - 1, U, C);
        int n_parts = 0;
        for (int cc = c_first; cc <= c_last; ++cc) n_parts += cta_has_units(cc, U, C) ? 1 : 0;
        if (tid == 0) {
          __threadfence();  // the partial of every consumer is visible before the count
          bars->last = atomicAdd(&dec_cnt[ig], 1) == n_parts - 1;
        }
        consumers_sync();
        if (bars->last) {
          __threadfence();
          for (int idx = tid; idx < G * D; idx += kDecWarps * 32) {
            const int h = idx / D, dd = idx - h * D;
            float M = -INFINITY, Ls = 0.f, oo = 0.f;
            for (int c0 = c_first; c0 <= c_last; c0 += 8) {
              float mp[8], lp[8], op[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {  // issue every load of the batch first
                const int cc = c0 + j;
                const bool use = cc <= c_last && cta_has_units(cc, U, C);
                const float *pp = partials + ((size_t)(ig + (use ? cc : c_first)) * G + h) * (D + 2);
                mp[j] = use ? __ldcg(pp) : -INFINITY;
                lp[j] = use ? __ldcg(pp + 1) : 0.f;
                op[j] = use ? __ldcg(pp + 2 + dd) : 0.f;
              }
              float Mn = M;
#pragma unroll
              for (int j = 0; j < 8; ++j) Mn = fmaxf(Mn, mp[j]);
              const float fo = M == -INFINITY ? 0.f : exp2_approx(M - Mn);
              Ls *= fo;
              oo *= fo;
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float f = mp[j] == -INFINITY ? 0.f : exp2_approx(mp[j] - Mn);
                Ls += f * lp[j];
                oo += f * op[j];
              }
              M = Mn;
            }
            a.out[((size_t)cit.tok * a.Hq + cit.g * G + h) * D + dd] =
                __half_as_ushort(__float2half_rn(Ls > 0.f ? oo / Ls : 0.f));
          }
          if (tid == 0) dec_cnt[ig] = 0;  // ready for the next run of this plan
        }
      } else if (!direct && tid == 0) {
        // hand the cross-CTA combine to the combining warp
        const int q = n_jobs % kJobs;
        if (dec_wait(&bars->job_empty[q], ((n_jobs / kJobs) & 1) ^ 1, err, abort)) {
          const int64_t ub = seg_begin, ue = ub + seg_units;
          DecJob job;
          job.ig = ig;
          job.tok = cit.tok;
          job.g = cit.g;
          job.c_first = cta_of_unit(ub, U, C);
          job.c_last = cta_of_unit(ue - 1, U, C);
          bars->jobs[q] = job;
          mbar_arrive(&bars->job_full[q]);
        }
      }
      if (!direct && k != n - 1) ++n_jobs;
    }
    it_next(cit, v);
  }
  if (tid == 0) {  // no more jobs
    const int q = n_jobs % kJobs;
    if (dec_wait(&bars->job_empty[q], ((n_jobs / kJobs) & 1) ^ 1, err, abort)) {
      bars->jobs[q].ig = -1;
      mbar_arrive(&bars->job_full[q]);
    }
  }
}

template <int D, int G>
static cudaError_t launch_decode_t(const AttnArgs &a, int num_sms, const AttnMaps *maps,
                                   cudaStream_t s) {
  using Cfg = DecCfg<D, G>;
  static bool attr_set = false;
  if (!attr_set) {
    // setmaxnreg.inc can only draw on registers the block was launched with: refuse to
    // launch (rather than wait forever) if the compiled allocation does not cover the split
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, k_decode<D, G>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * kDecThreads < kDecRegsSplitTotal) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(k_decode<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
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
  return cudaLaunchKernelEx(&cfg, k_decode<D, G>, a, *maps);
}

cudaError_t launch_decode(const AttnArgs &a, int num_sms, const void *tmaps, cudaStream_t s) {
  const AttnMaps *maps = static_cast<const AttnMaps *>(tmaps);
  const int G = a.Hq / a.Hkv;
#define PA_DEC_CASE(DD, GG) \
  if (a.D == DD && G == GG) return launch_decode_t<DD, GG>(a, num_sms, maps, s);
  PA_DEC_CASE(128, 1) PA_DEC_CASE(128, 2) PA_DEC_CASE(128, 4) PA_DEC_CASE(128, 8)
  PA_DEC_CASE(64, 1) PA_DEC_CASE(64, 2) PA_DEC_CASE(64, 4) PA_DEC_CASE(64, 8)
#undef PA_DEC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pa
