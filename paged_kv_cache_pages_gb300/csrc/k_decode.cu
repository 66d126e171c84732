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
// Inside a CTA (12 warps: 8 consumers, 1 producer, 1 combining warp, 2 idle; the consumers take
// a larger register share with setmaxnreg) one producer thread streams, for every unit, the 128 K rows and
// 128 V rows of the block (contiguous runs of the pool: one per page) and, at
// the start of each (i, g), the G query rows, with 1-D bulk async copies into a
// ring of stages; it runs up to NS units ahead of the consumers.  Eight
// consumer warps each take 16 of the block's keys and compute the G = Hq/Hkv
// query heads of the group against them (GQA grouping: every K/V byte is read
// from HBM once per KV head).  Scores use fp32 FMAs; the softmax keeps a lazy
// running max per head (one warp vote per block decides whether the max has to
// move), per-lane partial row sums, and merges the warps at segment ends.
#include "kernels.cuh"

namespace pa {

constexpr int kDecWarps = 16;                      // consumer warps (warpgroups 0-3)
constexpr int kDecThreads = 20 * 32;               // warpgroup 4: producer, combiner, 2 idle
constexpr int kDecRegsConsumer = 104;              // setmaxnreg split (per thread)
constexpr int kDecRegsOther = 64;
// registers the split needs from the launch; checked on the host before launching
constexpr int kDecRegsSplitTotal = 512 * kDecRegsConsumer + 128 * kDecRegsOther;
constexpr int kKeysPerWarp = KB / kDecWarps;       // 8
constexpr float kDecRescale = 8.0f;                // lazy max: rescale when it grows by > 2^8
static_assert(kKeysPerWarp == 8, "warp key slice is 8 rows");

template <int D, int G>
struct DecCfg {
  static constexpr int kBlk = KB * D * 2;                     // one block of K (or V)
  static constexpr int kQ = ((G * D * 2) + 127) / 128 * 128;  // the group's query rows
  static constexpr int kStage = 2 * kBlk + kQ;
  static constexpr int kSbuf = kDecWarps * kKeysPerWarp * G * 4;
  static constexpr int kMergeDims = 64;  // the warps merge 64 dims at a time
  static constexpr int kMerge = kDecWarps * G * (kMergeDims + 2) * 4;
  static constexpr int kFixed = kSbuf + kMerge + 512;  // + barriers, jobs, flags, stage rows
  static constexpr int kBudget = 227 * 1024 - 1024;
  static constexpr int NS0 = (kBudget - kFixed) / kStage;
  static constexpr int NS = NS0 > 6 ? 6 : NS0;
  static_assert(NS >= 2, "at least two stages");
  static constexpr int kSmem = NS * kStage + kFixed;
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
  int rows[6];   // valid keys of the block held by each stage
  int abort;
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

// Iterator at the CTA's first unit, as placed by the planner: (i, g, kb).
__device__ __forceinline__ void it_start(UnitIt &it, int4 st, const DecView &v) {
  it_token(it, st.x, v);
  it.g = st.y;
  it.kb = st.z;
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

// Sum-reduce-scatter across the 8 lanes of a key group (xor 4, 2, 1).
template <int N>
__device__ __forceinline__ void rs_step(float *v, bool up, int m) {
#pragma unroll
  for (int j = 0; j < N / 2; ++j) {
    float send = up ? v[j] : v[j + N / 2];
    float keep = up ? v[j + N / 2] : v[j];
    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
  }
}

// Reductions over the lanes that hold the same heads (equal bit 0 of the lane).
__device__ __forceinline__ float red_max_heads(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
  return x;
}
__device__ __forceinline__ float red_sum_heads(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  x += __shfl_xor_sync(0xffffffffu, x, 8);
  x += __shfl_xor_sync(0xffffffffu, x, 16);
  return x;
}

// Barrier of the eight consumer warps only (the producer warp never joins).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecWarps * 32) : "memory");
}

// Sum (or max) of one value per head over all lanes of the warp: every lane
// passes, for each head, its contribution (0 / -inf when it holds none).
template <int G>
__device__ __forceinline__ void warp_sum_heads(float (&x)[G]) {
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x[h] += __shfl_xor_sync(0xffffffffu, x[h], m);
}
template <int G>
__device__ __forceinline__ void warp_max_heads(float (&x)[G]) {
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) x[h] = fmaxf(x[h], __shfl_xor_sync(0xffffffffu, x[h], m));
}

template <int D, int G>
__global__ void __launch_bounds__(kDecThreads, 1) k_decode(AttnArgs a) {
  using Cfg = DecCfg<D, G>;
  constexpr int NS = Cfg::NS;
  constexpr int LPK = D / 8;                // lanes per key row (one 16-byte chunk = 8 dims each)
  constexpr int KPS = 32 / LPK;             // keys per step of the warp
  constexpr int STEPS = kKeysPerWarp / KPS; // steps per unit
  constexpr int DPL = D / 32;               // output dims per lane in the PV product
  constexpr int NV = STEPS * G;             // partial scores per lane before the reduction
  constexpr int NF = NV >= LPK ? NV / LPK : 1;  // scores per lane after the reduce-scatter

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *ring = smem;
  float *sbuf_all = reinterpret_cast<float *>(smem + NS * Cfg::kStage);
  float *merge = reinterpret_cast<float *>(smem + NS * Cfg::kStage + Cfg::kSbuf);
  DecBars *bars =
      reinterpret_cast<DecBars *>(smem + NS * Cfg::kStage + Cfg::kSbuf + Cfg::kMerge);

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
  const int4 start = reinterpret_cast<const int4 *>(a.ws + a.lay.dec_start)[c];

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
  __syncthreads();
  volatile int *abort = &bars->abort;

  if (w >= kDecWarps) {
    // ------------------------------------------------------------------ producer
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kDecRegsOther));
    if (w == kDecWarps && lane == 0) {
      UnitIt pit;
      it_start(pit, start, v);
      int issued = 0;
      for (int k = 0; k < n; ++k) {
        const int st = k % NS;
        if (!dec_wait(&bars->empty[st], ((k / NS) & 1) ^ 1, err, abort)) break;
        unsigned char *stage = ring + st * Cfg::kStage;
        const int key0 = pit.kb * KB;
        int rows = min(KB, pit.L - key0);
        // all pages of the block must exist, else the block is skipped (and flagged)
        const int32_t *row = a.tpt + (size_t)pit.tok * a.max_pages + key0 / a.P;
        const int npg = (rows + a.P - 1) / a.P;
        for (int j = 0; j < npg; ++j) {
          const int page = row[j];
          if (page < 0 || page >= a.num_pages) {
            atomicOr(err, PA_ERR_PAGE_RANGE);
            rows = 0;
            break;
          }
        }
        const bool seg_first = (k == 0) || pit.kb == 0;
        bars->rows[st] = rows;
        const uint32_t qbytes = seg_first ? (uint32_t)(G * D * 2) : 0u;
        mbar_arrive_expect_tx(&bars->full[st], 2u * rows * D * 2 + qbytes);
        for (int j = 0; rows > 0 && j < npg; ++j) {
          const int r = min(a.P, rows - j * a.P);
          const int64_t src = ((int64_t)row[j] * a.Hkv + pit.g) * a.P * D;
          bulk_g2s(stage + j * a.P * D * 2, a.k_pages + src, r * D * 2, &bars->full[st]);
          bulk_g2s(stage + Cfg::kBlk + j * a.P * D * 2, a.v_pages + src, r * D * 2,
                   &bars->full[st]);
        }
        if (seg_first)
          bulk_g2s(stage + 2 * Cfg::kBlk, a.q + ((size_t)pit.tok * a.Hq + pit.g * G) * D, qbytes,
                   &bars->full[st]);
        ++issued;
        it_next(pit, v);
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
  const int rl = lane % LPK, kq = lane / LPK;
  float *sbuf = sbuf_all + w * kKeysPerWarp * G;
  // After the reduce-scatter over the LPK lanes of a key, this lane holds NF
  // consecutive score indices starting at vbase (index = step * G + head); lanes
  // that differ only in bits of `dup` hold duplicates (levels where fewer values
  // than lanes were left are all-reduced instead of scattered).
  int vbase = 0, dup = 0;
  {
    int cnt = NV;
#pragma unroll
    for (int m = LPK / 2; m >= 1; m >>= 1) {
      if (cnt >= 2) {
        if (rl & m) vbase += cnt / 2;
        cnt /= 2;
      } else {
        dup |= m;
      }
    }
  }
  const bool primary = (rl & dup) == 0;

  UnitIt cit;
  it_start(cit, start, v);
  int seg_begin = 0;
  float qf[G][8];
  float m_run[G];    // running max per head (log2 domain), replicated in all lanes
  float l_part[G];   // this lane's partial row sums per head (primary lanes only)
  float acc[G][DPL];
  bool dead = false;
  int n_jobs = 0;  // partials handed to the combining warp

  for (int k = 0; k < n; ++k) {
    const int st = k % NS;
    unsigned char *stage = ring + st * Cfg::kStage;
    const bool seg_first = (k == 0) || cit.kb == 0;
    const bool seg_last = (k == n - 1) || cit.kb + 1 == cit.units;
    if (!dead) dead = !dec_wait(&bars->full[st], (k / NS) & 1, err, abort);
    const int rows = dead ? 0 : bars->rows[st];

    if (seg_first) {
      seg_begin = a.Hkv * v.tok_unit_off[cit.i] + cit.g * cit.units;
      const uint16_t *qs = reinterpret_cast<const uint16_t *>(stage + 2 * Cfg::kBlk);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        uint4 q4 = dead ? make_uint4(0, 0, 0, 0)
                        : *reinterpret_cast<const uint4 *>(qs + h * D + rl * 8);
        float2 f0 = h2_to_f2(q4.x), f1 = h2_to_f2(q4.y), f2 = h2_to_f2(q4.z), f3 = h2_to_f2(q4.w);
        qf[h][0] = f0.x * a.scale_log2; qf[h][1] = f0.y * a.scale_log2;
        qf[h][2] = f1.x * a.scale_log2; qf[h][3] = f1.y * a.scale_log2;
        qf[h][4] = f2.x * a.scale_log2; qf[h][5] = f2.y * a.scale_log2;
        qf[h][6] = f3.x * a.scale_log2; qf[h][7] = f3.y * a.scale_log2;
        m_run[h] = -INFINITY;
        l_part[h] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[h][e] = 0.f;
      }
    }

    const int nr = min(max(rows - w * kKeysPerWarp, 0), kKeysPerWarp);
    if (nr > 0) {
      const uint16_t *Ks = reinterpret_cast<const uint16_t *>(stage) + w * kKeysPerWarp * D;
      const uint16_t *Vs =
          reinterpret_cast<const uint16_t *>(stage + Cfg::kBlk) + w * kKeysPerWarp * D;
      // ---- scores: STEPS steps of KPS keys; LPK lanes per key, one 16-byte chunk each
      float vals[NV];
#pragma unroll
      for (int s = 0; s < STEPS; ++s) {
        const int r = s * KPS + kq;
        uint4 k4 = *reinterpret_cast<const uint4 *>(Ks + r * D + rl * 8);
        float2 k0 = h2_to_f2(k4.x), k1 = h2_to_f2(k4.y), k2 = h2_to_f2(k4.z), k3 = h2_to_f2(k4.w);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float2 p2 = make_float2(qf[h][0] * k0.x, qf[h][1] * k0.y);
          p2 = ffma2(make_float2(qf[h][2], qf[h][3]), k1, p2);
          p2 = ffma2(make_float2(qf[h][4], qf[h][5]), k2, p2);
          p2 = ffma2(make_float2(qf[h][6], qf[h][7]), k3, p2);
          vals[s * G + h] = p2.x + p2.y;
        }
      }
      // ---- sum over the LPK lanes of each key: scatter while values last, then all-reduce
      {
        int cnt = NV;
#pragma unroll
        for (int m = LPK / 2; m >= 1; m >>= 1) {
          if (cnt >= 2) {
            const bool up = (rl & m) != 0;
#pragma unroll
            for (int j = 0; j < NV / 2; ++j) {
              if (j < cnt / 2) {
                const float send = up ? vals[j] : vals[j + cnt / 2];
                const float keep = up ? vals[j + cnt / 2] : vals[j];
                vals[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
              }
            }
            cnt /= 2;
          } else {
            vals[0] += __shfl_xor_sync(0xffffffffu, vals[0], m);
          }
        }
      }
      // ---- masking (select, so stale or NaN rows never count) and the lazy max
      float x[NF];
      int hj[NF], kj[NF];
      bool need = false;
#pragma unroll
      for (int j = 0; j < NF; ++j) {
        const int vi = vbase + j;
        const int s = vi / G;
        hj[j] = vi - s * G;
        kj[j] = s * KPS + kq;
        x[j] = kj[j] < nr ? vals[j] : -INFINITY;
        float mr = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h)
          if (h == hj[j]) mr = m_run[h];
        need |= x[j] > mr + kDecRescale;  // also true while m_run is -inf
      }
      if (__any_sync(0xffffffffu, need)) {
        // the running max moves: exact block max per head, rescale what was summed
        float bm[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          bm[h] = -INFINITY;
#pragma unroll
          for (int j = 0; j < NF; ++j)
            if (hj[j] == h) bm[h] = fmaxf(bm[h], x[j]);
        }
        warp_max_heads<G>(bm);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float m_new = fmaxf(m_run[h], bm[h]);
          const float alpha = (m_run[h] == -INFINITY) ? 0.f : exp2_approx(m_run[h] - m_new);
          m_run[h] = m_new;
          l_part[h] *= alpha;
#pragma unroll
          for (int e = 0; e < DPL; ++e) acc[h][e] *= alpha;
        }
      }
      // ---- p = 2^(x - m) into the per-warp buffer; partial sums stay in the lane
#pragma unroll
      for (int j = 0; j < NF; ++j) {
        float mr = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h)
          if (h == hj[j]) mr = m_run[h];
        const float p = (x[j] == -INFINITY) ? 0.f : exp2_approx(x[j] - mr);
        if (primary) {
#pragma unroll
          for (int h = 0; h < G; ++h)
            if (h == hj[j]) l_part[h] += p;
          sbuf[kj[j] * G + hj[j]] = p;
        }
      }
      __syncwarp();
      // ---- PV: lane owns dims [DPL*lane, DPL*lane + DPL) of every head
#pragma unroll
      for (int jj = 0; jj < kKeysPerWarp; ++jj) {
        if (jj < nr) {
          float pr[G];
          if constexpr (G % 4 == 0) {
#pragma unroll
            for (int h = 0; h < G; h += 4) {
              float4 t4 = *reinterpret_cast<const float4 *>(sbuf + jj * G + h);
              pr[h] = t4.x; pr[h + 1] = t4.y; pr[h + 2] = t4.z; pr[h + 3] = t4.w;
            }
          } else if constexpr (G == 2) {
            float2 t2 = *reinterpret_cast<const float2 *>(sbuf + jj * 2);
            pr[0] = t2.x; pr[1] = t2.y;
          } else {
            pr[0] = sbuf[jj];
          }
          if constexpr (DPL == 4) {
            uint2 v2 = *reinterpret_cast<const uint2 *>(Vs + jj * D + 4 * lane);
            float2 v01 = h2_to_f2(v2.x), v23 = h2_to_f2(v2.y);
#pragma unroll
            for (int h = 0; h < G; ++h) {
              float2 a01 = ffma2(make_float2(pr[h], pr[h]), v01, make_float2(acc[h][0], acc[h][1]));
              float2 a23 = ffma2(make_float2(pr[h], pr[h]), v23, make_float2(acc[h][2], acc[h][3]));
              acc[h][0] = a01.x; acc[h][1] = a01.y; acc[h][2] = a23.x; acc[h][3] = a23.y;
            }
          } else {
            uint32_t v1 = *reinterpret_cast<const uint32_t *>(Vs + jj * D + 2 * lane);
            float2 v01 = h2_to_f2(v1);
#pragma unroll
            for (int h = 0; h < G; ++h) {
              float2 a01 = ffma2(make_float2(pr[h], pr[h]), v01, make_float2(acc[h][0], acc[h][1]));
              acc[h][0] = a01.x; acc[h][1] = a01.y;
            }
          }
        }
      }
    }
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
      float ls[G];
#pragma unroll
      for (int h = 0; h < G; ++h) ls[h] = l_part[h];
      warp_sum_heads<G>(ls);
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          mw[w * G + h] = m_run[h];
          lw[w * G + h] = ls[h];
        }
      }
      const int seg_units = cit.units;
      const bool direct = seg_begin >= u0 && seg_begin + seg_units <= u1;
      const int ig = cit.i * a.Hkv + cit.g;
      const int slot = ig + c;
#pragma unroll
      for (int d0 = 0; d0 < D; d0 += MD) {
        // lane owns dims [DPL*lane, DPL*lane + DPL): those inside [d0, d0 + MD) go in
        if (DPL * lane >= d0 && DPL * lane < d0 + MD) {
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < DPL; ++e) aw[(w * G + h) * MD + DPL * lane - d0 + e] = acc[h][e];
        }
        consumers_sync();
        for (int idx = tid; idx < G * MD; idx += kDecWarps * 32) {
          const int h = idx / MD, dd = d0 + (idx - h * MD);
          float M = -INFINITY;
#pragma unroll
          for (int xw = 0; xw < kDecWarps; ++xw) M = fmaxf(M, mw[xw * G + h]);
          float o = 0.f, Ls = 0.f;
          if (M != -INFINITY) {
#pragma unroll
            for (int xw = 0; xw < kDecWarps; ++xw) {
              const float mx = mw[xw * G + h];
              const float f = mx == -INFINITY ? 0.f : exp2_approx(mx - M);
              o += f * aw[(xw * G + h) * MD + dd - d0];
              Ls += f * lw[xw * G + h];
            }
          }
          if (direct) {
            const float r = Ls > 0.f ? o / Ls : 0.f;
            a.out[((size_t)cit.tok * a.Hq + cit.g * G + h) * D + dd] =
                __half_as_ushort(__float2half_rn(r));
          } else {
            float *pp = partials + ((size_t)slot * G + h) * (D + 2);
            pp[2 + dd] = o;
            if (dd == 0) { pp[0] = M; pp[1] = Ls; }
          }
        }
        consumers_sync();  // the merge area may be rewritten
      }
      if (!direct && tid == 0) {
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
      if (!direct) ++n_jobs;
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
static cudaError_t launch_decode_t(const AttnArgs &a, int num_sms, cudaStream_t s) {
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
  k_decode<D, G><<<num_sms, kDecThreads, Cfg::kSmem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode(const AttnArgs &a, int num_sms, cudaStream_t s) {
  const int G = a.Hq / a.Hkv;
#define PA_DEC_CASE(DD, GG) \
  if (a.D == DD && G == GG) return launch_decode_t<DD, GG>(a, num_sms, s);
  PA_DEC_CASE(128, 1) PA_DEC_CASE(128, 2) PA_DEC_CASE(128, 4) PA_DEC_CASE(128, 8)
  PA_DEC_CASE(64, 1) PA_DEC_CASE(64, 2) PA_DEC_CASE(64, 4) PA_DEC_CASE(64, 8)
#undef PA_DEC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pa
