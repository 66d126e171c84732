// Split-KV decode attention and its log-sum-exp reduce (sm_103a).
//
// The work is the planned decode tokens.  Each (token i, KV head g) owns
// ceil(kv_len / 128) key blocks ("units"); all units of all (i, g) are laid end
// to end and cut into gridDim.x equal contiguous ranges, one per CTA (one CTA
// per SM), so every SM streams the same number of KV bytes whatever the length
// mix.  A (i, g) whose units fall in one CTA is finished there; one that spans
// CTAs leaves one partial (m, l, acc) per CTA, combined by k_reduce (the
// partition + reduce scheme of the CacheFlow page, section 核心架构 3, "Paged
// Attention V2").
//
// Inside a CTA, warp w owns keys [16w, 16w+16) of every 128-key block: it
// streams exactly those K and V rows of the page (one contiguous run of
// 16 * d halves each, since 16 divides the page size) with 1-D bulk async
// copies into its own 3-stage shared-memory ring, and computes the G = Hq/Hkv
// query heads of the group against each key once (GQA grouping: every K/V byte
// is read from HBM once per KV head).  Scores use fp32 FMAs; the softmax is
// online per warp with warp-shuffle reductions; warps merge at the end.
#include "kernels.cuh"

namespace pa {

constexpr int kDecWarps = 8;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kKeysPerWarp = KB / kDecWarps;  // 16
static_assert(kKeysPerWarp == 16, "warp key slice is 16 rows");

template <int D, int G, int NS>
struct DecCfg {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kStageBytes = 2 * kKeysPerWarp * kRowBytes;     // K rows then V rows
  static constexpr int kRing = kDecWarps * NS * kStageBytes;
  static constexpr int kSbuf = kDecWarps * kKeysPerWarp * G * 4;         // scores / probs
  static constexpr int kMerge = kDecWarps * G * (D + 2) * 4;              // m, l, acc per warp
  static constexpr int kBars = kDecWarps * NS * 8;
  static constexpr int kSmem = kRing + kSbuf + kMerge + kBars;
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

// Rows of warp w's slice in unit `it` and the page they live in.
__device__ __forceinline__ int warp_rows(const UnitIt &it, int w, const AttnArgs &a, int64_t *src,
                                         int *err) {
  int key0 = it.kb * KB + w * kKeysPerWarp;
  int n = min(kKeysPerWarp, it.L - key0);
  if (n <= 0) return 0;
  int page = a.tpt[(size_t)it.tok * a.max_pages + key0 / a.P];
  if (page < 0 || page >= a.num_pages) {
    if (err) atomicOr(err, PA_ERR_PAGE_RANGE);
    return 0;
  }
  *src = (((int64_t)page * a.Hkv + it.g) * a.P + (key0 % a.P)) * a.D;
  return n;
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

template <int D, int G, int NS>
__global__ void __launch_bounds__(kDecThreads, 1) k_decode(AttnArgs a) {
  using Cfg = DecCfg<D, G, NS>;
  constexpr int NCH = D / 64;    // 16-byte chunks of a key row per lane (8 dims each)
  constexpr int DPL = D / 32;    // output dims per lane in the PV product
  constexpr int NV = 4 * G;      // partial scores per lane (4 keys x G heads)
  constexpr int HPL = (G + 1) / 2;  // heads per lane in the softmax (16 keys x 2 halves)

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *ring = smem;
  float *sbuf_all = reinterpret_cast<float *>(smem + Cfg::kRing);
  float *merge = reinterpret_cast<float *>(smem + Cfg::kRing + Cfg::kSbuf);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kRing + Cfg::kSbuf + Cfg::kMerge);

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

  const int U = hdr->n_units;
  const int C = gridDim.x, c = blockIdx.x;
  const int u0 = (int)((int64_t)c * U / C), u1 = (int)((int64_t)(c + 1) * U / C);
  if (u0 >= u1) return;
  const int n = u1 - u0;

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int r8 = lane & 7, kq = lane >> 3;
  unsigned char *my_ring = ring + w * NS * Cfg::kStageBytes;
  uint64_t *my_bars = bars + w * NS;
  float *sbuf = sbuf_all + w * kKeysPerWarp * G;

  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&my_bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // producer state (lane 0 of every warp walks the same unit sequence)
  const int4 start = reinterpret_cast<const int4 *>(a.ws + a.lay.dec_start)[c];
  UnitIt pit;
  it_start(pit, start, v);
  int issued = 0;      // units whose copies lane 0 has started
  int k_dead = n;      // first unit whose wait gave up
  auto issue = [&](int k) {
    uint64_t *bar = &my_bars[k % NS];
    unsigned char *st = my_ring + (k % NS) * Cfg::kStageBytes;
    int64_t src = 0;
    int rows = warp_rows(pit, w, a, &src, err);
    if (rows > 0) {
      uint32_t bytes = rows * Cfg::kRowBytes;
      mbar_arrive_expect_tx(bar, 2 * bytes);
      bulk_g2s(st, a.k_pages + src, bytes, bar);
      bulk_g2s(st + kKeysPerWarp * Cfg::kRowBytes, a.v_pages + src, bytes, bar);
    } else {
      mbar_arrive(bar);
    }
    it_next(pit, v);
    ++issued;
  };
  if (lane == 0) {
    for (int k = 0; k < NS && k < n; ++k) issue(k);
  }

  UnitIt cit;
  it_start(cit, start, v);
  int seg_i = -1, seg_g = -1, seg_begin = 0, seg_units = 0, seg_tok = 0;
  float qf[G][NCH][8];
  float m_run[G], l_run[G];
  float acc[G][DPL];
  bool dead = false;

  auto finish_segment = [&]() {
    // per-warp state -> shared, then merge over warps
    float *mw = merge;                          // [warps][G]
    float *lw = merge + kDecWarps * G;          // [warps][G]
    float *aw = merge + 2 * kDecWarps * G;      // [warps][G][D]
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) { mw[w * G + h] = m_run[h]; lw[w * G + h] = l_run[h]; }
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < DPL; ++e) aw[(w * G + h) * D + DPL * lane + e] = acc[h][e];
    __syncthreads();
    const bool direct = seg_begin >= u0 && seg_begin + seg_units <= u1;
    const int slot = seg_i * a.Hkv + seg_g + c;
    for (int idx = tid; idx < G * D; idx += kDecThreads) {
      int h = idx / D, dd = idx - h * D;
      float M = -INFINITY;
#pragma unroll
      for (int x = 0; x < kDecWarps; ++x) M = fmaxf(M, mw[x * G + h]);
      float o = 0.f, Ls = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int x = 0; x < kDecWarps; ++x) {
          float f = exp2_approx(mw[x * G + h] - M);
          o += f * aw[(x * G + h) * D + dd];
          Ls += f * lw[x * G + h];
        }
      }
      if (direct) {
        float r = Ls > 0.f ? o / Ls : 0.f;
        a.out[((size_t)seg_tok * a.Hq + seg_g * G + h) * D + dd] = __half_as_ushort(__float2half_rn(r));
      } else {
        float *pp = partials + ((size_t)slot * G + h) * (D + 2);
        pp[2 + dd] = o;
        if (dd == 0) { pp[0] = M; pp[1] = Ls; }
      }
    }
    __syncthreads();
  };

  for (int k = 0; k < n; ++k) {
    // ---- segment change: finish the previous (i, g), load q of the new one
    if (cit.i != seg_i || cit.g != seg_g) {
      if (seg_i >= 0) finish_segment();
      seg_i = cit.i;
      seg_g = cit.g;
      seg_tok = cit.tok;
      seg_units = cit.units;
      seg_begin = a.Hkv * v.tok_unit_off[cit.i] + cit.g * cit.units;
      const uint16_t *qrow = a.q + ((size_t)cit.tok * a.Hq + cit.g * G) * D;
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
          uint4 q4 = *reinterpret_cast<const uint4 *>(qrow + h * D + (r8 + 8 * ch) * 8);
          float2 f0 = h2_to_f2(q4.x), f1 = h2_to_f2(q4.y), f2 = h2_to_f2(q4.z), f3 = h2_to_f2(q4.w);
          qf[h][ch][0] = f0.x * a.scale_log2; qf[h][ch][1] = f0.y * a.scale_log2;
          qf[h][ch][2] = f1.x * a.scale_log2; qf[h][ch][3] = f1.y * a.scale_log2;
          qf[h][ch][4] = f2.x * a.scale_log2; qf[h][ch][5] = f2.y * a.scale_log2;
          qf[h][ch][6] = f3.x * a.scale_log2; qf[h][ch][7] = f3.y * a.scale_log2;
        }
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[h][e] = 0.f;
      }
    }

    // ---- wait for this warp's rows of unit k
    const int stage = k % NS;
    const uint32_t parity = (uint32_t)(k / NS) & 1u;
    if (!dead) {
      dead = !mbar_wait(&my_bars[stage], parity, err);
      if (dead) k_dead = k;
    }
    int64_t src_unused;
    const int rows = dead ? 0 : warp_rows(cit, w, a, &src_unused, nullptr);
    const unsigned char *st = my_ring + stage * Cfg::kStageBytes;
    const uint16_t *Ks = reinterpret_cast<const uint16_t *>(st);
    const uint16_t *Vs = reinterpret_cast<const uint16_t *>(st + kKeysPerWarp * Cfg::kRowBytes);

    if (rows > 0) {
      // ---- scores: 4 steps of 4 keys; 8 lanes per key, NCH 16-byte chunks per lane
      float vals[NV];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int r = 4 * s + kq;
        float2 p2[G];
#pragma unroll
        for (int h = 0; h < G; ++h) p2[h] = make_float2(0.f, 0.f);
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
          uint4 k4 = *reinterpret_cast<const uint4 *>(Ks + r * D + (r8 + 8 * ch) * 8);
          float2 k0 = h2_to_f2(k4.x), k1 = h2_to_f2(k4.y), k2 = h2_to_f2(k4.z), k3 = h2_to_f2(k4.w);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            p2[h] = ffma2(make_float2(qf[h][ch][0], qf[h][ch][1]), k0, p2[h]);
            p2[h] = ffma2(make_float2(qf[h][ch][2], qf[h][ch][3]), k1, p2[h]);
            p2[h] = ffma2(make_float2(qf[h][ch][4], qf[h][ch][5]), k2, p2[h]);
            p2[h] = ffma2(make_float2(qf[h][ch][6], qf[h][ch][7]), k3, p2[h]);
          }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) vals[s * G + h] = p2[h].x + p2[h].y;
      }
      rs_step<NV>(vals, (r8 & 4) != 0, 4);
      rs_step<NV / 2>(vals, (r8 & 2) != 0, 2);
      if constexpr (NV >= 8) {
        rs_step<NV / 4>(vals, (r8 & 1) != 0, 1);
      } else {
        vals[0] += __shfl_xor_sync(0xffffffffu, vals[0], 1);
      }
      constexpr int NF = NV >= 8 ? NV / 8 : 1;
      const int base = ((r8 & 4) ? NV / 2 : 0) + ((r8 & 2) ? NV / 4 : 0) +
                       ((NV >= 8 && (r8 & 1)) ? NV / 8 : 0);
      if (NV >= 8 || (r8 & 1) == 0) {
#pragma unroll
        for (int j = 0; j < NF; ++j) {
          int vi = base + j;
          int s = vi / G, h = vi - s * G;
          sbuf[(4 * s + kq) * G + h] = vals[j];
        }
      }
      __syncwarp();

      // ---- online softmax over this warp's 16 keys (lanes: key = lane & 15)
      const int j = lane & 15, half = lane >> 4;
      float x[HPL], mx[HPL];
#pragma unroll
      for (int i = 0; i < HPL; ++i) {
        int h = half + 2 * i;
        bool ok = (h < G) && (j < rows);
        x[i] = ok ? sbuf[j * G + (h < G ? h : 0)] : -INFINITY;
        float m = x[i];
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        mx[i] = m;
      }
      float m_new[G], alpha[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float bm = __shfl_sync(0xffffffffu, mx[h / 2], (h & 1) * 16);
        m_new[h] = fmaxf(m_run[h], bm);
        alpha[h] = (m_run[h] == -INFINITY) ? 0.f : exp2_approx(m_run[h] - m_new[h]);
      }
      float ps[HPL];
#pragma unroll
      for (int i = 0; i < HPL; ++i) {
        int h = half + 2 * i;
        float mref = 0.f;
#pragma unroll
        for (int hh = 0; hh < G; ++hh)
          if (hh == h) mref = m_new[hh];
        float p = (x[i] == -INFINITY) ? 0.f : exp2_approx(x[i] - mref);
        if (h < G) sbuf[j * G + h] = p;
        float sm = p;
        sm += __shfl_xor_sync(0xffffffffu, sm, 8);
        sm += __shfl_xor_sync(0xffffffffu, sm, 4);
        sm += __shfl_xor_sync(0xffffffffu, sm, 2);
        sm += __shfl_xor_sync(0xffffffffu, sm, 1);
        ps[i] = sm;
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float bs = __shfl_sync(0xffffffffu, ps[h / 2], (h & 1) * 16);
        l_run[h] = l_run[h] * alpha[h] + bs;
        m_run[h] = m_new[h];
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[h][e] *= alpha[h];
      }
      __syncwarp();

      // ---- PV: lane owns dims [DPL*lane, DPL*lane + DPL) of every head
      for (int jj = 0; jj < rows; ++jj) {
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
#pragma unroll
          for (int h = 0; h < G; ++h) pr[h] = sbuf[jj * G + h];
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
    __syncwarp();
    // ---- refill this stage with unit k + NS
    if (lane == 0 && k + NS < n && !dead) {
      fence_proxy_async();
      issue(k + NS);
    }
    __syncwarp();
    it_next(cit, v);
  }
  finish_segment();
  // a warp that gave up on a wait still lets its copies in flight land
  // (bounded) before the CTA's shared memory is released
  if (dead && lane == 0) {
    for (int kk = k_dead; kk < issued; ++kk) {
      uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&my_bars[kk % NS], (uint32_t)(kk / NS) & 1u) &&
             globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Reduce: combine the partials of every (decode token, KV head) that spans
// several CTAs.  out = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c.
// ---------------------------------------------------------------------------
template <int D, int G>
__global__ void __launch_bounds__(128) k_reduce(AttnArgs a, int C) {
  WsHeader *hdr = reinterpret_cast<WsHeader *>(a.ws);
  const int *dec_tok = reinterpret_cast<const int *>(a.ws + a.lay.dec_tok);
  const int *off = reinterpret_cast<const int *>(a.ws + a.lay.tok_unit_off);
  const float *partials = reinterpret_cast<const float *>(a.ws + a.lay.partials);
  const int n_ig = hdr->n_dec * a.Hkv;
  const int64_t U = hdr->n_units;
  for (int ig = blockIdx.x; ig < n_ig; ig += gridDim.x) {
    const int i = ig / a.Hkv, g = ig - i * a.Hkv;
    const int units = off[i + 1] - off[i];
    const int tok = dec_tok[i];
    uint16_t *orow = a.out + ((size_t)tok * a.Hq + g * G) * D;
    if (units == 0) {
      for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) orow[idx] = 0;
      continue;
    }
    const int64_t ub = (int64_t)a.Hkv * off[i] + (int64_t)g * units, ue = ub + units;
    // CTA c covers [floor(cU/C), floor((c+1)U/C)); first/last CTA touching [ub, ue)
    const int c_first = (int)(((ub + 1) * C + U - 1) / U) - 1;
    const int c_last = (int)((ue * C + U - 1) / U) - 1;
    if (c_first == c_last) continue;  // finished inside one CTA
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
      const int h = idx / D, dd = idx - h * D;
      // only CTAs whose unit range is non-empty wrote a partial (with fewer units
      // than CTAs, some CTAs in [c_first, c_last] own no unit at all)
      auto has_units = [&](int cc) {
        return (int64_t)(cc + 1) * U / C > (int64_t)cc * U / C;
      };
      float M = -INFINITY;
      for (int cc = c_first; cc <= c_last; ++cc)
        if (has_units(cc)) M = fmaxf(M, partials[((size_t)(ig + cc) * G + h) * (D + 2)]);
      float o = 0.f, Ls = 0.f;
      if (M != -INFINITY) {
        for (int cc = c_first; cc <= c_last; ++cc) {
          if (!has_units(cc)) continue;
          const float *pp = partials + ((size_t)(ig + cc) * G + h) * (D + 2);
          float f = exp2_approx(pp[0] - M);
          o += f * pp[2 + dd];
          Ls += f * pp[1];
        }
      }
      orow[idx] = __half_as_ushort(__float2half_rn(Ls > 0.f ? o / Ls : 0.f));
    }
  }
}

template <int D, int G>
static cudaError_t launch_decode_t(const AttnArgs &a, int num_sms, cudaStream_t s) {
  constexpr int NS = (D == 128 && G == 8) ? 2 : 3;
  using Cfg = DecCfg<D, G, NS>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_decode<D, G, NS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  k_decode<D, G, NS><<<num_sms, kDecThreads, Cfg::kSmem, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_reduce<D, G><<<num_sms * 4, 128, 0, s>>>(a, num_sms);
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
