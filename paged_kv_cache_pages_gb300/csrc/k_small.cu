// Small kernels of the paged-attention path (sm_103a):
//   k_expand   per-token expansion of the page table and true KV length
//              (UA-PagedAttention page, section 作品简介)
//   k_append   reshape-and-cache: scatter new K/V rows into their page slots
//              (CacheFlow page, section 核心架构 3)
//   k_validate table check without trapping
//   k_plan     one-CTA device planner: same-row runs -> tensor-core tiles,
//              short runs -> split-KV decode work
#include "kernels.cuh"

namespace pa {

// ---------------------------------------------------------------------------
// Expansion.  One warp per token: the row copy is 128-byte coalesced.
// ---------------------------------------------------------------------------
__global__ void k_expand(const int32_t *__restrict__ seq_pt, int n_seq, int max_pages,
                         const int32_t *__restrict__ tok_seq, const int32_t *__restrict__ tok_pos,
                         int T, int P, int32_t *__restrict__ tok_pt, int32_t *__restrict__ tok_kv,
                         int64_t *__restrict__ slot, int *err) {
  int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int t = warp; t < T; t += nwarps) {
    int s = tok_seq[t];
    int p = tok_pos[t];
    bool bad = s >= n_seq || (s >= 0 && (p < 0 || p / P >= max_pages));
    if (bad && lane == 0 && err) atomicOr(err, PA_ERR_SEQ_RANGE);
    int32_t *row = tok_pt + (size_t)t * max_pages;
    if (s < 0 || bad) {
      for (int i = lane; i < max_pages; i += 32) row[i] = -1;
      if (lane == 0) { tok_kv[t] = 0; slot[t] = -1; }
      continue;
    }
    const int32_t *srow = seq_pt + (size_t)s * max_pages;
    for (int i = lane; i < max_pages; i += 32) row[i] = srow[i];
    if (lane == 0) {
      tok_kv[t] = p + 1;
      int page = srow[p / P];
      slot[t] = page < 0 ? -1 : (int64_t)page * P + (p % P);
    }
  }
}

// ---------------------------------------------------------------------------
// Append.  One thread per 16-byte chunk of a (token, kv head) row; K and V in
// the same thread.  Consecutive threads cover consecutive bytes of a row.
// ---------------------------------------------------------------------------
// Page copy for copy-on-write forks: blockIdx.y walks the pairs, the x threads the
// 16-byte units of one page (K and V).
__global__ void k_copy_pages(const int32_t *__restrict__ src, const int32_t *__restrict__ dst,
                             int n, uint4 *__restrict__ kp, uint4 *__restrict__ vp,
                             int num_pages, long long page_units, int *err) {
  for (int pr = blockIdx.y; pr < n; pr += gridDim.y) {
    const int s = src[pr], d = dst[pr];
    if (s < 0 || s >= num_pages || d < 0 || d >= num_pages) {
      if (err && blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err, PA_ERR_PAGE_RANGE);
      continue;
    }
    const uint4 *ks = kp + (size_t)s * page_units, *vs = vp + (size_t)s * page_units;
    uint4 *kd = kp + (size_t)d * page_units, *vd = vp + (size_t)d * page_units;
    for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < page_units;
         u += (long long)gridDim.x * blockDim.x) {
      const uint4 a = ks[u], b = vs[u];
      kd[u] = a;
      vd[u] = b;
    }
  }
}

// FP8 E4M3 code of a binary32 value: nearest, ties to even, saturating at +-448.
// The same value goes into both halves of the pair, so the byte order of the pair
// does not matter.
__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(r) : "f"(x));
  return static_cast<uint8_t>(r & 0xFF);
}

// Quantising reshape-and-cache into FP8 pages (one warp per (token, KV head) row):
// scale = amax / 448 over the row (1 for an all-zero row), code = E4M3(x / scale).
// K rows go to k8 [page][h][offset][d]; V rows to v8t [page][h][d][offset]
// (transposed inside each (page, head) block); the scales to [page][h][offset].
__global__ void k_append_fp8(const uint16_t *__restrict__ k, const uint16_t *__restrict__ v,
                             const int64_t *__restrict__ slot, int T, uint8_t *__restrict__ k8,
                             uint8_t *__restrict__ v8t, float *__restrict__ ks,
                             float *__restrict__ vs, int num_pages, int Hkv, int P, int d,
                             int *err) {
  const int lane = threadIdx.x & 31;
  const long long nw = (long long)gridDim.x * blockDim.x / 32;
  for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 32;
       r < (long long)T * Hkv; r += nw) {
    const int t = (int)(r / Hkv), h = (int)(r % Hkv);
    const int64_t sl = slot[t];
    if (sl < 0) continue;
    if (sl >= (int64_t)num_pages * P) {
      if (err && lane == 0) atomicOr(err, PA_ERR_SLOT_RANGE);
      continue;
    }
    const int64_t page = sl / P, off = sl % P;
    const size_t row = ((size_t)page * Hkv + h) * P + off;
    for (int which = 0; which < 2; ++which) {
      const uint16_t *src = (which ? v : k) + ((size_t)t * Hkv + h) * d;
      float x[4];
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = lane + 32 * j;
        x[j] = i < d ? __half2float(__ushort_as_half(src[i])) : 0.f;
        amax = fmaxf(amax, fabsf(x[j]));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float scale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = lane + 32 * j;
        if (i >= d) break;
        const uint8_t c = f32_to_e4m3(__fdiv_rn(x[j], scale));
        if (which == 0)
          k8[row * d + i] = c;
        else
          v8t[(((size_t)page * Hkv + h) * d + i) * P + off] = c;
      }
      if (lane == 0) (which ? vs : ks)[row] = scale;
    }
  }
}

__global__ void k_append(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                         const int64_t *__restrict__ slot, int T, uint4 *__restrict__ kp,
                         uint4 *__restrict__ vp, int num_pages, int Hkv, int P, int chunks_per_row,
                         int *err) {
  // a following attention kernel may be launched now; it waits for this grid's
  // results (griddepcontrol.wait) before it reads the pool
  asm volatile("griddepcontrol.launch_dependents;");
  int64_t total = (int64_t)T * Hkv * chunks_per_row;
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    int c = (int)(i % chunks_per_row);
    int64_t th = i / chunks_per_row;
    int h = (int)(th % Hkv);
    int t = (int)(th / Hkv);
    int64_t s = slot[t];
    if (s < 0) continue;
    if (s >= (int64_t)num_pages * P) {
      if (h == 0 && c == 0 && err) atomicOr(err, PA_ERR_SLOT_RANGE);
      continue;
    }
    int64_t page = s / P, off = s % P;
    int64_t dst = (((page * Hkv) + h) * P + off) * chunks_per_row + c;
    kp[dst] = k[i];
    vp[dst] = v[i];
  }
}

// ---------------------------------------------------------------------------
// Validation: every page a token needs must exist; kv_len within the row.
// ---------------------------------------------------------------------------
__global__ void k_validate(const int32_t *__restrict__ tpt, int max_pages,
                           const int32_t *__restrict__ kv, int T, int P, int num_pages, int *err) {
  int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int t = warp; t < T; t += nwarps) {
    int L = kv[t];
    if (L < 0 || L > max_pages * P) {
      if (lane == 0) atomicOr(err, PA_ERR_KV_RANGE);
      continue;
    }
    int np = (L + P - 1) / P;
    bool bad = false;
    for (int i = lane; i < np; i += 32) {
      int pg = tpt[(size_t)t * max_pages + i];
      bad |= (pg < 0 || pg >= num_pages);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(err, PA_ERR_PAGE_RANGE);
  }
}

// ---------------------------------------------------------------------------
// Planner, part 1 (many CTAs): flags[t] = 1 if token t starts a run, i.e. its
// page-table row differs from row t-1 in any byte.  One warp per token.
// ---------------------------------------------------------------------------
__global__ void k_plan_mark(const int32_t *__restrict__ tpt, int max_pages, int T,
                            unsigned char *ws, WsLayout lay) {
  int *flags = reinterpret_cast<int *>(ws + lay.flags);
  int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int t = warp; t < T; t += nwarps) {
    bool d = (t == 0);
    if (!d) {
      const int32_t *a = tpt + (size_t)t * max_pages;
      const int32_t *b = a - max_pages;
      bool x = false;
      for (int i = lane; i < max_pages; i += 32) x |= (a[i] != b[i]);
      d = __any_sync(0xffffffffu, x);
    }
    if (lane == 0) flags[t] = d ? 1 : 0;
  }
}

// ---------------------------------------------------------------------------
// Planner, part 2 (one CTA of 1024 threads).
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;

// Exclusive scan across the block; returns the prefix of `v` and writes the
// block total to *total.  All threads must call it.
__device__ int block_excl_scan(int v, int *total, int *sh) {
  int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[w] = x;
  __syncthreads();
  if (w == 0) {
    int s = lane < (kPlanThreads / 32) ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    sh[lane] = s;  // inclusive prefix of warp sums
  }
  __syncthreads();
  int warp_prefix = w > 0 ? sh[w - 1] : 0;
  *total = sh[kPlanThreads / 32 - 1];
  __syncthreads();
  return warp_prefix + x - v;
}

// Largest i in [0, n] with off[i] * scale <= u (off non-decreasing, off[0] = 0).
__device__ __forceinline__ int upper_index(const int *off, int n, long long u, long long scale) {
  int lo = 0, hi = n;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if ((long long)off[mid] * scale <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kPlanThreads, 1)
k_plan(const int32_t *__restrict__ tpt, int max_pages, const int32_t *__restrict__ kv, int T,
       int P, int Hkv, int NP, int min_run, int C, unsigned char *ws, WsLayout lay) {
  __shared__ int sh[32];
  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
  int4 *tiles = reinterpret_cast<int4 *>(ws + lay.tiles);
  int *dec_tok = reinterpret_cast<int *>(ws + lay.dec_tok);
  int *tok_unit_off = reinterpret_cast<int *>(ws + lay.tok_unit_off);
  int *flags = reinterpret_cast<int *>(ws + lay.flags);
  int *runs = reinterpret_cast<int *>(ws + lay.runs);
  int *tile_off = reinterpret_cast<int *>(ws + lay.tile_off);
  int4 *dec_start = reinterpret_cast<int4 *>(ws + lay.dec_start);
  int4 *pf_start = reinterpret_cast<int4 *>(ws + lay.pf_start);
  int *pf_cnt = reinterpret_cast<int *>(ws + lay.pf_cnt);
  int *dec_cnt = reinterpret_cast<int *>(ws + lay.dec_cnt);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cap = max_pages * P;

  if (tid == 0) hdr->err = 0;

  // 1. run ids by a scan of the start flags; runs[r] = first token of run r
  int n_runs = 0;
  for (int c0 = 0; c0 < T; c0 += kPlanThreads) {
    int t = c0 + tid;
    int f = t < T ? flags[t] : 0;
    int tot;
    int rid = block_excl_scan(f, &tot, sh) + n_runs;
    if (f) runs[rid] = t;
    n_runs += tot;
  }
  if (tid == 0) runs[n_runs] = T;
  __syncthreads();

  // 2. runs of >= min_run tokens become tiles of <= 128 tokens (near-equal
  //    split); shorter runs become decode tokens.
  int tile_base = 0, dec_base = 0;
  for (int c0 = 0; c0 < n_runs; c0 += kPlanThreads) {
    int r = c0 + tid;
    int a = 0, len = 0;
    if (r < n_runs) { a = runs[r]; len = runs[r + 1] - a; }
    bool prefill_run = r < n_runs && len >= min_run;
    int n_tiles = prefill_run ? (len + KB - 1) / KB : 0;
    int n_dec = (r < n_runs && !prefill_run) ? len : 0;
    int tot_tiles, tot_dec;
    int tile_off0 = block_excl_scan(n_tiles, &tot_tiles, sh) + tile_base;
    int dec_off = block_excl_scan(n_dec, &tot_dec, sh) + dec_base;
    for (int i = 0; i < n_tiles; ++i) {
      int b0 = a + (int)((int64_t)len * i / n_tiles);
      int b1 = a + (int)((int64_t)len * (i + 1) / n_tiles);
      tiles[tile_off0 + i] = make_int4(b0, b1 - b0, 0, 0);
    }
    for (int i = 0; i < n_dec; ++i) dec_tok[dec_off + i] = a + i;
    tile_base += tot_tiles;
    dec_base += tot_dec;
  }
  __syncthreads();

  // arrival counters of this plan's prefill items start at zero (the combining
  // part resets its counter after use, so later runs of the plan find zeros too)
  for (int i = tid; i < tile_base * Hkv * NP * 8; i += kPlanThreads) pf_cnt[i] = 0;
  for (int i = tid; i < dec_base * Hkv; i += kPlanThreads) dec_cnt[i] = 0;

  // 3. key blocks of each tile: ceil(max kv_len over its tokens / 128); one warp per tile
  for (int i = warp; i < tile_base; i += kPlanThreads / 32) {
    int4 tl = tiles[i];
    int mx = 0;
    bool bad = false;
    for (int u = tl.x + lane; u < tl.x + tl.y; u += 32) {
      int L = kv[u];
      bad |= (L < 0 || L > cap);
      mx = max(mx, min(max(L, 0), cap));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&hdr->err, PA_ERR_KV_RANGE);
    if (lane == 0) {
      tiles[i].z = (mx + KB - 1) / KB;
      tiles[i].w = mx;
    }
  }
  __syncthreads();

  // 4. prefill work prefix over tiles: each tile holds Hkv * NP items of
  //    pf_item_units(n_kblocks) units (key blocks, at least kPfMinItemUnits)
  int work_base = 0;
  for (int c0 = 0; c0 < tile_base; c0 += kPlanThreads) {
    int i = c0 + tid;
    int wk = i < tile_base ? pf_item_units(tiles[i].z) * Hkv * NP : 0;
    int tot;
    int off = block_excl_scan(wk, &tot, sh) + work_base;
    if (i < tile_base) tile_off[i] = off;
    work_base += tot;
  }
  if (tid == 0) tile_off[tile_base] = work_base;

  // 5. decode units: 128-key blocks per decode token, prefix-summed
  int unit_base = 0;
  for (int c0 = 0; c0 < dec_base; c0 += kPlanThreads) {
    int i = c0 + tid;
    int units = 0;
    if (i < dec_base) {
      int L = kv[dec_tok[i]];
      if (L < 0 || L > cap) { atomicOr(&hdr->err, PA_ERR_KV_RANGE); L = L < 0 ? 0 : cap; }
      units = (L + KB - 1) / KB;
    }
    int tot;
    int off = block_excl_scan(units, &tot, sh) + unit_base;
    if (i < dec_base) tok_unit_off[i] = off;
    unit_base += tot;
  }
  if (tid == 0) tok_unit_off[dec_base] = unit_base;
  __syncthreads();

  // 6. where each of the C CTAs starts in the decode and in the prefill work.  The
  // decode work goes to min(C, U) CTAs, so that each of them owns at least one unit.
  const long long U = (long long)unit_base * Hkv, W = work_base;
  const int Cd = U < C ? (int)U : C;
  for (int c = tid; c < C; c += kPlanThreads) {
    if (c < Cd) {
      long long u = (long long)c * U / Cd;
      int i = upper_index(tok_unit_off, dec_base, u, Hkv);
      if (i >= dec_base) i = dec_base - 1;
      int units = tok_unit_off[i + 1] - tok_unit_off[i];
      while (units == 0 && i + 1 < dec_base) {  // tokens without keys own no unit
        ++i;
        units = tok_unit_off[i + 1] - tok_unit_off[i];
      }
      long long r = u - (long long)Hkv * tok_unit_off[i];
      int g = units > 0 ? (int)(r / units) : 0;
      const int tok = dec_tok[i];
      const int L = min(max(kv[tok], 0), cap);
      const int kb = units > 0 ? (int)(r - (long long)g * units) : 0;
      dec_start[4 * c] = make_int4(i, g, kb, tok);
      dec_start[4 * c + 1] = make_int4(units, L, tok_unit_off[i], 0);
      // page ids of the first key block, so the first copy needs no table lookup
      int pg[8];
      const int key0 = kb * KB, npg = (min(KB, L - key0) + P - 1) / P;
      const int32_t *row = tpt + (size_t)tok * max_pages + key0 / P;
      for (int j = 0; j < 8; ++j) pg[j] = j < npg ? row[j] : -1;
      dec_start[4 * c + 2] = make_int4(pg[0], pg[1], pg[2], pg[3]);
      dec_start[4 * c + 3] = make_int4(pg[4], pg[5], pg[6], pg[7]);
    }
    if (W > 0) {
      long long w = (long long)c * W / C;
      int t = upper_index(tile_off, tile_base, w, 1);
      if (t >= tile_base) t = tile_base - 1;
      while (tiles[t].z == 0 && t + 1 < tile_base) ++t;
      int nkb = tiles[t].z;
      long long r = w - tile_off[t];
      int j = nkb > 0 ? (int)(r / pf_item_units(nkb)) : 0;
      // and the item holding the CTA's last unit, tile * Hkv * NP + item (the prefill
      // kernel runs the segment of that item first, so that both parts of every split
      // item are done early and their combine stays off the end of the launch)
      long long wl = (long long)(c + 1) * W / C - 1;
      if (wl < w) wl = w;
      int tl = upper_index(tile_off, tile_base, wl, 1);
      if (tl >= tile_base) tl = tile_base - 1;
      while (tiles[tl].z == 0 && tl + 1 < tile_base) ++tl;
      const int nkl = tiles[tl].z;
      const int jl = nkl > 0 ? (int)((wl - tile_off[tl]) / pf_item_units(nkl)) : 0;
      pf_start[c] = make_int4(t, j, nkb > 0 ? (int)(r - (long long)j * pf_item_units(nkb)) : 0,
                              tl * Hkv * NP + jl);
    }
  }
  if (tid == 0) {
    hdr->n_tiles = tile_base;
    hdr->n_dec = dec_base;
    hdr->n_units = (int)U;
    hdr->pf_work = work_base;
    hdr->C = C;
    hdr->T = T;
    hdr->Hkv = Hkv;
    hdr->P = P;
    hdr->max_pages = max_pages;
  }
}

}  // namespace pa
