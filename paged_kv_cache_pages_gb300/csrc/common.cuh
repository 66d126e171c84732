// Device-side helpers shared by the paged-attention kernels (sm_103a).
// Inline PTX for mbarriers, bulk/tensor async copies and bounded waits.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/paged_attn.h"

namespace pa {

// ----------------------------------------------------------------------------
// Workspace layout (device memory owned by the caller).
//
//   [0, 256)       WsHeader
//   tiles          int4 [T]      (tok_start, n_tok, n_kblocks, max kv_len)
//   dec_tok        int  [T]      decode token indices
//   tok_unit_off   int  [T + 1]  prefix sums of decode key blocks per token
//   flags          int  [T]      plan scratch: run-start flags
//   runs           int  [T + 1]  plan scratch: first token of each run
//   tile_off       int  [T + 1]  prefix sums of prefill work (key blocks x items) per tile
//   dec_start      int4 [4C]     first decode unit of each CTA: (i, g, kb, token), (units, kv_len, first block of i, -),
//                                  then the page ids of that unit's key block (8 ints, -1 past its end)
//   pf_start       int4 [C]      first prefill unit of each CTA: (tile, item in tile, kb,
//                                  tile * items per tile + item of the CTA's last unit)
//   pf_cnt         int  [T * Hkv * NP * 2 * 4]  arrival counters of split prefill items,
//                                  one per (item, softmax warpgroup, warp)
//   dec_cnt        int  [T * Hkv]   arrival counters of decode segments split over CTAs
//   partials       union of
//                    decode split partials  float [(T*Hkv + C)][G][D + 2]
//                    prefill split parts    float [2C][2][128][D + 4]  (16-byte rows)
// The decode and prefill kernels of one ubatch run one after the other on a
// stream, so their partials share one region.
// ----------------------------------------------------------------------------
struct WsHeader {
  int err;        // PA_ERR_* bits
  int n_tiles;    // prefill tiles
  int n_dec;      // decode tokens
  int n_units;    // decode work units (token, kv head, 128-key block)
  int pf_work;    // prefill work units (item, 128-key block)
  int C;          // CTAs the plan was cut for (= SM count)
  int T, Hq, Hkv, D, P, max_pages;
  int pad[52];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

constexpr int KB = 128;  // keys per block (decode unit and prefill key tile)
// Prefill work units a tile item counts when the planner cuts the work into equal CTA
// ranges: its key blocks, but at least kPfMinItemUnits.  An item of a few blocks never
// fills the MMA/softmax pipeline and still pays a whole item switch (epilogue, next Q
// tiles), so a range of many such items would take far longer than its blocks say.
// The units past an item's last block are virtual: they hold no work.
constexpr int kPfMinItemUnits = 6;
__host__ __device__ inline int pf_item_units(int nkb) {
  return nkb > 0 ? (nkb > kPfMinItemUnits ? nkb : kPfMinItemUnits) : 0;
}

struct WsLayout {
  size_t tiles, dec_tok, tok_unit_off, flags, runs, tile_off, dec_start, pf_start, pf_cnt;
  size_t dec_cnt;
  size_t partials, total;
  int n_cnt;  // entries of pf_cnt
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WsLayout ws_layout(int T, int Hq, int Hkv, int D, int C) {
  WsLayout l;
  size_t o = sizeof(WsHeader);
  size_t Tm = T > 0 ? (size_t)T : 1;
  size_t G = (size_t)(Hq / Hkv);
  size_t NP = G >= 2 ? G / 2 : 1;
  l.tiles = o;        o = align_up(o + Tm * 16, 256);
  l.dec_tok = o;      o = align_up(o + Tm * 4, 256);
  l.tok_unit_off = o; o = align_up(o + (Tm + 1) * 4, 256);
  l.flags = o;        o = align_up(o + Tm * 4, 256);
  l.runs = o;         o = align_up(o + (Tm + 1) * 4, 256);
  l.tile_off = o;     o = align_up(o + (Tm + 1) * 4, 256);
  l.dec_start = o;    o = align_up(o + (size_t)C * 64, 256);
  l.pf_start = o;     o = align_up(o + (size_t)C * 16, 256);
  l.n_cnt = (int)(Tm * Hkv * NP * 8);
  l.pf_cnt = o;       o = align_up(o + (size_t)l.n_cnt * 4, 256);
  l.dec_cnt = o;      o = align_up(o + Tm * Hkv * 4, 256);
  l.partials = o;
  size_t dec_part = (Tm * Hkv + (size_t)C) * G * (D + 2) * 4;
  size_t pf_part = (size_t)2 * C * 2 * 128 * (D + 4) * 4;
  o = align_up(o + (dec_part > pf_part ? dec_part : pf_part), 256);
  l.total = o;
  return l;
}

// The CTA (of C, each owning [floor(cW/C), floor((c+1)W/C))) that owns unit u.
__host__ __device__ inline int cta_of_unit(long long u, long long W, int C) {
  return (int)(((u + 1) * C + W - 1) / W) - 1;
}
__host__ __device__ inline bool cta_has_units(int c, long long W, int C) {
  return (long long)(c + 1) * W / C > (long long)c * W / C;
}

// ----------------------------------------------------------------------------
// PTX helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase.  Returns false (and sets PA_ERR_TIMEOUT in
// *err) if the phase did not complete within ~2 s of wall time.  (The split-KV decode
// kernel takes its limit from the host, default the same 2 s.)
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// Bound of the waits that let a kernel's own copies in flight land before it exits
// (never shortened: the copies must land).
constexpr uint64_t kDrainLimitNs = 2000000000ull;

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *err) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u) {
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicOr(err, PA_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// 1-D bulk async copy global -> shared, completion signalled on an mbarrier.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Bring `bytes` (a multiple of 16, 16-byte aligned address) of global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 FMAs in one instruction (sm_100+ packed f32x2); operands are packed
// inside the asm so no local ever needs an address.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// Two fp32 adds in one instruction (sm_100+ packed f32x2).
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// Two fp32 multiplies in one instruction (sm_100+ packed f32x2).
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// max of three floats in one instruction (sm_100+).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float2 h2_to_f2(uint32_t h) {
  __half2 v = *reinterpret_cast<__half2 *>(&h);
  return __half22float2(v);
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace pa
