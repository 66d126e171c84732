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
//   [0, 256)            WsHeader
//   tiles               int4 [T]        (tok_start, n_tok, n_kblocks, max kv_len)
//   dec_tok             int  [T]        decode token indices
//   tok_unit_off        int  [T + 1]    prefix sums of decode key-blocks per token
//   flags               int  [T]        plan scratch: run-start flags
//   runs                int  [T + 1]    plan scratch: first token of each run
//   partials            float[(T*Hkv + C)][G][D + 2]   split-KV partial results
// ----------------------------------------------------------------------------
struct WsHeader {
  int err;           // PA_ERR_* bits
  int n_tiles;       // prefill tiles
  int n_dec;         // decode tokens
  int n_units;       // decode work units (token, kv head, 128-key block)
  int tile_next;     // dynamic prefill scheduler: next work item
  int tile_done;     // CTAs finished (last one resets tile_next)
  int T, Hq, Hkv, D, P, max_pages;
  int pad[52];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

constexpr int KB = 128;  // keys per block (decode unit and prefill key tile)

struct WsLayout {
  size_t tiles, dec_tok, tok_unit_off, flags, runs, partials, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WsLayout ws_layout(int T, int Hq, int Hkv, int D, int C) {
  WsLayout l;
  size_t o = sizeof(WsHeader);
  size_t Tm = T > 0 ? (size_t)T : 1;
  l.tiles = o;        o = align_up(o + Tm * 16, 256);
  l.dec_tok = o;      o = align_up(o + Tm * 4, 256);
  l.tok_unit_off = o; o = align_up(o + (Tm + 1) * 4, 256);
  l.flags = o;        o = align_up(o + Tm * 4, 256);
  l.runs = o;         o = align_up(o + (Tm + 1) * 4, 256);
  l.partials = o;
  size_t G = (size_t)(Hq / Hkv);
  o = align_up(o + (Tm * Hkv + (size_t)C) * G * (D + 2) * 4, 256);
  l.total = o;
  return l;
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
// *err) if the phase did not complete within ~2 s of wall time.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

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

__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 FMAs in one instruction (sm_100+ packed f32x2).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t ra = *reinterpret_cast<uint64_t *>(&a);
  uint64_t rb = *reinterpret_cast<uint64_t *>(&b);
  uint64_t rc = *reinterpret_cast<uint64_t *>(&c);
  uint64_t rd;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  return *reinterpret_cast<float2 *>(&rd);
}

__device__ __forceinline__ float2 h2_to_f2(uint32_t h) {
  __half2 v = *reinterpret_cast<__half2 *>(&h);
  return __half22float2(v);
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace pa
