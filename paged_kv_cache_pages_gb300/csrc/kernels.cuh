// Kernel declarations and launch parameters shared by the translation units.
#pragma once

#include <atomic>

#include "common.cuh"

namespace pa {

__global__ void k_expand(const int32_t *seq_pt, int n_seq, int max_pages, const int32_t *tok_seq,
                         const int32_t *tok_pos, int T, int P, int32_t *tok_pt, int32_t *tok_kv,
                         int64_t *slot, int *err);
__global__ void k_append(const uint4 *k, const uint4 *v, const int64_t *slot, int T, uint4 *kp,
                         uint4 *vp, int num_pages, int Hkv, int P, int chunks_per_row, int *err);
__global__ void k_append_fp8(const uint16_t *k, const uint16_t *v, const int64_t *slot, int T,
                             uint8_t *k8, uint8_t *v8t, float *ks, float *vs, int num_pages,
                             int Hkv, int P, int d, int *err);
__global__ void k_copy_pages(const int32_t *src, const int32_t *dst, int n, uint4 *kp, uint4 *vp,
                             int num_pages, long long page_units, int *err);
__global__ void k_validate(const int32_t *tpt, int max_pages, const int32_t *kv, int T, int P,
                           int num_pages, int *err);
__global__ void k_plan_mark(const int32_t *tpt, int max_pages, int T, unsigned char *ws,
                            WsLayout lay);
__global__ void k_plan(const int32_t *tpt, int max_pages, const int32_t *kv, int T, int P, int Hkv,
                       int NP, int min_run, int C, unsigned char *ws, WsLayout lay);

// Per-device flags of a kernel's one-time launch setup (function attributes are per
// device).  Returns true for the first caller on the current device, which then
// does the setup; a race makes two callers do the same idempotent setup.
struct PerDeviceOnce {
  std::atomic<unsigned long long> done{0};
  bool first() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return true;
    const unsigned long long bit = 1ull << dev;
    return (done.load(std::memory_order_acquire) & bit) == 0;
  }
  void mark() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return;
    done.fetch_or(1ull << dev, std::memory_order_release);
  }
};

// Arguments of the attention kernels (passed by value).
struct AttnArgs {
  const uint16_t *q;
  const uint16_t *k_pages;
  const uint16_t *v_pages;
  const int32_t *tpt;
  const int32_t *kv;
  uint16_t *out;
  unsigned char *ws;
  WsLayout lay;
  int max_pages, T, Hq, Hkv, P, D, num_pages;
  float scale_log2;  // scale * log2(e): softmax evaluated with exp2
  // masked decode (unified-span baseline) only, else null: (sequence, position) of
  // every slot of the pool and of every token
  const int32_t *cell_seq, *cell_pos, *tok_seq, *tok_pos;
  // FP8 pages only, else null: the binary32 scale of every cached (page, head, row)
  const float *k_scale, *v_scale;
  // bounded-wait limit of the split-KV decode kernel, in ns (paged_attn_set_decode_wait_limit)
  unsigned long long wait_ns;
  // decode with the append fused (f16 pages only), else null: the layer's new K/V rows
  // [T][Hkv][d] and their slots
  const uint16_t *k_new, *v_new;
  const int64_t *slot;
};

// Decode: split-KV over all SMs plus the log-sum-exp reduce.  Returns a
// cudaError_t from the launches.
cudaError_t launch_decode(const AttnArgs &a, int num_sms, const void *tmaps, cudaStream_t s);

// Prefill: tcgen05 tensor-core tiles.
cudaError_t launch_prefill(const AttnArgs &a, int num_sms, const void *tmaps, cudaStream_t s);

}  // namespace pa
