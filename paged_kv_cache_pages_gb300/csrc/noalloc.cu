// paged_attn_forward_noalloc: the whole attention of one ubatch without any
// device allocation by the caller or by the library.
//
// Some callers cannot call cudaMalloc: code running inside a host framework
// that owns all device memory and forbids outside allocations, runtimes with
// a fixed device-memory budget decided up front, and latency-critical paths
// where an allocation could synchronise the device.  They still own q, the
// pools, the tables and out; only the scratch that paged_attn_forward takes as
// `workspace` is replaced here by one fixed array in device memory.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes.  Each
// GPU that loads this library holds it until the process exits.  Host code may
// not use the array's name as a device address (on the host it names a
// stand-in object), so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current; make that first call
// before any stream capture.  All calls share the array and it keeps the last
// call's contents: the planning kernel clears everything a later kernel of the
// same call reads (error word, counters, work lists), and calls whose work
// overlaps on the GPU (different streams, or different host threads) race on
// it and must be serialised by the caller.
#include <mutex>

#include "kernels.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_for_current_device(void **addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ELAUNCH;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PA_ELAUNCH;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" int paged_attn_forward_noalloc(const uint16_t *q, const uint16_t *k_pages,
                                          const uint16_t *v_pages, const int32_t *tok_page_table,
                                          int max_pages, const int32_t *tok_kv_len, int T, int Hq,
                                          int Hkv, int P, int d, int num_pages, float scale,
                                          uint16_t *out, void *stream) {
  // The argument and shape checks of paged_attn_forward, in its order: with no
  // workspace it returns their first failure, PA_OK for an empty ubatch, or
  // PA_EWORKSPACE once everything but the workspace is acceptable.  So every input
  // gets the same status from both calls.
  int st = paged_attn_forward(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq,
                              Hkv, P, d, num_pages, scale, out, nullptr, 0, stream);
  if (st != PA_EWORKSPACE) return st;
  const size_t need = paged_attn_workspace_size(T, Hq, Hkv, d);
  if (need == 0) return PA_EUNSUPPORTED;
  if (need > kNoAllocScratchBytes) return PA_EWORKSPACE;  // ubatch too large for the fixed scratch
  void *scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != PA_OK) return st;
  return paged_attn_forward(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv,
                            P, d, num_pages, scale, out, scratch, kNoAllocScratchBytes, stream);
}
