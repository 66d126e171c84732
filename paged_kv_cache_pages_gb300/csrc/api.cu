// C-ABI entry points of libpagedattn.so (declared in include/paged_attn.h).
// Host-side argument checks, workspace layout, tensor-map encoding and launches.
#include <atomic>
#include <climits>
#include <cstdio>
#include <cuda.h>
#include <nvtx3/nvToolsExt.h>

#include "kernels.cuh"
#include "tmap.cuh"

using namespace pa;

namespace {

// Each launching entry point opens an NVTX range named after itself, so a profiler
// timeline (nsys, ncu's NVTX filter) shows which call launched which kernels.  With
// no tool attached the calls return at once (header-only NVTX3, no link dependency).
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};

std::atomic<int> g_min_run{16};
std::atomic<unsigned long long> g_decode_wait_ns{kWaitLimitNs};

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cached[64] = {0};
  if (dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool pow2_in(int x, int lo, int hi) { return x >= lo && x <= hi && (x & (x - 1)) == 0; }

int check_shape(int Hq, int Hkv, int P, int d) {
  if (Hq <= 0 || Hkv <= 0 || P <= 0 || d <= 0) return PA_EINVAL;
  if (Hq % Hkv != 0) return PA_EUNSUPPORTED;
  int G = Hq / Hkv;
  if (!(G == 1 || G == 2 || G == 4 || G == 8)) return PA_EUNSUPPORTED;
  if (!(d == 64 || d == 128)) return PA_EUNSUPPORTED;
  if (!pow2_in(P, 16, 128)) return PA_EUNSUPPORTED;
  return PA_OK;
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ELAUNCH; }

// Common checks of the attention calls.
int check_attn(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
               const int32_t *tpt, int max_pages, const int32_t *kv, int T, int Hq, int Hkv, int P,
               int d, int num_pages, const uint16_t *out, const void *ws, size_t ws_bytes,
               bool need_data) {
  if (T < 0 || max_pages < 0 || num_pages < 0) return PA_EINVAL;
  int st = check_shape(Hq, Hkv, P, d);
  if (st != PA_OK) return st;
  if ((int64_t)max_pages * P > INT_MAX / 2) return PA_EUNSUPPORTED;
  if ((int64_t)T * Hq > INT_MAX / 256) return PA_EUNSUPPORTED;
  if (T == 0) return PA_OK;
  if (!tpt || !kv || (max_pages == 0)) return PA_EINVAL;
  if (need_data && (!q || !k_pages || !v_pages || !out || num_pages == 0)) return PA_EINVAL;
  if (!ws) return PA_EWORKSPACE;
  int C = sm_count();
  if (C <= 0) return PA_ELAUNCH;
  if (ws_bytes < ws_layout(T, Hq, Hkv, d, C).total) return PA_EWORKSPACE;
  if (!aligned16(ws) || !aligned16(tpt) || !aligned16(kv)) return PA_EALIGN;
  if (need_data && (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out)))
    return PA_EALIGN;
  return PA_OK;
}

AttnArgs make_args(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                   const int32_t *tpt, int max_pages, const int32_t *kv, int T, int Hq, int Hkv,
                   int P, int d, int num_pages, float scale, uint16_t *out, void *ws) {
  AttnArgs a;
  a.q = q;
  a.k_pages = k_pages;
  a.v_pages = v_pages;
  a.tpt = tpt;
  a.kv = kv;
  a.out = out;
  a.ws = static_cast<unsigned char *>(ws);
  a.lay = ws_layout(T, Hq, Hkv, d, sm_count());
  a.max_pages = max_pages;
  a.T = T;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.P = P;
  a.D = d;
  a.num_pages = num_pages;
  a.scale_log2 = scale * kLog2e;
  a.cell_seq = a.cell_pos = a.tok_seq = a.tok_pos = nullptr;
  a.k_scale = a.v_scale = nullptr;
  a.wait_ns = g_decode_wait_ns.load();
  a.k_new = a.v_new = nullptr;
  a.slot = nullptr;
  return a;
}

}  // namespace

extern "C" {

const char *paged_attn_strerror(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_EINVAL: return "invalid argument (null pointer, negative or inconsistent size)";
    case PA_EUNSUPPORTED: return "unsupported shape (d in {64,128}, P in {16,32,64,128}, Hq/Hkv in {1,2,4,8})";
    case PA_EWORKSPACE: return "workspace missing or too small";
    case PA_ELAUNCH: return "CUDA launch or runtime call failed";
    case PA_EDEVICE: return "device-side error word is set (page id, kv_len, slot or wait timeout)";
    case PA_EALIGN: return "device pointer not 16-byte aligned";
    case PA_ENOSPACE: return "page pool has too few free pages";
    default: return "unknown status";
  }
}

int paged_attn_version(void) { return 100; }

int paged_expand_ubatch(const int32_t *seq_page_table, int n_seq, int max_pages,
                        const int32_t *tok_seq, const int32_t *tok_pos, int T, int P,
                        int32_t *tok_page_table, int32_t *tok_kv_len, int64_t *slot_mapping,
                        int *err, void *stream) {
  NvtxRange nvtx_range("paged_expand_ubatch");
  if (T < 0 || n_seq < 0 || max_pages <= 0 || P <= 0) return PA_EINVAL;
  if (T == 0) return PA_OK;
  if (!tok_seq || !tok_pos || !tok_page_table || !tok_kv_len || !slot_mapping) return PA_EINVAL;
  if (n_seq > 0 && !seq_page_table) return PA_EINVAL;
  int blocks = (T + 7) / 8;
  if (blocks > 65535) blocks = 65535;
  k_expand<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      seq_page_table, n_seq, max_pages, tok_seq, tok_pos, T, P, tok_page_table, tok_kv_len,
      slot_mapping, err);
  return launch_status(cudaGetLastError());
}

int paged_kv_append(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping, int T,
                    uint16_t *k_pages, uint16_t *v_pages, int num_pages, int Hkv, int P, int d,
                    int *err, void *stream) {
  NvtxRange nvtx_range("paged_kv_append");
  if (T < 0 || num_pages < 0 || Hkv <= 0 || P <= 0 || d <= 0) return PA_EINVAL;
  if (d % 8 != 0) return PA_EUNSUPPORTED;
  if (T == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_pages || !v_pages) return PA_EINVAL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pages) || !aligned16(v_pages))
    return PA_EALIGN;
  int cpr = d / 8;
  int64_t total = (int64_t)T * Hkv * cpr;
  int64_t blocks = (total + 255) / 256;
  int cap = sm_count() * 8;
  if (cap <= 0) cap = 1024;
  if (blocks > cap) blocks = cap;
  k_append<<<(int)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const uint4 *>(k), reinterpret_cast<const uint4 *>(v), slot_mapping, T,
      reinterpret_cast<uint4 *>(k_pages), reinterpret_cast<uint4 *>(v_pages), num_pages, Hkv, P,
      cpr, err);
  return launch_status(cudaGetLastError());
}

static int plan_with(const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                     int T, int Hq, int Hkv, int P, int d, void *workspace,
                     size_t workspace_bytes, void *stream, int min_run);

int paged_kv_append_fp8(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping, int T,
                        uint8_t *k8_pages, uint8_t *v8t_pages, float *k_scale, float *v_scale,
                        int num_pages, int Hkv, int P, int d, int *err, void *stream) {
  NvtxRange nvtx_range("paged_kv_append_fp8");
  if (T < 0 || num_pages < 0 || Hkv <= 0 || P <= 0 || d <= 0) return PA_EINVAL;
  if (d > 128 || d % 32 != 0) return PA_EUNSUPPORTED;
  if (T == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k8_pages || !v8t_pages || !k_scale || !v_scale)
    return PA_EINVAL;
  const long long rows = (long long)T * Hkv;
  int blocks = (int)std::min<long long>((rows + 7) / 8, (long long)sm_count() * 16);
  if (blocks < 1) blocks = 1;
  k_append_fp8<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      k, v, slot_mapping, T, k8_pages, v8t_pages, k_scale, v_scale, num_pages, Hkv, P, d, err);
  return launch_status(cudaGetLastError());
}

// Checks and launch arguments shared by the FP8-page attention entry points.  Returns
// PA_OK with *a and *maps set, or the status to return (PA_OK with T == 0: nothing to do).
static int fp8_setup(const uint16_t *q, const uint8_t *k8_pages, const uint8_t *v8t_pages,
                     const float *k_scale, const float *v_scale, const int32_t *tok_page_table,
                     int max_pages, const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P,
                     int d, int num_pages, float scale, uint16_t *out, void *workspace,
                     size_t workspace_bytes, AttnArgs *a, AttnMaps *maps) {
  const uint16_t *kp = reinterpret_cast<const uint16_t *>(k8_pages);
  const uint16_t *vp = reinterpret_cast<const uint16_t *>(v8t_pages);
  int st = check_attn(q, kp, vp, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P, d,
                      num_pages, out, workspace, workspace_bytes, true);
  if (st != PA_OK || T == 0) return st;
  if (P != 128 || d != 128) return PA_EUNSUPPORTED;
  if (!k_scale || !v_scale) return PA_EINVAL;
  if (!aligned16(k_scale) || !aligned16(v_scale)) return PA_EALIGN;
  *a = make_args(q, kp, vp, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P, d, num_pages,
                 scale, out, workspace);
  a->k_scale = k_scale;
  a->v_scale = v_scale;
  return encode_attn_maps_fp8(*a, maps);
}

int paged_attn_decode_fp8(const uint16_t *q, const uint8_t *k8_pages, const uint8_t *v8t_pages,
                          const float *k_scale, const float *v_scale,
                          const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                          int T, int Hq, int Hkv, int P, int d, int num_pages, float scale,
                          uint16_t *out, void *workspace, size_t workspace_bytes, void *stream) {
  NvtxRange nvtx_range("paged_attn_decode_fp8");
  AttnArgs a;
  AttnMaps maps;
  int st = fp8_setup(q, k8_pages, v8t_pages, k_scale, v_scale, tok_page_table, max_pages,
                     tok_kv_len, T, Hq, Hkv, P, d, num_pages, scale, out, workspace,
                     workspace_bytes, &a, &maps);
  if (st != PA_OK || T == 0) return st;
  return launch_status(launch_decode(a, sm_count(), &maps, static_cast<cudaStream_t>(stream)));
}

int paged_attn_prefill_fp8(const uint16_t *q, const uint8_t *k8_pages, const uint8_t *v8t_pages,
                           const float *k_scale, const float *v_scale,
                           const int32_t *tok_page_table, int max_pages,
                           const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                           int num_pages, float scale, uint16_t *out, void *workspace,
                           size_t workspace_bytes, void *stream) {
  NvtxRange nvtx_range("paged_attn_prefill_fp8");
  AttnArgs a;
  AttnMaps maps;
  int st = fp8_setup(q, k8_pages, v8t_pages, k_scale, v_scale, tok_page_table, max_pages,
                     tok_kv_len, T, Hq, Hkv, P, d, num_pages, scale, out, workspace,
                     workspace_bytes, &a, &maps);
  if (st != PA_OK || T == 0) return st;
  return launch_status(launch_prefill(a, sm_count(), &maps, static_cast<cudaStream_t>(stream)));
}

int paged_attn_forward_fp8(const uint16_t *q, const uint8_t *k8_pages, const uint8_t *v8t_pages,
                           const float *k_scale, const float *v_scale,
                           const int32_t *tok_page_table, int max_pages,
                           const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                           int num_pages, float scale, uint16_t *out, void *workspace,
                           size_t workspace_bytes, void *stream) {
  NvtxRange nvtx_range("paged_attn_forward_fp8");
  AttnArgs a;
  AttnMaps maps;
  int st = fp8_setup(q, k8_pages, v8t_pages, k_scale, v_scale, tok_page_table, max_pages,
                     tok_kv_len, T, Hq, Hkv, P, d, num_pages, scale, out, workspace,
                     workspace_bytes, &a, &maps);
  if (st != PA_OK || T == 0) return st;
  st = paged_attn_plan(tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P, d, workspace,
                       workspace_bytes, stream);
  if (st != PA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = launch_status(launch_prefill(a, sm_count(), &maps, s));
  if (st != PA_OK) return st;
  return launch_status(launch_decode(a, sm_count(), &maps, s));
}

int paged_copy_pages(const int32_t *src, const int32_t *dst, int n, uint16_t *k_pages,
                     uint16_t *v_pages, int num_pages, int Hkv, int P, int d, int *err,
                     void *stream) {
  NvtxRange nvtx_range("paged_copy_pages");
  if (n < 0 || num_pages < 0 || Hkv <= 0 || P <= 0 || d <= 0) return PA_EINVAL;
  const long long page_halves = (long long)Hkv * P * d;
  if (page_halves % 8 != 0) return PA_EUNSUPPORTED;
  if (n == 0) return PA_OK;
  if (!src || !dst || !k_pages || !v_pages) return PA_EINVAL;
  if (!aligned16(k_pages) || !aligned16(v_pages)) return PA_EALIGN;
  const long long units = page_halves / 8;
  int bx = (int)std::min<long long>((units + 255) / 256, 64);
  dim3 grid(bx, (unsigned)std::min(n, 65535));
  k_copy_pages<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      src, dst, n, reinterpret_cast<uint4 *>(k_pages), reinterpret_cast<uint4 *>(v_pages),
      num_pages, units, err);
  return launch_status(cudaGetLastError());
}

size_t paged_attn_workspace_size(int T, int Hq, int Hkv, int d) {
  if (T < 0 || check_shape(Hq, Hkv, 16, d) != PA_OK) return 0;
  int C = sm_count();
  if (C <= 0) C = 256;  // no device visible: size for the largest plausible SM count
  return ws_layout(T, Hq, Hkv, d, C).total;
}

static int plan_with(const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                     int T, int Hq, int Hkv, int P, int d, void *workspace,
                     size_t workspace_bytes, void *stream, int min_run) {
  int st = check_attn(nullptr, nullptr, nullptr, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv,
                      P, d, 1, nullptr, workspace, workspace_bytes, false);
  if (st != PA_OK) return st;
  if (T == 0) return PA_OK;
  const int C = sm_count();
  WsLayout lay = ws_layout(T, Hq, Hkv, d, C);
  const int G = Hq / Hkv;
  const int NP = G >= 2 ? G / 2 : 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  int blocks = (T + 7) / 8;
  if (blocks > 65535) blocks = 65535;
  k_plan_mark<<<blocks, 256, 0, s>>>(tok_page_table, max_pages, T, ws, lay);
  if (cudaGetLastError() != cudaSuccess) return PA_ELAUNCH;
  k_plan<<<1, 1024, 0, s>>>(tok_page_table, max_pages, tok_kv_len, T, P, Hkv, NP, min_run, C, ws,
                            lay);
  return launch_status(cudaGetLastError());
}

int paged_attn_plan(const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                    int T, int Hq, int Hkv, int P, int d, void *workspace, size_t workspace_bytes,
                    void *stream) {
  NvtxRange nvtx_range("paged_attn_plan");
  return plan_with(tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P, d, workspace,
                   workspace_bytes, stream, g_min_run.load());
}

int paged_attn_plan_decode(const int32_t *tok_page_table, int max_pages,
                           const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                           void *workspace, size_t workspace_bytes, void *stream) {
  NvtxRange nvtx_range("paged_attn_plan_decode");
  return plan_with(tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P, d, workspace,
                   workspace_bytes, stream, INT_MAX);
}

int paged_attn_plan_prefill(const int32_t *tok_page_table, int max_pages,
                            const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                            void *workspace, size_t workspace_bytes, void *stream) {
  NvtxRange nvtx_range("paged_attn_plan_prefill");
  return plan_with(tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P, d, workspace,
                   workspace_bytes, stream, 1);
}

int paged_attn_masked_prefill(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                              const int32_t *tok_page_table, int max_pages,
                              const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                              int num_pages, float scale, const int32_t *cell_seq,
                              const int32_t *cell_pos, const int32_t *tok_seq,
                              const int32_t *tok_pos, uint16_t *out, void *workspace,
                              size_t workspace_bytes, void *stream) {
  NvtxRange nvtx_range("paged_attn_masked_prefill");
  int st = check_attn(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P, d,
                      num_pages, out, workspace, workspace_bytes, true);
  if (st != PA_OK || T == 0) return st;
  if (!cell_seq || !cell_pos || !tok_seq || !tok_pos) return PA_EINVAL;
  AttnArgs a = make_args(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P,
                         d, num_pages, scale, out, workspace);
  a.cell_seq = cell_seq;
  a.cell_pos = cell_pos;
  a.tok_seq = tok_seq;
  a.tok_pos = tok_pos;
  AttnMaps maps;
  st = encode_attn_maps(a, &maps);
  if (st != PA_OK) return st;
  return launch_status(launch_prefill(a, sm_count(), &maps, static_cast<cudaStream_t>(stream)));
}

int paged_attn_masked_decode(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                             const int32_t *tok_page_table, int max_pages,
                             const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                             int num_pages, float scale, const int32_t *cell_seq,
                             const int32_t *cell_pos, const int32_t *tok_seq,
                             const int32_t *tok_pos, uint16_t *out, void *workspace,
                             size_t workspace_bytes, void *stream) {
  NvtxRange nvtx_range("paged_attn_masked_decode");
  int st = check_attn(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P, d,
                      num_pages, out, workspace, workspace_bytes, true);
  if (st != PA_OK || T == 0) return st;
  if (!cell_seq || !cell_pos || !tok_seq || !tok_pos) return PA_EINVAL;
  if (!aligned16(cell_seq) || !aligned16(cell_pos)) return PA_EALIGN;
  AttnArgs a = make_args(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P,
                         d, num_pages, scale, out, workspace);
  a.cell_seq = cell_seq;
  a.cell_pos = cell_pos;
  a.tok_seq = tok_seq;
  a.tok_pos = tok_pos;
  AttnMaps maps;
  st = encode_attn_maps(a, &maps);
  if (st != PA_OK) return st;
  return launch_status(launch_decode(a, sm_count(), &maps, static_cast<cudaStream_t>(stream)));
}

int paged_attn_prefill(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                       const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                       int T, int Hq, int Hkv, int P, int d, int num_pages, float scale,
                       uint16_t *out, void *workspace, size_t workspace_bytes, void *stream) {
  NvtxRange nvtx_range("paged_attn_prefill");
  int st = check_attn(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P, d,
                      num_pages, out, workspace, workspace_bytes, true);
  if (st != PA_OK || T == 0) return st;
  AttnArgs a = make_args(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P,
                         d, num_pages, scale, out, workspace);
  AttnMaps maps;
  st = encode_attn_maps(a, &maps);
  if (st != PA_OK) return st;
  return launch_status(launch_prefill(a, sm_count(), &maps, static_cast<cudaStream_t>(stream)));
}

int paged_attn_decode(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                      const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                      int T, int Hq, int Hkv, int P, int d, int num_pages, float scale,
                      uint16_t *out, void *workspace, size_t workspace_bytes, void *stream) {
  NvtxRange nvtx_range("paged_attn_decode");
  int st = check_attn(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P, d,
                      num_pages, out, workspace, workspace_bytes, true);
  if (st != PA_OK || T == 0) return st;
  AttnArgs a = make_args(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P,
                         d, num_pages, scale, out, workspace);
  AttnMaps maps;
  st = encode_attn_maps(a, &maps);
  if (st != PA_OK) return st;
  return launch_status(launch_decode(a, sm_count(), &maps, static_cast<cudaStream_t>(stream)));
}

int paged_attn_decode_append(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                             const int64_t *slot_mapping, uint16_t *k_pages, uint16_t *v_pages,
                             const int32_t *tok_page_table, int max_pages,
                             const int32_t *tok_kv_len, int T, int Hq, int Hkv, int P, int d,
                             int num_pages, float scale, uint16_t *out, void *workspace,
                             size_t workspace_bytes, void *stream) {
  NvtxRange nvtx_range("paged_attn_decode_append");
  int st = check_attn(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P, d,
                      num_pages, out, workspace, workspace_bytes, true);
  if (st != PA_OK || T == 0) return st;
  if (!k_new || !v_new || !slot_mapping) return PA_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new)) return PA_EALIGN;
  AttnArgs a = make_args(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P,
                         d, num_pages, scale, out, workspace);
  a.k_new = k_new;
  a.v_new = v_new;
  a.slot = slot_mapping;
  AttnMaps maps;
  st = encode_attn_maps(a, &maps);
  if (st != PA_OK) return st;
  return launch_status(launch_decode(a, sm_count(), &maps, static_cast<cudaStream_t>(stream)));
}

int paged_attn_run(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                   const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len, int T,
                   int Hq, int Hkv, int P, int d, int num_pages, float scale, uint16_t *out,
                   void *workspace, size_t workspace_bytes, void *stream) {
  NvtxRange nvtx_range("paged_attn_run");
  int st = paged_attn_prefill(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq,
                              Hkv, P, d, num_pages, scale, out, workspace, workspace_bytes, stream);
  if (st != PA_OK) return st;
  return paged_attn_decode(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv,
                           P, d, num_pages, scale, out, workspace, workspace_bytes, stream);
}

int paged_attn_forward(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                       const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                       int T, int Hq, int Hkv, int P, int d, int num_pages, float scale,
                       uint16_t *out, void *workspace, size_t workspace_bytes, void *stream) {
  NvtxRange nvtx_range("paged_attn_forward");
  int st = check_attn(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P, d,
                      num_pages, out, workspace, workspace_bytes, true);
  if (st != PA_OK || T == 0) return st;
  st = paged_attn_plan(tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P, d, workspace,
                       workspace_bytes, stream);
  if (st != PA_OK) return st;
  return paged_attn_run(q, k_pages, v_pages, tok_page_table, max_pages, tok_kv_len, T, Hq, Hkv, P,
                        d, num_pages, scale, out, workspace, workspace_bytes, stream);
}

int paged_attn_validate(const int32_t *tok_page_table, int max_pages, const int32_t *tok_kv_len,
                        int T, int P, int num_pages, int *err, void *stream) {
  NvtxRange nvtx_range("paged_attn_validate");
  if (T < 0 || max_pages <= 0 || P <= 0 || num_pages < 0) return PA_EINVAL;
  if (T == 0) return PA_OK;
  if (!tok_page_table || !tok_kv_len || !err) return PA_EINVAL;
  int blocks = (T + 7) / 8;
  if (blocks > 65535) blocks = 65535;
  k_validate<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      tok_page_table, max_pages, tok_kv_len, T, P, num_pages, err);
  return launch_status(cudaGetLastError());
}

int paged_attn_read_error(const void *workspace, int *err_host, void *stream) {
  if (!workspace || !err_host) return PA_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PA_ELAUNCH;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ELAUNCH;
  *err_host = v;
  return v == 0 ? PA_OK : PA_EDEVICE;
}

unsigned long long paged_attn_set_decode_wait_limit(unsigned long long ns) {
  if (ns == 0) ns = kWaitLimitNs;
  if (ns < 1000ull) ns = 1000ull;
  return g_decode_wait_ns.exchange(ns);
}

int paged_attn_set_prefill_min_run(int min_run) {
  if (min_run < 1) min_run = 1;
  return g_min_run.exchange(min_run);
}

}  // extern "C"
