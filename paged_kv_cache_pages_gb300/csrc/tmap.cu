// Tensor-map encoding for the prefill kernel.
#include <cudaTypedefs.h>
#include <mutex>

#include "tmap.cuh"

namespace pa {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

int encode_attn_maps(const AttnArgs &a, AttnMaps *m) {
  auto enc = get_encode();
  if (!enc) return PA_ELAUNCH;
  const cuuint32_t estr[3] = {1, 1, 1};
  {
    cuuint64_t dims[3] = {(cuuint64_t)a.D, (cuuint64_t)a.Hq, (cuuint64_t)a.T};
    cuuint64_t strides[2] = {(cuuint64_t)a.D * 2, (cuuint64_t)a.Hq * a.D * 2};
    cuuint32_t box[3] = {64, 1, 128};
    CUresult r = enc(&m->q, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<uint16_t *>(a.q), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return PA_ELAUNCH;
  }
  const uint16_t *src[2] = {a.k_pages, a.v_pages};
  CUtensorMap *dst[2] = {&m->k, &m->v};
  for (int i = 0; i < 2; ++i) {
    cuuint64_t dims[2] = {(cuuint64_t)a.D, (cuuint64_t)a.num_pages * a.Hkv * a.P};
    cuuint64_t strides[1] = {(cuuint64_t)a.D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)a.P};
    CUresult r = enc(dst[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(src[i]),
                     dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return PA_ELAUNCH;
  }
  return PA_OK;
}

int encode_attn_maps_fp8(const AttnArgs &a, AttnMaps *m) {
  auto enc = get_encode();
  if (!enc) return PA_ELAUNCH;
  const cuuint32_t estr[3] = {1, 1, 1};
  {
    cuuint64_t dims[3] = {(cuuint64_t)a.D, (cuuint64_t)a.Hq, (cuuint64_t)a.T};
    cuuint64_t strides[2] = {(cuuint64_t)a.D * 2, (cuuint64_t)a.Hq * a.D * 2};
    cuuint32_t box[3] = {64, 1, 128};
    CUresult r = enc(&m->q, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<uint16_t *>(a.q), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return PA_ELAUNCH;
  }
  // K codes: rows of d bytes, one per cached token; V codes: rows of P bytes, one per
  // (page, head, dim).  Both read as 128 x 128-byte boxes.
  {
    cuuint64_t dims[2] = {(cuuint64_t)a.D, (cuuint64_t)a.num_pages * a.Hkv * a.P};
    cuuint64_t strides[1] = {(cuuint64_t)a.D};
    cuuint32_t box[2] = {128, 128};
    CUresult r = enc(&m->k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint16_t *>(a.k_pages),
                     dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return PA_ELAUNCH;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)a.P, (cuuint64_t)a.num_pages * a.Hkv * a.D};
    cuuint64_t strides[1] = {(cuuint64_t)a.P};
    cuuint32_t box[2] = {128, 128};
    CUresult r = enc(&m->v, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint16_t *>(a.v_pages),
                     dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return PA_ELAUNCH;
  }
  return PA_OK;
}

}  // namespace pa
