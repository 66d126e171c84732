// TMA tensor maps of the attention kernels (host-side encoding through the
// driver entry point, so the library needs no link-time libcuda).
#pragma once

#include <cuda.h>

#include "kernels.cuh"

namespace pa {

struct AttnMaps {
  CUtensorMap q;  // 3-D {d, Hq, T}, box {64, 1, 128}, 128-byte swizzle
  CUtensorMap k;  // 2-D {d, num_pages * Hkv * P}, box {64, P}, 128-byte swizzle
  CUtensorMap v;
};

int encode_attn_maps(const AttnArgs &a, AttnMaps *m);
// FP8 pages (page size 128, d 128): K {d bytes, rows}, V transposed {P bytes, rows},
// both in 128 x 128-byte boxes with 128-byte swizzle; q as above.
int encode_attn_maps_fp8(const AttnArgs &a, AttnMaps *m);

}  // namespace pa
