// Prefill attention on tcgen05 tensor cores (sm_103a).  Placeholder until the
// tensor-core kernel lands: flags any planned tile as unsupported.
#include "tmap.cuh"

namespace pa {

__global__ void k_prefill_stub(AttnArgs a) {
  WsHeader *hdr = reinterpret_cast<WsHeader *>(a.ws);
  if (hdr->n_tiles > 0 && threadIdx.x == 0) atomicOr(&hdr->err, PA_ERR_TIMEOUT);
}

cudaError_t launch_prefill(const AttnArgs &a, int num_sms, const void *tmaps, cudaStream_t s) {
  (void)num_sms;
  (void)tmaps;
  k_prefill_stub<<<1, 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace pa
