// mla_prefill_sm103a.cu -- ragged causal MLA prefill with a cached-prefix offset (sm_103a).
#include "mla_internal.h"
#include "sm103a_ptx.cuh"

namespace mla {
cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, cudaStream_t stream) {
  (void)p; (void)tm_q; (void)tm_k; (void)tm_v; (void)stream;
  return cudaErrorNotSupported;
}
}  // namespace mla
