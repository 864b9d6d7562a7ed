// prefill.cu -- causal grouped-query prefill (placeholder until the tcgen05 kernel lands).
#include "common.cuh"
#include "internal.h"

namespace gqa {
cudaError_t launch_prefill_causal(const PrefillParams&, const CUtensorMap&, const CUtensorMap&,
                                  const CUtensorMap&, int, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace gqa
