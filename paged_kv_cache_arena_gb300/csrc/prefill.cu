// Chunked-prefill attention on tcgen05 tensor cores (not yet built: every
// prefill-class call reports cudaErrorNotSupported).
#include "common.cuh"
#include "internal.h"

namespace kshipra {

cudaError_t launch_prefill(const AttnArgs&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                           cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace kshipra
