// Tensor-core append / prefill attention (tcgen05 + TMEM) — under construction.
#include "pka_internal.h"

namespace pka {

cudaError_t launch_prefill(const AttnArgs&, int, int, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace pka
