// Paged extend (suffix prefill) -- placeholder until the tcgen05 kernel lands.
#include "internal.h"

namespace pkv {

bool extend_supported(int, int, int, int) { return false; }

cudaError_t launch_extend(const CUtensorMap&, const CUtensorMap&, const ExtendParams&, int, int,
                          int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace pkv
