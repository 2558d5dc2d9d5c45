// Prompt-chunk attention (tcgen05/TMEM); the kernel is not built yet.
#include "params.h"

namespace tfpa {
cudaError_t launch_prefill(const PrefillParams&, bool, int, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace tfpa
