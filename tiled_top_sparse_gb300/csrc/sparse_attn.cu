// Paged sparse attention (placeholder until the kernel lands).
#include "internal.h"

namespace tts {
cudaError_t launch_sparse_attn(const SparseArgs&, int*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace tts
