// Backward kernels (D preprocessing, main recomputing kernel, dQ finalize).
#include "fa_internal.h"

namespace fa {
size_t backward_smem_bytes(int) { return 0; }
cudaError_t launch_backward(const AttnShape&, const BwdArgs&, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace fa
