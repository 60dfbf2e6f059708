// Attention backward (placeholder until the tcgen05 kernels land).
#include "fa_internal.h"

namespace fa {
cudaError_t launch_backward(const BwdParams &, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace fa
