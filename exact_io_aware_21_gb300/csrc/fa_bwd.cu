// Backward kernels (placeholder until the tcgen05 backward lands).
#include "fa_kernels.h"

namespace fa {
cudaError_t launch_bwd(const BwdLaunch&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace fa
