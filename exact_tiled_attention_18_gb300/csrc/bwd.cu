// Backward kernels (placeholder until the tcgen05 backward lands).
#include <cuda_runtime.h>

#include "internal.h"

namespace fa {

cudaError_t launch_bwd(const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace fa
