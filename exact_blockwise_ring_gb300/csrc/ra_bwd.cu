// ra_bwd.cu -- backward kernel (placeholder until the tensor-core kernel lands).
#include "ra_internal.h"

namespace ra {
cudaError_t launch_bwd(const BwdArgs&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                       const CUtensorMap&, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace ra
