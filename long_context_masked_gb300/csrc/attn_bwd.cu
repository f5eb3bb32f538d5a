// Backward pass of mask-aware exact softmax attention on sm_103a (placeholder until
// the dK/dV and dQ kernels land).
#include <cuda_runtime.h>

#include "attn_kernels.h"
#include "lca_device.cuh"

namespace lca {

cudaError_t launch_bwd_preprocess(const BwdArgs&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_bwd_dkdv(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                            const CUtensorMap&, const BwdArgs&, int, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t launch_bwd_dq(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                          const CUtensorMap&, const BwdArgs&, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace lca
