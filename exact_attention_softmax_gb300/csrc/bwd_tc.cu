// bwd_tc.cu -- placeholder until the tensor-core backward lands.
#include "common.cuh"

namespace sdpa {
cudaError_t launch_bwd_tc(const BwdProblem&, int, const BwdMaps&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace sdpa
