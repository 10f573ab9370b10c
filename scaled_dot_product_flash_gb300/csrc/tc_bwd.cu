// Tensor-core backward (dQ and dK/dV kernels): not built yet; the tiled backward of
// fp16/bf16 inputs runs on the CUDA-core kernels meanwhile.
#include "launch.h"

namespace sdpa {

bool tensor_bwd_supported(const Problem&, int) { return false; }
cudaError_t launch_tc_dq(const Problem&, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_dkdv(const Problem&, int, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace sdpa
