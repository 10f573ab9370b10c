// Tensor-core path (TMA + tcgen05): not built yet; every call reports "unsupported".
#include "launch.h"

namespace sdpa {

bool tensor_supported(const Problem&, int) { return false; }

cudaError_t launch_tc_fwd(const Problem&, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_dq(const Problem&, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_tc_dkdv(const Problem&, int, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace sdpa
