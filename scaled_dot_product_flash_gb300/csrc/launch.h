// Internal launchers (not part of the C ABI).  Each enqueues exactly one kernel on the
// given stream and returns the CUDA error of that launch.
#pragma once

#include "common.cuh"

namespace sdpa {

// CUDA-core tiled path: every dtype, D in {32, 64, 96, 128, 256}.
cudaError_t launch_simt_fwd(const Problem& p, int dtype, cudaStream_t s);
cudaError_t launch_simt_dq(const Problem& p, int dtype, cudaStream_t s);
cudaError_t launch_simt_dkdv(const Problem& p, int dtype, cudaStream_t s);

// δ = rowsum(dO ∘ O) pre-pass, every dtype and D.
cudaError_t launch_delta(const Problem& p, int dtype, cudaStream_t s);

// Sink-logit gradients from lse and δ (any dtype: both are fp32).
cudaError_t launch_sink_grad(const Problem& p, cudaStream_t s);

// Short-query path (Lq <= 8, G·Lq <= 32): thread-block clusters split Lkv.
bool vector_supported(const Problem& p, int dtype);
cudaError_t launch_vector_fwd(const Problem& p, int dtype, cudaStream_t s);
cudaError_t launch_vector_bwd(const Problem& p, int dtype, cudaStream_t s);
// Its warp-level-MMA kernels for fp16/bf16 with D in {64, 128}.
bool vector_mma_supported(const Problem& p, int dtype);
cudaError_t launch_vector_mma_fwd(const Problem& p, int dtype, cudaStream_t s);
cudaError_t launch_vector_mma_bwd(const Problem& p, int dtype, cudaStream_t s);

// Tensor-core path (TMA + tcgen05), fp16/bf16: forward with D in {32, 64, 96, 128, 256},
// backward with D in {32, 64, 96, 128} (tc_bwd.cu) and 256 (tc_bwd256.cu).
bool tensor_supported(const Problem& p, int dtype);
bool tensor_bwd_supported(const Problem& p, int dtype);
bool tensor_bwd256_supported(const Problem& p, int dtype);
cudaError_t launch_tc_fwd(const Problem& p, int dtype, cudaStream_t s);
cudaError_t launch_tc_dq(const Problem& p, int dtype, cudaStream_t s);
cudaError_t launch_tc_dkdv(const Problem& p, int dtype, cudaStream_t s);
cudaError_t launch_tc_dq256(const Problem& p, int dtype, cudaStream_t s);
cudaError_t launch_tc_dkdv256(const Problem& p, int dtype, cudaStream_t s);

}  // namespace sdpa
