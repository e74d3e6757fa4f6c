// Launchers of the device kernels (internal to the library).
#pragma once
#include "common.cuh"

namespace smla {

// CUDA-core decode kernel (decode_cuda_core.cu)
int cuda_core_smem_bytes();
int cuda_core_threads();
int cuda_core_ctas_per_split(int H);
cudaError_t launch_decode_cuda_core(const DecodeParams& p, int grid, cudaStream_t stream);

// Split-K log-sum-exp combine (combine.cu)
cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream);

}  // namespace smla
