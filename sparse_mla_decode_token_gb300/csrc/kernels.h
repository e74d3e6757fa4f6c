// Launchers of the device kernels (internal to the library).
#pragma once
#include "common.cuh"

namespace smla {

// CUDA-core decode kernel (decode_cuda_core.cu)
int cuda_core_smem_bytes();
int cuda_core_threads();
int cuda_core_ctas_per_split(int H);
cudaError_t launch_decode_cuda_core(const DecodeParams& p, int grid, cudaStream_t stream);

// Sets the text smla_last_error() returns on this thread; returns st (smla_api.cu).
smla_status record_error(smla_status st, const char* msg);

// tcgen05 decode kernel (decode_tcgen05.cu): a 2-CTA cluster per (token, split);
// each CTA stages at most SMLA_TC_MAX_SPLIT_COLS index columns of its split.
#define SMLA_TC_MAX_SPLIT_COLS 2304
int tc_smem_bytes(int dtype);
int tc_threads();
cudaError_t launch_decode_tc(const DecodeParams& p, int grid, cudaStream_t stream);

// tcgen05 decode kernel for E4M3 rows with head-owned softmax
// (decode_tc_head_owned.cu): a 2-CTA cluster per (token, split), same column limit.
int tc_head_owned_smem_bytes();
int tc_head_owned_threads();
cudaError_t launch_decode_tc_head_owned(const DecodeParams& p, int grid, cudaStream_t stream);

// Split-K log-sum-exp combine (combine.cu)
cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream);

}  // namespace smla
