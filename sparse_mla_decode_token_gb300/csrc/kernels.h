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

// tcgen05 decode kernel, grid schedule (decode_tc_grid.cu): a 2-CTA cluster
// per (token, split) of at most SMLA_TC_MAX_SPLIT_COLS columns (BF16, E4M3
// and the packed forms, the last through BF16 tiles); pair = true
// (H = 64 only): per (token pair, split), grid = 2 ceil(T / 2) S, the two
// tokens' heads in one 128-row MMA tile over the union of their rows.
int tc_grid_smem_bytes(int dtype, bool pair);
int tc_grid_threads();
cudaError_t launch_decode_tc_grid(const DecodeParams& p, int grid, bool pair, cudaStream_t stream);

// tcgen05 decode kernel, balanced schedule (decode_tcgen05.cu): 2-CTA clusters working through
// units of at most SMLA_TC_MAX_SPLIT_COLS index columns of one token, at most
// SMLA_TC_MAX_UNITS per cluster.  clusters == 0: one unit per (token, split)
// (grid = 2 T S); clusters = P > 0: balanced mode, cluster c takes the c-th of
// P equal shares of the T x W columns (grid = 2 P); the pieces of cut tokens
// go through piece_o [P][2][H][512], piece_lse [P][2][2][H] and piece_cnt
// [P][2] (zero at launch), and the last piece of each token merges them.
#define SMLA_TC_MAX_SPLIT_COLS 2304
#define SMLA_TC_MAX_UNITS 16
int tc_smem_bytes(int dtype);
int tc_threads();
cudaError_t launch_decode_tc(const DecodeParams& p, int grid, int clusters, __nv_bfloat16* piece_o, float* piece_lse,
                             uint32_t* piece_cnt, cudaStream_t stream);

// tcgen05 decode kernel for E4M3 rows with head-owned softmax
// (decode_tc_head_owned.cu): a 2-CTA cluster per (token, split), same column limit.
int tc_head_owned_smem_bytes();
int tc_head_owned_threads();
cudaError_t launch_decode_tc_head_owned(const DecodeParams& p, int grid, cudaStream_t stream);

// tcgen05 decode kernel for E4M3 rows with the slot-split pair
// (decode_tc_slot.cu): a 2-CTA cluster per (token, split), same column limit;
// each CTA computes the full logits of its half of every 128-slot tile.
// pair = true (H = 64 only): per (token pair, split) over the union of the two
// tokens' rows, at most SMLA_TC_MAX_SPLIT_COLS / 2 columns of each token per
// split; grid = 2 ceil(T / 2) S.
int tc_slot_smem_bytes();
int tc_slot_threads();
cudaError_t launch_decode_tc_slot(const DecodeParams& p, int grid, bool pair, cudaStream_t stream);

// Split-K log-sum-exp combine (combine.cu)
cudaError_t launch_combine(const DecodeParams& p, cudaStream_t stream);

}  // namespace smla
