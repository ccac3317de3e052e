// Host-side launch entry points of the sm_103a kernels (one translation unit
// per element type instantiates them).
#pragma once

#include <cuda_runtime.h>

#include "gemm_params.h"

namespace g15 {

// Persistent tcgen05 GEMM: one-SM tiles of 128 x BN (CG = 1, BN = 64, 128 or
// 256) or SM-pair tiles of 256 x BN (CG = 2, clusters of two CTAs; grid even);
// SF selects a block-scaled MMA kind (one-SM tiles of BN = 128 or 256, or
// SM-pair 256 x 256 tiles).
template <int ELEM, int BN, int CG = 1, int SF = SF_NONE>
cudaError_t launch_gemm(const GemmParams& p, int grid, cudaStream_t stream);

// Largest number of SM-pair clusters of the CG = 2 kernel resident at once
// (0 if the query fails).
int gemm_max_pair_clusters(int elem);

// Split-K reduction / K == 0 epilogue (ELEM selects the 16-bit C/D type):
// `grid` blocks of `groups` warps (1..REDUCE_MAX_GROUPS).
template <int ELEM>
cudaError_t launch_reduce(const ReduceParams& p, int grid, int groups, cudaStream_t stream);

// Grid and warps per block of the reduction for its parameters.
void reduce_shape(const ReduceParams& p, int num_sms, int* grid, int* groups);

// Pipeline depth of the block-scaled kernel of a scale kind, tile width and
// CTA group.
int gemm_scaled_stages(int sf, int bn, int cg);

// Shared-memory bytes and pipeline depth of a GEMM instantiation.
int gemm_smem_bytes(int elem, int bn, int cg);
int gemm_stages(int elem, int bn, int cg);

}  // namespace g15
