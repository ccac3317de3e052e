// Definitions of the launch helpers, included by each instantiation unit.
#pragma once

#include "gemm_kernel.cuh"
#include "launch.h"

namespace g15 {

template <int ELEM, int BN>
cudaError_t launch_gemm(const GemmParams& p, int grid, cudaStream_t stream) {
    using TR = Traits<ELEM, BN>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        err = cudaFuncSetAttribute(gemm_tc_kernel<ELEM, BN>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, TR::SMEM_BYTES);
        if (err != cudaSuccess) return err;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    gemm_tc_kernel<ELEM, BN><<<grid, NUM_THREADS, TR::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

template <int ELEM>
cudaError_t launch_reduce(const ReduceParams& p, int grid, cudaStream_t stream) {
    splitk_reduce_kernel<ELEM><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace g15
