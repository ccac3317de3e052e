// Definitions of the launch helpers, included by each instantiation unit.
#pragma once

#include "gemm_kernel.cuh"
#include "launch.h"

namespace g15 {

template <int ELEM, int BN, int CG, int SF>
cudaError_t launch_gemm(const GemmParams& p, int grid, cudaStream_t stream) {
    using TR = Traits<ELEM, BN, CG, SF>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        err = cudaFuncSetAttribute(gemm_tc_kernel<ELEM, BN, CG, SF>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, TR::SMEM_BYTES);
        if (err != cudaSuccess) return err;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    // A programmatic dependent launch: when the kernel before it in the stream
    // triggers (every GEMM kernel does at entry), this grid's CTAs may start
    // as SMs free up, run their set-up, and wait (griddepcontrol.wait) before
    // touching global memory until that kernel has completed.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = TR::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = CG;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CG == 2 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<ELEM, BN, CG, SF>, p);
}

template <int ELEM>
int max_pair_clusters() {
    using TR = Traits<ELEM, 256, 2>;
    if (cudaFuncSetAttribute(gemm_tc_kernel<ELEM, 256, 2, SF_NONE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TR::SMEM_BYTES) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = TR::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<ELEM, 256, 2, SF_NONE>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <int ELEM>
cudaError_t launch_reduce(const ReduceParams& p, int grid, int groups, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(32 * groups), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    // programmatic dependent launch: scheduled while the GEMM kernel before it
    // runs, the kernel itself waits for that grid (griddepcontrol.wait)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<ELEM>, p);
}

}  // namespace g15
