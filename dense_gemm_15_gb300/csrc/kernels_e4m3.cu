// Instantiations of the sm_103a GEMM kernels for e4m3 operands.
#include "launch_impl.cuh"

namespace g15 {
template cudaError_t launch_gemm<ELEM_E4M3, 128>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<ELEM_E4M3, 256>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<ELEM_E4M3, 256, 2>(const GemmParams&, int, cudaStream_t);
template int max_pair_clusters<ELEM_E4M3>();

int gemm_smem_bytes(int elem, int bn, int cg) {
    if (cg == 2) return bn == 128 ? Traits<ELEM_F16, 128, 2>::SMEM_BYTES : Traits<ELEM_F16, 256, 2>::SMEM_BYTES;
    if (elem == ELEM_E4M3) return bn == 128 ? Traits<ELEM_E4M3, 128>::SMEM_BYTES : Traits<ELEM_E4M3, 256>::SMEM_BYTES;
    if (bn == 64) return Traits<ELEM_F16, 64>::SMEM_BYTES;
    return bn == 128 ? Traits<ELEM_F16, 128>::SMEM_BYTES : Traits<ELEM_F16, 256>::SMEM_BYTES;
}
int gemm_stages(int elem, int bn, int cg) {
    if (cg == 2) {
        if (elem == ELEM_E4M3) return Traits<ELEM_E4M3, 256, 2>::STAGES;
        return bn == 128 ? Traits<ELEM_F16, 128, 2>::STAGES : Traits<ELEM_F16, 256, 2>::STAGES;
    }
    if (elem == ELEM_E4M3) return bn == 128 ? Traits<ELEM_E4M3, 128>::STAGES : Traits<ELEM_E4M3, 256>::STAGES;
    if (bn == 64) return Traits<ELEM_F16, 64>::STAGES;
    return bn == 128 ? Traits<ELEM_F16, 128>::STAGES : Traits<ELEM_F16, 256>::STAGES;
}
int gemm_max_pair_clusters(int elem) {
    if (elem == ELEM_E4M3) return max_pair_clusters<ELEM_E4M3>();
    if (elem == ELEM_BF16) return max_pair_clusters<ELEM_BF16>();
    return max_pair_clusters<ELEM_F16>();
}
}  // namespace g15
