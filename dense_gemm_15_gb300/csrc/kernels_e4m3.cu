// Instantiations of the sm_103a GEMM kernels for e4m3 operands.
#include "launch_impl.cuh"

namespace g15 {
template cudaError_t launch_gemm<ELEM_E4M3, 128>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<ELEM_E4M3, 256>(const GemmParams&, int, cudaStream_t);

int gemm_smem_bytes(int elem, int bn) {
    if (elem == ELEM_E4M3) return bn == 128 ? Traits<ELEM_E4M3, 128>::SMEM_BYTES : Traits<ELEM_E4M3, 256>::SMEM_BYTES;
    return bn == 128 ? Traits<ELEM_F16, 128>::SMEM_BYTES : Traits<ELEM_F16, 256>::SMEM_BYTES;
}
int gemm_stages(int elem, int bn) {
    if (elem == ELEM_E4M3) return bn == 128 ? Traits<ELEM_E4M3, 128>::STAGES : Traits<ELEM_E4M3, 256>::STAGES;
    return bn == 128 ? Traits<ELEM_F16, 128>::STAGES : Traits<ELEM_F16, 256>::STAGES;
}
}  // namespace g15
