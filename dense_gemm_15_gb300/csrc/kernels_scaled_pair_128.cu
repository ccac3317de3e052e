// Instantiations of the block-scaled sm_103a GEMM kernels on SM-pair 256 x 128
// tiles (tcgen05 cta_group::2, two accumulators per CTA): MXFP8 with E4M3 or E5M2
// elements, MXFP4 and NVFP4 with packed E2M1 elements.
#include "launch_impl.cuh"

namespace g15 {
template cudaError_t launch_gemm<ELEM_E4M3, 128, 2, SF_MXF8>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<ELEM_E5M2, 128, 2, SF_MXF8>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<ELEM_E2M1, 128, 2, SF_MXF4>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<ELEM_E2M1, 128, 2, SF_NVF4>(const GemmParams&, int, cudaStream_t);
}  // namespace g15
