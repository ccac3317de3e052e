// Instantiations of the sm_103a GEMM kernels for bf16 operands.
#include "launch_impl.cuh"

namespace g15 {
template cudaError_t launch_gemm<ELEM_BF16, 64>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<ELEM_BF16, 128>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<ELEM_BF16, 256>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<ELEM_BF16, 256, 2>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<ELEM_BF16, 128, 2>(const GemmParams&, int, cudaStream_t);
template int max_pair_clusters<ELEM_BF16>();
template cudaError_t launch_reduce<ELEM_BF16>(const ReduceParams&, int, int, cudaStream_t);
}  // namespace g15
