// Instantiations of the block-scaled sm_103a GEMM kernels on one-SM 128 x 256
// tiles with one accumulator (MXFP8 with E4M3 or E5M2 elements, MXFP4 and NVFP4
// with packed E2M1 elements), and the pipeline depth of every block-scaled form.
#include "launch_impl.cuh"

namespace g15 {
template cudaError_t launch_gemm<ELEM_E4M3, 256, 1, SF_MXF8>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<ELEM_E5M2, 256, 1, SF_MXF8>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<ELEM_E2M1, 256, 1, SF_MXF4>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_gemm<ELEM_E2M1, 256, 1, SF_NVF4>(const GemmParams&, int, cudaStream_t);

int gemm_scaled_stages(int sf, int bn, int cg) {
    if (cg == 2 && bn == 128) {
        switch (sf) {
            case SF_MXF8: return Traits<ELEM_E4M3, 128, 2, SF_MXF8>::STAGES;
            case SF_MXF4: return Traits<ELEM_E2M1, 128, 2, SF_MXF4>::STAGES;
            default: return Traits<ELEM_E2M1, 128, 2, SF_NVF4>::STAGES;
        }
    }
    if (cg == 2) {
        switch (sf) {
            case SF_MXF8: return Traits<ELEM_E4M3, 256, 2, SF_MXF8>::STAGES;
            case SF_MXF4: return Traits<ELEM_E2M1, 256, 2, SF_MXF4>::STAGES;
            default: return Traits<ELEM_E2M1, 256, 2, SF_NVF4>::STAGES;
        }
    }
    if (bn == 128) {
        switch (sf) {
            case SF_MXF8: return Traits<ELEM_E4M3, 128, 1, SF_MXF8>::STAGES;
            case SF_MXF4: return Traits<ELEM_E2M1, 128, 1, SF_MXF4>::STAGES;
            default: return Traits<ELEM_E2M1, 128, 1, SF_NVF4>::STAGES;
        }
    }
    switch (sf) {
        case SF_MXF8: return Traits<ELEM_E4M3, 256, 1, SF_MXF8>::STAGES;
        case SF_MXF4: return Traits<ELEM_E2M1, 256, 1, SF_MXF4>::STAGES;
        default: return Traits<ELEM_E2M1, 256, 1, SF_NVF4>::STAGES;
    }
}
}  // namespace g15
