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
void reduce_shape(const ReduceParams& p, int num_sms, int* grid, int* groups) {
    // split groups: one warp per partial up to REDUCE_MAX_GROUPS (balanced
    // split-K: a tile's holders vary, four groups)
    int g = p.units > 0 ? 4 : (p.splits > 0 ? p.splits : 1);
    g = g < 1 ? 1 : (g > REDUCE_MAX_GROUPS ? REDUCE_MAX_GROUPS : g);
    const int64_t elems = static_cast<int64_t>(p.M) * ((p.N + REDUCE_COLS - 1) / REDUCE_COLS);
    const int64_t batches = (elems + 31) / 32;
    const int64_t cap = static_cast<int64_t>(num_sms) * (64 / g);  // 64 warps per SM
    const int64_t b = batches < cap ? batches : cap;
    *grid = static_cast<int>(b < 1 ? 1 : b);
    *groups = g;
}

int gemm_max_pair_clusters(int elem) {
    if (elem == ELEM_E4M3) return max_pair_clusters<ELEM_E4M3>();
    if (elem == ELEM_BF16) return max_pair_clusters<ELEM_BF16>();
    return max_pair_clusters<ELEM_F16>();
}
}  // namespace g15
