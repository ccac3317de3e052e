// gemm_run_splitk_noalloc: the split-K GEMM for callers that must not
// allocate device memory.
//
// Who needs this: code that runs inside a host application which owns all
// device memory (an inference server or a plugin handed a fixed memory
// budget, where an outside cudaMalloc either fails or breaks the host's
// accounting), and latency-critical loops where a cudaMalloc / cudaFree is not
// acceptable because it can block and synchronise the whole device.  Plans
// allocate their workspace on demand, so such callers cannot use them for a
// split-K run.  This entry point takes no plan: its partial tiles live in a
// fixed, file-scope device array that every GPU loading the library holds
// until the process exits.
//
// Sharing: every call uses the same array.  Calls that may run at the same
// time on the GPU (different streams, or several host threads) race on it and
// give wrong results; serialise them (one stream, or events).  Partial tiles
// are fully written before they are read, so the array needs no clearing; the
// status word is cleared on the stream at the start of every call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/gemm15.h"
#include "gemm_params.h"
#include "launch.h"

using namespace g15;

namespace {

constexpr size_t STATUS_BYTES = 256;  // the first 256 bytes hold the status word
constexpr size_t SCRATCH_BYTES = GEMM15_NOALLOC_SCRATCH_BYTES;
constexpr int MAX_DEVICES = 64;

}  // namespace

// The scratch: status word, then fp32 partial tiles of the split-K kernel.
static __device__ __align__(256) float g15_noalloc_scratch[SCRATCH_BYTES / sizeof(float)];

namespace {

struct DeviceSetup {
    bool done = false;
    gemm15_status_t status = GEMM15_OK;
    float* scratch = nullptr;  // device address of g15_noalloc_scratch on this device
    int num_sms = 0;
};

std::mutex g_setup_lock;
DeviceSetup g_setup[MAX_DEVICES];

// Resolves the scratch's device address once per device, with that device
// current (the host-side symbol is only a stand-in, not a device address).
gemm15_status_t setup_device(int dev, DeviceSetup** out) {
    if (dev < 0 || dev >= MAX_DEVICES) return GEMM15_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_setup_lock);
    DeviceSetup& s = g_setup[dev];
    if (!s.done) {
        s.done = true;
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
            s.status = GEMM15_ERR_CUDA;
        } else if (prop.major != 10 || prop.minor != 3) {
            s.status = GEMM15_ERR_NO_DEVICE;
        } else {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g15_noalloc_scratch) != cudaSuccess || p == nullptr) {
                cudaGetLastError();
                s.status = GEMM15_ERR_CUDA;
            } else {
                s.scratch = static_cast<float*>(p);
                s.num_sms = prop.multiProcessorCount;
            }
        }
    }
    *out = &s;
    return s.status;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

bool tmap(CUtensorMap* m, int elem, const void* ptr, uint64_t inner, uint64_t outer,
          uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
    auto fn = encoder();
    if (!fn) return false;
    const CUtensorMapDataType t = elem == ELEM_F16    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                  : elem == ELEM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, t, 2, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" gemm15_status_t gemm_run_splitk_noalloc(
    const gemm15_plan_desc_t* desc, const void* A, int64_t lda, const void* B, int64_t ldb,
    const void* C, int64_t ldc, void* D, int64_t ldd, int64_t M, int64_t N, int64_t K,
    float alpha, float beta, const float* scale_a, const float* scale_b, int32_t splits,
    int32_t* status, void* stream) {
    if (!desc) return GEMM15_ERR_INVALID_ARG;
    const gemm15_plan_desc_t& d = *desc;
    int elem, out_elem;
    if (d.acc != GEMM15_F32 || d.a != d.b) return GEMM15_ERR_UNSUPPORTED;
    if (d.a == GEMM15_F16 && d.c == GEMM15_F16 && d.d == GEMM15_F16) {
        elem = out_elem = ELEM_F16;
    } else if (d.a == GEMM15_BF16 && d.c == GEMM15_BF16 && d.d == GEMM15_BF16) {
        elem = out_elem = ELEM_BF16;
    } else if (d.a == GEMM15_E4M3 && d.c == GEMM15_BF16 && d.d == GEMM15_BF16) {
        elem = ELEM_E4M3;
        out_elem = ELEM_BF16;
    } else {
        return GEMM15_ERR_UNSUPPORTED;
    }
    const auto is_layout = [](int l) { return l == GEMM15_ROW_MAJOR || l == GEMM15_COL_MAJOR; };
    if (!is_layout(d.layout_a) || !is_layout(d.layout_b) || !is_layout(d.layout_cd) ||
        (d.epilogue < GEMM15_EPI_LINEAR || d.epilogue > GEMM15_EPI_TANH))
        return GEMM15_ERR_INVALID_ARG;
    if ((scale_a || scale_b) && elem != ELEM_E4M3) return GEMM15_ERR_INVALID_ARG;
    if (splits < 1 || M < 0 || N < 0 || K < 0) return GEMM15_ERR_INVALID_ARG;
    if (M > (1ll << 31) - 256 || N > (1ll << 31) - 256 || K > (1ll << 31) - 256)
        return GEMM15_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM15_OK;

    // every argument check comes before the first device call
    // column-major C/D: compute D^T = B^T . A^T (row-major N x M)
    const bool a_row = d.layout_a == GEMM15_ROW_MAJOR;
    const bool b_row = d.layout_b == GEMM15_ROW_MAJOR;
    int64_t m = M, n = N;
    const void* pa = A;
    const void* pb = B;
    int64_t la = lda, lb = ldb;
    bool a_k = a_row, b_k = !b_row;
    if (d.layout_cd == GEMM15_COL_MAJOR) {
        m = N;
        n = M;
        pa = B;
        la = ldb;
        a_k = !b_row;
        pb = A;
        lb = lda;
        b_k = a_row;
    }
    const int es = elem == ELEM_E4M3 ? 1 : 2;
    const bool has_c = beta != 0.0f;
    if (!D || (has_c && !C) || (K > 0 && (!pa || !pb))) return GEMM15_ERR_INVALID_ARG;
    if (ldd < n || (has_c && ldc < n)) return GEMM15_ERR_INVALID_ARG;
    if (!aligned(D) || (ldd * 2) % 16 || (has_c && (!aligned(C) || (ldc * 2) % 16)))
        return GEMM15_ERR_ALIGNMENT;
    if (K > 0) {
        if (la < (a_k ? K : m) || lb < (b_k ? K : n)) return GEMM15_ERR_INVALID_ARG;
        if (!aligned(pa) || !aligned(pb) || (la * es) % 16 || (lb * es) % 16)
            return GEMM15_ERR_ALIGNMENT;
    }

    const int bn = n <= 128 ? 128 : 256;
    const int bk = 128 / es;
    const int64_t m_blocks = (m + TILE_M - 1) / TILE_M;
    const int64_t n_blocks = (n + bn - 1) / bn;
    const int64_t tiles = m_blocks * n_blocks;
    const int64_t k_blocks = (K + bk - 1) / bk;
    const int64_t sp = K > 0 ? std::min<int64_t>(splits, k_blocks) : 0;
    const size_t need = STATUS_BYTES + static_cast<size_t>(tiles) * sp * TILE_M * bn * sizeof(float);
    if (need > SCRATCH_BYTES) return GEMM15_ERR_UNSUPPORTED;  // beyond the fixed scratch

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM15_ERR_CUDA;
    DeviceSetup* ds = nullptr;
    gemm15_status_t st = setup_device(dev, &ds);
    if (st != GEMM15_OK) return st;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* dev_status = status ? status : reinterpret_cast<int32_t*>(ds->scratch);
    if (cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s) != cudaSuccess) return GEMM15_ERR_CUDA;
    float* partials = ds->scratch + STATUS_BYTES / sizeof(float);
    const int act = static_cast<int>(d.epilogue);

    if (K > 0) {
        GemmParams gp;
        std::memset(&gp, 0, sizeof(gp));
        const uint32_t w = 128 / es;
        bool ok = a_k ? tmap(&gp.tmA, elem, pa, K, m, la * es, bk, TILE_M)
                      : tmap(&gp.tmA, elem, pa, m, K, la * es, w, bk);
        ok = ok && (b_k ? tmap(&gp.tmB, elem, pb, K, n, lb * es, bk, bn)
                        : tmap(&gp.tmB, elem, pb, n, K, lb * es, w, bk));
        ok = ok && tmap(&gp.tmD, out_elem, D, n, m, ldd * 2, EPI_COLS, 32);
        if (!ok) return GEMM15_ERR_CUDA;
        gp.D = D;
        gp.ldd = ldd;
        gp.C = nullptr;  // split-K parts never read C; the reduction does
        gp.ldc = 0;
        gp.M = static_cast<int32_t>(m);
        gp.N = static_cast<int32_t>(n);
        gp.K = static_cast<int32_t>(K);
        gp.k_blocks = static_cast<int32_t>(k_blocks);
        gp.m_blocks = static_cast<int32_t>(m_blocks);
        gp.n_blocks = static_cast<int32_t>(n_blocks);
        gp.tiles = static_cast<int32_t>(tiles);
        gp.raster = static_cast<int32_t>(std::min<int64_t>(m_blocks, 16));
        gp.sched = SCHED_SPLIT;
        gp.splits = static_cast<int32_t>(sp);
        gp.has_c = 0;  // the reduction reads C
        gp.alpha = alpha;
        gp.beta = beta;
        gp.act = act;
        // shared-memory operand layouts (128-byte swizzle) and the MMA descriptor
        const uint32_t mn_box = static_cast<uint32_t>(128 * bk);
        const uint32_t umma_k = 32 / es;
        gp.a_kmajor = a_k;
        gp.b_kmajor = b_k;
        gp.a_lbo = a_k ? 16u : mn_box;
        gp.a_sbo = 1024u;
        gp.a_kstep = a_k ? 32u : umma_k * 128;
        gp.b_lbo = b_k ? 16u : mn_box;
        gp.b_sbo = 1024u;
        gp.b_kstep = b_k ? 32u : umma_k * 128;
        const uint32_t fmt = elem == ELEM_BF16 ? 1u : 0u;
        gp.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((a_k ? 0u : 1u) << 15) |
                   ((b_k ? 0u : 1u) << 16) | (static_cast<uint32_t>(bn >> 3) << 17) |
                   (static_cast<uint32_t>(TILE_M >> 4) << 24);
        gp.ws = partials;
        gp.flags = nullptr;  // split-K never waits on other CTAs
        gp.status = dev_status;
        gp.epoch = 1;
        gp.timeout_ns = 2000000000ull;
        gp.fault_skip_flag = -1;
        const int grid = static_cast<int>(std::min<int64_t>(ds->num_sms, tiles * sp));
        set_sched_divisors(gp, grid);
        cudaError_t e;
        if (elem == ELEM_F16)
            e = bn == 128 ? launch_gemm<ELEM_F16, 128>(gp, grid, s) : launch_gemm<ELEM_F16, 256>(gp, grid, s);
        else if (elem == ELEM_BF16)
            e = bn == 128 ? launch_gemm<ELEM_BF16, 128>(gp, grid, s) : launch_gemm<ELEM_BF16, 256>(gp, grid, s);
        else
            e = bn == 128 ? launch_gemm<ELEM_E4M3, 128>(gp, grid, s) : launch_gemm<ELEM_E4M3, 256>(gp, grid, s);
        if (e != cudaSuccess) return GEMM15_ERR_CUDA;
    }
    ReduceParams rp{};
    rp.ws = partials;
    rp.splits = static_cast<int32_t>(sp);
    rp.tile_n = bn;
    rp.n_blocks = static_cast<int32_t>(n_blocks);
    rp.M = static_cast<int32_t>(m);
    rp.N = static_cast<int32_t>(n);
    rp.C = C;
    rp.ldc = ldc;
    rp.D = D;
    rp.ldd = ldd;
    rp.alpha = alpha;
    rp.beta = beta;
    rp.scale_a = scale_a;
    rp.scale_b = scale_b;
    rp.act = act;
    rp.has_c = has_c;
    int rgrid = 1, groups = 1;
    reduce_shape(rp, ds->num_sms, &rgrid, &groups);
    const cudaError_t e = out_elem == ELEM_F16 ? launch_reduce<ELEM_F16>(rp, rgrid, groups, s)
                                               : launch_reduce<ELEM_BF16>(rp, rgrid, groups, s);
    return e == cudaSuccess ? GEMM15_OK : GEMM15_ERR_CUDA;
}
