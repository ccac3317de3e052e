// C-ABI of gemm15: plans, validation, the host planner (tile shape, schedule,
// grid, workspace), tensor-map encoding and kernel launches.  See
// include/gemm15.h for the contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <map>
#include <tuple>
#include <vector>

#include "../../include/gemm15.h"
#include "gemm_params.h"
#include "launch.h"

using namespace g15;

namespace {

constexpr uint32_t PLAN_MAGIC = 0x67313570u;  // "g15p"
constexpr uint32_t PLAN_DEAD = 0xdeadbeefu;

struct Options {
    int schedule = 0;
    int splits = 0;
    int cta_group = 0;
    int tile_n = 0;
    int raster = 0;
    int grid = 0;
    int64_t timeout_us = 2000000;  // 2 s
    int fault_skip_flag = -1;
    int sk_dp_waves = -1;
    int trace_items = 0;
    int swap_ab = 0;  // 0 automatic, 1 never, 2 always (dense problems)
    int splitk_inline = 0;  // split-K reduced by the last split: 0 automatic, 1 never, 2 always
    int l2_hints = 0;       // operand L2 policies: 0 none, 1 A evict-last, 2 and B evict-first
};

// Kernel choice fixed by gemm_plan_autotune for one problem shape.
struct Tuned {
    int schedule, cta_group, tile_n, sk_dp_waves, splits, swap_ab;
};

}  // namespace

struct gemm15_plan {
    uint32_t magic = PLAN_MAGIC;
    gemm15_plan_desc_t desc{};
    int device = 0;
    int num_sms = 0;
    int elem = ELEM_F16;       // operand kind
    int out_elem = ELEM_F16;   // C/D 16-bit kind
    int32_t* d_status = nullptr;
    uint32_t* d_flags = nullptr;
    int flags_cap = 0;
    float* d_ws = nullptr;
    size_t ws_cap = 0;
    GroupEntry* d_groups = nullptr;
    GroupEntry* h_groups = nullptr;  // pinned staging
    int groups_cap = 0;
    cudaEvent_t groups_done = nullptr;
    // the problems the device table currently describes (a call with the same
    // problems, C use and tile width reuses it without encoding or copying)
    std::vector<gemm15_problem_t> groups_key;
    bool groups_key_c = false;
    int groups_key_bn = 0;
    int groups_key_raster = 0;
    int groups_key_cg = 0;
    int32_t groups_tiles = 0;
    int groups_ng = 0;
    void* d_host_path[3] = {nullptr, nullptr, nullptr};  // A, B, C|D for gemm_run_host
    size_t host_path_cap[3] = {0, 0, 0};
    float* d_scales = nullptr;  // two floats for gemm_run_host
    uint32_t epoch = 0;
    int pair_clusters = -1;  // resident SM-pair clusters (queried on first use)
    uint64_t* d_trace = nullptr;  // timeline of the last traced launch
    size_t trace_cap = 0;         // bytes
    int trace_ctas = 0;
    Options opt;
    gemm15_config_t last{};
    // autotuned choices per computed problem shape (M, N, K after normalisation)
    std::map<std::tuple<int64_t, int64_t, int64_t>, Tuned> tuned;
    uint64_t tuned_gen = 0;  // bumped whenever `tuned` changes
    // ordering of calls across streams: the plan's device state (workspace,
    // flags, status, grouped table, host-path buffers) is used by every call,
    // so a call on another stream than the previous one first waits for the
    // work the previous call enqueued (recorded in done_ev)
    cudaEvent_t done_ev = nullptr;
    cudaStream_t last_stream = nullptr;
    bool has_last = false;
    // gemm_run_host: a second stream for the B copy, with fork / join events;
    // for the column-chunked pipeline a stream for the D downloads and events
    // per chunk (B chunk uploaded, D chunk computed)
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
    cudaStream_t d2h_stream = nullptr;
    cudaEvent_t a_ev = nullptr, d2h_ev = nullptr;
    cudaEvent_t up_ev[8] = {}, done_evs[8] = {};
    // launch parameters of recent dense problems (see LaunchCache)
    void* cache = nullptr;
};

namespace {

// ------------------------------------------------------------------ helpers

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool plan_ok(const gemm15_plan* p) { return p != nullptr && p->magic == PLAN_MAGIC; }

// Orders this call after the previous call of the plan when the two use
// different streams (same stream: stream order already does it).
gemm15_status_t order_after_previous(gemm15_plan* plan, cudaStream_t s) {
    if (plan->has_last && plan->last_stream != s) {
        if (cudaStreamWaitEvent(s, plan->done_ev, 0) != cudaSuccess) return GEMM15_ERR_CUDA;
    }
    return GEMM15_OK;
}

// Records the end of this call's work on `s` for the next call's ordering.
gemm15_status_t mark_done(gemm15_plan* plan, cudaStream_t s) {
    if (cudaEventRecord(plan->done_ev, s) != cudaSuccess) return GEMM15_ERR_CUDA;
    plan->last_stream = s;
    plan->has_last = true;
    return GEMM15_OK;
}

int esize_of(gemm15_dtype_t t) {
    switch (t) {
        case GEMM15_F16:
        case GEMM15_BF16: return 2;
        case GEMM15_F32: return 4;
        case GEMM15_E4M3: return 1;
    }
    return 0;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

CUtensorMapDataType tmap_type(int elem16_or_8) {
    switch (elem16_or_8) {
        case ELEM_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        case ELEM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        default: return CU_TENSOR_MAP_DATA_TYPE_UINT8;  // fp8 bytes
    }
}

// 2-D tiled tensor map with 128-byte swizzle (or none) and zero fill out of bounds.
bool make_tmap(CUtensorMap* map, int elem, const void* ptr, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle = true) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, tmap_type(elem), 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// One problem after layout normalisation: D is row-major M x N.
struct Prob {
    int64_t M, N, K;
    const void* A;
    int64_t lda;
    bool a_kmajor;  // row-major A (K contiguous)
    const void* B;
    int64_t ldb;
    bool b_kmajor;  // column-major B (K contiguous)
    const void* C;
    int64_t ldc;
    void* D;
    int64_t ldd;
    const void* bias = nullptr;  // per output column of the user's D, or null
    bool bias_rows = false;      // the bias runs along the computed rows (D^T)
    const void* aux = nullptr;   // auxiliary tensor Z (layout of C / D), or null
    int64_t ldaux = 0;
    int aux_op = 0;
    void* pre = nullptr;         // pre-activation output Y (layout of D), or null
    int64_t ldpre = 0;
    bool out_trans = false;      // computed (r, c) is stored at C / D / Z / Y + c * ld + r
};

// Column-major C/D: compute D^T = B^T . A^T, which is row-major N x M.
Prob normalise(const gemm15_plan* plan, int64_t M, int64_t N, int64_t K, const void* A,
               int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc, void* D,
               int64_t ldd) {
    const bool a_row = plan->desc.layout_a == GEMM15_ROW_MAJOR;
    const bool b_row = plan->desc.layout_b == GEMM15_ROW_MAJOR;
    Prob p{};
    if (plan->desc.layout_cd == GEMM15_ROW_MAJOR) {
        p = Prob{M, N, K, A, lda, a_row, B, ldb, !b_row, C, ldc, D, ldd};
    } else {
        // A' = B^T (N x K): K contiguous iff B is column-major.
        // B' = A^T (K x M): K contiguous iff A is row-major.
        p = Prob{N, M, K, B, ldb, !b_row, A, lda, a_row, C, ldc, D, ldd};
        p.bias_rows = true;  // the user's columns are the computed rows
    }
    return p;
}

// Swap-AB: the same product computed as its transpose, D^T = B^T . A^T, so
// that a short M becomes the narrow N side of the MMA and the long N side
// fills its 128 rows; the tile is then stored transposed.
Prob swapped(const Prob& p) {
    Prob q = p;
    q.M = p.N;
    q.N = p.M;
    q.A = p.B;
    q.lda = p.ldb;
    q.a_kmajor = p.b_kmajor;
    q.B = p.A;
    q.ldb = p.lda;
    q.b_kmajor = p.a_kmajor;
    q.bias_rows = !p.bias_rows;
    q.out_trans = !p.out_trans;
    return q;
}

gemm15_status_t check_operands(const gemm15_plan* plan, const Prob& p, float beta) {
    const int es = esize_of(plan->desc.a);
    const int eo = esize_of(plan->desc.d);
    if (p.M < 0 || p.N < 0 || p.K < 0) return GEMM15_ERR_INVALID_ARG;
    if (p.M > (1ll << 31) - 256 || p.N > (1ll << 31) - 256 || p.K > (1ll << 31) - 256)
        return GEMM15_ERR_INVALID_ARG;
    if (p.M == 0 || p.N == 0) return GEMM15_OK;
    if (!p.D) return GEMM15_ERR_INVALID_ARG;
    if (beta != 0.0f && !p.C) return GEMM15_ERR_INVALID_ARG;
    if (p.K > 0 && (!p.A || !p.B)) return GEMM15_ERR_INVALID_ARG;
    // leading dimensions must cover the contiguous extent
    if (p.K > 0) {
        if (p.lda < (p.a_kmajor ? p.K : p.M)) return GEMM15_ERR_INVALID_ARG;
        if (p.ldb < (p.b_kmajor ? p.K : p.N)) return GEMM15_ERR_INVALID_ARG;
        if (!aligned16(p.A) || !aligned16(p.B)) return GEMM15_ERR_ALIGNMENT;
        if ((p.lda * es) % 16 || (p.ldb * es) % 16) return GEMM15_ERR_ALIGNMENT;
    }
    if (p.ldd < p.N) return GEMM15_ERR_INVALID_ARG;
    if (!aligned16(p.D) || (p.ldd * eo) % 16) return GEMM15_ERR_ALIGNMENT;
    if (beta != 0.0f) {
        if (p.ldc < p.N) return GEMM15_ERR_INVALID_ARG;
        if (!aligned16(p.C) || (p.ldc * eo) % 16) return GEMM15_ERR_ALIGNMENT;
    }
    if (p.bias && !aligned16(p.bias)) return GEMM15_ERR_ALIGNMENT;
    if (p.aux_op < 0 || p.aux_op > 4) return GEMM15_ERR_INVALID_ARG;
    if (p.aux_op) {
        if (!p.aux || p.ldaux < p.N) return GEMM15_ERR_INVALID_ARG;
        if (!aligned16(p.aux) || (p.ldaux * eo) % 16) return GEMM15_ERR_ALIGNMENT;
    }
    if (p.pre) {
        if (p.ldpre < p.N) return GEMM15_ERR_INVALID_ARG;
        if (!aligned16(p.pre) || (p.ldpre * eo) % 16) return GEMM15_ERR_ALIGNMENT;
    }
    return GEMM15_OK;
}

// ------------------------------------------------------------------ planner

struct Decision {
    int cg = 1;
    int bn = 256;
    int bk = 64;
    int sched = SCHED_DP;
    int grid = 1;
    int32_t m_blocks = 0, n_blocks = 0, tiles = 0, k_blocks = 0;
    int32_t dp_tiles = 0, splits = 1, raster = 1;
    int64_t sk_units = 0;
    bool balanced = false;  // split-K over a stream-K partition of all units
    bool inline_split = false;  // split-K reduced inside the GEMM kernel (last split)
    size_t ws_bytes = 0;
    int flags = 0;
};

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int pair_clusters(gemm15_plan* plan) {
    if (plan->pair_clusters < 0) plan->pair_clusters = gemm_max_pair_clusters(plan->elem);
    return plan->pair_clusters;
}

// Picks the tile shape, schedule and grid for one problem (thresholds set
// from measurements of the target shapes on GB300):
//   - SM-pair 256 x 256 tiles (cta_group::2) when there is at least one full
//     wave of them: they halve each SM's share of B traffic;
//   - at least one wave: data-parallel when the last wave is at least 95%
//     full, or at least 80% full while A and B together exceed 64 MiB (then
//     stream-K's units, which sweep different k ranges of tiles that share
//     operands at the same time, lose more to L2 misses than the tail wave
//     costs); stream-K over the tail waves otherwise;
//   - less than one wave: split-K with a separate reduction when at least two
//     splits per tile fit (stream-K otherwise), on SM-pair tiles when M >= 512
//     and on 128-wide tiles when more than 16 splits per tile fit; unless K
//     is short (fewer than 32 k-blocks), where data-parallel 128 x 128 tiles
//     win.
// The plan's options with an autotuned choice for this shape filled in where
// the option is left automatic.
Options effective_options(const gemm15_plan* plan, int64_t M, int64_t N, int64_t K) {
    Options o = plan->opt;
    const auto it = plan->tuned.find(std::make_tuple(M, N, K));
    if (it == plan->tuned.end()) return o;
    const Tuned& t = it->second;
    if (o.schedule == 0) {
        o.schedule = t.schedule;
        if (o.sk_dp_waves < 0) o.sk_dp_waves = t.sk_dp_waves;
        if (o.splits == 0) o.splits = t.splits;
    }
    if (o.cta_group == 0) o.cta_group = t.cta_group;
    if (o.tile_n == 0) o.tile_n = t.tile_n;
    if (o.swap_ab == 0) o.swap_ab = t.swap_ab;
    return o;
}

// Swap-AB for a short computed M against a long N (decode-size token counts
// against a weight matrix): unless the plan's option says otherwise.
bool use_swap(const Options& o, const Prob& p) {
    if (o.swap_ab == 1) return false;
    if (o.swap_ab == 2) return true;
    return p.M <= 128 && p.N >= 1024 && p.K >= 256;
}

// With `swap` the problem is a swapped one (swap-AB): single-SM tiles whose N
// covers the short side, 64 wide for 16-bit operands when it fits (the
// narrowest B stage that is a whole 128-byte swizzle row), else 128.
Decision decide(gemm15_plan* plan, int64_t M, int64_t N, int64_t K, const Options& o,
                bool swap = false) {
    Decision d;
    d.bk = plan->elem == ELEM_E4M3 ? 128 : 64;
    d.bn = o.tile_n ? o.tile_n : (N <= 128 ? 128 : 256);
    if (swap) d.bn = (plan->elem != ELEM_E4M3 && N <= 64) ? 64 : 128;
    const int G1 = o.grid > 0 ? std::min(o.grid, plan->num_sms) : plan->num_sms;
    int cg = 1;
    // SM-pair tiles 256 x 128 exist for 16-bit operands only (an fp8 half-tile
    // of B would be narrower than one 128-byte swizzle row)
    // swap-AB tiles pair only when asked (16-bit, 128 tokens wide: each CTA of
    // the pair stages 64 of them)
    const bool pair_ok = swap ? (o.cta_group == 2 && d.bn == 128 && plan->elem != ELEM_E4M3)
                              : (d.bn == 256 || plan->elem != ELEM_E4M3);
    const int clusters = std::min(pair_clusters(plan), G1 / 2);
    if (pair_ok && o.cta_group != 1) {
        const int64_t tiles2 = cdiv(M, 2 * TILE_M) * cdiv(N, 256);
        if (clusters > 0 && (o.cta_group == 2 || (d.bn == 256 && M >= 512 && tiles2 >= clusters))) cg = 2;
    }
    int G = cg == 2 ? clusters : G1;  // scheduling units
    d.k_blocks = static_cast<int32_t>(cdiv(K, d.bk));
    auto set_tiles = [&]() {
        d.m_blocks = static_cast<int32_t>(cdiv(M, TILE_M * cg));
        d.n_blocks = static_cast<int32_t>(cdiv(N, d.bn));
        d.tiles = d.m_blocks * d.n_blocks;
    };
    set_tiles();

    int sched = o.schedule;
    if (sched == 0) {
        if (d.tiles >= G) {
            const int64_t waves = cdiv(d.tiles, G);
            const double eff = static_cast<double>(d.tiles) / static_cast<double>(waves * G);
            const int64_t esize = plan->elem == ELEM_E4M3 ? 1 : 2;
            const bool operands_fit_l2 = (M + N) * K * esize <= (int64_t{64} << 20);
            const bool dp = eff >= 0.95 || (eff >= 0.8 && !operands_fit_l2) || d.k_blocks < 8;
            sched = dp ? SCHED_DP : SCHED_SK;
        } else if (d.k_blocks < 32) {
            sched = SCHED_DP;
            if (!o.tile_n && cg == 1 && d.bn == 256) {
                d.bn = 128;  // twice the tiles to spread a short-K problem
                set_tiles();
            }
        } else {
            // swap-AB decode shapes: stream-K (one launch; measured equal or better
            // than split-K on every Llama-70B layer at M 16 and 128: o_proj M 128
            // 48 against 54 us, down M 128 97 against 104)
            sched = (G / d.tiles >= 2 && !swap) ? SCHED_SPLIT : SCHED_SK;
            if (sched == SCHED_SPLIT && o.cta_group == 0 && cg == 1 && pair_ok && d.bn == 256 &&
                M >= 512 && clusters > 0) {
                // pair tiles share each B tile across the pair at the same
                // number of split units
                cg = 2;
                G = clusters;
                set_tiles();
            }
            if (sched == SCHED_SPLIT && !o.tile_n && cg == 1 && d.bn == 256 && G / d.tiles > 16) {
                // many splits: half-width tiles halve the fp32 partial traffic
                d.bn = 128;
                set_tiles();
            }
        }
    }
    d.cg = cg;
    d.sched = sched;
    // balanced split-K (option splits = -1): the k iterations of all tiles cut
    // evenly over every unit (pieces may straddle two tiles); the reduction
    // kernel finds each tile's pieces from the partition.  Measured slower than
    // whole splits per tile on the GB300 decode shapes (each unit leaves up to
    // two partial tiles), so it is never chosen automatically.
    d.balanced = sched == SCHED_SPLIT && cg == 1 && o.splits == -1 && d.tiles < G;
    d.raster = o.raster > 0 ? std::min<int32_t>(o.raster, d.m_blocks)
                            : std::min<int32_t>(d.m_blocks, cg == 2 ? 8 : 16);
    const size_t half_tile = static_cast<size_t>(TILE_M) * d.bn * sizeof(float);
    int units = 1;
    if (sched == SCHED_DP) {
        units = static_cast<int>(std::min<int64_t>(G, d.tiles));
    } else if (sched == SCHED_SK) {
        if (o.sk_dp_waves >= 0)
            d.dp_tiles = static_cast<int32_t>(std::min<int64_t>(o.sk_dp_waves, d.tiles / G)) * G;
        else
            d.dp_tiles = d.tiles >= 2 * G ? (d.tiles / G - 1) * G : 0;
        if (d.dp_tiles >= d.tiles) d.dp_tiles = d.tiles - 1;
        d.sk_units = static_cast<int64_t>(d.tiles - d.dp_tiles) * d.k_blocks;
        units = static_cast<int>(std::min<int64_t>(G, d.sk_units));
        // per unit and CTA: a tail piece and a head piece may each leave a partial tile
        d.ws_bytes = static_cast<size_t>(2 * units) * cg * half_tile;
        d.flags = 2 * units * cg;
    } else if (d.balanced) {
        d.sk_units = static_cast<int64_t>(d.tiles) * d.k_blocks;
        units = static_cast<int>(std::min<int64_t>(G, d.sk_units));
        d.splits = 0;
        d.ws_bytes = static_cast<size_t>(2 * units) * half_tile;  // a tail and a head piece per unit
    } else {
        int splits = o.splits > 0 ? o.splits : std::max(1, G / std::max<int32_t>(d.tiles, 1));
        splits = static_cast<int>(std::min<int64_t>(splits, d.k_blocks));
        splits = std::max(splits, 1);
        d.splits = splits;
        units = static_cast<int>(std::min<int64_t>(G, static_cast<int64_t>(d.tiles) * splits));
        d.ws_bytes = static_cast<size_t>(d.tiles) * cg * splits * half_tile;
        // the last split of a tile adds the partials itself when they are few
        // (one CTA reads them all: at most 256 KiB) and the tile is stored
        // as computed; else a reduction kernel (measured on GB300: 1536^2 x
        // 16384 on SM-pair tiles 91 -> 75 us in-kernel, while swap-AB decode
        // shapes, whose transposed stores make the last split's pass long,
        // were 4 us faster with the kernel)
        d.inline_split = o.splitk_inline == 2 ||
                         (o.splitk_inline == 0 && !swap &&
                          static_cast<size_t>(splits) * half_tile <= (256u << 10));
        if (d.inline_split) d.flags = 2 * d.tiles * cg;  // one 64-bit arrival counter per tile half
    }
    d.grid = units * cg;
    return d;
}

gemm15_status_t ensure_ws(gemm15_plan* plan, size_t bytes, int flags) {
    if (bytes > plan->ws_cap) {
        if (plan->d_ws) cudaFree(plan->d_ws);
        plan->d_ws = nullptr;
        plan->ws_cap = 0;
        size_t cap = std::max(bytes, static_cast<size_t>(1) << 20);
        if (cudaMalloc(&plan->d_ws, cap) != cudaSuccess) {
            cudaGetLastError();
            return GEMM15_ERR_OOM;
        }
        plan->ws_cap = cap;
    }
    if (flags > plan->flags_cap) {
        if (plan->d_flags) cudaFree(plan->d_flags);
        plan->d_flags = nullptr;
        plan->flags_cap = 0;
        int cap = std::max(flags, 1024);
        if (cudaMalloc(&plan->d_flags, cap * sizeof(uint32_t)) != cudaSuccess) {
            cudaGetLastError();
            return GEMM15_ERR_OOM;
        }
        if (cudaMemset(plan->d_flags, 0, cap * sizeof(uint32_t)) != cudaSuccess)
            return GEMM15_ERR_CUDA;
        plan->flags_cap = cap;
    }
    return GEMM15_OK;
}

cudaError_t launch_kernel(int elem, int bn, int cg, const GemmParams& gp, int grid, cudaStream_t s) {
    if (cg == 2) {
        if (elem == ELEM_F16) return bn == 128 ? launch_gemm<ELEM_F16, 128, 2>(gp, grid, s) : launch_gemm<ELEM_F16, 256, 2>(gp, grid, s);
        if (elem == ELEM_BF16) return bn == 128 ? launch_gemm<ELEM_BF16, 128, 2>(gp, grid, s) : launch_gemm<ELEM_BF16, 256, 2>(gp, grid, s);
        return launch_gemm<ELEM_E4M3, 256, 2>(gp, grid, s);
    }
    if (elem == ELEM_F16) {
        if (bn == 64) return launch_gemm<ELEM_F16, 64>(gp, grid, s);
        return bn == 128 ? launch_gemm<ELEM_F16, 128>(gp, grid, s) : launch_gemm<ELEM_F16, 256>(gp, grid, s);
    }
    if (elem == ELEM_BF16) {
        if (bn == 64) return launch_gemm<ELEM_BF16, 64>(gp, grid, s);
        return bn == 128 ? launch_gemm<ELEM_BF16, 128>(gp, grid, s) : launch_gemm<ELEM_BF16, 256>(gp, grid, s);
    }
    return bn == 128 ? launch_gemm<ELEM_E4M3, 128>(gp, grid, s) : launch_gemm<ELEM_E4M3, 256>(gp, grid, s);
}

cudaError_t launch_reduce_kernel(int out_elem, const ReduceParams& rp, cudaStream_t s, int num_sms) {
    int grid = 1, groups = 1;
    reduce_shape(rp, num_sms, &grid, &groups);
    return out_elem == ELEM_F16 ? launch_reduce<ELEM_F16>(rp, grid, groups, s)
                                : launch_reduce<ELEM_BF16>(rp, grid, groups, s);
}

// Fills the operand-layout part of the kernel parameters.
void fill_layout(const gemm15_plan* plan, GemmParams& gp, bool a_kmajor, bool b_kmajor, int bn,
                 int cg = 1) {
    const bool f8 = plan->elem == ELEM_E4M3;
    const int es = f8 ? 1 : 2;
    const int bk = 128 / es;
    const int umma_k = 32 / es;
    gp.a_kmajor = a_kmajor;
    gp.b_kmajor = b_kmajor;
    // K-major, 128-byte swizzle: rows of 128 B, 8-row groups 1024 B apart;
    // one MMA step along K advances 32 bytes inside the swizzle row.
    // MN-major, 128-byte swizzle: 128-byte MN chunks (one TMA box of BK rows
    // each) LBO apart, 8-row K groups 1024 B apart; one MMA step along K
    // advances UMMA_K rows of 128 B.
    const uint32_t mn_box = static_cast<uint32_t>((128 / es) * bk * es);
    gp.a_lbo = a_kmajor ? 16u : mn_box;
    gp.a_sbo = 1024u;
    gp.a_kstep = a_kmajor ? 32u : static_cast<uint32_t>(umma_k * 128);
    gp.b_lbo = b_kmajor ? 16u : mn_box;
    gp.b_sbo = 1024u;
    gp.b_kstep = b_kmajor ? 32u : static_cast<uint32_t>(umma_k * 128);
    // instruction descriptor: A/B format 0 = f16 / e4m3, 1 = bf16
    const uint32_t fmt = plan->elem == ELEM_BF16 ? 1u : 0u;
    uint32_t idesc = 0;
    idesc |= 1u << 4;                      // D format f32
    idesc |= fmt << 7;                     // A format
    idesc |= fmt << 10;                    // B format
    idesc |= (a_kmajor ? 0u : 1u) << 15;   // A MN-major
    idesc |= (b_kmajor ? 0u : 1u) << 16;   // B MN-major
    idesc |= static_cast<uint32_t>(bn >> 3) << 17;
    idesc |= static_cast<uint32_t>((TILE_M * cg) >> 4) << 24;  // M = 128 or 256 (SM pair)
    gp.idesc = idesc;
}

// bn_box: columns of B one CTA stages (the tile width, or half of it for SM pairs).
bool operand_maps(const gemm15_plan* plan, const Prob& p, int bn_box, CUtensorMap* tA, CUtensorMap* tB) {
    const bool f8 = plan->elem == ELEM_E4M3;
    const int es = f8 ? 1 : 2;
    const uint32_t bk = 128 / es, w = 128 / es;
    bool ok = true;
    if (p.a_kmajor)
        ok &= make_tmap(tA, plan->elem, p.A, p.K, p.M, p.lda * es, bk, TILE_M);
    else
        ok &= make_tmap(tA, plan->elem, p.A, p.M, p.K, p.lda * es, w, bk);
    if (p.b_kmajor)
        ok &= make_tmap(tB, plan->elem, p.B, p.K, p.N, p.ldb * es, bk, bn_box);
    else
        ok &= make_tmap(tB, plan->elem, p.B, p.N, p.K, p.ldb * es, w, bk);
    return ok;
}

bool output_maps(const gemm15_plan* plan, const Prob& p, bool has_c, CUtensorMap* tC, CUtensorMap* tD) {
    bool ok = make_tmap(tD, plan->out_elem, p.D, p.N, p.M, p.ldd * 2, EPI_COLS, 32);
    if (has_c) ok &= make_tmap(tC, plan->out_elem, p.C, p.N, p.M, p.ldc * 2, EPI_COLS, 32);
    else std::memset(tC, 0, sizeof(*tC));
    return ok;
}

void record_config(gemm15_plan* plan, const Decision& d, int launches) {
    gemm15_config_t& c = plan->last;
    c.cta_group = d.cg;
    c.tile_m = TILE_M * d.cg;
    c.tile_n = d.bn;
    c.tile_k = d.bk;
    c.stages = gemm_stages(plan->elem, d.bn, d.cg);
    c.schedule = d.sched;
    c.grid = d.grid;
    c.tiles = d.tiles;
    c.splits = d.sched == SCHED_SPLIT ? d.splits : 1;
    c.raster = d.raster;
    c.launches = launches;
    c.swap_ab = plan->desc.layout_cd == GEMM15_COL_MAJOR ? 1 : 0;
}

// Points the kernel at a zeroed timeline buffer when tracing is on.
gemm15_status_t attach_trace(gemm15_plan* plan, GemmParams& gp, int grid, cudaStream_t s) {
    gp.trace = nullptr;
    gp.trace_items = 0;
    if (plan->opt.trace_items <= 0) return GEMM15_OK;
    const size_t bytes = static_cast<size_t>(grid) * (plan->opt.trace_items + 1) * TRACE_WORDS * 8;
    if (bytes > plan->trace_cap) {
        cudaFree(plan->d_trace);
        plan->d_trace = nullptr;
        plan->trace_cap = 0;
        if (cudaMalloc(&plan->d_trace, bytes) != cudaSuccess) {
            cudaGetLastError();
            return GEMM15_ERR_OOM;
        }
        plan->trace_cap = bytes;
    }
    if (cudaMemsetAsync(plan->d_trace, 0, bytes, s) != cudaSuccess) return GEMM15_ERR_CUDA;
    gp.trace = plan->d_trace;
    gp.trace_items = plan->opt.trace_items;
    plan->trace_ctas = grid;
    return GEMM15_OK;
}

// Launch parameters of one dense problem, computed once and reused while the
// same problem (pointers, shape, leading dimensions, epilogue operands) is run
// again with the same options: the per-call work is then a lookup and the
// launch, with the tensor maps already encoded.
struct LaunchEntry {
    bool valid = false;
    Prob p{};            // the caller's problem (after layout normalisation)
    Prob pe{};           // the problem the kernel computes (swapped for swap-AB)
    bool swap = false;
    bool has_c = false;
    Options opt{};       // the decision-relevant options at encoding time
    uint64_t tuned_gen = 0;
    Decision d{};
    GemmParams gp{};     // every field that does not change from call to call
};

constexpr int CACHE_ENTRIES = 8;
struct LaunchCache {
    LaunchEntry e[CACHE_ENTRIES];
    int next = 0;
};

bool same_prob(const Prob& a, const Prob& b) {
    return a.M == b.M && a.N == b.N && a.K == b.K && a.A == b.A && a.lda == b.lda &&
           a.a_kmajor == b.a_kmajor && a.B == b.B && a.ldb == b.ldb && a.b_kmajor == b.b_kmajor &&
           a.C == b.C && a.ldc == b.ldc && a.D == b.D && a.ldd == b.ldd && a.bias == b.bias &&
           a.bias_rows == b.bias_rows && a.aux == b.aux && a.ldaux == b.ldaux &&
           a.aux_op == b.aux_op && a.pre == b.pre && a.ldpre == b.ldpre &&
           a.out_trans == b.out_trans;
}

bool same_choice_options(const Options& a, const Options& b) {
    return a.schedule == b.schedule && a.splits == b.splits && a.cta_group == b.cta_group &&
           a.tile_n == b.tile_n && a.raster == b.raster && a.grid == b.grid &&
           a.sk_dp_waves == b.sk_dp_waves && a.swap_ab == b.swap_ab &&
           a.splitk_inline == b.splitk_inline;
}

// Finds or builds the launch parameters of problem p (nullptr on an encoding
// failure).
const LaunchEntry* launch_entry(gemm15_plan* plan, const Prob& key, bool has_c) {
    if (!plan->cache) plan->cache = new (std::nothrow) LaunchCache();
    LaunchCache* cache = static_cast<LaunchCache*>(plan->cache);
    if (!cache) return nullptr;
    for (const LaunchEntry& e : cache->e)
        if (e.valid && e.has_c == has_c && e.tuned_gen == plan->tuned_gen &&
            same_choice_options(e.opt, plan->opt) && same_prob(e.p, key))
            return &e;
    LaunchEntry& e = cache->e[cache->next];
    cache->next = (cache->next + 1) % CACHE_ENTRIES;
    e.valid = false;
    // options with this shape's autotuned choice filled in
    const Options o = effective_options(plan, key.M, key.N, key.K);
    const bool swap = use_swap(o, key);
    const Prob p = swap ? swapped(key) : key;  // the problem the kernel computes
    const Decision d = decide(plan, p.M, p.N, p.K, o, swap);
    GemmParams& gp = e.gp;
    std::memset(&gp, 0, sizeof(gp));
    if (!operand_maps(plan, p, d.bn / d.cg, &gp.tmA, &gp.tmB)) return nullptr;
    // a transposed output: C, Z and Y element-wise; D through a tensor map of
    // its storage seen transposed (inner dimension = the computed rows), stored
    // from 32 x 64 boxes that the epilogue fills transposed
    if (!p.out_trans && !output_maps(plan, p, has_c, &gp.tmC, &gp.tmD)) return nullptr;
    if (p.out_trans) {
        if (!make_tmap(&gp.tmD, plan->out_elem, p.D, p.M, p.N, p.ldd * 2, 32, EPI_COLS, false))
            return nullptr;
        gp.out_tma = 1;
    }
    gp.out_trans = p.out_trans ? 1 : 0;
    gp.D = p.D;
    gp.ldd = p.ldd;
    gp.C = has_c ? p.C : nullptr;
    gp.ldc = p.ldc;
    gp.M = static_cast<int32_t>(p.M);
    gp.N = static_cast<int32_t>(p.N);
    gp.K = static_cast<int32_t>(p.K);
    gp.k_blocks = d.k_blocks;
    gp.m_blocks = d.m_blocks;
    gp.n_blocks = d.n_blocks;
    gp.tiles = d.tiles;
    gp.raster = d.raster;
    gp.sched = d.balanced ? SCHED_SK : d.sched;
    gp.sk_partials_only = d.balanced ? 1 : 0;
    gp.dp_tiles = d.dp_tiles;
    gp.splits = d.splits;
    // split-K with a reduction kernel: that kernel reads C and applies the epilogue
    const bool epi_here = d.sched != SCHED_SPLIT || d.inline_split;
    gp.splitk_inline = d.inline_split ? 1 : 0;
    gp.has_c = has_c && epi_here;
    gp.sk_units = d.sk_units;
    gp.act = static_cast<int>(plan->desc.epilogue);
    gp.bias = epi_here ? p.bias : nullptr;
    gp.bias_rows = p.bias_rows;
    gp.aux = p.aux;
    gp.ldaux = p.ldaux;
    gp.aux_op = epi_here ? p.aux_op : 0;
    gp.pre = epi_here ? p.pre : nullptr;
    gp.ldpre = p.ldpre;
    fill_layout(plan, gp, p.a_kmajor, p.b_kmajor, d.bn, d.cg);
    gp.groups = nullptr;
    gp.num_groups = 0;
    set_sched_divisors(gp, d.grid / d.cg);
    e.p = key;
    e.pe = p;
    e.swap = swap;
    e.has_c = has_c;
    e.opt = plan->opt;
    e.tuned_gen = plan->tuned_gen;
    e.d = d;
    e.valid = true;
    return &e;
}

// Element types whose plans run only the block-scaled entry point.
bool block_scaled_only(const gemm15_plan* plan) {
    return plan->elem == ELEM_E5M2 || plan->elem == ELEM_E2M1;
}

gemm15_status_t run_dense(gemm15_plan* plan, const Prob& p, float alpha, float beta,
                          const float* scale_a, const float* scale_b, cudaStream_t s) {
    if (block_scaled_only(plan)) return GEMM15_ERR_UNSUPPORTED;
    gemm15_status_t st = check_operands(plan, p, beta);
    if (st != GEMM15_OK) return st;
    if (p.M == 0 || p.N == 0) {
        std::memset(&plan->last, 0, sizeof(plan->last));
        return GEMM15_OK;
    }
    st = order_after_previous(plan, s);
    if (st != GEMM15_OK) return st;
    const bool has_c = beta != 0.0f;
    const int act = static_cast<int>(plan->desc.epilogue);
    if (p.K == 0) {
        ReduceParams rp{};
        rp.ws = nullptr;
        rp.splits = 0;
        rp.tile_n = 256;
        rp.n_blocks = 1;
        rp.M = static_cast<int32_t>(p.M);
        rp.N = static_cast<int32_t>(p.N);
        rp.C = p.C;
        rp.ldc = p.ldc;
        rp.D = p.D;
        rp.ldd = p.ldd;
        rp.alpha = alpha;
        rp.beta = beta;
        rp.act = act;
        rp.has_c = has_c;
        rp.bias = p.bias;
        rp.bias_rows = p.bias_rows;
        rp.aux = p.aux;
        rp.ldaux = p.ldaux;
        rp.aux_op = p.aux_op;
        rp.pre = p.pre;
        rp.ldpre = p.ldpre;
        if (launch_reduce_kernel(plan->out_elem, rp, s, plan->num_sms) != cudaSuccess) return GEMM15_ERR_CUDA;
        Decision d;
        d.sched = SCHED_SPLIT;
        d.splits = 0;
        record_config(plan, d, 1);
        plan->last.grid = 0;
        return mark_done(plan, s);
    }
    const LaunchEntry* le = launch_entry(plan, p, has_c);
    if (!le) return GEMM15_ERR_CUDA;
    const Decision& d = le->d;
    const Prob& pe = le->pe;
    st = ensure_ws(plan, d.ws_bytes, d.flags);
    if (st != GEMM15_OK) return st;

    GemmParams gp = le->gp;
    gp.alpha = alpha;
    gp.beta = beta;
    gp.scale_a = scale_a;
    gp.scale_b = scale_b;
    gp.ws = plan->d_ws;
    gp.flags = plan->d_flags;
    gp.status = plan->d_status;
    gp.epoch = ++plan->epoch == 0 ? ++plan->epoch : plan->epoch;
    gp.timeout_ns = static_cast<uint64_t>(plan->opt.timeout_us) * 1000ull;
    gp.fault_skip_flag = plan->opt.fault_skip_flag;
    gp.l2_hints = plan->opt.l2_hints;
    st = attach_trace(plan, gp, d.grid, s);
    if (st != GEMM15_OK) return st;
    if (launch_kernel(plan->elem, d.bn, d.cg, gp, d.grid, s) != cudaSuccess) return GEMM15_ERR_CUDA;
    int launches = 1;
    if (d.sched == SCHED_SPLIT && !d.inline_split) {
        ReduceParams rp{};
        rp.ws = plan->d_ws;
        rp.splits = d.splits;
        rp.tile_n = d.bn;
        rp.n_blocks = d.n_blocks;
        rp.M = gp.M;
        rp.N = gp.N;
        rp.C = pe.C;
        rp.ldc = pe.ldc;
        rp.D = pe.D;
        rp.ldd = pe.ldd;
        rp.alpha = alpha;
        rp.beta = beta;
        rp.scale_a = scale_a;
        rp.scale_b = scale_b;
        rp.act = act;
        rp.has_c = has_c;
        rp.bias = pe.bias;
        rp.bias_rows = pe.bias_rows;
        rp.aux = pe.aux;
        rp.ldaux = pe.ldaux;
        rp.aux_op = pe.aux_op;
        rp.pre = pe.pre;
        rp.ldpre = pe.ldpre;
        rp.out_trans = pe.out_trans ? 1 : 0;
        if (d.balanced) {
            rp.units = d.grid;
            rp.sk_units = d.sk_units;
            rp.k_blocks = d.k_blocks;
            rp.m_blocks = d.m_blocks;
            rp.raster = d.raster;
        }
        if (launch_reduce_kernel(plan->out_elem, rp, s, plan->num_sms) != cudaSuccess) return GEMM15_ERR_CUDA;
        ++launches;
    }
    record_config(plan, d, launches);
    if (le->swap) plan->last.swap_ab ^= 1;
    return mark_done(plan, s);
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

const char* gemm15_status_string(gemm15_status_t s) {
    switch (s) {
        case GEMM15_OK: return "ok";
        case GEMM15_ERR_INVALID_ARG: return "invalid argument";
        case GEMM15_ERR_UNSUPPORTED: return "unsupported type or layout combination";
        case GEMM15_ERR_ALIGNMENT: return "pointer or leading dimension not 16-byte aligned";
        case GEMM15_ERR_CUDA: return "CUDA call failed";
        case GEMM15_ERR_TIMEOUT: return "a bounded device-side wait ran out";
        case GEMM15_ERR_OOM: return "device memory allocation failed";
        case GEMM15_ERR_DEVICE_FAULT: return "device reported an internal error";
        case GEMM15_ERR_NO_DEVICE: return "no sm_103 device available";
        case GEMM15_ERR_BAD_PLAN: return "invalid or destroyed plan handle";
    }
    return "unknown status";
}

gemm15_status_t gemm_plan_create(gemm15_plan_t* out, const gemm15_plan_desc_t* desc) {
    if (!out || !desc) return GEMM15_ERR_INVALID_ARG;
    *out = nullptr;
    const gemm15_plan_desc_t& d = *desc;
    auto valid_t = [](int t) { return t >= GEMM15_F16 && t <= GEMM15_E2M1; };
    auto valid_l = [](int l) { return l == GEMM15_ROW_MAJOR || l == GEMM15_COL_MAJOR; };
    if (!valid_t(d.a) || !valid_t(d.b) || !valid_t(d.c) || !valid_t(d.d) || !valid_t(d.acc) ||
        !valid_l(d.layout_a) || !valid_l(d.layout_b) || !valid_l(d.layout_cd) ||
        (d.epilogue < GEMM15_EPI_LINEAR || d.epilogue > GEMM15_EPI_TANH))
        return GEMM15_ERR_INVALID_ARG;
    if (d.acc != GEMM15_F32 || d.a != d.b) return GEMM15_ERR_UNSUPPORTED;
    int elem, out_elem;
    if (d.a == GEMM15_F16 && d.c == GEMM15_F16 && d.d == GEMM15_F16) {
        elem = out_elem = ELEM_F16;
    } else if (d.a == GEMM15_BF16 && d.c == GEMM15_BF16 && d.d == GEMM15_BF16) {
        elem = out_elem = ELEM_BF16;
    } else if (d.a == GEMM15_E4M3 && d.c == GEMM15_BF16 && d.d == GEMM15_BF16) {
        elem = ELEM_E4M3;
        out_elem = ELEM_BF16;
    } else if ((d.a == GEMM15_E5M2 || d.a == GEMM15_E2M1) && d.c == GEMM15_BF16 && d.d == GEMM15_BF16) {
        elem = d.a == GEMM15_E5M2 ? ELEM_E5M2 : ELEM_E2M1;  // block-scaled runs only
        out_elem = ELEM_BF16;
    } else {
        return GEMM15_ERR_UNSUPPORTED;
    }
    int dev = 0, count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
        cudaGetLastError();
        return GEMM15_ERR_NO_DEVICE;
    }
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM15_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return GEMM15_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return GEMM15_ERR_NO_DEVICE;
    if (!encode_fn()) return GEMM15_ERR_CUDA;

    gemm15_plan* p = new (std::nothrow) gemm15_plan();
    if (!p) return GEMM15_ERR_OOM;
    p->desc = d;
    p->device = dev;
    p->num_sms = prop.multiProcessorCount;
    p->elem = elem;
    p->out_elem = out_elem;
    if (cudaMalloc(&p->d_status, sizeof(int32_t)) != cudaSuccess ||
        cudaMemset(p->d_status, 0, sizeof(int32_t)) != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return GEMM15_ERR_OOM;
    }
    if (ensure_ws(p, 0, p->num_sms) != GEMM15_OK) {
        cudaFree(p->d_status);
        delete p;
        return GEMM15_ERR_OOM;
    }
    if (cudaEventCreateWithFlags(&p->done_ev, cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(p->d_status);
        cudaFree(p->d_flags);
        cudaFree(p->d_ws);
        delete p;
        return GEMM15_ERR_CUDA;
    }
    *out = p;
    return GEMM15_OK;
}

gemm15_status_t gemm_plan_destroy(gemm15_plan_t plan) {
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    DeviceGuard g(plan->device);
    if (plan->groups_done) {
        cudaEventSynchronize(plan->groups_done);
        cudaEventDestroy(plan->groups_done);
    }
    cudaFree(plan->d_status);
    cudaFree(plan->d_flags);
    cudaFree(plan->d_ws);
    cudaFree(plan->d_groups);
    if (plan->h_groups) cudaFreeHost(plan->h_groups);
    for (void* b : plan->d_host_path) cudaFree(b);
    cudaFree(plan->d_scales);
    cudaFree(plan->d_trace);
    if (plan->done_ev) cudaEventDestroy(plan->done_ev);
    if (plan->fork_ev) cudaEventDestroy(plan->fork_ev);
    if (plan->join_ev) cudaEventDestroy(plan->join_ev);
    if (plan->copy_stream) cudaStreamDestroy(plan->copy_stream);
    if (plan->d2h_stream) cudaStreamDestroy(plan->d2h_stream);
    if (plan->a_ev) cudaEventDestroy(plan->a_ev);
    if (plan->d2h_ev) cudaEventDestroy(plan->d2h_ev);
    for (int i = 0; i < 8; ++i) {
        if (plan->up_ev[i]) cudaEventDestroy(plan->up_ev[i]);
        if (plan->done_evs[i]) cudaEventDestroy(plan->done_evs[i]);
    }
    delete static_cast<LaunchCache*>(plan->cache);
    plan->magic = PLAN_DEAD;
    delete plan;
    return GEMM15_OK;
}

gemm15_status_t gemm_run_ex(gemm15_plan_t plan, const void* A, int64_t lda, const void* B,
                            int64_t ldb, const void* C, int64_t ldc, void* D, int64_t ldd,
                            int64_t M, int64_t N, int64_t K, float alpha, float beta,
                            const float* scale_a, const float* scale_b, void* stream) {
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    if ((scale_a || scale_b) && plan->elem != ELEM_E4M3) return GEMM15_ERR_INVALID_ARG;
    DeviceGuard g(plan->device);
    if (!g.ok) return GEMM15_ERR_CUDA;
    Prob p = normalise(plan, M, N, K, A, lda, B, ldb, C, ldc, D, ldd);
    return run_dense(plan, p, alpha, beta, scale_a, scale_b, static_cast<cudaStream_t>(stream));
}

gemm15_status_t gemm_run_args(gemm15_plan_t plan, const gemm15_args_t* a, void* stream) {
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    if (!a) return GEMM15_ERR_INVALID_ARG;
    if ((a->scale_a || a->scale_b) && plan->elem != ELEM_E4M3) return GEMM15_ERR_INVALID_ARG;
    DeviceGuard g(plan->device);
    if (!g.ok) return GEMM15_ERR_CUDA;
    const bool a_row = plan->desc.layout_a == GEMM15_ROW_MAJOR;
    const bool b_row = plan->desc.layout_b == GEMM15_ROW_MAJOR;
    const bool cd_row = plan->desc.layout_cd == GEMM15_ROW_MAJOR;
    const int64_t lda = a->lda ? a->lda : (a_row ? a->K : a->M);
    const int64_t ldb = a->ldb ? a->ldb : (b_row ? a->N : a->K);
    const int64_t ldc = a->ldc ? a->ldc : (cd_row ? a->N : a->M);
    const int64_t ldd = a->ldd ? a->ldd : (cd_row ? a->N : a->M);
    Prob p = normalise(plan, a->M, a->N, a->K, a->A, lda, a->B, ldb, a->C, ldc, a->D, ldd);
    p.bias = a->bias;
    p.aux_op = a->aux_op;
    p.aux = a->aux_op ? a->aux : nullptr;
    p.ldaux = a->ldaux ? a->ldaux : (cd_row ? a->N : a->M);
    p.pre = a->pre;
    p.ldpre = a->ldpre ? a->ldpre : (cd_row ? a->N : a->M);
    return run_dense(plan, p, a->alpha, a->beta, a->scale_a, a->scale_b,
                     static_cast<cudaStream_t>(stream));
}

gemm15_status_t gemm_plan_autotune(gemm15_plan_t plan, const gemm15_args_t* a, int32_t iterations,
                                   gemm15_tune_result_t* results, int32_t capacity, int32_t* count,
                                   void* stream) {
    if (count) *count = 0;
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    if (!a || iterations < 1 || capacity < 0 || (capacity > 0 && !results))
        return GEMM15_ERR_INVALID_ARG;
    if ((a->scale_a || a->scale_b) && plan->elem != ELEM_E4M3) return GEMM15_ERR_INVALID_ARG;
    DeviceGuard g(plan->device);
    if (!g.ok) return GEMM15_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool a_row = plan->desc.layout_a == GEMM15_ROW_MAJOR;
    const bool b_row = plan->desc.layout_b == GEMM15_ROW_MAJOR;
    const bool cd_row = plan->desc.layout_cd == GEMM15_ROW_MAJOR;
    Prob p = normalise(plan, a->M, a->N, a->K, a->A, a->lda ? a->lda : (a_row ? a->K : a->M), a->B,
                       a->ldb ? a->ldb : (b_row ? a->N : a->K), a->C,
                       a->ldc ? a->ldc : (cd_row ? a->N : a->M), a->D,
                       a->ldd ? a->ldd : (cd_row ? a->N : a->M));
    p.bias = a->bias;
    p.aux_op = a->aux_op;
    p.aux = a->aux_op ? a->aux : nullptr;
    p.ldaux = a->ldaux ? a->ldaux : (cd_row ? a->N : a->M);
    p.pre = a->pre;
    p.ldpre = a->ldpre ? a->ldpre : (cd_row ? a->N : a->M);
    gemm15_status_t st = check_operands(plan, p, a->beta);
    if (st != GEMM15_OK) return st;
    if (p.M == 0 || p.N == 0 || p.K == 0) return GEMM15_OK;  // one fixed path: nothing to choose
    const auto key = std::make_tuple(p.M, p.N, p.K);
    plan->tuned.erase(key);
    ++plan->tuned_gen;

    // candidates: every schedule on each tile shape, stream-K with and without
    // its data-parallel waves
    std::vector<Tuned> cands;
    for (int sched : {SCHED_DP, SCHED_SK, SCHED_SPLIT})
        for (int cg : {1, 2})
            for (int bn : {128, 256}) {
                if (cg == 2 && bn == 128 && plan->elem == ELEM_E4M3) continue;
                if (sched == SCHED_SK) {
                    for (int w : {-1, 0}) cands.push_back(Tuned{sched, cg, bn, w, 0, 1});
                } else {
                    cands.push_back(Tuned{sched, cg, bn, -1, 0, 1});
                }
            }
    // swap-AB (its own tile shape), each schedule once, where one side is short
    if (std::min(p.M, p.N) <= 256)
        for (int sched : {SCHED_DP, SCHED_SK, SCHED_SPLIT}) cands.push_back(Tuned{sched, 1, 0, -1, 0, 2});
    const Options saved = plan->opt;
    // every timed run starts from an L2 that holds none of the operands (a
    // write of twice the L2 size), as when they do not stay in L2 between uses
    int l2_bytes = 0;
    cudaDeviceGetAttribute(&l2_bytes, cudaDevAttrL2CacheSize, plan->device);
    const size_t flush_bytes = std::max<size_t>(2 * static_cast<size_t>(l2_bytes), 64u << 20);
    void* flush = nullptr;
    if (cudaMalloc(&flush, flush_bytes) != cudaSuccess) {
        cudaGetLastError();
        return GEMM15_ERR_OOM;
    }
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        if (e0) cudaEventDestroy(e0);
        cudaFree(flush);
        return GEMM15_ERR_CUDA;
    }
    std::vector<gemm15_tune_result_t> res;
    int best = -1;
    for (size_t i = 0; i < cands.size(); ++i) {
        const Tuned& c = cands[i];
        plan->opt = saved;
        plan->opt.schedule = c.schedule;
        plan->opt.cta_group = c.cta_group;
        plan->opt.tile_n = c.tile_n;
        plan->opt.sk_dp_waves = c.sk_dp_waves;
        plan->opt.splits = c.splits;
        plan->opt.swap_ab = c.swap_ab;
        gemm15_tune_result_t r{};
        r.sk_dp_waves = c.sk_dp_waves;
        r.us = -1.0f;
        r.status = run_dense(plan, p, a->alpha, a->beta, a->scale_a, a->scale_b, s);  // warm-up
        r.config = plan->last;
        float total_ms = 0.0f;
        for (int it = 0; it < iterations && r.status == GEMM15_OK; ++it) {
            float ms = 0.0f;
            if (cudaMemsetAsync(flush, it & 0xff, flush_bytes, s) != cudaSuccess ||
                cudaEventRecord(e0, s) != cudaSuccess) {
                r.status = GEMM15_ERR_CUDA;
                break;
            }
            r.status = run_dense(plan, p, a->alpha, a->beta, a->scale_a, a->scale_b, s);
            if (r.status != GEMM15_OK) break;
            if (cudaEventRecord(e1, s) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
                cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) {
                r.status = GEMM15_ERR_CUDA;
                break;
            }
            total_ms += ms;
        }
        if (r.status == GEMM15_OK) {
            r.us = 1000.0f * total_ms / iterations;
            const gemm15_status_t dev = gemm_plan_query_error(plan);
            if (dev != GEMM15_OK) r.status = dev;
        }
        if (r.status == GEMM15_OK && (best < 0 || r.us < res[best].us)) best = static_cast<int>(res.size());
        res.push_back(r);
    }
    plan->opt = saved;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaStreamSynchronize(s);
    cudaFree(flush);
    if (best < 0) return GEMM15_ERR_CUDA;
    plan->tuned[key] = cands[best];
    ++plan->tuned_gen;
    // leave D holding the chosen configuration's result (and plan->last its config)
    st = run_dense(plan, p, a->alpha, a->beta, a->scale_a, a->scale_b, s);
    if (st != GEMM15_OK) return st;
    std::stable_sort(res.begin(), res.end(), [](const gemm15_tune_result_t& x, const gemm15_tune_result_t& y) {
        const bool xo = x.status == GEMM15_OK, yo = y.status == GEMM15_OK;
        if (xo != yo) return xo;
        return xo && x.us < y.us;
    });
    const int32_t n = static_cast<int32_t>(res.size());
    for (int32_t i = 0; i < std::min(n, capacity); ++i) results[i] = res[i];
    if (count) *count = n;
    return GEMM15_OK;
}

gemm15_status_t gemm_plan_forget_tuning(gemm15_plan_t plan) {
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    plan->tuned.clear();
    ++plan->tuned_gen;
    return GEMM15_OK;
}

gemm15_status_t gemm_run(gemm15_plan_t plan, const void* A, const void* B, const void* C, void* D,
                         int64_t M, int64_t N, int64_t K, float alpha, float beta, void* stream) {
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    const bool a_row = plan->desc.layout_a == GEMM15_ROW_MAJOR;
    const bool b_row = plan->desc.layout_b == GEMM15_ROW_MAJOR;
    const bool cd_row = plan->desc.layout_cd == GEMM15_ROW_MAJOR;
    return gemm_run_ex(plan, A, a_row ? K : M, B, b_row ? N : K, C, cd_row ? N : M, D,
                       cd_row ? N : M, M, N, K, alpha, beta, nullptr, nullptr, stream);
}

gemm15_status_t gemm_run_host(gemm15_plan_t plan, const void* hA, const void* hB, const void* hC,
                              void* hD, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                              float scale_a, float scale_b, void* stream) {
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    if (block_scaled_only(plan)) return GEMM15_ERR_UNSUPPORTED;
    if (M < 0 || N < 0 || K < 0) return GEMM15_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM15_OK;
    if (!hD || (K > 0 && (!hA || !hB)) || (beta != 0.0f && !hC)) return GEMM15_ERR_INVALID_ARG;
    DeviceGuard g(plan->device);
    if (!g.ok) return GEMM15_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int es = esize_of(plan->desc.a), eo = esize_of(plan->desc.d);
    const size_t bytes[3] = {static_cast<size_t>(M * K * es), static_cast<size_t>(K * N * es),
                             static_cast<size_t>(M * N * eo)};
    // the plan's device state may still be in use by its previous call
    if (order_after_previous(plan, s) != GEMM15_OK) return GEMM15_ERR_CUDA;
    for (int i = 0; i < 3; ++i) {
        const size_t need = (bytes[i] + 255) & ~static_cast<size_t>(255);
        if (need > plan->host_path_cap[i]) {
            cudaFree(plan->d_host_path[i]);
            plan->d_host_path[i] = nullptr;
            plan->host_path_cap[i] = 0;
            if (cudaMalloc(&plan->d_host_path[i], std::max<size_t>(need, 256)) != cudaSuccess) {
                cudaGetLastError();
                return GEMM15_ERR_OOM;
            }
            plan->host_path_cap[i] = std::max<size_t>(need, 256);
        }
    }
    if (!plan->d_scales && cudaMalloc(&plan->d_scales, 2 * sizeof(float)) != cudaSuccess)
        return GEMM15_ERR_OOM;
    if (!plan->copy_stream) {
        if (cudaStreamCreateWithFlags(&plan->copy_stream, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&plan->fork_ev, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&plan->join_ev, cudaEventDisableTiming) != cudaSuccess)
            return GEMM15_ERR_CUDA;
    }
    void* dA = plan->d_host_path[0];
    void* dB = plan->d_host_path[1];
    void* dCD = plan->d_host_path[2];  // C is copied in and D overwrites it in place
    const bool a_row = plan->desc.layout_a == GEMM15_ROW_MAJOR;
    const bool b_row = plan->desc.layout_b == GEMM15_ROW_MAJOR;
    const bool cd_row = plan->desc.layout_cd == GEMM15_ROW_MAJOR;

    // Large row-major problems: a pipeline over column chunks of B, C and D.
    // The copy stream uploads A, then each chunk of B (and C) with a strided
    // copy; `stream` computes chunk k once its columns are up; a third stream
    // downloads chunk k of D while chunk k + 1 computes.  Four chunks of whole
    // 256-column tiles (the last takes the rest): a strided copy moves long rows
    // faster (on GB300 940 MB of B went up at 193 GB/s in 28 KB rows, 152 GB/s
    // in 14 KB rows), and the fill and drain of the pipeline grow with the chunk:
    // Llama-70B gate+up end to end 8.2 ms with four equal chunks, 8.7 with
    // eight, 9.3 with an eighth, two wide chunks and an eighth
    const bool pipeline = a_row && b_row && cd_row && K > 0 && N >= 4096 &&
                          bytes[1] + bytes[2] >= (static_cast<size_t>(64) << 20);
    if (pipeline && plan->elem != ELEM_E4M3) {
        if (!plan->d2h_stream) {
            if (cudaStreamCreateWithFlags(&plan->d2h_stream, cudaStreamNonBlocking) != cudaSuccess ||
                cudaEventCreateWithFlags(&plan->a_ev, cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&plan->d2h_ev, cudaEventDisableTiming) != cudaSuccess)
                return GEMM15_ERR_CUDA;
            for (int i = 0; i < 8; ++i)
                if (cudaEventCreateWithFlags(&plan->up_ev[i], cudaEventDisableTiming) != cudaSuccess ||
                    cudaEventCreateWithFlags(&plan->done_evs[i], cudaEventDisableTiming) != cudaSuccess)
                    return GEMM15_ERR_CUDA;
        }
        const int64_t T = cdiv(N, 256);
        const int64_t q = (T + 3) / 4 * 256;
        const int64_t widths[4] = {q, q, q, q};
        const size_t ea = static_cast<size_t>(es), ed = static_cast<size_t>(eo);
        if (cudaEventRecord(plan->fork_ev, s) != cudaSuccess ||
            cudaStreamWaitEvent(plan->copy_stream, plan->fork_ev, 0) != cudaSuccess ||
            cudaStreamWaitEvent(plan->d2h_stream, plan->fork_ev, 0) != cudaSuccess ||
            cudaMemcpyAsync(dA, hA, bytes[0], cudaMemcpyHostToDevice, plan->copy_stream) != cudaSuccess ||
            cudaEventRecord(plan->a_ev, plan->copy_stream) != cudaSuccess ||
            cudaStreamWaitEvent(s, plan->a_ev, 0) != cudaSuccess)
            return GEMM15_ERR_CUDA;
        int64_t n0 = 0;
        for (int nc = 0; nc < 4 && n0 < N; n0 += widths[nc], ++nc) {
            const int64_t cw = std::min<int64_t>(widths[nc], N - n0);
            auto colp = [&](const void* base, size_t e) {
                return static_cast<const uint8_t*>(base) + static_cast<size_t>(n0) * e;
            };
            if (cudaMemcpy2DAsync(const_cast<uint8_t*>(colp(dB, ea)), N * ea, colp(hB, ea), N * ea, cw * ea, K,
                                  cudaMemcpyHostToDevice, plan->copy_stream) != cudaSuccess)
                return GEMM15_ERR_CUDA;
            if (beta != 0.0f &&
                cudaMemcpy2DAsync(const_cast<uint8_t*>(colp(dCD, ed)), N * ed, colp(hC, ed), N * ed, cw * ed, M,
                                  cudaMemcpyHostToDevice, plan->copy_stream) != cudaSuccess)
                return GEMM15_ERR_CUDA;
            if (cudaEventRecord(plan->up_ev[nc], plan->copy_stream) != cudaSuccess ||
                cudaStreamWaitEvent(s, plan->up_ev[nc], 0) != cudaSuccess)
                return GEMM15_ERR_CUDA;
            void* dchunk = const_cast<uint8_t*>(colp(dCD, ed));
            Prob p = normalise(plan, M, cw, K, dA, K, colp(dB, ea), N, dchunk, N, dchunk, N);
            gemm15_status_t st = run_dense(plan, p, alpha, beta, nullptr, nullptr, s);
            if (st != GEMM15_OK) return st;
            if (cudaEventRecord(plan->done_evs[nc], s) != cudaSuccess ||
                cudaStreamWaitEvent(plan->d2h_stream, plan->done_evs[nc], 0) != cudaSuccess ||
                cudaMemcpy2DAsync(static_cast<uint8_t*>(hD) + static_cast<size_t>(n0) * ed, N * ed, dchunk,
                                  N * ed, cw * ed, M, cudaMemcpyDeviceToHost, plan->d2h_stream) != cudaSuccess)
                return GEMM15_ERR_CUDA;
        }
        if (cudaEventRecord(plan->d2h_ev, plan->d2h_stream) != cudaSuccess ||
            cudaStreamWaitEvent(s, plan->d2h_ev, 0) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return GEMM15_ERR_CUDA;
        int32_t status = 0;
        if (cudaMemcpy(&status, plan->d_status, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess)
            return GEMM15_ERR_CUDA;
        if (status != 0) {
            if (cudaMemset(plan->d_status, 0, sizeof(int32_t)) != cudaSuccess) return GEMM15_ERR_CUDA;
            if (status < 0 || status > GEMM15_ERR_BAD_PLAN) return GEMM15_ERR_DEVICE_FAULT;
        }
        return static_cast<gemm15_status_t>(status);
    }

    // B goes up on the plan's copy stream while A (and C) go up on `stream`
    if (K > 0) {
        if (cudaEventRecord(plan->fork_ev, s) != cudaSuccess ||
            cudaStreamWaitEvent(plan->copy_stream, plan->fork_ev, 0) != cudaSuccess ||
            cudaMemcpyAsync(dB, hB, bytes[1], cudaMemcpyHostToDevice, plan->copy_stream) != cudaSuccess ||
            cudaEventRecord(plan->join_ev, plan->copy_stream) != cudaSuccess ||
            cudaMemcpyAsync(dA, hA, bytes[0], cudaMemcpyHostToDevice, s) != cudaSuccess)
            return GEMM15_ERR_CUDA;
    }
    if (beta != 0.0f &&
        cudaMemcpyAsync(dCD, hC, bytes[2], cudaMemcpyHostToDevice, s) != cudaSuccess)
        return GEMM15_ERR_CUDA;
    if (K > 0 && cudaStreamWaitEvent(s, plan->join_ev, 0) != cudaSuccess) return GEMM15_ERR_CUDA;
    const float* sa = nullptr;
    const float* sb = nullptr;
    if (plan->elem == ELEM_E4M3) {
        float hs[2] = {scale_a, scale_b};
        // cudaMemcpyAsync from pageable memory completes the host read before returning
        if (cudaMemcpyAsync(plan->d_scales, hs, sizeof(hs), cudaMemcpyHostToDevice, s) != cudaSuccess)
            return GEMM15_ERR_CUDA;
        sa = plan->d_scales;
        sb = plan->d_scales + 1;
    }
    Prob p = normalise(plan, M, N, K, dA, a_row ? K : M, dB, b_row ? N : K, dCD, cd_row ? N : M,
                       dCD, cd_row ? N : M);
    gemm15_status_t st = run_dense(plan, p, alpha, beta, sa, sb, s);
    if (st != GEMM15_OK) return st;
    if (cudaMemcpyAsync(hD, dCD, bytes[2], cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return GEMM15_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GEMM15_ERR_CUDA;
    // read and clear the status word, as gemm_plan_query_error does
    int32_t status = 0;
    if (cudaMemcpy(&status, plan->d_status, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM15_ERR_CUDA;
    if (status != 0) {
        if (cudaMemset(plan->d_status, 0, sizeof(int32_t)) != cudaSuccess) return GEMM15_ERR_CUDA;
        if (status < 0 || status > GEMM15_ERR_BAD_PLAN) return GEMM15_ERR_DEVICE_FAULT;
    }
    return static_cast<gemm15_status_t>(status);
}

gemm15_status_t grouped_gemm_run(gemm15_plan_t plan, const gemm15_problem_t* problems,
                                 int32_t count, float alpha, float beta, void* stream) {
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    if (count < 0 || (count > 0 && !problems)) return GEMM15_ERR_INVALID_ARG;
    if (block_scaled_only(plan)) return GEMM15_ERR_UNSUPPORTED;
    DeviceGuard g(plan->device);
    if (!g.ok) return GEMM15_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool has_c = beta != 0.0f;
    const bool a_row = plan->desc.layout_a == GEMM15_ROW_MAJOR;
    const bool b_row = plan->desc.layout_b == GEMM15_ROW_MAJOR;
    const bool cd_row = plan->desc.layout_cd == GEMM15_ROW_MAJOR;
    const int bn = plan->opt.tile_n ? plan->opt.tile_n : 256;
    const int bk = plan->elem == ELEM_E4M3 ? 128 : 64;

    // validate every group first: nothing is launched on an argument error
    std::vector<Prob> probs;
    std::vector<const gemm15_problem_t*> src;  // the problem each entry of probs came from
    probs.reserve(count);
    src.reserve(count);
    for (int32_t i = 0; i < count; ++i) {
        const gemm15_problem_t& q = problems[i];
        if (q.M < 0 || q.N < 0 || q.K < 0) return GEMM15_ERR_INVALID_ARG;
        if ((q.scale_a || q.scale_b) && plan->elem != ELEM_E4M3) return GEMM15_ERR_INVALID_ARG;
        if (q.M == 0 || q.N == 0) continue;
        if (q.K == 0) return GEMM15_ERR_UNSUPPORTED;
        const int64_t lda = q.lda ? q.lda : (a_row ? q.K : q.M);
        const int64_t ldb = q.ldb ? q.ldb : (b_row ? q.N : q.K);
        const int64_t ldc = q.ldc ? q.ldc : (cd_row ? q.N : q.M);
        const int64_t ldd = q.ldd ? q.ldd : (cd_row ? q.N : q.M);
        Prob p = normalise(plan, q.M, q.N, q.K, q.A, lda, q.B, ldb, q.C, ldc, q.D, ldd);
        gemm15_status_t st = check_operands(plan, p, beta);
        if (st != GEMM15_OK) return st;
        probs.push_back(p);
        src.push_back(&q);
    }
    const int ng = static_cast<int>(probs.size());
    if (ng == 0) {
        std::memset(&plan->last, 0, sizeof(plan->last));
        return GEMM15_OK;
    }
    const int G1 = plan->opt.grid > 0 ? std::min(plan->opt.grid, plan->num_sms) : plan->num_sms;
    // SM-pair tiles when the groups fill a wave of them and rounding each group's
    // rows up to 256 instead of 128 adds at most ~15% rows
    int cg = 1;
    const int clusters = std::min(pair_clusters(plan), G1 / 2);
    const bool pair_ok = bn == 256 || plan->elem != ELEM_E4M3;
    if (clusters > 0 && pair_ok && plan->opt.cta_group != 1) {
        int64_t tiles2 = 0, rows1 = 0, rows2 = 0;
        for (const Prob& p : probs) {
            tiles2 += cdiv(p.M, 2 * TILE_M) * cdiv(p.N, bn);
            rows1 += cdiv(p.M, TILE_M) * TILE_M;
            rows2 += cdiv(p.M, 2 * TILE_M) * 2 * TILE_M;
        }
        if (plan->opt.cta_group == 2 ||
            (bn == 256 && tiles2 >= clusters && rows2 * 100 <= rows1 * 115))
            cg = 2;
    }
    const int G = cg == 2 ? clusters : G1;  // scheduling units
    if (order_after_previous(plan, s) != GEMM15_OK) return GEMM15_ERR_CUDA;
    int32_t tiles = 0;
    const bool reuse = plan->d_groups && plan->groups_ng == ng && plan->groups_key_c == has_c &&
                       plan->groups_key_bn == bn && plan->groups_key_raster == plan->opt.raster &&
                       plan->groups_key_cg == cg &&
                       plan->groups_key.size() == static_cast<size_t>(count) &&
                       std::memcmp(plan->groups_key.data(), problems,
                                   sizeof(gemm15_problem_t) * static_cast<size_t>(count)) == 0;
    if (reuse) {
        tiles = plan->groups_tiles;
        // the copy that wrote the table may have been enqueued on another stream
        if (cudaStreamWaitEvent(s, plan->groups_done, 0) != cudaSuccess) return GEMM15_ERR_CUDA;
    } else {
        plan->groups_key.clear();  // the table is about to change
        plan->groups_ng = 0;
        if (ng > plan->groups_cap) {
            if (plan->groups_done) cudaEventSynchronize(plan->groups_done);
            cudaFree(plan->d_groups);
            if (plan->h_groups) cudaFreeHost(plan->h_groups);
            plan->d_groups = nullptr;
            plan->h_groups = nullptr;
            plan->groups_cap = 0;
            const int cap = std::max(ng, 64);
            if (cudaMalloc(&plan->d_groups, cap * sizeof(GroupEntry)) != cudaSuccess ||
                cudaMallocHost(&plan->h_groups, cap * sizeof(GroupEntry)) != cudaSuccess) {
                cudaGetLastError();
                return GEMM15_ERR_OOM;
            }
            plan->groups_cap = cap;
        }
        if (!plan->groups_done &&
            cudaEventCreateWithFlags(&plan->groups_done, cudaEventDisableTiming) != cudaSuccess)
            return GEMM15_ERR_CUDA;
        // the previous grouped call's copy must have read the staging buffer
        if (cudaEventSynchronize(plan->groups_done) != cudaSuccess) return GEMM15_ERR_CUDA;

        bool mixed_layout = false;
        for (int i = 0; i < ng; ++i) {
            const Prob& p = probs[i];
            if (p.a_kmajor != probs[0].a_kmajor || p.b_kmajor != probs[0].b_kmajor) mixed_layout = true;
            GroupEntry& e = plan->h_groups[i];
            std::memset(&e, 0, sizeof(e));
            if (!operand_maps(plan, p, bn / cg, &e.tmA, &e.tmB)) return GEMM15_ERR_CUDA;
            if (!output_maps(plan, p, has_c, &e.tmC, &e.tmD)) return GEMM15_ERR_CUDA;
            e.M = static_cast<int32_t>(p.M);
            e.N = static_cast<int32_t>(p.N);
            e.K = static_cast<int32_t>(p.K);
            e.k_blocks = static_cast<int32_t>(cdiv(p.K, bk));
            e.m_blocks = static_cast<int32_t>(cdiv(p.M, TILE_M * cg));
            e.n_blocks = static_cast<int32_t>(cdiv(p.N, bn));
            e.tile_start = tiles;
            e.has_c = has_c;
            e.D = p.D;
            e.ldd = p.ldd;
            e.C = has_c ? p.C : nullptr;
            e.ldc = p.ldc;
            // (s_a * s_b is symmetric: a group computed as D^T = B^T A^T keeps both)
            e.scale_a = src[i]->scale_a;
            e.scale_b = src[i]->scale_b;
            e.raster = plan->opt.raster > 0 ? std::min<int32_t>(plan->opt.raster, e.m_blocks)
                                            : std::min<int32_t>(e.m_blocks, cg == 2 ? 8 : 16);
            const int64_t t = static_cast<int64_t>(e.m_blocks) * e.n_blocks;
            if (tiles + t > (1ll << 30)) return GEMM15_ERR_INVALID_ARG;
            tiles += static_cast<int32_t>(t);
        }
        if (mixed_layout) return GEMM15_ERR_UNSUPPORTED;  // normalisation is per plan: cannot happen
        if (cudaMemcpyAsync(plan->d_groups, plan->h_groups, ng * sizeof(GroupEntry),
                            cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaEventRecord(plan->groups_done, s) != cudaSuccess)
            return GEMM15_ERR_CUDA;
        plan->groups_key.assign(problems, problems + count);
        plan->groups_key_c = has_c;
        plan->groups_key_bn = bn;
        plan->groups_key_raster = plan->opt.raster;
        plan->groups_key_cg = cg;
        plan->groups_tiles = tiles;
        plan->groups_ng = ng;
    }

    GemmParams gp;
    std::memset(&gp, 0, sizeof(gp));
    gp.tiles = tiles;
    gp.sched = SCHED_DP;
    gp.splits = 1;
    gp.k_blocks = 0;
    gp.alpha = alpha;
    gp.beta = beta;
    gp.act = static_cast<int>(plan->desc.epilogue);
    gp.has_c = has_c;
    fill_layout(plan, gp, probs[0].a_kmajor, probs[0].b_kmajor, bn, cg);
    gp.ws = plan->d_ws;
    gp.flags = plan->d_flags;
    gp.status = plan->d_status;
    gp.epoch = ++plan->epoch == 0 ? ++plan->epoch : plan->epoch;
    gp.timeout_ns = static_cast<uint64_t>(plan->opt.timeout_us) * 1000ull;
    gp.fault_skip_flag = -1;
    gp.groups = plan->d_groups;
    gp.num_groups = ng;
    const int grid = std::min(G, tiles) * cg;
    set_sched_divisors(gp, grid / cg);
    {
        gemm15_status_t tst = attach_trace(plan, gp, grid, s);
        if (tst != GEMM15_OK) return tst;
    }
    if (launch_kernel(plan->elem, bn, cg, gp, grid, s) != cudaSuccess) return GEMM15_ERR_CUDA;
    Decision d;
    d.bn = bn;
    d.bk = bk;
    d.cg = cg;
    d.sched = SCHED_DP;
    d.grid = grid;
    d.tiles = tiles;
    d.raster = cg == 2 ? 8 : 16;
    record_config(plan, d, 1);
    return mark_done(plan, s);
}

gemm15_status_t gemm_run_batched(gemm15_plan_t plan, const void* A, int64_t lda, int64_t stride_a,
                                 const void* B, int64_t ldb, int64_t stride_b, const void* C,
                                 int64_t ldc, int64_t stride_c, void* D, int64_t ldd,
                                 int64_t stride_d, int64_t M, int64_t N, int64_t K,
                                 int32_t batch, float alpha, float beta, void* stream) {
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    if (batch < 0 || stride_a < 0 || stride_b < 0 || stride_c < 0 || stride_d < 0)
        return GEMM15_ERR_INVALID_ARG;
    if (batch == 0 || M == 0 || N == 0) {
        std::memset(&plan->last, 0, sizeof(plan->last));
        return (M < 0 || N < 0 || K < 0) ? GEMM15_ERR_INVALID_ARG : GEMM15_OK;
    }
    const int64_t ea = plan->elem == ELEM_E4M3 ? 1 : 2;
    const int64_t ec = 2;  // C and D are 16-bit
    if ((stride_a * ea) % 16 || (stride_b * ea) % 16 || (stride_c * ec) % 16 || (stride_d * ec) % 16)
        return GEMM15_ERR_ALIGNMENT;
    std::vector<gemm15_problem_t> probs(static_cast<size_t>(batch));
    for (int32_t b = 0; b < batch; ++b) {
        gemm15_problem_t& q = probs[b];
        q.M = M;
        q.N = N;
        q.K = K;
        q.A = static_cast<const uint8_t*>(A) + b * stride_a * ea;
        q.B = static_cast<const uint8_t*>(B) + b * stride_b * ea;
        q.C = C ? static_cast<const uint8_t*>(C) + b * stride_c * ec : nullptr;
        q.D = static_cast<uint8_t*>(D) + b * stride_d * ec;
        q.lda = lda;
        q.ldb = ldb;
        q.ldc = ldc;
        q.ldd = ldd;
    }
    return grouped_gemm_run(plan, probs.data(), batch, alpha, beta, stream);
}

gemm15_status_t gemm_run_block_scaled(gemm15_plan_t plan, const gemm15_scaled_args_t* a,
                                      void* stream) {
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    if (!a) return GEMM15_ERR_INVALID_ARG;
    int sf = -1;
    if (plan->elem == ELEM_E4M3 || plan->elem == ELEM_E5M2) {
        if (a->scale_kind == GEMM15_SCALE_MX) sf = SF_MXF8;
    } else if (plan->elem == ELEM_E2M1) {
        if (a->scale_kind == GEMM15_SCALE_MX) sf = SF_MXF4;
        else if (a->scale_kind == GEMM15_SCALE_NV) sf = SF_NVF4;
    }
    if (a->scale_kind != GEMM15_SCALE_MX && a->scale_kind != GEMM15_SCALE_NV) return GEMM15_ERR_INVALID_ARG;
    if (sf < 0) return GEMM15_ERR_UNSUPPORTED;
    if (plan->desc.layout_a != GEMM15_ROW_MAJOR || plan->desc.layout_b != GEMM15_COL_MAJOR ||
        plan->desc.layout_cd != GEMM15_ROW_MAJOR)
        return GEMM15_ERR_UNSUPPORTED;
    const int64_t M = a->M, N = a->N, K = a->K;
    if (M < 0 || N < 0 || K < 0) return GEMM15_ERR_INVALID_ARG;
    if (M > (1ll << 31) - 256 || N > (1ll << 31) - 256 || K > (1ll << 31) - 256)
        return GEMM15_ERR_INVALID_ARG;
    if (M == 0 || N == 0) {
        std::memset(&plan->last, 0, sizeof(plan->last));
        return GEMM15_OK;
    }
    const bool fp4 = plan->elem == ELEM_E2M1;
    const int64_t bk = fp4 ? 256 : 128;  // elements of one 128-byte k-block
    if (K == 0 || K % bk) return GEMM15_ERR_UNSUPPORTED;
    const int64_t block = sf == SF_NVF4 ? 16 : 32;
    const int64_t lda = a->lda ? a->lda : K, ldb = a->ldb ? a->ldb : K;
    const int64_t ldd = a->ldd ? a->ldd : N, ldc = a->ldc ? a->ldc : N;
    const bool has_c = a->beta != 0.0f;
    if (!a->A || !a->B || !a->SFA || !a->SFB || !a->D || (has_c && !a->C)) return GEMM15_ERR_INVALID_ARG;
    if (lda < K || ldb < K || ldd < N || (has_c && ldc < N)) return GEMM15_ERR_INVALID_ARG;
    if (fp4 && (lda % 2 || ldb % 2)) return GEMM15_ERR_ALIGNMENT;
    const int64_t lda_b = fp4 ? lda / 2 : lda, ldb_b = fp4 ? ldb / 2 : ldb;  // bytes
    if (!aligned16(a->A) || !aligned16(a->B) || !aligned16(a->SFA) || !aligned16(a->SFB) ||
        !aligned16(a->D) || (has_c && !aligned16(a->C)) || (a->bias && !aligned16(a->bias)))
        return GEMM15_ERR_ALIGNMENT;
    if (lda_b % 16 || ldb_b % 16 || (ldd * 2) % 16 || (has_c && (ldc * 2) % 16))
        return GEMM15_ERR_ALIGNMENT;
    DeviceGuard g(plan->device);
    if (!g.ok) return GEMM15_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (order_after_previous(plan, s) != GEMM15_OK) return GEMM15_ERR_CUDA;

    // tile width: 256 columns (one accumulator per CTA) by default; 128-wide
    // tiles keep two accumulators but measured slower on GB300 (one SM, MXFP8
    // 8192^3: 686 against 531 us, NVFP4 508 against 381; SM pairs: MXFP8 755
    // against 484 us)
    const int BN = plan->opt.tile_n == 128 ? 128 : 256;
    const int G = plan->opt.grid > 0 ? std::min(plan->opt.grid, plan->num_sms) : plan->num_sms;
    // SM-pair 256 x 256 tiles (each CTA stages its 128 rows of A and 128 columns
    // of B, and all of B's scale atoms) for MXFP8, or when asked for; the fp4
    // kinds stay on one-SM tiles, where each CTA copies half as many scale
    // atoms per k-block (measured on GB300, 8192^3: MXFP8 484 us on pairs
    // against 514; MXFP4 306 against 320, NVFP4 377 against 405 on one SM)
    const int clusters = std::min(pair_clusters(plan), G / 2);
    const bool want_pair = plan->opt.cta_group == 2 || (plan->opt.cta_group == 0 && sf == SF_MXF8);
    const int cg = (clusters > 0 && want_pair && (BN == 256 || plan->opt.cta_group == 2)) ? 2 : 1;
    Decision d;
    d.cg = cg;
    d.bn = BN;
    d.bk = static_cast<int>(bk);
    d.sched = SCHED_DP;
    d.m_blocks = static_cast<int32_t>(cdiv(M, TILE_M * cg));
    d.n_blocks = static_cast<int32_t>(cdiv(N, BN));
    d.tiles = d.m_blocks * d.n_blocks;
    d.k_blocks = static_cast<int32_t>(K / bk);
    d.grid = cg == 2 ? 2 * static_cast<int>(std::min<int64_t>(clusters, d.tiles))
                     : static_cast<int>(std::min<int64_t>(G, d.tiles));
    d.raster = plan->opt.raster > 0 ? std::min<int32_t>(plan->opt.raster, d.m_blocks)
                                    : std::min<int32_t>(d.m_blocks, cg == 2 ? 8 : 16);

    GemmParams gp;
    std::memset(&gp, 0, sizeof(gp));
    // operands as bytes: 128-byte boxes of K, 128 rows of A and 256 of B
    const uint64_t kbytes = static_cast<uint64_t>(fp4 ? K / 2 : K);
    bool ok = make_tmap(&gp.tmA, ELEM_E4M3, a->A, kbytes, M, lda_b, 128, TILE_M);
    ok = ok && make_tmap(&gp.tmB, ELEM_E4M3, a->B, kbytes, N, ldb_b, 128, BN / cg);
    // scale atoms as rows of 128 bytes (4 per atom), no swizzle: a box of one
    // k-block's atoms (1, 2 or 4) lands in shared memory byte for byte
    const int apk = sf == SF_MXF8 ? 1 : sf == SF_MXF4 ? 2 : 4;
    const int64_t cb = K / block / 4;  // atoms per 128-row block
    ok = ok && make_tmap(&gp.tmSFA, ELEM_E4M3, a->SFA, 128, static_cast<uint64_t>(cdiv(M, TILE_M) * cb * 4),
                         128, 128, static_cast<uint32_t>(4 * apk), false);
    ok = ok && make_tmap(&gp.tmSFB, ELEM_E4M3, a->SFB, 128, static_cast<uint64_t>(cdiv(N, TILE_M) * cb * 4),
                         128, 128, static_cast<uint32_t>(4 * apk), false);
    Prob po{};
    po.M = M;
    po.N = N;
    po.D = a->D;
    po.ldd = ldd;
    po.C = a->C;
    po.ldc = ldc;
    ok = ok && output_maps(plan, po, has_c, &gp.tmC, &gp.tmD);
    if (!ok) return GEMM15_ERR_CUDA;
    gp.D = a->D;
    gp.ldd = ldd;
    gp.C = has_c ? a->C : nullptr;
    gp.ldc = ldc;
    gp.M = static_cast<int32_t>(M);
    gp.N = static_cast<int32_t>(N);
    gp.K = static_cast<int32_t>(K);
    gp.k_blocks = d.k_blocks;
    gp.m_blocks = d.m_blocks;
    gp.n_blocks = d.n_blocks;
    gp.tiles = d.tiles;
    gp.raster = d.raster;
    gp.sched = SCHED_DP;
    gp.splits = 1;
    gp.has_c = has_c;
    gp.alpha = a->alpha;
    gp.beta = a->beta;
    gp.act = static_cast<int>(plan->desc.epilogue);
    gp.bias = a->bias;
    gp.sf_cb = static_cast<int32_t>(cb);
    set_sched_divisors(gp, d.grid / cg);
    gp.a_kmajor = gp.b_kmajor = 1;
    gp.a_lbo = gp.b_lbo = 16;
    gp.a_sbo = gp.b_sbo = 1024;
    gp.a_kstep = gp.b_kstep = 32;
    // instruction descriptor of the block-scaled kinds: A / B format (E4M3 0,
    // E5M2 1; E2M1 1 for the fp4 kinds), K-major operands, N >> 3, scale
    // format (bit 23: 1 UE8M0, 0 UE4M3), M >> 4; the scale-factor IDs (bits
    // 29-30 and 4-5) are set per MMA by the kernel
    const uint32_t fmt = plan->elem == ELEM_E4M3 ? 0u : 1u;
    gp.idesc = (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
               ((sf == SF_NVF4 ? 0u : 1u) << 23) | (static_cast<uint32_t>((TILE_M * cg) >> 4) << 24);
    gp.ws = plan->d_ws;
    gp.flags = plan->d_flags;
    gp.status = plan->d_status;
    gp.epoch = ++plan->epoch == 0 ? ++plan->epoch : plan->epoch;
    gp.timeout_ns = static_cast<uint64_t>(plan->opt.timeout_us) * 1000ull;
    gp.fault_skip_flag = -1;
    gemm15_status_t st = attach_trace(plan, gp, d.grid, s);
    if (st != GEMM15_OK) return st;
    cudaError_t e;
    if (cg == 2 && BN == 128) {
        if (sf == SF_MXF8)
            e = plan->elem == ELEM_E4M3 ? launch_gemm<ELEM_E4M3, 128, 2, SF_MXF8>(gp, d.grid, s)
                                        : launch_gemm<ELEM_E5M2, 128, 2, SF_MXF8>(gp, d.grid, s);
        else if (sf == SF_MXF4)
            e = launch_gemm<ELEM_E2M1, 128, 2, SF_MXF4>(gp, d.grid, s);
        else
            e = launch_gemm<ELEM_E2M1, 128, 2, SF_NVF4>(gp, d.grid, s);
    } else if (cg == 2) {
        if (sf == SF_MXF8)
            e = plan->elem == ELEM_E4M3 ? launch_gemm<ELEM_E4M3, 256, 2, SF_MXF8>(gp, d.grid, s)
                                        : launch_gemm<ELEM_E5M2, 256, 2, SF_MXF8>(gp, d.grid, s);
        else if (sf == SF_MXF4)
            e = launch_gemm<ELEM_E2M1, 256, 2, SF_MXF4>(gp, d.grid, s);
        else
            e = launch_gemm<ELEM_E2M1, 256, 2, SF_NVF4>(gp, d.grid, s);
    } else if (BN == 256) {
        if (sf == SF_MXF8)
            e = plan->elem == ELEM_E4M3 ? launch_gemm<ELEM_E4M3, 256, 1, SF_MXF8>(gp, d.grid, s)
                                        : launch_gemm<ELEM_E5M2, 256, 1, SF_MXF8>(gp, d.grid, s);
        else if (sf == SF_MXF4)
            e = launch_gemm<ELEM_E2M1, 256, 1, SF_MXF4>(gp, d.grid, s);
        else
            e = launch_gemm<ELEM_E2M1, 256, 1, SF_NVF4>(gp, d.grid, s);
    } else {
        if (sf == SF_MXF8)
            e = plan->elem == ELEM_E4M3 ? launch_gemm<ELEM_E4M3, 128, 1, SF_MXF8>(gp, d.grid, s)
                                        : launch_gemm<ELEM_E5M2, 128, 1, SF_MXF8>(gp, d.grid, s);
        else if (sf == SF_MXF4)
            e = launch_gemm<ELEM_E2M1, 128, 1, SF_MXF4>(gp, d.grid, s);
        else
            e = launch_gemm<ELEM_E2M1, 128, 1, SF_NVF4>(gp, d.grid, s);
    }
    if (e != cudaSuccess) return GEMM15_ERR_CUDA;
    record_config(plan, d, 1);
    plan->last.stages = gemm_scaled_stages(sf, BN, cg);
    return mark_done(plan, s);
}

gemm15_status_t gemm_plan_query_error(gemm15_plan_t plan) {
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    DeviceGuard g(plan->device);
    if (!g.ok) return GEMM15_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return GEMM15_ERR_CUDA;
    int32_t status = 0;
    if (cudaMemcpy(&status, plan->d_status, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM15_ERR_CUDA;
    if (status != 0 && cudaMemset(plan->d_status, 0, sizeof(int32_t)) != cudaSuccess)
        return GEMM15_ERR_CUDA;
    if (status < 0 || status > GEMM15_ERR_BAD_PLAN) return GEMM15_ERR_DEVICE_FAULT;
    return static_cast<gemm15_status_t>(status);
}

gemm15_status_t gemm_plan_set_option(gemm15_plan_t plan, gemm15_option_t option, int64_t v) {
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    Options& o = plan->opt;
    switch (option) {
        case GEMM15_OPT_SCHEDULE:
            if (v < 0 || v > 3) return GEMM15_ERR_INVALID_ARG;
            o.schedule = static_cast<int>(v);
            return GEMM15_OK;
        case GEMM15_OPT_SPLITS:
            if (v < -1 || v > 4096) return GEMM15_ERR_INVALID_ARG;
            o.splits = static_cast<int>(v);
            return GEMM15_OK;
        case GEMM15_OPT_CTA_GROUP:
            if (v != 0 && v != 1 && v != 2) return GEMM15_ERR_INVALID_ARG;
            o.cta_group = static_cast<int>(v);
            return GEMM15_OK;
        case GEMM15_OPT_TILE_N:
            if (v != 0 && v != 128 && v != 256) return GEMM15_ERR_INVALID_ARG;
            o.tile_n = static_cast<int>(v);
            return GEMM15_OK;
        case GEMM15_OPT_RASTER:
            if (v < 0 || v > 4096) return GEMM15_ERR_INVALID_ARG;
            o.raster = static_cast<int>(v);
            return GEMM15_OK;
        case GEMM15_OPT_GRID:
            if (v < 0 || v > 100000) return GEMM15_ERR_INVALID_ARG;
            o.grid = static_cast<int>(v);
            return GEMM15_OK;
        case GEMM15_OPT_TIMEOUT_US:
            if (v < 1000 || v > 60000000) return GEMM15_ERR_INVALID_ARG;
            o.timeout_us = v;
            return GEMM15_OK;
        case GEMM15_OPT_SK_DP_WAVES:
            if (v < -1 || v > 100000) return GEMM15_ERR_INVALID_ARG;
            o.sk_dp_waves = static_cast<int>(v);
            return GEMM15_OK;
        case GEMM15_OPT_TRACE_ITEMS:
            if (v < 0 || v > 65536) return GEMM15_ERR_INVALID_ARG;
            o.trace_items = static_cast<int>(v);
            return GEMM15_OK;
        case GEMM15_OPT_SWAP_AB:
            if (v < 0 || v > 2) return GEMM15_ERR_INVALID_ARG;
            o.swap_ab = static_cast<int>(v);
            return GEMM15_OK;
        case GEMM15_OPT_SPLITK_INLINE:
            if (v < 0 || v > 2) return GEMM15_ERR_INVALID_ARG;
            o.splitk_inline = static_cast<int>(v);
            return GEMM15_OK;
        case GEMM15_OPT_L2_HINTS:
            if (v < 0 || v > 2) return GEMM15_ERR_INVALID_ARG;
            o.l2_hints = static_cast<int>(v);
            return GEMM15_OK;
        case GEMM15_OPT_FAULT_SKIP_FLAG:
            if (v < -1 || v > 100000) return GEMM15_ERR_INVALID_ARG;
            o.fault_skip_flag = static_cast<int>(v);
            return GEMM15_OK;
    }
    return GEMM15_ERR_INVALID_ARG;
}

gemm15_status_t gemm_plan_trace(gemm15_plan_t plan, void* out, int64_t capacity, int32_t* ctas,
                                int32_t* items) {
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    if (ctas) *ctas = plan->trace_ctas;
    if (items) *items = plan->opt.trace_items;
    if (!plan->d_trace || plan->opt.trace_items <= 0 || !out) return GEMM15_ERR_INVALID_ARG;
    const size_t bytes =
        static_cast<size_t>(plan->trace_ctas) * (plan->opt.trace_items + 1) * TRACE_WORDS * 8;
    if (capacity < 0 || static_cast<size_t>(capacity) < bytes || bytes > plan->trace_cap)
        return GEMM15_ERR_INVALID_ARG;
    DeviceGuard g(plan->device);
    if (!g.ok) return GEMM15_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return GEMM15_ERR_CUDA;
    if (cudaMemcpy(out, plan->d_trace, bytes, cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM15_ERR_CUDA;
    return GEMM15_OK;
}

gemm15_status_t gemm_plan_last_config(gemm15_plan_t plan, gemm15_config_t* out) {
    if (!plan_ok(plan)) return GEMM15_ERR_BAD_PLAN;
    if (!out) return GEMM15_ERR_INVALID_ARG;
    *out = plan->last;
    return GEMM15_OK;
}

}  // extern "C"
