// Kernel parameter blocks shared by the host planner and the sm_103a kernels.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace g15 {

enum ElemKind : int { ELEM_F16 = 0, ELEM_BF16 = 1, ELEM_E4M3 = 2, ELEM_E5M2 = 3, ELEM_E2M1 = 4 };
// block-scaled MMA kinds (tcgen05 .block_scale): scale factors per 32 or 16 K
enum ScaleKind : int {
    SF_NONE = 0,
    SF_MXF8 = 1,   // kind::mxf8f6f4, UE8M0 per 32, scale_vec::1X (E4M3 / E5M2 elements)
    SF_MXF4 = 2,   // kind::mxf4, UE8M0 per 32, scale_vec::2X (packed E2M1)
    SF_NVF4 = 3    // kind::mxf4nvf4, UE4M3 per 16, scale_vec::4X (packed E2M1)
};
enum Schedule : int { SCHED_DP = 1, SCHED_SK = 2, SCHED_SPLIT = 3 };
enum DeviceError : int { DEV_ERR_TIMEOUT = 5, DEV_ERR_FAULT = 7 };
// epilogue activation (values of gemm15_epilogue_t)
enum Activation : int { ACT_NONE = 0, ACT_RELU = 1, ACT_SIGMOID = 2, ACT_TANH = 3 };

constexpr int TILE_M = 128;         // rows of A per CTA (UMMA M for one SM)
constexpr int EPI_WARPS = 4;        // epilogue warps (one per 32-lane TMEM quarter)
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;  // warp 0 TMA, warp 1 MMA, then epilogue
constexpr int EPI_COLS = 64;        // output columns per epilogue chunk (128 B of 16-bit)
constexpr int EPI_BUF_BYTES = 32 * 128;  // one 32-row x 128-byte epilogue staging box
constexpr int REDUCE_COLS = 4;      // split-K reduction: output columns per element
constexpr int REDUCE_MAX_GROUPS = 8; // split-K reduction: warps (split groups) per block

// Division by a launch constant d (1 <= d) of dividends 0 <= n < 2^31 as a
// multiply and a shift: q = (n * mul) >> shift, shift = 31 + ceil(log2 d),
// mul = ceil(2^shift / d) (Granlund and Montgomery, "Division by invariant
// integers using multiplication").  With mul = 2^shift / d + e, 0 <= e < 1,
// the error n * e / 2^shift stays below 2^-ceil(log2 d) <= 1/d, which is not
// enough to reach the next integer above n / d: the floor is exact.  mul <=
// 2^32, so n * mul < 2^63.  Larger dividends fall back to a division by d.
struct FastDiv {
    uint64_t mul;
    int64_t d;
    uint32_t shift;
    uint32_t pad;
};

inline FastDiv make_fastdiv(int64_t d) {
    FastDiv f{};
    if (d < 1) d = 1;
    f.d = d;
    uint32_t l = 0;
    while ((int64_t{1} << l) < d) ++l;  // ceil(log2 d)
    f.shift = 31 + l;
    if (f.shift < 63) f.mul = ((uint64_t{1} << f.shift) + static_cast<uint64_t>(d) - 1) / static_cast<uint64_t>(d);
    return f;  // d >= 2^32: every dividend takes the fallback
}

// One group of a grouped GEMM as the kernel reads it from device memory.
struct alignas(128) GroupEntry {
    CUtensorMap tmA, tmB, tmC, tmD;
    int32_t M, N, K, k_blocks;
    int32_t m_blocks, n_blocks, tile_start, has_c;
    int32_t raster, pad0;
    void* D;                          // for the ragged last column chunk
    int64_t ldd;
    const void* C;                    // read directly by the epilogue
    int64_t ldc;
    const float* scale_a;             // fp8 per-tensor scales of A_g / B_g (device), or null
    const float* scale_b;
};

struct GemmParams {
    CUtensorMap tmA, tmB, tmC, tmD;  // dense problem (unused when grouped)
    void* D;                          // D and its leading dimension (elements), for
    int64_t ldd;                      // column chunks the TMA store cannot clip exactly
    const void* C;                    // C and its leading dimension (elements); the
    int64_t ldc;                      // epilogue reads C straight into registers
    int32_t M, N, K;
    int32_t k_blocks;                 // ceil(K / BK)
    int32_t m_blocks, n_blocks, tiles;
    int32_t raster;                   // M-blocks per raster band
    int32_t sched;                    // Schedule
    int32_t dp_tiles;                 // SK: tiles done whole before the stream-K region
    int32_t splits;                   // SPLIT: k-splits per tile
    int32_t has_c;                    // beta != 0 (C is read)
    int64_t sk_units;                 // SK: (tiles - dp_tiles) * k_blocks
    // the scheduler's divisors: scheduling units (CTAs or SM pairs), k_blocks,
    // sk_units, raster * n_blocks, raster, the last raster band's M-blocks, splits
    FastDiv fd_units, fd_kb, fd_sk, fd_band, fd_raster, fd_last, fd_splits;
    int32_t sk_partials_only;         // SK partition whose every piece leaves a partial tile
                                      // for the reduction kernel (balanced split-K)
    int32_t l2_hints;                 // operand loads: 0 default, 1 A evict-last, 2 A
                                      // evict-last and B evict-first
    int32_t splitk_inline;            // SPLIT: the split that finishes a tile last adds the
                                      // partials and writes it (no reduction kernel); the
                                      // arrival counters are 64-bit words in `flags`
    float alpha, beta;
    const float* scale_a;             // fp8 per-tensor scales (device), or null
    const float* scale_b;
    int32_t act;                      // Activation
    int32_t bias_rows;                // bias indexed by output row (1) or column (0)
    const void* bias;                 // 16-bit bias vector (device), or null
    const void* aux;                  // auxiliary tensor Z (output type, row-major), or null
    int64_t ldaux;
    int32_t aux_op;                   // 0 none, 1 add, 2 sub, 3 mul, 4 div
    void* pre;                        // pre-activation output Y (output type, layout of D),
    int64_t ldpre;                    // or null
    int32_t out_trans;                // 1: the computed tile is the transpose of the stored
                                      // one (swap-AB): element (r, c) of the computed output
                                      // lives at C / D / Z + c * ld + r
    int32_t out_tma;                  // out_trans: tmD maps the stored D transposed (inner
                                      // dimension = computed rows, 32 x 64 boxes, no swizzle)
    // block-scaled operands: scale factors in the 128 x 4 atom layout (512-byte
    // atoms, one per 128 rows and 4 consecutive scales along K; atom (rb, cb)
    // at (rb * sf_cb + cb) * 512), read through 2-D tensor maps of 128-byte
    // rows (an atom is 4 rows)
    CUtensorMap tmSFA, tmSFB;
    int32_t sf_cb;
    // operand layouts in shared memory (bytes) and the MMA instruction descriptor
    uint32_t a_kmajor, b_kmajor;
    uint32_t a_lbo, a_sbo, a_kstep;
    uint32_t b_lbo, b_sbo, b_kstep;
    uint32_t idesc;
    // workspace and status
    float* ws;                        // fp32 partial tiles
    uint32_t* flags;                  // SK partial-ready flags, two per CTA (tail, head piece)
    int32_t* status;                  // device status word (0 = ok)
    uint32_t epoch;                   // launch sequence number (flag value)
    uint64_t timeout_ns;              // bound of every wait
    int32_t fault_skip_flag;          // test hook (-1 = off)
    // grouped problems (device table) or null
    const GroupEntry* groups;
    int32_t num_groups;
    // optional timeline: per CTA a header record then one record per work
    // item, TRACE_WORDS 64-bit words each (null = off)
    uint64_t* trace;
    int32_t trace_items;
};

// Sets the scheduler's divisors from the schedule fields and the number of
// scheduling units the launch has (grid / CTAs per tile).
inline void set_sched_divisors(GemmParams& gp, int32_t units) {
    gp.fd_units = make_fastdiv(units);
    gp.fd_kb = make_fastdiv(gp.k_blocks);
    gp.fd_sk = make_fastdiv(gp.sk_units);
    const int32_t raster = gp.raster > 0 ? gp.raster : 1;
    gp.fd_band = make_fastdiv(static_cast<int64_t>(raster) * gp.n_blocks);
    gp.fd_raster = make_fastdiv(raster);
    gp.fd_last = make_fastdiv(gp.m_blocks > 0 ? gp.m_blocks - ((gp.m_blocks - 1) / raster) * raster : 1);
    gp.fd_splits = make_fastdiv(gp.splits);
}

constexpr int TRACE_WORDS = 8;
// header record: [0] globaltimer at kernel start, [1] SM id, [2] / [3]
// globaltimer after the final CTA barrier seen by thread 0 / the first
// epilogue thread, [4] 1 if thread 0 saw the first epilogue thread's
// pre-barrier write after the barrier.  item record: [0] tile | kind << 32, [1] kb0 | kb1 << 32,
// [2] MMA start, [3] MMA issue done, [4] accumulator ready (epilogue),
// [5] chunk loop start, [6] epilogue done, [7] partial published (stream-K
// peer) or the peers' partials of the first chunk added (owner).

struct ReduceParams {
    const float* ws;
    int32_t splits;                   // 0: no product term (K == 0)
    int32_t tile_n, n_blocks;
    int32_t M, N;
    const void* C;
    int64_t ldc;
    void* D;
    int64_t ldd;
    float alpha, beta;
    const float* scale_a;
    const float* scale_b;
    int32_t act, has_c;
    const void* bias;                 // as in GemmParams
    int32_t bias_rows;
    const void* aux;
    int64_t ldaux;
    int32_t aux_op;
    void* pre;                        // as in GemmParams
    int64_t ldpre;
    int32_t out_trans;                // as in GemmParams
    // balanced split-K: the partials come from a stream-K partition of
    // sk_units iterations over units units (0 = classic split-K layout)
    int32_t units;
    int64_t sk_units;
    int32_t k_blocks, m_blocks, raster;
};

}  // namespace g15
