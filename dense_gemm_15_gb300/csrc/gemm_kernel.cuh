// Persistent warp-specialised tcgen05 GEMM for sm_103a.
//
//   D = act(alpha * s_a * s_b * (A . B) + beta * C + bias) [op Z],
//   act in {identity, ReLU, sigmoid, tanh}, op in {+, -, *, /}
//
// The operation is the plan/run GEMM of the CUTLASS Python interface
// ("Python packages associated with CUTLASS", section "CUTLASS Python
// Interface"; alpha/beta as in the kwkr.cn blog "CUTLASS Python接口" section
// 3.3; ReLU fused in the epilogue as in "CUTLASS Python 接口全解析" section 2.3;
// the bias of that blog's section 5.2; sigmoid, tanh and the auxiliary tensor Z
// from the roadmap section of "Generating State-of-the-Art GEMMs with
// TorchInductor's CuteDSL backend").
// Stream-K and grouped scheduling are the variants listed under "Current
// functionality" of the CUTLASS README; this kernel is our own design for
// Blackwell (tcgen05 / TMEM / TMA), not the pre-SM90 kernels the pages use.
//
// One CTA per SM (CG = 1) or one SM pair per tile (CG = 2), 192 threads:
//   warp 0      TMA producer: A and B tiles into a STAGES-deep shared ring
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//   warps 2..5  epilogue: TMEM -> registers -> alpha/beta/C/bias/act/Z -> 16-bit ->
//               swizzled shared staging -> TMA store (one 32-row quarter each)
// The fp32 accumulator lives in TMEM, double-buffered (2 x TILE_N columns),
// so the epilogue of tile i overlaps the mainloop of tile i+1.
//
// Every wait is bounded (p.timeout_ns); when one runs out the kernel records
// DEV_ERR_TIMEOUT in the status word, every role leaves its loop, in-flight
// copies and MMAs are drained with a bounded wait, TMEM is freed, and the
// kernel returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "gemm_params.h"
#include "ptx.cuh"

namespace g15 {

// CG = 1: one CTA computes a 128 x BN tile.  CG = 2: an SM pair (a cluster of
// two CTAs) computes a 256 x BN tile with tcgen05 cta_group::2 -- each CTA
// stages its own 128 rows of A and its own BN/2 columns of B, and holds its
// 128 rows of the accumulator in its own TMEM.
template <int ELEM, int BN, int CG = 1, int SF = SF_NONE>
struct Traits {
    static constexpr bool FP4 = (ELEM == ELEM_E2M1);   // packed, two elements per byte
    static constexpr bool F8 = (ELEM == ELEM_E4M3 || ELEM == ELEM_E5M2 || FP4);
    static constexpr int ESIZE = F8 ? 1 : 2;           // bytes per A/B element (fp4: per pair)
    static constexpr int BK = FP4 ? 256 : 128 / ESIZE; // elements of one 128-byte swizzle row of K
    static constexpr int UMMA_K = FP4 ? 64 : 32 / ESIZE;  // K per tcgen05.mma (32 bytes)
    static constexpr int KSTEPS = BK / UMMA_K;         // MMAs per k-block (4)
    static constexpr int A_STAGE = TILE_M * 128;       // 16 KB
    static constexpr int B_COLS = BN / CG;             // B columns staged by one CTA
    static constexpr int B_STAGE = B_COLS * 128;       // 16 or 32 KB
    // block-scaled kinds: 512-byte scale atoms per k-block and 128 rows (1 for
    // the 4 scales of an MXFP8 k-block, 2 for MXFP4's 8, 4 for NVFP4's 16)
    static constexpr int SF_APK = SF == SF_NONE ? 0 : SF == SF_MXF8 ? 1 : SF == SF_MXF4 ? 2 : 4;
    static constexpr int SF_BROWS = BN / 128;          // 128-row blocks of B
    static constexpr int SF_STAGE = SF_APK * 512 * (1 + SF_BROWS);
    static constexpr int SF_COLS = SF_APK * 4 * (1 + SF_BROWS);  // TMEM columns per stage
    static constexpr int STAGE_BYTES = A_STAGE + B_STAGE + SF_STAGE;
    // accumulators in TMEM: two (the epilogue of one tile overlaps the next
    // tile's mainloop), or one when 256-wide block-scaled tiles leave the other
    // half of the 512 columns to their scale factors
    static constexpr int ACC_BUFS = (SF != SF_NONE && BN == 256) ? 1 : 2;
    // Epilogue staging: one 32 x 64 box per warp and output chunk of the tile
    // when that leaves room for six stages (the whole C tile is then fetched
    // as soon as the tile starts), else a ring of two boxes per warp (the rest
    // of the C tile is then prefetched into L2 when the tile starts).
    static constexpr int NCH = BN / EPI_COLS;          // output chunks per tile row
    static constexpr int SMEM_FIXED = 232448 - 1024 - 256;
    static constexpr int STAGES_WHOLE = (SMEM_FIXED - EPI_WARPS * NCH * EPI_BUF_BYTES) / STAGE_BYTES;
    static constexpr int EPI_BUFS = (NCH <= 2 || STAGES_WHOLE >= 6) ? NCH : 2;
    static constexpr bool EPI_WHOLE = EPI_BUFS == NCH;
    static constexpr int EPI_BYTES = EPI_WARPS * EPI_BUFS * EPI_BUF_BYTES;
    // as many stages as fit next to the epilogue staging (at most 8)
    static constexpr int STAGES_FIT = (SMEM_FIXED - EPI_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    // an N-major B stage is whole 128-byte swizzle rows of N
    // (block-scaled B is always K-major: any multiple of 8 rows)
    static_assert(SF != SF_NONE || (B_COLS * ESIZE >= 128 && (B_COLS * ESIZE) % 128 == 0),
                  "B columns per CTA");
    static_assert(EPI_BUFS <= 8, "C barrier parity bits");
    static_assert(SF == SF_NONE || BN % 128 == 0, "block-scaled tiles");
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_SF = OFF_B + STAGES * B_STAGE;
    // the epilogue's 128-byte-swizzled staging boxes start on a 1024-byte boundary
    static constexpr int OFF_EPI = OFF_SF + (STAGES * SF_STAGE + 1023) / 1024 * 1024;
    static_assert(OFF_EPI % 1024 == 0, "epilogue staging alignment");
    static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
    // barriers: full[S], empty[S], acc_full[2], acc_empty[2], cbar[4][EPI_BUFS], drain, epi
    static constexpr int NUM_BARS = 2 * STAGES + 4 + EPI_BUFS * EPI_WARPS + 2;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;  // tmem base, abort flag
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;      // + alignment slack
    // TMEM: the accumulators, then (block-scaled) one scale-factor slot per stage
    static constexpr uint32_t TMEM_COLS = SF == SF_NONE ? 2 * BN : 512;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(TMEM_COLS <= 512, "TMEM budget");
    static_assert(SF == SF_NONE || ACC_BUFS * BN + STAGES * SF_COLS <= 512, "TMEM scale-factor slots");
};

template <int ELEM>
struct OutType;
template <>
struct OutType<ELEM_F16> {
    using T = __half;
};
template <>
struct OutType<ELEM_BF16> {
    using T = __nv_bfloat16;
};
template <>
struct OutType<ELEM_E4M3> {
    using T = __nv_bfloat16;
};
template <>
struct OutType<ELEM_E5M2> {
    using T = __nv_bfloat16;
};
template <>
struct OutType<ELEM_E2M1> {
    using T = __nv_bfloat16;
};

// Packs two fp32 values into two 16-bit outputs (round to nearest even).
template <int ELEM>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (ELEM == ELEM_F16) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

template <int ELEM>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
    if constexpr (ELEM == ELEM_F16) {
        __half2 h = *reinterpret_cast<__half2*>(&v);
        return __half22float2(h);
    } else {
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&v);
        return __bfloat1622float2(h);
    }
}

// One stored 16-bit output-type value as float.
template <int ELEM>
__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
    if constexpr (ELEM == ELEM_F16) return __half2float(__ushort_as_half(h));
    else return __bfloat162float(__ushort_as_bfloat16(h));
}

// max(x, 0) that keeps NaN (one max.NaN instruction).
__device__ __forceinline__ float relu_nan(float x) {
    float r;
    asm("max.NaN.f32 %0, %1, 0f00000000;" : "=f"(r) : "f"(x));
    return r;
}

// Logistic sigmoid 1 / (1 + e^-x) from the exponential and fast-division
// intrinsics (its definition; x -> -inf gives 0, +inf gives 1, NaN stays NaN).
__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// tanh by the hardware approximation (PTX tanh.approx.f32, relative error
// below 2^-10.9, the order of one 16-bit output rounding).
__device__ __forceinline__ float tanh_f(float x) {
    float r;
    asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// The epilogue activation of one value (Activation).
__device__ __forceinline__ float activate(float x, int act) {
    switch (act) {
        case ACT_RELU: return relu_nan(x);
        case ACT_SIGMOID: return sigmoid_f(x);
        case ACT_TANH: return tanh_f(x);
        default: return x;
    }
}

// v op z for the auxiliary-tensor operation (1 add, 2 sub, 3 mul, 4 div).
__device__ __forceinline__ float aux_apply(float v, float z, int op) {
    switch (op) {
        case 1: return v + z;
        case 2: return v - z;
        case 3: return v * z;
        case 4: return v / z;
        default: return v;
    }
}

// Applies the activation to n values held in registers: one uniform branch,
// then straight-line code.
template <int NV>
__device__ __forceinline__ void activate_all(float (&v)[NV], int act) {
    if (act == ACT_RELU) {
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = relu_nan(v[i]);
    } else if (act == ACT_SIGMOID) {
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = sigmoid_f(v[i]);
    } else if (act == ACT_TANH) {
#pragma unroll
        for (int i = 0; i < NV; ++i) v[i] = tanh_f(v[i]);
    }
}

// Eight consecutive bias elements starting at column c (16-bit, zero past n),
// packed in pairs.
__device__ __forceinline__ uint4 load_bias8(const void* bias, int64_t c, int64_t n) {
    const uint16_t* b = static_cast<const uint16_t*>(bias);
    if (c + 8 <= n) return __ldg(reinterpret_cast<const uint4*>(b + c));
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    for (int t = 0; t < 8; ++t)
        if (c + t < n) w[t >> 1] |= static_cast<uint32_t>(__ldg(b + c + t)) << (16 * (t & 1));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Stores the first min(64, left) of 64 fp32 values, rounded to the 16-bit
// output type, at dst (a row of 64 elements starting on a 16-byte boundary):
// 16-byte stores when the row is whole, element stores otherwise.
template <int ELEM>
__device__ __forceinline__ void store_row64(uint16_t* dst, const float (&v)[64], int32_t left) {
    if (left >= 64) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(dst + 8 * j) =
                make_uint4(pack2<ELEM>(v[8 * j], v[8 * j + 1]), pack2<ELEM>(v[8 * j + 2], v[8 * j + 3]),
                           pack2<ELEM>(v[8 * j + 4], v[8 * j + 5]), pack2<ELEM>(v[8 * j + 6], v[8 * j + 7]));
    } else {
#pragma unroll
        for (int t = 0; t < 64; t += 2) {
            const uint32_t pr = pack2<ELEM>(v[t], v[t + 1]);
            if (t < left) dst[t] = static_cast<uint16_t>(pr);
            if (t + 1 < left) dst[t + 1] = static_cast<uint16_t>(pr >> 16);
        }
    }
}

// ------------------------------------------------------------------ errors

struct Ctl {
    volatile uint32_t* abort;  // shared flag: some role gave up
    int32_t* status;
    uint64_t timeout_ns;
};

__device__ __forceinline__ void raise_error(volatile uint32_t* abort, int32_t* status, int code) {
    atomicCAS(status, 0, code);
    *abort = 1u;
}

static __device__ __noinline__ bool wait_bar_slow(volatile uint32_t* abort, int32_t* status,
                                           uint64_t timeout_ns, uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                raise_error(abort, status, DEV_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Waits for the phase of parity `parity` of `bar`; false if the kernel is
// aborting or the wait ran out (which starts the abort).
__device__ __forceinline__ bool wait_bar(const Ctl& c, uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(c.abort, c.status, c.timeout_ns, bar, parity);
}

// Bounded wait used only while draining after an abort (ignores the flag).
static __device__ __noinline__ void drain_bar(uint32_t bar, uint32_t parity, uint64_t budget_ns) {
    const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > budget_ns) return;
    }
}

// ------------------------------------------------------------------ scheduling

// One unit of work of a CTA: k-blocks [kb0, kb1) of output tile `tile`.
struct Work {
    int32_t tile;      // linear tile id (within its group)
    int32_t group;     // group index (0 for dense)
    int32_t m_blk, n_blk;
    int32_t kb0, kb1;
    int32_t kind;      // WK_*
    int32_t slot;      // workspace slot (and flag) of a partial tile (128-row halves)
    int32_t h0, h1;    // stream-K: first and last unit holding a piece of this tile
};
// A stream-K tile split across units has one owner, the unit expected to
// finish its piece last, which adds the others' partial tiles (peers).
enum : int32_t { WK_FULL = 0, WK_PEER = 1, WK_OWNER = 2, WK_SPLIT = 3 };

// Scheduling works on "units": one CTA (CG = 1) or one SM pair (CG = 2).
struct Unit {
    int32_t id, count, rank, cg;
};

// A stream-K unit's range [u0, u_end) of (tile, k-block) iterations holds at
// most one tail piece (its start, inside a tile), whole tiles, and at most one
// head piece (its end: the k = 0 head of a tile).  The pieces are taken in the
// order tail, head, whole tiles, so that pieces of split tiles finish early
// and their fix-up overlaps the whole tiles' mainloop instead of trailing it.
struct SchedState {
    int32_t i;          // data-parallel / split item counter
    int32_t phase;      // 0 data-parallel, 1 stream-K, 2 done
    int32_t step;       // stream-K: 0 tail piece, 1 head piece, 2 whole tiles
    int64_t u0, u_end;  // stream-K range of this unit
    int64_t u;          // stream-K: end of the tail piece, then cursor over whole tiles
    int64_t o_begin;    // stream-K: start of the head piece (u_end if none)
};

// The rare 64-bit division, out of line so that the call sites stay short.
static __device__ __noinline__ int64_t div64(int64_t x, int64_t d) { return x / d; }

// x / d for 0 <= x and 0 < d, in 32-bit arithmetic when both fit: a 64-bit
// division is a long dependent software sequence.
__device__ __forceinline__ int64_t idiv(int64_t x, int64_t d) {
    if (((x | d) >> 31) == 0)
        return static_cast<int64_t>(static_cast<uint32_t>(x) / static_cast<uint32_t>(d));
    return div64(x, d);
}

// x / f.d for 0 <= x by the launch's precomputed multiplier (FastDiv): the
// scheduler divides a few dozen times before a CTA's first copy, and even a
// 32-bit division is a dependent chain of a few hundred cycles.
__device__ __forceinline__ int64_t fdiv(int64_t x, const FastDiv& f) {
    if (static_cast<uint64_t>(x) < (1ull << 31))
        return static_cast<int64_t>((static_cast<uint64_t>(x) * f.mul) >> f.shift);
    return div64(x, f.d);
}

__device__ __forceinline__ int64_t sk_begin(const GemmParams& p, const Unit& un, int64_t unit) {
    return fdiv(p.sk_units * unit, p.fd_units);
}

// The unit whose range holds stream-K iteration x.
__device__ __forceinline__ int32_t sk_unit_of(const GemmParams& p, const Unit& un, int64_t x) {
    int64_t u = fdiv(x * un.count, p.fd_sk);  // sk_begin(u) <= x up to rounding
    while (u > 0 && sk_begin(p, un, u) > x) --u;
    while (u + 1 < un.count && sk_begin(p, un, u + 1) <= x) ++u;
    return static_cast<int32_t>(u);
}

// Iterations unit v runs before its piece of the tile [t0, t0 + k_blocks) is
// done, in its piece order (tail piece, head piece, whole tiles): the piece's
// length, plus the unit's leading piece when this piece is the tile's head
// and the unit's range starts inside an earlier tile.
__device__ __forceinline__ int64_t sk_piece_finish(const GemmParams& p, const Unit& un, int32_t v,
                                                   int64_t t0) {
    const int64_t kb = p.k_blocks;
    const int64_t b = sk_begin(p, un, v), e = sk_begin(p, un, v + 1);
    const int64_t len = min(e, t0 + kb) - max(b, t0);
    const int64_t bt = fdiv(b, p.fd_kb);  // the tile b lies in
    if (b >= t0 || b == bt * kb) return len;
    return (min(e, (bt + 1) * kb) - b) + len;
}

// Workspace slot / flag of unit v's partial tile: each unit holds at most a
// tail piece (slot 2v) and a head piece (slot 2v + 1) of split tiles.
__device__ __forceinline__ int32_t sk_slot(const Unit& un, int32_t v, bool head) {
    return (2 * v + (head ? 1 : 0)) * un.cg + un.rank;
}

// Linear tile index of block (mb, nb) in the raster order of raster_coords.
__device__ __forceinline__ int32_t raster_tile(int32_t mb, int32_t nb, int32_t m_blocks,
                                               int32_t n_blocks, int32_t raster) {
    const int32_t band = mb / raster;
    const int32_t first_m = band * raster;
    const int32_t rows = min(raster, m_blocks - first_m);
    return band * raster * n_blocks + nb * rows + (mb - first_m);
}

__device__ __forceinline__ void raster_coords(int32_t tile, int32_t m_blocks, int32_t n_blocks,
                                              int32_t raster, int32_t& mb, int32_t& nb) {
    const int32_t band_tiles = raster * n_blocks;
    const int32_t band = tile / band_tiles;
    const int32_t first_m = band * raster;
    const int32_t rows = min(raster, m_blocks - first_m);
    const int32_t local = tile - band * band_tiles;
    mb = first_m + local % rows;
    nb = local / rows;
}

__device__ __forceinline__ void sched_init(const GemmParams& p, const Unit& un, SchedState& s) {
    s.i = 0;
    s.phase = 0;
    s.step = 0;
    s.u0 = s.u = s.u_end = s.o_begin = 0;
    if (p.sched == SCHED_SK) {
        const int64_t kb = p.k_blocks;
        s.u0 = sk_begin(p, un, un.id);
        s.u_end = sk_begin(p, un, un.id + 1);
        // end of the tail piece (u0 itself when the range starts on a tile)
        const int64_t first_tile = fdiv(s.u0, p.fd_kb) * kb;
        s.u = (s.u0 != first_tile) ? min(s.u_end, first_tile + kb) : s.u0;
        // start of the head piece (u_end when the range ends on a tile)
        const int64_t last_tile = fdiv(s.u_end, p.fd_kb) * kb;
        s.o_begin = (s.u_end != last_tile && last_tile >= s.u) ? last_tile : s.u_end;
    }
}

__device__ __forceinline__ void fill_coords(const GemmParams& p, Work& w) {
    if (p.groups) {
        // locate the group whose tile range holds w.tile (prefix sums ascend)
        int32_t lo = 0, hi = p.num_groups - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (p.groups[mid].tile_start <= w.tile) lo = mid; else hi = mid - 1;
        }
        const GroupEntry& g = p.groups[lo];
        w.group = lo;
        raster_coords(w.tile - g.tile_start, g.m_blocks, g.n_blocks, g.raster, w.m_blk, w.n_blk);
        w.kb0 = 0;
        w.kb1 = g.k_blocks;
    } else {
        // raster_coords with the launch's divisors
        w.group = 0;
        const int32_t band = static_cast<int32_t>(fdiv(w.tile, p.fd_band));
        const int32_t first_m = band * p.raster;
        const int32_t local = w.tile - band * p.raster * p.n_blocks;
        const bool full = first_m + p.raster <= p.m_blocks;
        const int32_t rows = full ? p.raster : p.m_blocks - first_m;
        const int32_t q = static_cast<int32_t>(full ? fdiv(local, p.fd_raster) : fdiv(local, p.fd_last));
        w.m_blk = first_m + (local - q * rows);
        w.n_blk = q;
    }
}

// OWNER = false skips who owns a split tile (h0, h1 and the kind of a piece),
// which only the epilogue reads.
template <bool OWNER = true>
__device__ __forceinline__ bool sched_next(const GemmParams& p, const Unit& un, SchedState& s,
                                           Work& w) {
    const int32_t G = un.count;
    if (p.sched == SCHED_SPLIT) {
        const int32_t j = un.id + s.i * G;
        if (j >= p.tiles * p.splits) return false;
        ++s.i;
        w.tile = static_cast<int32_t>(fdiv(j, p.fd_splits));
        const int32_t sp = j - w.tile * p.splits;
        fill_coords(p, w);
        w.kb0 = static_cast<int32_t>(fdiv(static_cast<int64_t>(p.k_blocks) * sp, p.fd_splits));
        w.kb1 = static_cast<int32_t>(fdiv(static_cast<int64_t>(p.k_blocks) * (sp + 1), p.fd_splits));
        w.kind = WK_SPLIT;
        w.h0 = w.h1 = un.id;
        // slots are indexed by 128-row block so the reduction sees one layout
        w.slot = ((w.m_blk * un.cg + un.rank) * p.n_blocks + w.n_blk) * p.splits + sp;
        return true;
    }
    const int32_t dp_limit = (p.sched == SCHED_SK) ? p.dp_tiles : p.tiles;
    if (s.phase == 0) {
        const int32_t t = un.id + s.i * G;
        if (t < dp_limit) {
            ++s.i;
            w.tile = t;
            w.kb0 = 0;
            w.kb1 = p.k_blocks;
            fill_coords(p, w);
            w.kind = WK_FULL;
            w.slot = 0;
            w.h0 = w.h1 = un.id;
            return true;
        }
        s.phase = (p.sched == SCHED_SK) ? 1 : 2;
    }
    if (s.phase == 1) {
        const int32_t kb = p.k_blocks;
        int64_t b0 = -1, b1 = -1;  // the next piece, [b0, b1) within one tile
        if (s.step == 0) {
            s.step = 1;
            if (s.u > s.u0) {
                b0 = s.u0;
                b1 = s.u;
            }
        }
        if (b0 < 0 && s.step == 1) {
            s.step = 2;
            if (s.o_begin < s.u_end) {
                b0 = s.o_begin;
                b1 = s.u_end;
            }
        }
        if (b0 < 0) {
            if (s.u >= s.o_begin) {
                s.phase = 2;
                return false;
            }
            b0 = s.u;
            b1 = s.u + kb;
            s.u = b1;
        }
        const int32_t rel = static_cast<int32_t>(fdiv(b0, p.fd_kb));
        const int64_t tile_u0 = static_cast<int64_t>(rel) * kb;
        w.tile = p.dp_tiles + rel;
        fill_coords(p, w);
        w.kb0 = static_cast<int32_t>(b0 - tile_u0);
        w.kb1 = static_cast<int32_t>(b1 - tile_u0);
        w.slot = sk_slot(un, un.id, w.kb0 == 0);
        w.h0 = w.h1 = un.id;
        if (w.kb0 == 0 && w.kb1 == kb) {
            w.kind = WK_FULL;
        } else if (!OWNER) {
            w.kind = WK_PEER;  // not known here
        } else {
            // owner: the holder with the latest expected finish (lowest unit on ties)
            w.h0 = sk_unit_of(p, un, tile_u0);
            w.h1 = sk_unit_of(p, un, tile_u0 + kb - 1);
            int32_t owner = w.h0;
            int64_t best = -1;
            for (int32_t v = w.h0; v <= w.h1; ++v) {
                const int64_t f = sk_piece_finish(p, un, v, tile_u0);
                if (f > best) {
                    best = f;
                    owner = v;
                }
            }
            w.kind = owner == un.id ? WK_OWNER : WK_PEER;
        }
        // balanced split-K: every piece goes to the workspace, the reduction adds them
        if (p.sk_partials_only) w.kind = WK_SPLIT;
        return true;
    }
    return false;
}

// True when the item sched_next returned last was a unit's final stream-K
// item (nothing follows it in this unit): no head piece still to come (it
// has been taken, or there is none) and no whole tile left.
__device__ __forceinline__ bool sched_sk_last(const SchedState& s) {
    return s.phase == 1 && (s.step == 2 || s.o_begin >= s.u_end) && s.u >= s.o_begin;
}

// ------------------------------------------------------------------ split-K arrivals

// Counts one arrival at a split tile's counter for launch `epoch` and returns
// the arrival number (1 = first).  The counter holds the launch epoch in its
// high word and the count in its low word, so values left by an earlier launch
// (one that stopped early) read as zero.  0 if the update never succeeded.
__device__ __forceinline__ uint32_t count_arrival(unsigned long long* ctr, uint32_t epoch) {
    unsigned long long old = atomicAdd(ctr, 0ull);
#pragma unroll 1
    for (int it = 0; it < (1 << 20); ++it) {
        const uint32_t cnt = static_cast<uint32_t>(old >> 32) == epoch ? static_cast<uint32_t>(old) : 0u;
        const unsigned long long nw = (static_cast<unsigned long long>(epoch) << 32) | (cnt + 1u);
        const unsigned long long prev = atomicCAS(ctr, old, nw);
        if (prev == old) return cnt + 1u;
        old = prev;
    }
    return 0u;
}

// ------------------------------------------------------------------ partial tiles

// Adds n fp32 partial chunks, in order, into acc (the first one assigned when
// `assign`).  src_of(j) is this thread's first float4 of partial j; its nq
// float4 groups lie 32 float4 apart (a warp's 512 contiguous bytes each).  The
// loads of 16 / NQP partials are in flight together, so n partials cost about
// n * NQP / 16 round trips to L2 instead of n.
template <int NQP, class SrcOf>
__device__ __forceinline__ void sum_partials_n(const SrcOf& src_of, int32_t n, int nq,
                                               float (&acc)[64], bool assign, uint64_t pol) {
    constexpr int P = 16 / NQP;
    for (int32_t j0 = 0; j0 < n; j0 += P) {
        float4 t[16];
#pragma unroll
        for (int jj = 0; jj < P; ++jj) {
            const bool live = j0 + jj < n;
            const float4* src = live ? src_of(j0 + jj) : nullptr;
#pragma unroll
            for (int i = 0; i < NQP; ++i)
                t[jj * NQP + i] = (live && i < nq) ? ld_global_cg_hint(src + 32 * i, pol)
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int jj = 0; jj < P; ++jj) {
            if (j0 + jj >= n) break;
            const bool first = assign && j0 + jj == 0;
#pragma unroll
            for (int i = 0; i < NQP; ++i) {
                if (i >= nq) continue;
                const float4 x = t[jj * NQP + i];
                if (first) {
                    acc[4 * i + 0] = x.x;
                    acc[4 * i + 1] = x.y;
                    acc[4 * i + 2] = x.z;
                    acc[4 * i + 3] = x.w;
                } else {
                    acc[4 * i + 0] += x.x;
                    acc[4 * i + 1] += x.y;
                    acc[4 * i + 2] += x.z;
                    acc[4 * i + 3] += x.w;
                }
            }
        }
    }
}

// The same for any nq <= 16: four partials at a time for chunks of at most
// four groups (a swap-AB tile of a 16-token problem), else one.
template <class SrcOf>
__device__ __forceinline__ void sum_partials(const SrcOf& src_of, int32_t n, int nq,
                                             float (&acc)[64], bool assign, uint64_t pol) {
    if (nq <= 4) sum_partials_n<4>(src_of, n, nq, acc, assign, pol);
    else sum_partials_n<16>(src_of, n, nq, acc, assign, pol);
}

// ------------------------------------------------------------------ four-column epilogue

// The epilogue of the REDUCE_COLS (4) computed outputs (m, n .. n + 3) from
// the sum of their products: D = act(alpha * acc + beta * C + bias) [op Z],
// Y (pre) = the value before act, columns past N skipped; each output stored
// as computed, or for a transposed output (swap-AB) at row n + t, column m.
// P is GemmParams or ReduceParams (the same field names).
template <int ELEM, class P>
__device__ __forceinline__ void epilogue_cols4(const P& p, float alpha, int32_t m, int32_t n, float4 acc) {
    constexpr int V = REDUCE_COLS;
    const float av[V] = {acc.x, acc.y, acc.z, acc.w};
    const int nvalid = min(V, p.N - n);
    float bias[V];
#pragma unroll
    for (int t = 0; t < V; ++t) bias[t] = 0.0f;
    if (p.bias) {
        const uint16_t* bv = static_cast<const uint16_t*>(p.bias);
#pragma unroll
        for (int t = 0; t < V; ++t) {
            if (p.bias_rows) bias[t] = half_bits_to_float<ELEM>(__ldg(bv + m));
            else if (t < nvalid) bias[t] = half_bits_to_float<ELEM>(__ldg(bv + n + t));
        }
    }
    auto at = [&](int64_t ld, int t) -> int64_t {
        return p.out_trans ? static_cast<int64_t>(n + t) * ld + m : static_cast<int64_t>(m) * ld + n + t;
    };
    const uint16_t* cb = static_cast<const uint16_t*>(p.C);
    uint16_t* db = static_cast<uint16_t*>(p.D);
    float o[V];
#pragma unroll
    for (int t = 0; t < V; ++t) {
        float x = alpha * av[t];
        if (p.has_c && t < nvalid) x = fmaf(p.beta, half_bits_to_float<ELEM>(cb[at(p.ldc, t)]), x);
        x += bias[t];
        if (p.pre && t < nvalid) {
            const uint32_t pr = pack2<ELEM>(x, x);
            static_cast<uint16_t*>(p.pre)[at(p.ldpre, t)] = static_cast<uint16_t>(pr);
        }
        o[t] = activate(x, p.act);
        if (p.aux_op && t < nvalid) {
            const uint16_t z = static_cast<const uint16_t*>(p.aux)[at(p.ldaux, t)];
            o[t] = aux_apply(o[t], half_bits_to_float<ELEM>(z), p.aux_op);
        }
    }
    const uint32_t pk[2] = {pack2<ELEM>(o[0], o[1]), pack2<ELEM>(o[2], o[3])};
    if (nvalid == V && !p.out_trans) {
        *reinterpret_cast<uint2*>(db + at(p.ldd, 0)) = make_uint2(pk[0], pk[1]);
    } else {
        for (int t = 0; t < nvalid; ++t) db[at(p.ldd, t)] = static_cast<uint16_t>(pk[t >> 1] >> (16 * (t & 1)));
    }
}

// ------------------------------------------------------------------ tracing

__device__ __forceinline__ uint64_t* trace_rec(const GemmParams& p, int32_t item) {
    if (!p.trace || item >= p.trace_items) return nullptr;
    return p.trace + (static_cast<size_t>(blockIdx.x) * (p.trace_items + 1) + 1 + item) * TRACE_WORDS;
}

// ------------------------------------------------------------------ the kernel

template <int ELEM, int BN, int CG, int SF>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ GemmParams p) {
    using TR = Traits<ELEM, BN, CG, SF>;
    constexpr int ACC_BUFS = TR::ACC_BUFS;
    using OutT = typename OutType<ELEM>::T;
    constexpr int STAGES = TR::STAGES;
    constexpr int TILE_ROWS = TILE_M * CG;  // output rows per tile

    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte-swizzled TMA / UMMA tiles
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sA = sbase + TR::OFF_A;
    const uint32_t sB = sbase + TR::OFF_B;
    const uint32_t sSF = sbase + TR::OFF_SF;
    const uint32_t sEpi = sbase + TR::OFF_EPI;
    const uint32_t bar0 = sbase + TR::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    constexpr int EPI_BUFS = TR::EPI_BUFS;
    auto c_bar = [&](int q, int b) { return bar0 + 8u * (2 * STAGES + 4 + EPI_BUFS * q + b); };
    const uint32_t drain = bar0 + 8u * (2 * STAGES + 4 + EPI_BUFS * EPI_WARPS);
    const uint32_t epi_bar = drain + 8u;  // bounded barrier of the 4 epilogue warps
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + TR::OFF_MISC);
    volatile uint32_t* tmem_slot = misc;
    volatile uint32_t* abort_flag = misc + 1;

    // a programmatic dependent (the split-K reduction, or the next GEMM) may be
    // scheduled now; it waits for this grid's completion before it touches
    // global memory.  This grid, itself launched as a programmatic dependent,
    // waits for the kernel before it (griddepcontrol.wait) before its first
    // global access: its roles do so after their set-up, a traced or grouped
    // launch (trace records, the problem table) here.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (p.trace || p.groups) asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    Ctl ctl{abort_flag, p.status, p.timeout_ns};
    Unit un;
    un.cg = CG;
    un.rank = CG == 2 ? static_cast<int32_t>(cluster_ctarank()) : 0;
    un.id = static_cast<int32_t>(blockIdx.x) / CG;
    un.count = static_cast<int32_t>(gridDim.x) / CG;
    const bool leader = un.rank == 0;
    uint64_t* trace_hdr =
        p.trace ? p.trace + static_cast<size_t>(blockIdx.x) * (p.trace_items + 1) * TRACE_WORDS : nullptr;
    if (trace_hdr && threadIdx.x == 0) {
        trace_hdr[0] = globaltimer_ns();
        trace_hdr[1] = smid();
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), EPI_WARPS * CG);  // both CTAs' epilogues release
        }
        for (int q = 0; q < EPI_WARPS; ++q)
            for (int b = 0; b < EPI_BUFS; ++b) mbar_init(c_bar(q, b), 1);
        mbar_init(drain, 1);
        mbar_init(epi_bar, EPI_WARPS);
        *abort_flag = 0u;
        misc[2] = 0u;  // set by the first epilogue thread just before the final barrier
        fence_mbar_init();
    }
    __syncwarp();
    if (warp == 1) {
        // with CG = 2 one warp of each CTA of the pair allocates collectively
        tmem_alloc<CG>(smem_u32(misc), TR::TMEM_COLS);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (CG == 2) cluster_sync();  // the peer's barriers are initialised
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ============================ TMA producer
        if (lane == 0) {
            if (!p.groups) {
                tma_prefetch_desc(&p.tmA);
                tma_prefetch_desc(&p.tmB);
            }
            if constexpr (SF != SF_NONE) {
                tma_prefetch_desc(&p.tmSFA);
                tma_prefetch_desc(&p.tmSFB);
            }
            // the raster band's A rows are read by every wave of the band: keep
            // them in L2 (evict-last) when asked; B then streams (evict-first)
            const uint64_t pol_a = p.l2_hints >= 1 ? l2_policy_evict_last() : 0ull;
            const uint64_t pol_b = p.l2_hints >= 2 ? l2_policy_evict_first() : 0ull;
            SchedState st;
            sched_init(p, un, st);
            Work w;
            uint32_t n_issued = 0;
            asm volatile("griddepcontrol.wait;" ::: "memory");
            bool ok = true;
            int last_group = -1;
            while (ok && sched_next<false>(p, un, st, w)) {
                const CUtensorMap* tA = &p.tmA;
                const CUtensorMap* tB = &p.tmB;
                if (p.groups) {
                    tA = &p.groups[w.group].tmA;
                    tB = &p.groups[w.group].tmB;
                    if (w.group != last_group) {
                        tensormap_acquire(tA);
                        tensormap_acquire(tB);
                        last_group = w.group;
                    }
                }
                const int32_t m0 = w.m_blk * TILE_ROWS + un.rank * TILE_M;
                const int32_t n0 = w.n_blk * BN + un.rank * TR::B_COLS;
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                    const int s = n_issued % STAGES;
                    const uint32_t ph = (n_issued / STAGES) & 1u;
                    if (!wait_bar(ctl, empty_bar(s), ph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    // CG = 2: both CTAs' copies complete on the leader's barrier,
                    // which the leader arms for the pair's bytes
                    uint32_t fb = full_bar(s);
                    if constexpr (CG == 2) fb = map_cluster(fb, 0);
                    if constexpr (SF != SF_NONE) {
                        // the stage's scale atoms (tensor maps of 128-byte rows, 4 per
                        // atom): this CTA's 128 rows of A, then every 128-row block of
                        // the tile's B (each CTA of a pair holds all of B's scales);
                        // blocks past M or N read as zeros, their outputs are not stored
                        constexpr uint32_t ATOMS = TR::SF_APK * 512u;
                        if (leader)
                            mbar_arrive_expect_tx(full_bar(s), CG * (TR::A_STAGE + TR::B_STAGE + ATOMS * (1 + TR::SF_BROWS)));
                        const uint32_t dS = sSF + s * TR::SF_STAGE;
                        const int32_t cb0 = kb * TR::SF_APK;
                        const int32_t rba = w.m_blk * CG + un.rank;
                        auto load_sf = [&](uint32_t dst, const CUtensorMap* t, int32_t row) {
                            if constexpr (CG == 2) tma_load_2d_pair(dst, t, fb, 0, row);
                            else tma_load_2d(dst, t, fb, 0, row);
                        };
                        load_sf(dS, &p.tmSFA, (rba * p.sf_cb + cb0) * 4);
#pragma unroll
                        for (int nb = 0; nb < TR::SF_BROWS; ++nb)
                            load_sf(dS + (1 + nb) * ATOMS, &p.tmSFB, ((w.n_blk * TR::SF_BROWS + nb) * p.sf_cb + cb0) * 4);
                    } else if (leader) {
                        mbar_arrive_expect_tx(full_bar(s), CG * TR::STAGE_BYTES);
                    }
                    const uint32_t dA = sA + s * TR::A_STAGE;
                    const uint32_t dB = sB + s * TR::B_STAGE;
                    // K coordinate in tensor-map units: elements, or bytes for packed fp4
                    const int32_t k0 = kb * (TR::FP4 ? 128 : TR::BK);
                    // operand loads, with an L2 policy when asked (pol 0 = none)
                    auto load = [&](uint32_t dst, const CUtensorMap* t, int32_t x, int32_t y, uint64_t pol) {
                        if constexpr (CG == 2) {
                            if (pol) tma_load_2d_pair_hint(dst, t, fb, x, y, pol);
                            else tma_load_2d_pair(dst, t, fb, x, y);
                        } else {
                            if (pol) tma_load_2d_hint(dst, t, fb, x, y, pol);
                            else tma_load_2d(dst, t, fb, x, y);
                        }
                    };
                    if (p.a_kmajor) {
                        load(dA, tA, k0, m0, pol_a);
                    } else {
                        constexpr int AW = 128 / TR::ESIZE;  // M elements per 128-byte row
#pragma unroll
                        for (int j = 0; j < TILE_M / AW; ++j) load(dA + j * AW * 128, tA, m0 + j * AW, k0, pol_a);
                    }
                    if (p.b_kmajor) {
                        load(dB, tB, k0, n0, pol_b);
                    } else {
                        constexpr int BW = 128 / TR::ESIZE;  // N elements per 128-byte row
#pragma unroll
                        for (int j = 0; j < TR::B_COLS / BW; ++j) load(dB + j * BW * 128, tB, n0 + j * BW, k0, pol_b);
                    }
                    ++n_issued;
                }
            }
            if (ok && !*abort_flag) {
                // producer tail: the MMA warp's releases of the last stages land in
                // this CTA's shared memory (for CG = 2, from the leader); wait for
                // them so that none arrives after the CTA has exited
                const uint32_t last = n_issued < STAGES ? n_issued : STAGES;
                for (uint32_t i = 0; i < last; ++i) {
                    const uint32_t n = n_issued - 1 - i;
                    if (!wait_bar(ctl, empty_bar(n % STAGES), (n / STAGES) & 1u)) break;
                }
            }
            if (!ok || *abort_flag) {
                // let every issued copy land before the CTA's shared memory goes away
                const uint32_t outstanding = n_issued < STAGES ? n_issued : STAGES;
                for (uint32_t i = 0; i < outstanding; ++i) {
                    const uint32_t n = n_issued - 1 - i;
                    if (CG == 1 || leader) drain_bar(full_bar(n % STAGES), (n / STAGES) & 1u, 200000000ull);
                }
                if (CG == 2 && !leader) {
                    // the peer's copies complete on the leader: give them time to land
                    const uint64_t t0 = globaltimer_ns();
                    while (globaltimer_ns() - t0 < 2000000ull) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ============================ MMA issuer (one thread of the leader CTA)
        if (lane == 0 && leader) {
            // no global access here, but the bounded waits below must not start
            // timing while the kernel before this one is still running
            asm volatile("griddepcontrol.wait;" ::: "memory");
            const uint64_t adesc0 = sdesc_base(p.a_lbo, p.a_sbo);
            const uint64_t bdesc0 = sdesc_base(p.b_lbo, p.b_sbo);
            SchedState st;
            sched_init(p, un, st);
            Work w;
            uint32_t n_used = 0, n_acc = 0;
            bool ok = true, issued = false;
            // completion signals go to the same barrier in every CTA of the pair
            auto commit = [&](uint32_t bar) {
                if constexpr (CG == 1) {
                    umma_commit(bar);
                } else {
                    umma_commit_pair(bar);
                    umma_commit_pair(map_cluster(bar, 1));
                }
            };
            while (ok && sched_next<false>(p, un, st, w)) {
                const uint32_t ab = ACC_BUFS == 2 ? (n_acc & 1u) : 0u;
                const uint32_t aph = ACC_BUFS == 2 ? ((n_acc >> 1) & 1u) : (n_acc & 1u);
                if (!wait_bar(ctl, acce_bar(ab), aph ^ 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint64_t* tr = trace_rec(p, static_cast<int32_t>(n_acc));
                if (tr) tr[2] = globaltimer_ns();
                const uint32_t d_tmem = tmem_base + ab * BN;
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
                    const int s = n_used % STAGES;
                    const uint32_t ph = (n_used / STAGES) & 1u;
                    if (!wait_bar(ctl, full_bar(s), ph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = sA + s * TR::A_STAGE;
                    const uint32_t b_addr = sB + s * TR::B_STAGE;
                    if constexpr (SF != SF_NONE) {
                        // the stage's scale atoms into its TMEM slot (after the
                        // accumulator): A's atom j at +4j, B's atom j of row block
                        // nb at +4*APK + 4*SF_BROWS*j + 4*nb
                        const uint32_t sf_t = tmem_base + ACC_BUFS * BN + s * TR::SF_COLS;
                        const uint32_t sfb_t = sf_t + 4 * TR::SF_APK;
                        const uint32_t dS = sSF + s * TR::SF_STAGE;
#pragma unroll
                        for (int j = 0; j < TR::SF_APK; ++j) {
                            tmem_cp_32x128b_x4<CG>(sf_t + 4 * j, sdesc_atom(dS + 512 * j));
#pragma unroll
                            for (int nb = 0; nb < TR::SF_BROWS; ++nb)
                                tmem_cp_32x128b_x4<CG>(sfb_t + 4 * TR::SF_BROWS * j + 4 * nb,
                                                       sdesc_atom(dS + (1 + nb) * 512 * TR::SF_APK + 512 * j));
                        }
#pragma unroll
                        for (int k = 0; k < TR::KSTEPS; ++k) {
                            // MXFP8: one scale per row and MMA, byte k of atom 0;
                            // MXFP4: two per MMA, bytes 2(k%2).. of atom k/2;
                            // NVFP4: four per MMA, atom k
                            uint32_t atom = 0, id = 0;
                            if constexpr (SF == SF_MXF8) { id = k; }
                            else if constexpr (SF == SF_MXF4) { atom = k >> 1; id = 2 * (k & 1); }
                            else { atom = k; }
                            const uint32_t idesc = p.idesc | (id << 29) | (id << 4);
                            umma_block_scaled<CG, SF>(d_tmem, sdesc_at(adesc0, a_addr + k * p.a_kstep),
                                                  sdesc_at(bdesc0, b_addr + k * p.b_kstep), idesc,
                                                  sf_t + 4 * atom, sfb_t + 4 * TR::SF_BROWS * atom,
                                                  (kb > w.kb0 || k > 0) ? 1u : 0u);
                        }
                    } else {
#pragma unroll
                    for (int k = 0; k < TR::KSTEPS; ++k) {
                        umma<CG, TR::F8>(d_tmem, sdesc_at(adesc0, a_addr + k * p.a_kstep),
                                         sdesc_at(bdesc0, b_addr + k * p.b_kstep), p.idesc,
                                         (kb > w.kb0 || k > 0) ? 1u : 0u);
                    }
                    }
                    issued = true;
                    commit(empty_bar(s));
                    ++n_used;
                }
                if (!ok) break;
                commit(accf_bar(ab));
                if (tr) tr[3] = globaltimer_ns();
                ++n_acc;
            }
            if (issued && (!ok || *abort_flag)) {
                if constexpr (CG == 1) umma_commit(drain);
                else umma_commit_pair(drain);
                drain_bar(drain, 0, 200000000ull);
            }
        }
    } else {
        // ============================ epilogue warps
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        const int e = warp - 2;                 // epilogue warp index (buffers)
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t ebuf0 = sEpi + e * EPI_BUFS * EPI_BUF_BYTES;
        asm volatile("griddepcontrol.wait;" ::: "memory");  // before any global access
        float alpha = p.alpha;
        if (p.scale_a) alpha *= __ldg(p.scale_a);
        if (p.scale_b) alpha *= __ldg(p.scale_b);
        const float beta = p.beta;
        const int act = p.act;
        const bool has_bias = p.bias != nullptr;
        // C, D and the peers' partial tiles are each touched once here: let L2
        // evict them before the A and B tiles that other CTAs still read
        const uint64_t pol_once = l2_policy_evict_first();
        constexpr int NCH = TR::NCH;
        constexpr bool WHOLE = TR::EPI_WHOLE;  // one staging box per chunk of the tile
        // Stream-K partial tiles are stored in groups of four columns: float4
        // (warp quarter q, column group g, lane) sits at (q * BN/4 + g) * 32 + lane,
        // so that each warp-wide float4 access covers 512 contiguous bytes.
        auto peer_off = [&](int32_t col0) -> size_t {
            return (static_cast<size_t>(q) * (BN / 4) + col0 / 4) * 32 + lane;
        };
        // this thread's first float4 of chunk col0 in peer unit v's partial tile
        // of the tile held by units [w.h0, w.h1] (h0 holds its head)
        auto peer_src = [&](const Work& w, int32_t v, int32_t col0) -> const float4* {
            const int32_t slot = sk_slot(un, v, v == w.h0);
            return reinterpret_cast<const float4*>(p.ws + static_cast<size_t>(slot) * TILE_M * BN) +
                   peer_off(col0);
        };
        // the peers of an owner item: units h0..h1 but this one, in unit order
        auto n_peers = [&](const Work& w) -> int32_t {
            return (w.h1 - w.h0 + 1) - ((un.id >= w.h0 && un.id <= w.h1) ? 1 : 0);
        };
        auto peer_at = [&](const Work& w, int32_t j) -> int32_t {
            const int32_t v = w.h0 + j;
            return (un.id >= w.h0 && v >= un.id) ? v + 1 : v;
        };

        // Bounded barrier of the four epilogue warps (mbarrier with count 4):
        // release/acquire at CTA scope, and it cannot hang if a warp gives up.
        uint32_t epi_phase = 0;
        auto epi_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(epi_bar);
            const bool r = wait_bar(ctl, epi_bar, epi_phase);
            epi_phase ^= 1u;
            return r;
        };

        SchedState st;
        sched_init(p, un, st);
        Work w;
        uint32_t n_acc = 0;
        uint32_t n_chunk = 0;      // chunks stored by this warp (ring buffer parity)
        uint32_t c_phase = 0;      // per-buffer C barrier parity bits
        uint32_t c_pending = 0;    // C loads issued and not yet waited for
        int last_group = -1;
        bool ok = true;
        while (ok && sched_next(p, un, st, w)) {
            const uint32_t ab = ACC_BUFS == 2 ? (n_acc & 1u) : 0u;
            const uint32_t aph = ACC_BUFS == 2 ? ((n_acc >> 1) & 1u) : (n_acc & 1u);

            int32_t M = p.M, N = p.N;
            const CUtensorMap* tC = &p.tmC;
            const CUtensorMap* tD = &p.tmD;
            int32_t has_c = p.has_c;
            OutT* Dptr = static_cast<OutT*>(p.D);
            int64_t ldd = p.ldd;
            if (p.groups) {
                const GroupEntry& g = p.groups[w.group];
                M = g.M;
                N = g.N;
                tC = &g.tmC;
                tD = &g.tmD;
                has_c = g.has_c;
                Dptr = static_cast<OutT*>(g.D);
                ldd = g.ldd;
                alpha = p.alpha;  // the group's own fp8 scales
                if (g.scale_a) alpha *= __ldg(g.scale_a);
                if (g.scale_b) alpha *= __ldg(g.scale_b);
                if (lane == 0 && w.group != last_group) {
                    tensormap_acquire(tC);
                    tensormap_acquire(tD);
                }
                last_group = w.group;
            }
            const int32_t m0 = w.m_blk * TILE_ROWS + un.rank * TILE_M;
            const int32_t n0 = w.n_blk * BN;
            const int32_t row0 = m0 + q * 32;      // first row of this warp
            const bool rows_live = row0 < M;
            const bool to_ws = (w.kind == WK_PEER || w.kind == WK_SPLIT);
            // a transposed output (swap-AB) reads C and writes D element-wise
            const bool stage_c = has_c && !to_ws && rows_live && !p.out_trans;
            const int nch = min(NCH, (N - n0 + EPI_COLS - 1) / EPI_COLS);
            // bias of this thread's row (bias indexed by output row)
            float bias_row = 0.0f;
            if (has_bias && p.bias_rows && row0 + lane < M)
                bias_row = half_bits_to_float<ELEM>(__ldg(static_cast<const uint16_t*>(p.bias) + row0 + lane));

            // C is fetched while the mainloop still runs: the whole tile when
            // every chunk has its own box, else the first chunk, with the rest
            // prefetched into L2
            auto issue_c = [&](bool to_ws_, bool stage_c_) {
                if (WHOLE && !to_ws_ && lane == 0) {
                    bulk_wait_read<0>();  // the previous tile's stores have read their boxes
                    if (stage_c_) {
                        for (int c = 0; c < nch; ++c) {
                            mbar_arrive_expect_tx(c_bar(e, c), EPI_BUF_BYTES);
                            tma_load_2d_hint(ebuf0 + c * EPI_BUF_BYTES, tC, c_bar(e, c), n0 + c * EPI_COLS, row0, pol_once);
                            c_pending |= 1u << c;
                        }
                    }
                } else if (!WHOLE && stage_c_ && lane == 0) {
                    // the latest store read the other box; the one before it read this one
                    const uint32_t b = n_chunk & 1u;
                    bulk_wait_read<1>();
                    mbar_arrive_expect_tx(c_bar(e, b), EPI_BUF_BYTES);
                    tma_load_2d_hint(ebuf0 + b * EPI_BUF_BYTES, tC, c_bar(e, b), n0, row0, pol_once);
                    c_pending |= 1u << b;
                    for (int c = 1; c < nch; ++c) tma_prefetch_l2_2d(tC, n0 + c * EPI_COLS, row0);
                }
                __syncwarp();  // lane 0's wait for the stores orders the warp's writes to the boxes
            };
            issue_c(to_ws, stage_c);

            // stream-K owner: wait until every peer unit's partial is published
            if (w.kind == WK_OWNER) {
                if (threadIdx.x >= 64 && threadIdx.x < 96) {
                    // one lane per peer: every flag is polled at the same time
                    const int32_t np = n_peers(w);
                    for (int32_t j0 = 0; j0 < np; j0 += 32) {
                        if (j0 + lane < np) {
                            const int32_t v = peer_at(w, j0 + lane);
                            const uint32_t* flag = p.flags + sk_slot(un, v, v == w.h0);
                            const uint64_t t0 = globaltimer_ns();
                            uint32_t it = 0;
                            while (ld_acquire_gpu(flag) != p.epoch) {
                                if ((++it & 15u) == 0) {
                                    if (*abort_flag) break;
                                    if (globaltimer_ns() - t0 > p.timeout_ns) {
                                        raise_error(ctl.abort, ctl.status, DEV_ERR_TIMEOUT);
                                        break;
                                    }
                                }
                            }
                        }
                        __syncwarp();
                        if (*abort_flag) break;
                    }
                }
                if (!epi_sync() || *abort_flag) ok = false;
            }

            // A stream-K owner item that ends its unit leaves the other TMEM
            // accumulator idle (the MMA warp has no further item): the sum of
            // the peers' partial tiles is loaded into it while this item's
            // mainloop still runs, so the fix-up reads TMEM instead of L2.
            const bool preload = ACC_BUFS == 2 && w.kind == WK_OWNER && n_peers(w) > 0 &&
                                 sched_sk_last(st) && ok;
            if (preload && rows_live) {
                for (int c = 0; c < nch; ++c) {
                    const int32_t col0 = c * EPI_COLS;
                    // float4 groups of the chunk inside N (partials past N are never written)
                    const int nq = min(16, (N - (n0 + col0) + 3) / 4);
                    float ps[64];
#pragma unroll
                    for (int i = 0; i < 64; ++i) ps[i] = 0.0f;
                    sum_partials([&](int32_t j) { return peer_src(w, peer_at(w, j), col0); },
                                 n_peers(w), nq, ps, true, pol_once);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t r[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(ps[32 * h + i]);
                        tmem_st32(tmem_base + lane_base + (ab ^ 1u) * BN + col0 + h * 32, r);
                    }
                }
                tmem_st_wait();
            }

            if (!wait_bar(ctl, accf_bar(ab), aph)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint64_t* tr = (threadIdx.x == 64) ? trace_rec(p, static_cast<int32_t>(n_acc)) : nullptr;
            if (tr) {
                tr[0] = static_cast<uint32_t>(w.tile) | (static_cast<uint64_t>(w.kind) << 32);
                tr[1] = static_cast<uint32_t>(w.kb0) | (static_cast<uint64_t>(w.kb1) << 32);
                tr[4] = globaltimer_ns();
                tr[7] = 0;
            }

            if (tr) tr[5] = globaltimer_ns();
            // the output chunks of this item: values from TMEM (plus stream-K
            // peers), or with from_ws the sum of the tile's split partials
            auto run_chunks = [&](bool from_ws, bool to_ws, bool stage_c) {
#pragma unroll 1
            for (int c = 0; ok && rows_live && c < nch; ++c) {
                const int32_t col0 = c * EPI_COLS;
                // float4 groups of the chunk inside N: partial tiles are written
                // and read only there (a swap-AB tile of a 16-token problem has 4)
                const int nq = min(16, (N - (n0 + col0) + 3) / 4);
                const uint32_t b = WHOLE ? static_cast<uint32_t>(c) : (n_chunk & 1u);
                const uint32_t buf = ebuf0 + b * EPI_BUF_BYTES;
                // bias by output column: lane j < 8 fetches columns 8j..8j+7 of the chunk
                uint4 bias8 = make_uint4(0u, 0u, 0u, 0u);
                if (has_bias && !p.bias_rows && !to_ws)
                    bias8 = load_bias8(p.bias, static_cast<int64_t>(n0) + col0 + 8 * (lane & 7), N);
                if (WHOLE) {
                    // nothing to wait for: the boxes were freed when the tile started
                } else if (stage_c) {
                    // prefetch C of the next chunk into the other buffer once the
                    // store that last used it has read it
                    if (c + 1 < nch && lane == 0) {
                        bulk_wait_read<0>();
                        mbar_arrive_expect_tx(c_bar(e, b ^ 1u), EPI_BUF_BYTES);
                        tma_load_2d_hint(ebuf0 + (b ^ 1u) * EPI_BUF_BYTES, tC, c_bar(e, b ^ 1u),
                                         n0 + col0 + EPI_COLS, row0, pol_once);
                        c_pending |= 1u << (b ^ 1u);
                    }
                    __syncwarp();
                } else if (!to_ws) {
                    // the store issued two chunks ago from this buffer must have read it
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                }
                float v[64];
                if (from_ws) {
                    // the tile's split partials in split order (this CTA's own included)
#pragma unroll
                    for (int i = 0; i < 64; ++i) v[i] = 0.0f;
                    const int32_t slot0 = (w.slot / p.splits) * p.splits;
                    sum_partials([&](int32_t sp) {
                                     return reinterpret_cast<const float4*>(
                                                p.ws + static_cast<size_t>(slot0 + sp) * TILE_M * BN) + peer_off(col0);
                                 },
                                 p.splits, nq, v, false, pol_once);
                } else {
                uint32_t r[2][32];
                const uint32_t taddr = tmem_base + lane_base + ab * BN + col0;
                tmem_ld32(taddr, r[0]);
                tmem_ld32(taddr + 32, r[1]);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v[i] = __uint_as_float(r[0][i]);
                    v[32 + i] = __uint_as_float(r[1][i]);
                }
                if (preload) {
                    // the peers' sum, staged in the idle accumulator
                    const uint32_t paddr = tmem_base + lane_base + (ab ^ 1u) * BN + col0;
                    tmem_ld32(paddr, r[0]);
                    tmem_ld32(paddr + 32, r[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        v[i] += __uint_as_float(r[0][i]);
                        v[32 + i] += __uint_as_float(r[1][i]);
                    }
                } else if (w.kind == WK_OWNER) {
                    // add the peer units' partial tiles in unit order (deterministic)
                    sum_partials([&](int32_t j) { return peer_src(w, peer_at(w, j), col0); },
                                 n_peers(w), nq, v, false, pol_once);
                }
                }  // from TMEM
                if (tr && w.kind == WK_OWNER && c == 0) tr[7] = globaltimer_ns();  // peers added
                if (to_ws) {
                    float4* dst = reinterpret_cast<float4*>(p.ws + static_cast<size_t>(w.slot) * TILE_M * BN);
                    if (w.kind == WK_PEER || p.splitk_inline) {
                        // read back by the owner's (or the last split's) epilogue, in the same layout
                        dst += peer_off(col0);
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (i < nq)
                                __stcg(dst + 32 * i, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
                    } else {
                        // split-K partials: row-major tiles, as the reduction kernel reads them
                        dst += (static_cast<size_t>(q * 32 + lane) * BN + col0) / 4;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (i < nq)
                                __stcg(dst + i, make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]));
                    }
                    continue;
                }
                if (p.out_trans) {
                    // swap-AB: computed element (row, n0 + col0 + i) is stored element
                    // (n0 + col0 + i, row) of C / D / Z; for a fixed i the warp's 32
                    // lanes touch 32 consecutive elements (64 bytes)
                    const int32_t my_row = row0 + lane;
                    const int32_t cvalid = N - (n0 + col0);  // columns of this chunk in range
                    const bool live = my_row < M;
                    const int64_t c0 = static_cast<int64_t>(n0) + col0;
                    if (has_c && live) {
                        const uint16_t* cb = static_cast<const uint16_t*>(p.C) + my_row;
#pragma unroll
                        for (int i = 0; i < 64; ++i) {
                            const float cv = i < cvalid ? half_bits_to_float<ELEM>(cb[(c0 + i) * p.ldc]) : 0.0f;
                            v[i] = fmaf(beta, cv, alpha * v[i]);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 64; ++i) v[i] *= alpha;
                    }
                    if (has_bias && p.bias_rows) {
#pragma unroll
                        for (int i = 0; i < 64; ++i) v[i] += bias_row;
                    } else if (has_bias) {
                        // bias by computed column: the same 64 elements for every lane
                        const uint16_t* bb = static_cast<const uint16_t*>(p.bias) + c0;
#pragma unroll
                        for (int i = 0; i < 64; ++i)
                            v[i] += i < cvalid ? half_bits_to_float<ELEM>(__ldg(bb + i)) : 0.0f;
                    }
                    if (p.pre && live) {
                        // the pre-activation output, transposed like D
                        uint16_t* yb = static_cast<uint16_t*>(p.pre) + my_row;
#pragma unroll
                        for (int i = 0; i < 64; i += 2) {
                            const uint32_t pr = pack2<ELEM>(v[i], v[i + 1]);
                            if (i < cvalid) yb[(c0 + i) * p.ldpre] = static_cast<uint16_t>(pr);
                            if (i + 1 < cvalid) yb[(c0 + i + 1) * p.ldpre] = static_cast<uint16_t>(pr >> 16);
                        }
                    }
                    activate_all(v, act);
                    if (p.aux_op && live) {
                        const uint16_t* zb = static_cast<const uint16_t*>(p.aux) + my_row;
#pragma unroll
                        for (int i = 0; i < 64; ++i) {
                            const float z = i < cvalid ? half_bits_to_float<ELEM>(zb[(c0 + i) * p.ldaux]) : 1.0f;
                            v[i] = aux_apply(v[i], z, p.aux_op);
                        }
                    }
                    if (p.out_tma) {
                        // the chunk transposed into the warp's staging box (row i = computed
                        // column i: this warp's 32 computed rows, 64 bytes; conflict-free),
                        // then one TMA store through the transposed tensor map, which
                        // clips rows and columns past the edges
#pragma unroll
                        for (int i = 0; i < 64; i += 2) {
                            const uint32_t pr = pack2<ELEM>(v[i], v[i + 1]);
                            st_shared_u16(buf + i * 64 + lane * 2, static_cast<uint16_t>(pr));
                            st_shared_u16(buf + (i + 1) * 64 + lane * 2, static_cast<uint16_t>(pr >> 16));
                        }
                        fence_async_shared();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d_hint(tD, buf, row0, n0 + col0, pol_once);
                            bulk_commit();
                        }
                        ++n_chunk;
                        __syncwarp();
                    } else if (live) {
                        uint16_t* db = reinterpret_cast<uint16_t*>(Dptr) + my_row;
#pragma unroll
                        for (int i = 0; i < 64; i += 2) {
                            const uint32_t pr = pack2<ELEM>(v[i], v[i + 1]);
                            if (i < cvalid) db[(c0 + i) * ldd] = static_cast<uint16_t>(pr);
                            if (i + 1 < cvalid) db[(c0 + i + 1) * ldd] = static_cast<uint16_t>(pr >> 16);
                        }
                    }
                    continue;
                }
                if (stage_c) {
                    if (!wait_bar(ctl, c_bar(e, b), (c_phase >> b) & 1u)) {
                        ok = false;
                        break;
                    }
                    c_phase ^= 1u << b;
                    c_pending &= ~(1u << b);
                }
                // The TMA store clips columns only at 16-byte granularity: a last
                // chunk that ends inside a 16-byte group is written element-wise.
                const int32_t left = N - (n0 + col0);
                const bool ragged = left < EPI_COLS && (left & 7) != 0;
                const int32_t my_row = row0 + lane;
                OutT* drow = Dptr + static_cast<int64_t>(my_row) * ldd + n0 + col0;
                // 128-byte swizzle: 16-byte chunk j of row `lane` sits at j ^ (lane % 8)
                auto slot_of = [&](int j) { return buf + lane * 128 + ((j ^ (lane & 7)) << 4); };
                // alpha * acc (+ beta * C), then the bias, then the activation, then
                // 16-bit pairs: each phase is straight-line code chosen by one
                // uniform branch, and all eight C loads come before any store
                if (stage_c) {
                    uint4 cvs[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) cvs[j] = ld_shared_v4(slot_of(j));
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t cw[4] = {cvs[j].x, cvs[j].y, cvs[j].z, cvs[j].w};
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const float2 f = unpack2<ELEM>(cw[t]);
                            v[8 * j + 2 * t] = fmaf(beta, f.x, alpha * v[8 * j + 2 * t]);
                            v[8 * j + 2 * t + 1] = fmaf(beta, f.y, alpha * v[8 * j + 2 * t + 1]);
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i) v[i] *= alpha;
                }
                if (has_bias) {
                    if (p.bias_rows) {
#pragma unroll
                        for (int i = 0; i < 64; ++i) v[i] += bias_row;
                    } else {
                        // lane j (< 8) holds columns 8j..8j+7 of this chunk
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint32_t bw[4] = {__shfl_sync(0xffffffffu, bias8.x, j),
                                                    __shfl_sync(0xffffffffu, bias8.y, j),
                                                    __shfl_sync(0xffffffffu, bias8.z, j),
                                                    __shfl_sync(0xffffffffu, bias8.w, j)};
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const float2 f = unpack2<ELEM>(bw[t]);
                                v[8 * j + 2 * t] += f.x;
                                v[8 * j + 2 * t + 1] += f.y;
                            }
                        }
                    }
                }
                if (p.pre && my_row < M)  // the pre-activation output
                    store_row64<ELEM>(static_cast<uint16_t*>(p.pre) + static_cast<int64_t>(my_row) * p.ldpre +
                                          n0 + col0, v, left);
                activate_all(v, act);
                if (p.aux_op && my_row < M) {
                    // the auxiliary tensor's 64 columns of this row, 16 bytes at a time
                    const uint16_t* zrow = static_cast<const uint16_t*>(p.aux) +
                                           static_cast<int64_t>(my_row) * p.ldaux + n0 + col0;
                    uint4 zv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) zv[j] = load_bias8(zrow + 8 * j, 0, left - 8 * j);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t zw[4] = {zv[j].x, zv[j].y, zv[j].z, zv[j].w};
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const float2 f = unpack2<ELEM>(zw[t]);
                            v[8 * j + 2 * t] = aux_apply(v[8 * j + 2 * t], f.x, p.aux_op);
                            v[8 * j + 2 * t + 1] = aux_apply(v[8 * j + 2 * t + 1], f.y, p.aux_op);
                        }
                    }
                }
                uint32_t pk[8][4];
#pragma unroll
                for (int j = 0; j < 8; ++j)
#pragma unroll
                    for (int t = 0; t < 4; ++t) pk[j][t] = pack2<ELEM>(v[8 * j + 2 * t], v[8 * j + 2 * t + 1]);
                if (!ragged) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) st_shared_v4(slot_of(j), pk[j][0], pk[j][1], pk[j][2], pk[j][3]);
                } else if (my_row < M) {
                    // the rounded values are stored element-wise from their 16-bit pairs
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
#pragma unroll
                        for (int t = 0; t < 8; ++t) {
                            if (8 * j + t < left) {
                                const uint16_t h = static_cast<uint16_t>(pk[j][t >> 1] >> (16 * (t & 1)));
                                reinterpret_cast<uint16_t*>(drow)[8 * j + t] = h;
                            }
                        }
                    }
                }
                if (!ragged) {
                    fence_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d_hint(tD, buf, n0 + col0, row0, pol_once);
                        bulk_commit();
                    }
                    ++n_chunk;  // only chunks that stored from their buffer flip it
                }
                __syncwarp();
            }
            };
            run_chunks(false, to_ws, stage_c);
            // accumulator fully read: hand the TMEM buffer back to the MMA warp
            // (the leader's barrier counts the epilogue warps of both CTAs)
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 1) mbar_arrive(acce_bar(ab));
                else mbar_arrive_cluster(acce_bar(ab), 0);
            }
            if (tr) tr[6] = globaltimer_ns();
            ++n_acc;

            if (w.kind == WK_PEER) {
                // publish this CTA's partial tile for the owner
                __threadfence();
                const bool synced = epi_sync();
                if (threadIdx.x == 64 && ok && synced && !*abort_flag &&
                    p.fault_skip_flag != un.id) {
                    st_release_gpu(p.flags + w.slot, p.epoch);
                    if (tr) tr[7] = globaltimer_ns();
                }
                if (!synced) ok = false;
            }
            if (w.kind == WK_SPLIT && p.splitk_inline && ok) {
                // this split's partial is written: count the tile's arrivals; the
                // split that arrives last adds every partial in split order and
                // writes the tile (no CTA waits for another)
                __threadfence();
                volatile uint32_t* last_flag = misc + 3;
                if (!epi_sync()) ok = false;
                if (ok && threadIdx.x == 64) {
                    unsigned long long* ctr =
                        reinterpret_cast<unsigned long long*>(p.flags) + (static_cast<int64_t>(w.tile) * CG + un.rank);
                    const uint32_t n = count_arrival(ctr, p.epoch);
                    if (n == 0u) raise_error(ctl.abort, ctl.status, DEV_ERR_TIMEOUT);
                    *last_flag = (n == static_cast<uint32_t>(p.splits)) ? 1u : 0u;
                }
                if (ok && !epi_sync()) ok = false;
                if (ok && *last_flag && !*abort_flag) {
                    __threadfence();
                    const bool sc = has_c && rows_live && !p.out_trans;
                    issue_c(false, sc);
                    run_chunks(true, false, sc);
                }
            }
            if (*abort_flag) ok = false;
        }
        // drain outstanding C loads; D stores must have read their boxes before
        // the shared memory goes away (their global writes complete with the grid)
        if (lane == 0) {
            for (int b = 0; b < EPI_BUFS; ++b)
                if (c_pending & (1u << b)) drain_bar(c_bar(e, b), (c_phase >> b) & 1u, 200000000ull);
            bulk_wait_read<0>();
        }
        __syncwarp();
    }

    // lanes 1..31 of the producer and MMA warps wait here for their lane 0, so
    // that every warp reaches the CTA barrier converged
    __syncwarp();
    if (trace_hdr && threadIdx.x == 64) *reinterpret_cast<volatile uint32_t*>(misc + 2) = 1u;
    tc_fence_before();
    __syncthreads();
    if (trace_hdr && threadIdx.x == 0) {
        // 1 if the first epilogue thread's write before the barrier is visible after it
        trace_hdr[4] = *reinterpret_cast<volatile uint32_t*>(misc + 2);
        trace_hdr[2] = globaltimer_ns();
    }
    if (trace_hdr && threadIdx.x == 64) trace_hdr[3] = globaltimer_ns();
    // the pair's MMAs read both CTAs' shared memory and write both TMEMs
    if constexpr (CG == 2) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, TR::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ split-K reduction

// D = act(alpha * sum_s partial_s + beta * C + bias) [op Z] for split-K runs
// (splits >= 1), or D = act(beta * C + bias) [op Z] when K == 0 (splits == 0);
// the value before the activation also goes to Y when requested.  A block is
// G warps (G = blockDim.x / 32, at most REDUCE_MAX_GROUPS) over 32 output
// elements of REDUCE_COLS consecutive columns: warp g sums its fixed share of
// the partials in order, then warp 0 adds the G group sums in order and runs
// the epilogue, so the result does not depend on timing.  Launched as a
// programmatic dependent of the GEMM kernel: it waits for that grid here.
template <int ELEM>
__global__ void __launch_bounds__(32 * REDUCE_MAX_GROUPS) splitk_reduce_kernel(const __grid_constant__ ReduceParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int V = REDUCE_COLS;
    __shared__ float4 group_sum[REDUCE_MAX_GROUPS][32];
    const int G = static_cast<int>(blockDim.x >> 5);
    const int g = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int64_t nv = (p.N + V - 1) / V;
    const int64_t total = static_cast<int64_t>(p.M) * nv;
    const int64_t batches = (total + 31) / 32;
    float alpha = p.alpha;
    if (p.scale_a) alpha *= __ldg(p.scale_a);
    if (p.scale_b) alpha *= __ldg(p.scale_b);
    const size_t tile_elems = static_cast<size_t>(TILE_M) * p.tile_n;
    for (int64_t bt = blockIdx.x; bt < batches; bt += gridDim.x) {  // uniform per block
        const int64_t idx = bt * 32 + lane;
        const bool live = idx < total;
        const int32_t m = live ? static_cast<int32_t>(idiv(idx, nv)) : 0;
        const int32_t n = live ? static_cast<int32_t>(idx - static_cast<int64_t>(m) * nv) * V : 0;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (live && (p.units > 0 || p.splits > 0)) {
            const int32_t mb = m / TILE_M, r = m - mb * TILE_M;
            const int32_t nb = n / p.tile_n, cc = n - nb * p.tile_n;
            const float* base = p.ws + static_cast<size_t>(r) * p.tile_n + cc;
            // the partials of this element in their fixed order: split order, or
            // for balanced split-K the unit order of the tile's holders h0..h1
            // (h0's piece, the tile's head, sits in slot 2*h0 + 1, the others' in 2*v)
            int64_t P, h0 = 0;
            if (p.units > 0) {
                const int64_t t0 = static_cast<int64_t>(raster_tile(mb, nb, p.m_blocks, p.n_blocks, p.raster)) * p.k_blocks;
                auto begin = [&](int64_t u) { return idiv(p.sk_units * u, p.units); };
                auto unit_of = [&](int64_t x) {
                    int64_t u = idiv(x * p.units, p.sk_units);
                    while (u > 0 && begin(u) > x) --u;
                    while (u + 1 < p.units && begin(u + 1) <= x) ++u;
                    return u;
                };
                h0 = unit_of(t0);
                P = unit_of(t0 + p.k_blocks - 1) - h0 + 1;
            } else {
                base += static_cast<size_t>(mb * p.n_blocks + nb) * p.splits * tile_elems;
                P = p.splits;
            }
            auto partial = [&](int64_t j) -> const float4* {
                const int64_t slot = p.units > 0 ? (j == 0 ? 2 * h0 + 1 : 2 * (h0 + j)) : j;
                return reinterpret_cast<const float4*>(base + slot * tile_elems);
            };
            const int64_t j0 = idiv(P * g, G), j1 = idiv(P * (g + 1), G);
            constexpr int U = 8;
            int64_t j = j0;
            for (; j + U <= j1; j += U) {
                float4 a[U];
#pragma unroll
                for (int u = 0; u < U; ++u) a[u] = __ldcg(partial(j + u));
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    acc.x += a[u].x; acc.y += a[u].y; acc.z += a[u].z; acc.w += a[u].w;
                }
            }
            for (; j < j1; ++j) {
                const float4 a = __ldcg(partial(j));
                acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
            }
        }
        if (g > 0) group_sum[g][lane] = acc;
        __syncthreads();
        if (g == 0 && live) {
            for (int gg = 1; gg < G; ++gg) {
                const float4 a = group_sum[gg][lane];
                acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
            }
            epilogue_cols4<ELEM>(p, alpha, m, n, acc);
        }
        __syncthreads();  // group_sum is reused by the next batch
    }
}

}  // namespace g15
