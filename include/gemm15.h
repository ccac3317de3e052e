/*
 * gemm15 -- dense GEMM D = act(alpha * (A . B) + beta * C) on one GB300
 * (sm_103a), behind a plain C ABI.
 *
 * The operation and the plan/run split follow the CUTLASS Python interface
 * as the pages describe it:
 *   - "Python packages associated with CUTLASS" (CUTLASS python/README.md),
 *     section "CUTLASS Python Interface": a plan is declared with element type
 *     and layout, then `plan.run(A, B, C, D)` computes D = A . B + C.
 *   - "CUTLASS Python 接口全解析", section 2.1: element_A/B/C/D/accumulator
 *     are bound separately at plan construction and cannot change afterwards;
 *     one plan runs tensors of any shape with matching types.  Section 2.2:
 *     compilation is separate from execution.  Section 2.3: an elementwise
 *     activation (ReLU) is fused into the epilogue, and `run()` is
 *     asynchronous with an explicit `sync()`.
 *   - kwkr.cn blog "CUTLASS Python接口", section 3.3: the linear combination
 *     D = alpha * A * B + beta * C with fp32 accumulation.
 *   - "Python packages associated with CUTLASS", section "Current
 *     functionality": stream-K and grouped GEMM variants.
 *   - "Generating State-of-the-Art GEMMs with TorchInductor's CuteDSL
 *     backend", section "CuteDSL 后端支持的功能": FP8 mm and grouped mm.
 *
 * Conventions for every entry point:
 *   - A is M x K, B is K x N, C and D are M x N.  Leading dimensions are in
 *     elements.  Row-major X with leading dimension ld stores X[i][j] at
 *     X + i*ld + j; column-major stores it at X + j*ld + i.
 *   - Matrix pointers are DEVICE pointers on the plan's device (except in
 *     gemm_run_host), owned by the caller, and must stay valid until the work
 *     enqueued on `stream` has finished.
 *   - Every pointer and every leading dimension * element size must be a
 *     multiple of 16 bytes (tensor-memory-accelerator rule); otherwise the call
 *     returns GEMM15_ERR_ALIGNMENT and launches nothing.  There is no fallback
 *     path.
 *   - Argument errors are returned synchronously and nothing is launched.
 *     Errors detected on the device (a bounded wait that ran out) are written
 *     to the plan's status word; read them with gemm_plan_query_error after
 *     synchronising the stream.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   - GEMM kernels are launched as programmatic dependents of the kernel
 *     before them in the stream: their set-up may overlap that kernel's tail,
 *     but they read and write no memory before it has completed, so stream
 *     order holds as usual.  They also allow the kernel after them to start
 *     early; a kernel that asks for that (programmatic stream serialization)
 *     must itself wait (griddepcontrol.wait / cudaGridDependencySynchronize)
 *     before reading what the GEMM wrote.
 *   - A plan may be used from one host thread at a time.  Its device state
 *     (workspace, stream-K flags, status word, grouped table, host-path
 *     buffers) serves every call, so calls on one plan never run concurrently
 *     on the GPU: a call enqueued on another stream than the plan's previous
 *     call first makes its stream wait for the previous call's work (an event
 *     the plan records after each call).  Independent GEMMs that should overlap
 *     on different streams need one plan each.
 */
#ifndef GEMM15_H_
#define GEMM15_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM15_F16 = 0,  /* IEEE binary16 */
    GEMM15_BF16 = 1, /* bfloat16 */
    GEMM15_F32 = 2,  /* binary32: accumulator type only */
    GEMM15_E4M3 = 3, /* OCP fp8 e4m3 (finite-only variant), A and B only */
    GEMM15_E5M2 = 4, /* OCP fp8 e5m2, A and B only, block-scaled runs only */
    GEMM15_E2M1 = 5  /* OCP fp4 e2m1, two per byte (element 2i in the low nibble),
                        A and B only, block-scaled runs only */
} gemm15_dtype_t;

typedef enum { GEMM15_ROW_MAJOR = 0, GEMM15_COL_MAJOR = 1 } gemm15_layout_t;

/* Epilogue activation, applied last, to alpha*(A.B) + beta*C (+ bias)
 * ("CUTLASS Python 接口全解析" section 2.3 fuses an activation into the
 * epilogue; the kwkr.cn blog "CUTLASS Python接口" section 5.2 applies ReLU to
 * alpha*(A.B) + beta*C + bias; "Generating State-of-the-Art GEMMs with
 * TorchInductor's CuteDSL backend", roadmap section, lists ReLU, Sigmoid and
 * Tanh as epilogue activations).  NaN propagates through every activation.
 *   SIGMOID: 1 / (1 + exp(-x)), with the fast exponential and division;
 *   TANH:    the hardware approximation (relative error below 2^-10.9, the
 *            order of one fp16 rounding). */
typedef enum {
    GEMM15_EPI_LINEAR = 0,
    GEMM15_EPI_RELU = 1,
    GEMM15_EPI_SIGMOID = 2,
    GEMM15_EPI_TANH = 3
} gemm15_epilogue_t;

typedef enum {
    GEMM15_OK = 0,
    GEMM15_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad enum, ... */
    GEMM15_ERR_UNSUPPORTED = 2,  /* type / layout combination not provided */
    GEMM15_ERR_ALIGNMENT = 3,    /* pointer or leading dimension not 16-byte aligned */
    GEMM15_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed */
    GEMM15_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out */
    GEMM15_ERR_OOM = 6,          /* plan workspace could not be allocated */
    GEMM15_ERR_DEVICE_FAULT = 7, /* the device reported an internal error */
    GEMM15_ERR_NO_DEVICE = 8,    /* no sm_103 device available */
    GEMM15_ERR_BAD_PLAN = 9      /* null, destroyed or foreign plan handle */
} gemm15_status_t;

typedef struct gemm15_plan* gemm15_plan_t;

/* Plan description: element types and layouts, fixed for the plan's life.
 * Supported: a == b in {F16, BF16} with c == d == a; or a == b in {E4M3,
 * E5M2, E2M1} with c == d == BF16 (E5M2 and E2M1 plans run only
 * gemm_run_block_scaled).  acc must be F32.  layout_a / layout_b are free;
 * layout_cd applies to both C and D. */
typedef struct {
    gemm15_dtype_t a, b, c, d, acc;
    gemm15_layout_t layout_a, layout_b, layout_cd;
    gemm15_epilogue_t epilogue;
} gemm15_plan_desc_t;

/* Creates a plan on the current CUDA device: validates the description,
 * allocates the plan's small device state (status word, stream-K flags) and
 * resolves the tensor-map encoder.  Kernels are compiled ahead of time into
 * this library, so this is the whole "compile" step ("CUTLASS Python 接口全解析"
 * section 2.2).  *out receives the handle, owned by the caller until
 * gemm_plan_destroy.  Errors: INVALID_ARG (null), UNSUPPORTED (types),
 * NO_DEVICE, CUDA, OOM. */
gemm15_status_t gemm_plan_create(gemm15_plan_t* out, const gemm15_plan_desc_t* desc);

/* Frees the plan and all device / pinned memory it owns.  The caller must have
 * synchronised every stream the plan was used on.  BAD_PLAN for null or
 * already destroyed handles. */
gemm15_status_t gemm_plan_destroy(gemm15_plan_t plan);

/* D = act(alpha * (A . B) + beta * C) with packed leading dimensions (lda = K
 * for row-major A, M for column-major; ldb = N or K; ldc = ldd = N for
 * row-major C/D, M for column-major).  Asynchronous on `stream`.
 * M == 0 or N == 0: nothing to do, returns OK.  K == 0: D = act(beta * C).
 * beta == 0: C is never read and may be NULL.  The plan's workspace grows on
 * demand (a cudaMalloc outside the stream); do not call a growing shape for the
 * first time inside stream capture. */
gemm15_status_t gemm_run(gemm15_plan_t plan, const void* A, const void* B, const void* C,
                         void* D, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                         void* stream);

/* gemm_run with explicit leading dimensions and, for E4M3 plans, per-tensor
 * fp32 dequantisation scales: the real value of an fp8 operand element is
 * scale * stored value, so D = act(alpha * s_a * s_b * (A_q . B_q) + beta * C).
 * scale_a / scale_b are DEVICE pointers to one float each, or NULL for 1.0;
 * they are read by the kernel, so they may change between enqueued runs. */
gemm15_status_t gemm_run_ex(gemm15_plan_t plan, const void* A, int64_t lda, const void* B,
                            int64_t ldb, const void* C, int64_t ldc, void* D, int64_t ldd,
                            int64_t M, int64_t N, int64_t K, float alpha, float beta,
                            const float* scale_a, const float* scale_b, void* stream);

/* Elementwise operation of an auxiliary tensor Z with the activated value
 * (the EFC epilogue operations -- auxiliary tensor loads, elementwise add /
 * sub / mul / div -- of the roadmap section of "Generating State-of-the-Art
 * GEMMs with TorchInductor's CuteDSL backend"). */
typedef enum {
    GEMM15_AUX_NONE = 0,
    GEMM15_AUX_ADD = 1, /* D = act(...) + Z */
    GEMM15_AUX_SUB = 2, /* D = act(...) - Z */
    GEMM15_AUX_MUL = 3, /* D = act(...) * Z */
    GEMM15_AUX_DIV = 4  /* D = act(...) / Z (IEEE division) */
} gemm15_aux_op_t;

/* Per-run arguments of gemm_run_args (leading dimensions 0 = packed, as in
 * gemm_run). */
typedef struct {
    const void* A;
    int64_t lda;
    const void* B;
    int64_t ldb;
    const void* C;
    int64_t ldc;
    void* D;
    int64_t ldd;
    int64_t M, N, K;
    float alpha, beta;
    const float* scale_a; /* E4M3 plans: DEVICE float, NULL = 1 (as gemm_run_ex) */
    const float* scale_b;
    const void* bias;     /* DEVICE vector of N elements of D's type, or NULL */
    const void* aux;      /* DEVICE M x N tensor Z of D's type and layout, or NULL */
    int64_t ldaux;        /* its leading dimension (0 = packed) */
    int32_t aux_op;       /* gemm15_aux_op_t; GEMM15_AUX_NONE ignores aux */
    void* pre;            /* DEVICE M x N output Y of D's type and layout receiving the
                             pre-activation alpha * s_a * s_b * (A . B) + beta * C + bias
                             (rounded once to D's type), or NULL */
    int64_t ldpre;        /* its leading dimension (0 = packed) */
} gemm15_args_t;

/* D = act(alpha * s_a * s_b * (A . B) + beta * C + bias) [op Z], bias[j]
 * added to every element of column j of D -- the LinearCombinationBiasReLU
 * epilogue of the kwkr.cn blog "CUTLASS Python接口", section 5.2 (bias vector of
 * length N in the output type, fp32 arithmetic, activation last) -- and an
 * optional auxiliary tensor Z entering the activated value by aux_op.  With
 * `pre` set, the epilogue also stores the value before the activation to Y
 * (the auxiliary tensor store of the EFC epilogue operations in the roadmap
 * section of "Generating State-of-the-Art GEMMs with TorchInductor's CuteDSL
 * backend"; what a backward pass through the activation needs).  Y follows
 * the rules of Z: 16-byte aligned pointer and ldpre * 2 (ALIGNMENT otherwise),
 * ldpre >= the contiguous extent (INVALID_ARG otherwise).
 * Everything else as gemm_run_ex; the bias and aux pointers and ldaux * 2 must
 * be 16-byte aligned (ALIGNMENT otherwise), ldaux >= the contiguous extent
 * (INVALID_ARG otherwise).  With K == 0, D = act(beta * C + bias) [op Z]. */
gemm15_status_t gemm_run_args(gemm15_plan_t plan, const gemm15_args_t* args, void* stream);

/* End-to-end variant for callers holding HOST buffers (packed layouts as in
 * gemm_run; pinned memory recommended).  Copies A, B (and C when beta != 0)
 * into plan-owned device buffers, runs the GEMM and copies D back, then
 * synchronises `stream` and returns (and clears) the device status.  Large
 * 16-bit row-major problems (B and D together at least 64 MiB, N >= 4096)
 * run as a pipeline over 4 column chunks: the chunks of B and C go up on
 * a plan-owned copy stream, each chunk's GEMM runs on `stream` as soon as its
 * columns are up, and its D comes back on another plan-owned stream while the
 * next chunk computes.  scale_a / scale_b are HOST floats here (1.0 for 16-bit
 * plans). */
gemm15_status_t gemm_run_host(gemm15_plan_t plan, const void* hA, const void* hB,
                              const void* hC, void* hD, int64_t M, int64_t N, int64_t K,
                              float alpha, float beta, float scale_a, float scale_b,
                              void* stream);

/* One problem of a grouped GEMM (device pointers, leading dimensions as in
 * gemm_run_ex; 0 means packed). */
typedef struct {
    int64_t M, N, K;
    const void* A;
    const void* B;
    const void* C;
    void* D;
    int64_t lda, ldb, ldc, ldd;
    const float* scale_a; /* E4M3 plans: DEVICE floats, the per-tensor scales of */
    const float* scale_b; /* A_g and B_g (NULL = 1); other plans: NULL */
} gemm15_problem_t;

/* Grouped GEMM: D_g = act(alpha * s_a,g * s_b,g * (A_g . B_g) + beta * C_g) for every g in one
 * launch ("Python packages associated with CUTLASS", "Current functionality";
 * "Generating State-of-the-Art GEMMs with TorchInductor's CuteDSL backend",
 * grouped mm).  `problems` is a HOST array of `count` entries, read during the
 * call only.  The plan copies a problem table (shapes, pointers, tensor maps)
 * to device memory on `stream`.  Groups with M, N == 0 are skipped; K == 0
 * groups are not supported (UNSUPPORTED).  Every group must pass the same
 * alignment rules as gemm_run_ex.  E4M3 plans take per-group fp32 scales of
 * A_g and B_g (the grouped fp8 mm of the CuteDSL page, section 5.1), read by
 * the kernel like gemm_run_ex's; a scale on a 16-bit plan is INVALID_ARG. */
gemm15_status_t grouped_gemm_run(gemm15_plan_t plan, const gemm15_problem_t* problems,
                                 int32_t count, float alpha, float beta, void* stream);

/* Batched GEMM: `batch` independent problems of one shape, problem b reading
 * A + b*stride_a, B + b*stride_b, C + b*stride_c and writing D + b*stride_d
 * (strides in elements), D_b = act(alpha * (A_b . B_b) + beta * C_b) -- the
 * batch_count / batch_stride arguments of the kwkr.cn blog "CUTLASS
 * Python接口", section 6.3, where the strides of packed batches are M*K, K*N
 * and M*N.  A stride of 0 shares that operand across the batch (one weight
 * matrix for every batch entry); the D matrices must not overlap.  Leading
 * dimensions as in gemm_run_ex (0 = packed).  Every stride * element size must
 * be a multiple of 16 bytes (ALIGNMENT otherwise).  Runs as one grouped launch
 * (same device table and rules as grouped_gemm_run: K == 0 is UNSUPPORTED);
 * batch == 0, M == 0 or N == 0 do nothing.  INVALID_ARG for batch < 0 or
 * negative strides. */
gemm15_status_t gemm_run_batched(gemm15_plan_t plan, const void* A, int64_t lda, int64_t stride_a,
                                 const void* B, int64_t ldb, int64_t stride_b, const void* C,
                                 int64_t ldc, int64_t stride_c, void* D, int64_t ldd,
                                 int64_t stride_d, int64_t M, int64_t N, int64_t K,
                                 int32_t batch, float alpha, float beta, void* stream);

/* Reads and clears the plan's device status word (GEMM15_OK if no device-side
 * error was recorded).  Synchronises the plan's device; call it after the
 * enqueued work has finished, like `args.sync()` ("CUTLASS Python 接口全解析"
 * section 2.3). */
gemm15_status_t gemm_plan_query_error(gemm15_plan_t plan);

/* Static description of a status code (never NULL). */
const char* gemm15_status_string(gemm15_status_t status);

/* Tuning / test options (defaults are the library's own choices). */
typedef enum {
    GEMM15_OPT_SCHEDULE = 0,     /* 0 auto, 1 data-parallel, 2 stream-K, 3 split-K + reduce */
    GEMM15_OPT_SPLITS = 1,       /* split-K: splits per tile (0 = auto; -1 = balanced:
                                    the k iterations of all tiles cut evenly over
                                    every SM, single-SM tiles only) */
    GEMM15_OPT_CTA_GROUP = 2,    /* 0 auto, 1 one-SM tiles, 2 SM-pair tiles */
    GEMM15_OPT_TILE_N = 3,       /* 0 auto, 128 or 256 */
    GEMM15_OPT_RASTER = 4,       /* 0 auto, else M-blocks per raster band */
    GEMM15_OPT_GRID = 5,         /* 0 auto (one CTA per SM), else max CTAs */
    GEMM15_OPT_TIMEOUT_US = 6,   /* bound of every device-side wait, microseconds */
    GEMM15_OPT_FAULT_SKIP_FLAG = 7, /* test hook: stream-K peer unit that skips its
                                       partial-ready flag (-1 = none) */
    GEMM15_OPT_SK_DP_WAVES = 8,    /* stream-K: full waves run data-parallel before
                                      the stream-K region (-1 = auto) */
    GEMM15_OPT_TRACE_ITEMS = 9,    /* record a per-CTA timeline of up to this many
                                      work items per launch (0 = off); read it
                                      with gemm_plan_trace */
    GEMM15_OPT_SWAP_AB = 10,       /* dense runs: 0 auto (swap-AB when the computed
                                      M <= 128 against N >= 1024 and K >= 256),
                                      1 never, 2 always.  Swap-AB computes
                                      D^T = B^T . A^T on 128 x 64 (16-bit, M <= 64)
                                      or 128 x 128 single-SM tiles and stores the
                                      tile transposed; GEMM15_OPT_TILE_N does not
                                      apply to it, GEMM15_OPT_CTA_GROUP = 2 puts
                                      16-bit 128-wide swap tiles on SM pairs
                                      (256 x 128) */
    GEMM15_OPT_SPLITK_INLINE = 11, /* split-K: 0 auto (when a tile's partials total at
                                      most 256 KiB), 1 never, 2 always: the split that
                                      finishes a tile last (a per-tile arrival
                                      counter) adds all partials in split order and
                                      writes the tile, instead of a separate
                                      reduction kernel; no CTA waits for another */
    GEMM15_OPT_L2_HINTS = 12       /* L2 policies of the operand loads: 0 none, 1 A
                                      (the rows a raster band shares) evict-last,
                                      2 also B evict-first */
} gemm15_option_t;

/* Sets an option on the plan; INVALID_ARG for unknown options or values. */
gemm15_status_t gemm_plan_set_option(gemm15_plan_t plan, gemm15_option_t option, int64_t value);

/* The configuration the last run of the plan launched. */
typedef struct {
    int32_t cta_group;   /* 1 or 2 */
    int32_t tile_m, tile_n, tile_k;
    int32_t stages;
    int32_t schedule;    /* 1 data-parallel, 2 stream-K, 3 split-K + reduce */
    int32_t grid;        /* CTAs launched by the GEMM kernel */
    int32_t tiles;       /* output tiles */
    int32_t splits;      /* split-K splits per tile (1 otherwise; 0 for balanced split-K:
                            the k iterations of all tiles cut evenly over every SM, a
                            piece may straddle two tiles, the reduction kernel finds
                            each tile's pieces) */
    int32_t raster;      /* M-blocks per raster band */
    int32_t launches;    /* kernels launched by the run */
    int32_t swap_ab;     /* 1 if the kernel computed the transpose of the stored
                            product with A and B swapped: D^T = B^T . A^T for
                            row-major C/D under swap-AB, or column-major C/D
                            without it */
} gemm15_config_t;

gemm15_status_t gemm_plan_last_config(gemm15_plan_t plan, gemm15_config_t* out);

/* One candidate measured by gemm_plan_autotune. */
typedef struct {
    gemm15_config_t config;  /* what the candidate launched */
    int32_t sk_dp_waves;     /* stream-K option the candidate forced (-1 = automatic) */
    float us;                /* mean time per run in microseconds (-1 if it failed) */
    gemm15_status_t status;  /* GEMM15_OK, or why the candidate could not run */
} gemm15_tune_result_t;

/* Autotuning: the kwkr.cn blog "CUTLASS Python接口", section 6.2, profiles
 * each kernel configuration for the problem size and data types with its
 * GemmProfiler and keeps the fastest; "Generating State-of-the-Art GEMMs with
 * TorchInductor's CuteDSL backend", section 6.2, autotunes over candidate
 * configurations.  This call runs each candidate the library can launch for this problem
 * -- data-parallel, stream-K (with and without its data-parallel waves) and
 * split-K schedules on single-SM and SM-pair tiles 128 and 256 wide -- once to
 * warm up and then `iterations` times, each timed with CUDA events on
 * `stream` after the L2 cache has been cleared (a write of twice its size to
 * a scratch buffer the call allocates and frees), as when the operands do not
 * stay in L2 between uses; the call synchronises the stream.  The fastest is kept in the plan for
 * this (M, N, K): later gemm_run / gemm_run_ex / gemm_run_args calls of that
 * shape use it wherever the corresponding plan options are left automatic.
 * The operands are used as in gemm_run_args (D is written many times; it ends
 * holding the chosen configuration's result).  The first min(count,
 * capacity) results, fastest first (failed candidates last), go to the HOST
 * array `results`; *count receives the number of candidates.  M, N or K == 0:
 * nothing to choose, OK.  Argument errors as gemm_run_args. */
gemm15_status_t gemm_plan_autotune(gemm15_plan_t plan, const gemm15_args_t* args,
                                   int32_t iterations, gemm15_tune_result_t* results,
                                   int32_t capacity, int32_t* count, void* stream);

/* Drops every autotuned choice of the plan. */
gemm15_status_t gemm_plan_forget_tuning(gemm15_plan_t plan);

/* Copies the timeline of the plan's last traced GEMM-kernel launch (see
 * GEMM15_OPT_TRACE_ITEMS) into the HOST buffer `out` of `capacity` bytes, after
 * synchronising the plan's device.  Layout: for each of *ctas CTAs, one header
 * record then *items item records, 8 uint64 each (globaltimer nanoseconds).
 * Header: start, SM id, time after the final CTA barrier seen by thread 0 and
 * by the first epilogue thread, 1 if thread 0 saw after that barrier a value
 * the first epilogue thread wrote before it.  Item: tile | kind << 32 (0 whole tile, 1
 * stream-K peer part, 2 stream-K owner part, 3 split-K part), kb0 | kb1 << 32,
 * MMA start, MMA issued, accumulator ready, epilogue chunks start, epilogue
 * done, partial published (stream-K peer part) or the peers' partials of the
 * first chunk added (owner part); unused items are zero.  INVALID_ARG if tracing is
 * off or `capacity` is too small (*ctas and *items are still set). */
gemm15_status_t gemm_plan_trace(gemm15_plan_t plan, void* out, int64_t capacity, int32_t* ctas,
                                int32_t* items);

/* Block scaling of fp8 / fp4 operands: one scale per `block` consecutive K
 * elements of a row of A and of a column of B (the _scaled_mm formats MXFP8,
 * MXFP4 and NVFP4 of "Generating State-of-the-Art GEMMs with TorchInductor's
 * CuteDSL backend", section 5.1; their scale types and block sizes are the
 * OCP MX and NVFP4 definitions). */
typedef enum {
    GEMM15_SCALE_MX = 1, /* UE8M0 scales (2^(e-127)) per 32 elements: MXFP8 (E4M3 /
                            E5M2 plans) and MXFP4 (E2M1 plans) */
    GEMM15_SCALE_NV = 2  /* UE4M3 scales (e4m3 bits, positive) per 16 elements:
                            NVFP4 (E2M1 plans); a per-tensor fp32 scale goes in alpha */
} gemm15_scale_kind_t;

/* Arguments of gemm_run_block_scaled.  A is M x K row-major (K contiguous),
 * B is K x N column-major (stored as N rows of K contiguous elements): the
 * "TN" layout.  lda / ldb are in elements (0 = K); for E2M1 they count 4-bit
 * elements and must be even.  SFA holds the M x K/block scales of A, SFB the
 * N x K/block scales of B, both in the 128 x 4 blocked layout the tensor
 * cores read: 512-byte atoms, one per 128 rows (row block rb) and 4
 * consecutive scales along K (column block cb), atom (rb, cb) at byte
 * (rb * K/(4*block) + cb) * 512, the scale of row r, column c at byte
 * 16 * (r % 32) + 4 * ((r % 128) / 32) + c % 4 inside it; rows beyond M (N)
 * up to the next multiple of 128 are padding (any value).  C, D are M x N
 * bf16 row-major (ldc / ldd 0 = N), bias an optional N-vector of bf16. */
typedef struct {
    const void* A;
    int64_t lda;
    const void* B;
    int64_t ldb;
    const void* SFA;
    const void* SFB;
    int32_t scale_kind;  /* gemm15_scale_kind_t */
    const void* C;
    int64_t ldc;
    void* D;
    int64_t ldd;
    int64_t M, N, K;
    float alpha, beta;
    const void* bias;
} gemm15_scaled_args_t;

/* D = act(alpha * sum_k (A[i,k] * SFA[i, k/block]) * (B[k,j] * SFB[j, k/block])
 *        + beta * C + bias): the block-scaled GEMM, on tcgen05 block-scaled MMAs
 * (kind::mxf8f6f4 for MXFP8, kind::mxf4 for MXFP4, kind::mxf4nvf4 for NVFP4;
 * scale factors copied to tensor memory beside the accumulator).  Tiles: SM-pair
 * 256 x 256 (cta_group::2) for MXFP8 and one-SM 128 x 256 for the fp4 kinds by
 * default; GEMM15_OPT_CTA_GROUP = 1 / 2 forces one-SM / SM-pair tiles and
 * GEMM15_OPT_TILE_N = 128 selects 128 x 128 (one SM) or 256 x 128 (SM pair)
 * tiles.  The plan
 * must have layout_a ROW_MAJOR, layout_b COL_MAJOR, layout_cd ROW_MAJOR
 * (UNSUPPORTED otherwise).  K must be a multiple of 128 (fp8) or 256 (fp4)
 * (UNSUPPORTED otherwise); pointers 16-byte aligned and leading dimensions
 * whole multiples of 16 bytes (ALIGNMENT otherwise).  M == 0 or N == 0: OK,
 * nothing launched; K == 0: UNSUPPORTED.  Asynchronous on `stream`. */
gemm15_status_t gemm_run_block_scaled(gemm15_plan_t plan, const gemm15_scaled_args_t* args,
                                      void* stream);

/* ---- Split-K GEMM that allocates nothing.  The pages have no counterpart of
 * this entry point; it exists for callers that cannot call cudaMalloc: code
 * living inside a host application that owns every byte of device memory (an
 * inference server or plugin with a fixed budget), and latency-critical loops
 * where an allocation, which can block and synchronise the device, is not
 * acceptable.  Plans grow their workspace on demand, so such callers use this
 * instead.
 *
 * Computes the same D = act(alpha * s_a * s_b * (A . B) + beta * C) as
 * gemm_run_ex, always as split-K: each output tile's K range is cut into
 * `splits` parts (clamped to the number of K blocks), whose fp32 partial tiles
 * a second kernel sums in a fixed order.  The partial tiles live in one
 * file-scope device array of GEMM15_NOALLOC_SCRATCH_BYTES that every GPU which
 * loads this library holds until the process exits; nothing is allocated per
 * call.  The arguments are those of gemm_run_ex, with the element types and
 * layouts taken from `desc` (no plan), plus:
 *   splits  >= 1; tiles * splits * 128 * tile_n * 4 bytes + 256 must fit in
 *           GEMM15_NOALLOC_SCRATCH_BYTES (tile_n = 128 if N <= 128, else 256;
 *           tiles = ceil(M/128) * ceil(N/tile_n)), otherwise the call returns
 *           GEMM15_ERR_UNSUPPORTED and launches nothing;
 *   status  optional DEVICE pointer to an int32 that the call clears and the
 *           kernels set to GEMM15_ERR_TIMEOUT if a bounded wait runs out; NULL
 *           keeps that word inside the scratch, unreported.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the array and keep the last call's partials, so
 * calls that overlap on the GPU (other streams, other host threads) race and
 * give wrong results: serialise them.  Errors as for gemm_run_ex. */
#define GEMM15_NOALLOC_SCRATCH_BYTES (32u << 20)

gemm15_status_t gemm_run_splitk_noalloc(const gemm15_plan_desc_t* desc, const void* A,
                                        int64_t lda, const void* B, int64_t ldb, const void* C,
                                        int64_t ldc, void* D, int64_t ldd, int64_t M, int64_t N,
                                        int64_t K, float alpha, float beta, const float* scale_a,
                                        const float* scale_b, int32_t splits, int32_t* status,
                                        void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM15_H_ */
