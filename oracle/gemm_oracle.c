/*
 * Oracle for the dense GEMM hot path -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark may load this library.  The GPU product path never links, loads
 * or calls it, and it shares no code with the CUDA sources.
 *
 * What it computes (plain definition, no blocking, no reordering of the sum):
 *
 *     D[i,j] = act( alpha * s_a * s_b * sum_{k=0..K-1} x(A[i,k]) * x(B[k,j])
 *                   + beta * x(C[i,j]) + x(bias[j]) )  [op x(Z[i,j])]
 *
 *   - "D = A*B + C" for a RowMajor fp16 plan is the worked example of
 *     "Python packages associated with CUTLASS" (CUTLASS python/README.md),
 *     section "CUTLASS Python Interface".
 *   - alpha and beta are the linear-combination coefficients of the
 *     GemmArguments in the kwkr.cn blog "CUTLASS Python接口", section 3.3
 *     (D = alpha * A * B + beta * C), which also states fp32 accumulation.
 *   - act is identity, ReLU, sigmoid or tanh, applied to the whole sum, after
 *     the beta*C and bias adds ("CUTLASS Python 接口全解析" section 2.3 fuses the
 *     activation into the epilogue; the kwkr.cn blog section 5.2 applies ReLU
 *     to alpha*(A*B) + beta*C + bias, with a bias vector of length N added to
 *     every row; "Generating State-of-the-Art GEMMs with TorchInductor's
 *     CuteDSL backend", roadmap section, names ReLU, Sigmoid and Tanh as
 *     epilogue activations).  sigmoid(v) = 1 / (1 + e^-v); tanh is the C
 *     library's.  The bias is optional (absent = 0).
 *   - op is an optional elementwise operation with an auxiliary M x N tensor Z
 *     (add, subtract, multiply, divide), applied to the activated value: the
 *     EFC epilogue operations listed in the roadmap section of the CuteDSL page
 *     (auxiliary tensor loads, elementwise add / mul / sub / div, activations).
 *   - s_a, s_b are per-tensor dequantisation scales of fp8 operands (real value
 *     = s * stored value); they are 1 for 16-bit operands.  FP8 mm support is
 *     listed in "Generating State-of-the-Art GEMMs with TorchInductor's CuteDSL
 *     backend", section "CuteDSL 后端支持的功能 / 功能清单".
 *   - element types of A, B, C are bound separately ("CUTLASS Python 接口全解析"
 *     section 2.1); each stored value is decoded exactly to double by x().
 *   - block-scaled operands (the _scaled_mm formats MXFP8 / MXFP4 / NVFP4 of the
 *     CuteDSL page's "功能清单", whose scale types and block sizes that page
 *     leaves to the formats' definitions): every element is multiplied by the
 *     decoded scale of its block of `block` consecutive K indices before the
 *     product -- x(A[i,k]) * x(SA[i, k/block]) and x(B[k,j]) * x(SB[k/block, j]).
 *     MX formats: E4M3 / E5M2 / E2M1 elements, E8M0 scales, block 32; NVFP4:
 *     E2M1 elements, E4M3 scales, block 16 (a per-tensor scale is alpha).
 *
 * The sum runs in double precision in increasing k.  Threads split the rows
 * of D; each row is computed by exactly one thread with the same arithmetic,
 * so the result does not depend on the thread count.
 *
 * Output rounding (double -> fp16 / bf16, round to nearest even) is provided
 * separately for the cases whose expected value is bit-exact.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F16 = 0, OR_BF16 = 1, OR_F32 = 2, OR_E4M3 = 3, OR_F64 = 4,
       OR_E5M2 = 5, OR_E2M1 = 6, OR_UE8M0 = 7 };

/* ---- decoding stored element bits to double, from the format definitions */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^-14 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
double oracle_decode_bf16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133); /* f * 2^-7 * 2^-126 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134); /* (1 + f/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

/* OCP 8-bit E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 fraction bits;
 * no infinities, S.1111.111 is NaN, largest finite magnitude 448. */
double oracle_decode_e4m3(uint8_t q) {
    int sign = (q >> 7) & 1;
    int e = (q >> 3) & 0xf;
    int f = q & 0x7;
    double v;
    if (e == 15 && f == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, -9); /* f * 2^-3 * 2^-6 */
    else
        v = ldexp((double)(8 + f), e - 10); /* (1 + f/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* OCP 8-bit E5M2: 1 sign, 5 exponent (bias 15), 2 fraction bits, with
 * infinities and NaN as in binary16 (it is binary16's top byte). */
double oracle_decode_e5m2(uint8_t q) {
    return oracle_decode_f16((uint16_t)((uint16_t)q << 8));
}

/* OCP 4-bit E2M1 (the element type of MXFP4 / NVFP4), stored one per byte in
 * the low nibble: 1 sign, 2 exponent (bias 1), 1 fraction bit, no infinity or
 * NaN; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double oracle_decode_e2m1(uint8_t q) {
    int sign = (q >> 3) & 1;
    int e = (q >> 1) & 0x3;
    int f = q & 0x1;
    double v = e == 0 ? 0.5 * f : ldexp(1.0 + 0.5 * f, e - 1);
    return sign ? -v : v;
}

/* OCP E8M0 block scale (UE8M0): 8 exponent bits, no sign or fraction; value
 * 2^(e - 127), 0xFF is NaN. */
double oracle_decode_ue8m0(uint8_t q) {
    return q == 0xFF ? NAN : ldexp(1.0, (int)q - 127);
}

static double load_elem(const void* p, int dtype, int64_t idx) {
    switch (dtype) {
    case OR_F16: return oracle_decode_f16(((const uint16_t*)p)[idx]);
    case OR_BF16: return oracle_decode_bf16(((const uint16_t*)p)[idx]);
    case OR_E4M3: return oracle_decode_e4m3(((const uint8_t*)p)[idx]);
    case OR_F32: return (double)((const float*)p)[idx];
    case OR_E5M2: return oracle_decode_e5m2(((const uint8_t*)p)[idx]);
    case OR_E2M1: return oracle_decode_e2m1(((const uint8_t*)p)[idx]);
    case OR_UE8M0: return oracle_decode_ue8m0(((const uint8_t*)p)[idx]);
    default: return ((const double*)p)[idx];
    }
}

/* ---- rounding double -> 16-bit formats, round to nearest, ties to even */

/* Round a finite positive double to a multiple of 2^q (q = quantum exponent),
 * ties to even, returning the integer multiple. */
static double rne_multiple(double a, int q) {
    double m = ldexp(a, -q); /* exact: scaling by a power of two */
    double fl = floor(m);
    double r = m - fl;
    if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    return fl;
}

uint16_t oracle_round_f16(double x) {
    if (isnan(x)) return 0x7e00;
    uint16_t s = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return s;
    int e;
    frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) -> unbiased exponent e-1 */
    int ue = e - 1;
    if (ue < -14) ue = -14; /* subnormal range shares the quantum 2^-24 */
    int q = ue - 10;        /* spacing of representable values */
    double n = rne_multiple(a, q);
    double v = ldexp(n, q); /* rounded magnitude */
    if (v >= 65536.0) return s | 0x7c00; /* beyond max finite 65504 -> inf */
    if (v < ldexp(1.0, -14)) return s | (uint16_t)n; /* subnormal (or zero) */
    int ve;
    frexp(v, &ve);
    int E = ve - 1;
    uint16_t frac = (uint16_t)(ldexp(v, -E) * 1024.0 - 1024.0);
    return s | (uint16_t)((E + 15) << 10) | frac;
}

uint16_t oracle_round_bf16(double x) {
    if (isnan(x)) return 0x7fc0;
    uint16_t s = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return s;
    int e;
    frexp(a, &e);
    int ue = e - 1;
    if (ue < -126) ue = -126;
    int q = ue - 7;
    double n = rne_multiple(a, q);
    double v = ldexp(n, q);
    if (v >= ldexp(1.0, 128)) return s | 0x7f80;
    if (v < ldexp(1.0, -126)) return s | (uint16_t)n;
    int ve;
    frexp(v, &ve);
    int E = ve - 1;
    uint16_t frac = (uint16_t)(ldexp(v, -E) * 128.0 - 128.0);
    return s | (uint16_t)((E + 127) << 7) | frac;
}

void oracle_round_f16_array(const double* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_f16(x[i]);
}
void oracle_round_bf16_array(const double* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(x[i]);
}
void oracle_decode_array(const void* p, int dtype, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = load_elem(p, dtype, i);
}

/* ---- the GEMM definition */

typedef struct {
    const void* A; int a_dtype; int64_t lda; int a_col_major;
    const void* B; int b_dtype; int64_t ldb; int b_col_major;
    const void* C; int c_dtype; int64_t ldc;
    double* D; int64_t ldd;      /* D[(i - row_begin) * ldd + j] */
    int64_t M, N, K;
    double alpha, beta, scale_a, scale_b;
    int act;                     /* 0 identity, 1 ReLU, 2 sigmoid, 3 tanh */
    const void* bias; int bias_dtype;  /* N elements, or NULL */
    const void* aux; int aux_dtype; int64_t ldaux; int aux_op;  /* Z, row-major; op 0 none,
                                                                   1 add, 2 sub, 3 mul, 4 div */
    /* block scales: A[i,k] is scaled by SA[i, k / block] (M x ceil(K/block),
     * row-major), B[k,j] by SB[k / block, j] (ceil(K/block) x N, row-major) */
    const void* sa; const void* sb; int s_dtype; int64_t block;
    int absolute;                /* 1: compute sum |a||b| (error bound), no epilogue */
    int64_t row_begin, row_end;
    const double* Bd;            /* B decoded to double, K x N row-major, or NULL */
    int64_t next_row;            /* shared work counter */
    pthread_mutex_t lock;
} oracle_job;

static int64_t a_index(const oracle_job* j, int64_t i, int64_t k) {
    return j->a_col_major ? k * j->lda + i : i * j->lda + k;
}
static int64_t b_index(const oracle_job* j, int64_t k, int64_t n) {
    return j->b_col_major ? n * j->ldb + k : k * j->ldb + n;
}

/* One row of D.  acc is scratch of N doubles.  Loop order i-k-j: for a fixed
 * (i, j) the terms are still added in increasing k. */
static void oracle_row(const oracle_job* j, int64_t i, double* acc) {
    for (int64_t n = 0; n < j->N; ++n) acc[n] = 0.0;
    const int64_t kblocks = j->block > 0 ? (j->K + j->block - 1) / j->block : 0;
    for (int64_t k = 0; k < j->K; ++k) {
        double a = load_elem(j->A, j->a_dtype, a_index(j, i, k));
        if (j->sa) a *= load_elem(j->sa, j->s_dtype, i * kblocks + k / j->block);
        if (j->absolute) a = fabs(a);
        if (j->Bd) {
            const double* brow = j->Bd + k * j->N;
            if (j->absolute)
                for (int64_t n = 0; n < j->N; ++n) acc[n] += a * fabs(brow[n]);
            else
                for (int64_t n = 0; n < j->N; ++n) acc[n] += a * brow[n];
        } else {
            for (int64_t n = 0; n < j->N; ++n) {
                double b = load_elem(j->B, j->b_dtype, b_index(j, k, n));
                if (j->sb) b *= load_elem(j->sb, j->s_dtype, (k / j->block) * j->N + n);
                if (j->absolute) b = fabs(b);
                acc[n] += a * b;
            }
        }
    }
    double* out = j->D + (i - j->row_begin) * j->ldd;
    if (j->absolute) {
        for (int64_t n = 0; n < j->N; ++n) out[n] = acc[n];
        return;
    }
    for (int64_t n = 0; n < j->N; ++n) {
        double v = j->alpha * (j->scale_a * j->scale_b * acc[n]);
        if (j->beta != 0.0) v += j->beta * load_elem(j->C, j->c_dtype, i * j->ldc + n);
        if (j->bias) v += load_elem(j->bias, j->bias_dtype, n);
        switch (j->act) {
        case 1: if (v < 0.0) v = 0.0; break; /* NaN propagates (NaN < 0 is false) */
        case 2: v = 1.0 / (1.0 + exp(-v)); break;
        case 3: v = tanh(v); break;
        default: break;
        }
        if (j->aux_op) {
            const double z = load_elem(j->aux, j->aux_dtype, i * j->ldaux + n);
            switch (j->aux_op) {
            case 1: v = v + z; break;
            case 2: v = v - z; break;
            case 3: v = v * z; break;
            case 4: v = v / z; break;
            default: break;
            }
        }
        out[n] = v;
    }
}

static void* oracle_worker(void* arg) {
    oracle_job* j = (oracle_job*)arg;
    double* acc = (double*)malloc(sizeof(double) * (size_t)(j->N > 0 ? j->N : 1));
    if (!acc) return (void*)1;
    for (;;) {
        pthread_mutex_lock(&j->lock);
        int64_t i = j->next_row++;
        pthread_mutex_unlock(&j->lock);
        if (i >= j->row_end) break;
        oracle_row(j, i, acc);
    }
    free(acc);
    return NULL;
}

/* Computes rows [row_begin, row_end) of D into D_out (fp64, row stride ldd).
 * C may be NULL when beta == 0 (it is then never read).
 * Returns 0 on success, nonzero on bad arguments or allocation failure. */
int oracle_gemm(const void* A, int a_dtype, int64_t lda, int a_col_major,
                const void* B, int b_dtype, int64_t ldb, int b_col_major,
                const void* C, int c_dtype, int64_t ldc,
                double* D_out, int64_t ldd,
                int64_t M, int64_t N, int64_t K,
                double alpha, double beta, double scale_a, double scale_b,
                int act, const void* bias, int bias_dtype,
                const void* aux, int aux_dtype, int64_t ldaux, int aux_op,
                const void* sa, const void* sb, int s_dtype, int64_t block,
                int absolute, int64_t row_begin, int64_t row_end,
                int nthreads) {
    if (M < 0 || N < 0 || K < 0 || row_begin < 0 || row_end > M || row_begin > row_end)
        return 1;
    if (!D_out || (K > 0 && (!A || !B)) || (beta != 0.0 && !absolute && !C)) return 1;
    oracle_job j;
    memset(&j, 0, sizeof(j));
    j.A = A; j.a_dtype = a_dtype; j.lda = lda; j.a_col_major = a_col_major;
    j.B = B; j.b_dtype = b_dtype; j.ldb = ldb; j.b_col_major = b_col_major;
    j.C = C; j.c_dtype = c_dtype; j.ldc = ldc;
    j.D = D_out; j.ldd = ldd;
    j.M = M; j.N = N; j.K = K;
    j.alpha = alpha; j.beta = beta; j.scale_a = scale_a; j.scale_b = scale_b;
    if (act < 0 || act > 3 || aux_op < 0 || aux_op > 4 || (aux_op && !aux)) return 1;
    j.act = act; j.bias = bias; j.bias_dtype = bias_dtype; j.absolute = absolute;
    j.aux = aux; j.aux_dtype = aux_dtype; j.ldaux = ldaux; j.aux_op = aux_op;
    if ((sa || sb) && block < 1) return 1;
    j.sa = sa; j.sb = sb; j.s_dtype = s_dtype; j.block = block;
    j.row_begin = row_begin; j.row_end = row_end; j.next_row = row_begin;
    /* Decode B once (the same exact values load_elem would produce); if the
     * copy does not fit in memory, decode element by element instead. */
    double* bd = NULL;
    if (K > 0 && N > 0 && (double)K * (double)N * 8.0 < 8.0e9) {
        bd = (double*)malloc(sizeof(double) * (size_t)K * (size_t)N);
        if (bd)
            for (int64_t k = 0; k < K; ++k)
                for (int64_t n = 0; n < N; ++n) {
                    double b = load_elem(B, b_dtype, b_index(&j, k, n));
                    if (j.sb) b *= load_elem(j.sb, j.s_dtype, (k / j.block) * N + n);
                    bd[k * N + n] = b;
                }
    }
    j.Bd = bd;
    pthread_mutex_init(&j.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int started = 0, rc = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[started], NULL, oracle_worker, &j) != 0) break;
        ++started;
    }
    if (oracle_worker(&j) != NULL) rc = 2;
    for (int t = 0; t < started; ++t) {
        void* r = NULL;
        pthread_join(th[t], &r);
        if (r != NULL) rc = 2;
    }
    pthread_mutex_destroy(&j.lock);
    free(bd);
    return rc;
}
