/*
 * gemm_oracle.c -- the CPU oracle for the GEMM path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load or call this code.  The
 * library (tiled_tensor_core_persistent_gb300) never does, and it shares no
 * code, header, table or constant with it.
 *
 * What it computes (the plain definition, no blocking, fusion or reordering):
 *
 *   D_ref(i,j) = act( alpha * sA * sB * sum_{k=0}^{K-1} a(i,k) * b(k,j)
 *                     + [beta != 0] * beta * c(i,j)
 *                     + bias(j) )
 *
 *   - "CUTLASS" (stanleyjacob.dev), Part I, the one-GEMM identity
 *     D = alpha * (A @ B) + beta * C with A M x K, B K x N, D M x N.
 *   - same page, Part II (LinearCombination epilogue: alpha * acc + beta * C)
 *     and Part VII Lab 4 (ReLU or GELU applied after alpha*AB + beta*C).
 *   - same page, Part IV Stage 5 (bias add, GELU and a dequantisation scale
 *     fused into the epilogue): the bias is added before the activation, and
 *     the FP8 per-tensor scales sA, sB multiply the raw sum.
 *
 * The FP8 per-tensor scales may be refined by optional per-row (i) and
 * per-column (j) fp32 scale vectors, multiplying the raw sum the same way
 * (the per-channel dequantisation scale of the same Stage 5 paragraph).
 *
 * Block-scaled operands (same page, Part V "data types and quantization":
 * narrow formats in which a few neighbouring elements share one scale, an
 * operand handled together with its scales): each run of `blk`
 * consecutive k of row i of A shares the scale sa(i, k / blk), and likewise
 * for column j of B with sb(j, k / blk).  The operand values are then
 * sa(i, k/blk) * a(i,k) and sb(j, k/blk) * b(k,j), and the sum runs over those
 * products.  The scale factors are the 8-bit exponents of the OCP Microscaling
 * formats (E8M0: value 2^(e - 127), e = 255 is NaN) with blk = 32, or the
 * unsigned E4M3 scales of NVFP4 with blk = 16, the readings taken where the
 * page names no format.  The four-bit elements are FP4 E2M1 (OCP MX), two per
 * byte, the even element of each pair in the low nibble.
 *
 * Readings where the pages are silent:
 *   - bias is indexed by the output column j and added before act;
 *   - GELU is the exact erf form 0.5*x*(1+erf(x/sqrt(2)));
 *   - ReLU is x > 0 ? x : 0;
 *   - beta == 0 means C is not read at all (a NaN in C does not propagate).
 *
 * Arithmetic: every stored input is decoded to its exact value (bf16 and e4m3
 * values are exact in double), the dot product is summed in double in
 * increasing k, and the result is returned in double, unrounded.
 *
 * Operand storage (the "layout" of the logical M x K matrix A and K x N
 * matrix B): ROW = row-major with leading dimension ld, COL = column-major.
 * C is row-major M x N with leading dimension ldc.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { OR_ROW = 0, OR_COL = 1 };
enum { OR_BF16 = 0, OR_E4M3 = 1, OR_F32 = 2, OR_F16 = 3, OR_E5M2 = 4, OR_E2M1 = 5 };
enum { OR_SF_E8M0 = 0, OR_SF_UE4M3 = 1 };
enum { OR_ACT_NONE = 0, OR_ACT_RELU = 1, OR_ACT_GELU = 2 };

/* ------------------------------------------------------------------------ */
/* Exact decoders, written from the bit-level definitions of the formats.   */
/* ------------------------------------------------------------------------ */

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 * Normal: (-1)^s * 2^(e-127) * (1 + f/128); subnormal (e = 0):
 * (-1)^s * 2^(-126) * (f/128); e = 255: infinity (f = 0) or NaN. */
double oracle_decode_bf16(uint16_t bits) {
    int s = (bits >> 15) & 1;
    int e = (bits >> 7) & 0xFF;
    int f = bits & 0x7F;
    double v;
    if (e == 0xFF) {
        v = (f == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)f / 128.0, -126);
    } else {
        v = ldexp(1.0 + (double)f / 128.0, e - 127);
    }
    return s ? -v : v;
}

/* float8 e4m3 ("fn" variant from the FP8 formats paper cited on the CUTLASS
 * page, Part XI item 11): 1 sign, 4 exponent bits (bias 7), 3 fraction bits,
 * no infinities, NaN only for exponent 15 with fraction 7, largest finite
 * value 448.  Subnormal (e = 0): (-1)^s * 2^(-6) * (f/8). */
double oracle_decode_e4m3(uint8_t bits) {
    int s = (bits >> 7) & 1;
    int e = (bits >> 3) & 0xF;
    int f = bits & 0x7;
    double v;
    if (e == 0xF && f == 0x7) {
        v = NAN;
    } else if (e == 0) {
        v = ldexp((double)f / 8.0, -6);
    } else {
        v = ldexp(1.0 + (double)f / 8.0, e - 7);
    }
    return s ? -v : v;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Normal: (-1)^s 2^(e-15) (1 + f/1024); subnormal: (-1)^s 2^(-14) (f/1024);
 * e = 31: infinity (f = 0) or NaN. */
double oracle_decode_f16(uint16_t bits) {
    int s = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1F;
    int f = bits & 0x3FF;
    double v;
    if (e == 0x1F) {
        v = (f == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)f / 1024.0, -14);
    } else {
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    }
    return s ? -v : v;
}

/* float8 e5m2 (FP8 formats paper): 1 sign, 5 exponent bits (bias 15), 2
 * fraction bits, IEEE-like specials: e = 31 is infinity (f = 0) or NaN;
 * subnormal (e = 0): (-1)^s 2^(-14) (f/4); largest finite value 57344. */
double oracle_decode_e5m2(uint8_t bits) {
    int s = (bits >> 7) & 1;
    int e = (bits >> 2) & 0x1F;
    int f = bits & 0x3;
    double v;
    if (e == 0x1F) {
        v = (f == 0) ? INFINITY : NAN;
    } else if (e == 0) {
        v = ldexp((double)f / 4.0, -14);
    } else {
        v = ldexp(1.0 + (double)f / 4.0, e - 15);
    }
    return s ? -v : v;
}

/* IEEE binary32, decoded through its bits for the same reason. */
static double decode_f32(const void* p) {
    float x;
    memcpy(&x, p, sizeof x);
    return (double)x;
}

/* FP4 E2M1 (OCP Microscaling formats): 1 sign, 2 exponent bits (bias 1),
 * 1 fraction bit; normal (e > 0): (-1)^s 2^(e-1) (1 + f/2); subnormal
 * (e = 0): (-1)^s (f/2).  No infinities or NaN; largest value 6. */
double oracle_decode_e2m1(uint8_t nibble) {
    int s = (nibble >> 3) & 1;
    int e = (nibble >> 1) & 3;
    int f = nibble & 1;
    double v = (e == 0) ? 0.5 * (double)f : ldexp(1.0 + 0.5 * (double)f, e - 1);
    return s ? -v : v;
}

/* Unsigned E4M3 scale of NVFP4: the E4M3 encoding without its sign bit
 * (4 exponent bits, bias 7, 3 fraction bits); 0x7F is NaN, bit 7 ignored. */
double oracle_decode_ue4m3(uint8_t bits) {
    return oracle_decode_e4m3((uint8_t)(bits & 0x7F));
}

/* E8M0 scale factor of the OCP Microscaling formats: an unsigned 8-bit
 * exponent with bias 127 and no mantissa; 0xFF is NaN. */
double oracle_decode_e8m0(uint8_t bits) {
    if (bits == 0xFF) return NAN;
    return ldexp(1.0, (int)bits - 127);
}

static double decode_scale(int fmt, uint8_t bits) {
    return fmt == OR_SF_UE4M3 ? oracle_decode_ue4m3(bits) : oracle_decode_e8m0(bits);
}

static double g_bf16_table[65536];
static double g_f16_table[65536];
static double g_e4m3_table[256];
static double g_e5m2_table[256];
static pthread_once_t g_tables_once = PTHREAD_ONCE_INIT;

static void build_tables(void) {
    for (int i = 0; i < 65536; ++i) g_bf16_table[i] = oracle_decode_bf16((uint16_t)i);
    for (int i = 0; i < 65536; ++i) g_f16_table[i] = oracle_decode_f16((uint16_t)i);
    for (int i = 0; i < 256; ++i) g_e4m3_table[i] = oracle_decode_e4m3((uint8_t)i);
    for (int i = 0; i < 256; ++i) g_e5m2_table[i] = oracle_decode_e5m2((uint8_t)i);
}

/* ------------------------------------------------------------------------ */
/* Activation functions.                                                     */
/* ------------------------------------------------------------------------ */

double oracle_act(int act, double x) {
    switch (act) {
    case OR_ACT_RELU:
        return x > 0.0 ? x : 0.0;
    case OR_ACT_GELU:
        return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
    default:
        return x;
    }
}

/* ------------------------------------------------------------------------ */
/* The problem description shared by the entry points.                       */
/* ------------------------------------------------------------------------ */

typedef struct {
    int M, N, K;
    double alpha, beta, scale_a, scale_b;
    const void* A; long long lda; int opA;
    const void* B; long long ldb; int opB;
    int ab_dtype;
    const void* C; long long ldc; int c_dtype;
    const void* bias; int bias_dtype;
    int act;
    /* optional per-row (length M) and per-column (length N) fp32 scales */
    const float* row_scale;
    const float* col_scale;
    /* optional block scale factors (E8M0 bytes): sfa[i * ld_sfa + k / blk],
     * sfb[j * ld_sfb + k / blk] */
    const uint8_t* sfa; long long ld_sfa;
    const uint8_t* sfb; long long ld_sfb;
    int blk;
    int sf_fmt;
    /* optional instrumented operation counter (tiny problems only) */
    int count_ops;
} oracle_problem;

static double load_ab(const void* base, int dtype, long long idx) {
    switch (dtype) {
    case OR_E4M3: return g_e4m3_table[((const uint8_t*)base)[idx]];
    case OR_E5M2: return g_e5m2_table[((const uint8_t*)base)[idx]];
    case OR_E2M1: {
        uint8_t byte = ((const uint8_t*)base)[idx >> 1];
        return oracle_decode_e2m1((uint8_t)((idx & 1) ? (byte >> 4) : (byte & 0xF)));
    }
    case OR_F16: return g_f16_table[((const uint16_t*)base)[idx]];
    case OR_F32: return decode_f32((const float*)base + idx);
    default: return g_bf16_table[((const uint16_t*)base)[idx]];
    }
}

static double load_vec(const void* base, int dtype, long long idx) {
    if (dtype == OR_F32) return decode_f32((const float*)base + idx);
    if (dtype == OR_F16) return g_f16_table[((const uint16_t*)base)[idx]];
    return g_bf16_table[((const uint16_t*)base)[idx]];
}

/* Element (i,k) of the logical A and element (k,j) of the logical B. */
static long long a_index(const oracle_problem* p, int i, int k) {
    return p->opA == OR_ROW ? (long long)i * p->lda + k : (long long)k * p->lda + i;
}
static long long b_index(const oracle_problem* p, int k, int j) {
    return p->opB == OR_ROW ? (long long)k * p->ldb + j : (long long)j * p->ldb + k;
}

/* One output element, straight from the definition. */
static double element(const oracle_problem* p, int i, int j, long long* n_mul, long long* n_add) {
    double s = 0.0;
    for (int k = 0; k < p->K; ++k) {
        double a = load_ab(p->A, p->ab_dtype, a_index(p, i, k));
        double b = load_ab(p->B, p->ab_dtype, b_index(p, k, j));
        if (p->sfa) {
            a = decode_scale(p->sf_fmt, p->sfa[(long long)i * p->ld_sfa + k / p->blk]) * a;
            b = decode_scale(p->sf_fmt, p->sfb[(long long)j * p->ld_sfb + k / p->blk]) * b;
        }
        s = s + a * b;
        if (p->count_ops) { ++*n_mul; ++*n_add; }
    }
    double scale = p->alpha * p->scale_a * p->scale_b;
    if (p->row_scale) scale *= decode_f32(p->row_scale + i);
    if (p->col_scale) scale *= decode_f32(p->col_scale + j);
    double d = scale * s;
    if (p->beta != 0.0) d += p->beta * load_vec(p->C, p->c_dtype, (long long)i * p->ldc + j);
    if (p->bias) d += load_vec(p->bias, p->bias_dtype, j);
    return oracle_act(p->act, d);
}

/* ------------------------------------------------------------------------ */
/* Threaded drivers over a list of (row, col) output positions.              */
/* ------------------------------------------------------------------------ */

typedef struct {
    const oracle_problem* p;
    const int* rows; int nrows;   /* output positions: rows[r] x cols[c] */
    const int* cols; int ncols;
    double* out;                  /* nrows x ncols, row-major */
    long long begin, end;         /* flattened range for this worker */
    long long n_mul, n_add;
} work_item;

static void* worker(void* arg) {
    work_item* w = (work_item*)arg;
    for (long long t = w->begin; t < w->end; ++t) {
        int r = (int)(t / w->ncols), c = (int)(t % w->ncols);
        w->out[t] = element(w->p, w->rows[r], w->cols[c], &w->n_mul, &w->n_add);
    }
    return NULL;
}

static int resolve_threads(int nthreads) {
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static long long run_positions(const oracle_problem* p, const int* rows, int nrows,
                               const int* cols, int ncols, double* out, int nthreads,
                               long long* n_mul, long long* n_add) {
    pthread_once(&g_tables_once, build_tables);
    long long total = (long long)nrows * ncols;
    if (total <= 0) return 0;
    int nt = resolve_threads(nthreads);
    if ((long long)nt > total) nt = (int)total;
    work_item* items = (work_item*)calloc((size_t)nt, sizeof(work_item));
    pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
    if (!items || !th) { free(items); free(th); return -1; }
    for (int t = 0; t < nt; ++t) {
        items[t].p = p;
        items[t].rows = rows; items[t].nrows = nrows;
        items[t].cols = cols; items[t].ncols = ncols;
        items[t].out = out;
        items[t].begin = total * t / nt;
        items[t].end = total * (t + 1) / nt;
    }
    for (int t = 1; t < nt; ++t) pthread_create(&th[t], NULL, worker, &items[t]);
    worker(&items[0]);
    for (int t = 1; t < nt; ++t) pthread_join(th[t], NULL);
    long long m = 0, a = 0;
    for (int t = 0; t < nt; ++t) { m += items[t].n_mul; a += items[t].n_add; }
    if (n_mul) *n_mul = m;
    if (n_add) *n_add = a;
    free(items); free(th);
    return total;
}

/* ------------------------------------------------------------------------ */
/* Exported entry points (called through ctypes from oracle/__init__.py).    */
/* ------------------------------------------------------------------------ */

#define PROBLEM_ARGS                                                          \
    int M, int N, int K, double alpha, const void* A, long long lda, int opA, \
    const void* B, long long ldb, int opB, int ab_dtype, double beta,          \
    const void* C, long long ldc, int c_dtype, const void* bias,               \
    int bias_dtype, int act, double scale_a, double scale_b

static oracle_problem make_problem(PROBLEM_ARGS) {
    oracle_problem p;
    memset(&p, 0, sizeof p);
    p.M = M; p.N = N; p.K = K;
    p.alpha = alpha; p.beta = beta; p.scale_a = scale_a; p.scale_b = scale_b;
    p.A = A; p.lda = lda; p.opA = opA;
    p.B = B; p.ldb = ldb; p.opB = opB;
    p.ab_dtype = ab_dtype;
    p.C = C; p.ldc = ldc; p.c_dtype = c_dtype;
    p.bias = bias; p.bias_dtype = bias_dtype;
    p.act = act;
    return p;
}

/* Per-row / per-column dequantisation scales for the next oracle_gemm_*
 * call on this thread (NULL = none).  The vectors are fp32, length M and N. */
static _Thread_local const float* g_row_scale = NULL;
static _Thread_local const float* g_col_scale = NULL;
void oracle_set_channel_scales(const float* row_scale, const float* col_scale) {
    g_row_scale = row_scale;
    g_col_scale = col_scale;
}

/* Block scale factors for the next oracle_gemm_* call on this thread (NULL =
 * none): E8M0 bytes, sfa[i * ld_sfa + kb] for row i of A and k-block kb,
 * sfb[j * ld_sfb + kb] for column j of B, blocks of blk consecutive k. */
static _Thread_local const uint8_t* g_sfa = NULL;
static _Thread_local const uint8_t* g_sfb = NULL;
static _Thread_local long long g_ld_sfa = 0, g_ld_sfb = 0;
static _Thread_local int g_blk = 32;
static _Thread_local int g_sf_fmt = OR_SF_E8M0;
void oracle_set_block_scales(const uint8_t* sfa, long long ld_sfa, const uint8_t* sfb, long long ld_sfb,
                             int blk, int sf_fmt) {
    g_sfa = sfa; g_ld_sfa = ld_sfa;
    g_sfb = sfb; g_ld_sfb = ld_sfb;
    g_blk = blk > 0 ? blk : 32;
    g_sf_fmt = sf_fmt;
}

static void attach_thread_state(oracle_problem* p) {
    p->row_scale = g_row_scale;
    p->col_scale = g_col_scale;
    if (g_sfa && g_sfb) {
        p->sfa = g_sfa; p->ld_sfa = g_ld_sfa;
        p->sfb = g_sfb; p->ld_sfb = g_ld_sfb;
        p->blk = g_blk;
        p->sf_fmt = g_sf_fmt;
    }
}

/* Selected rows x selected columns of D_ref, written to out (nrows x ncols).
 * Returns the number of elements computed, or -1 on allocation failure. */
long long oracle_gemm_select(PROBLEM_ARGS, const int* rows, int nrows,
                             const int* cols, int ncols, double* out, int nthreads) {
    oracle_problem p = make_problem(M, N, K, alpha, A, lda, opA, B, ldb, opB, ab_dtype,
                                    beta, C, ldc, c_dtype, bias, bias_dtype, act,
                                    scale_a, scale_b);
    attach_thread_state(&p);
    return run_positions(&p, rows, nrows, cols, ncols, out, nthreads, NULL, NULL);
}

/* The whole M x N result, row-major in out.  When count_ops is non-zero the
 * scalar multiplies and adds of the dot products are counted one by one into
 * *n_mul and *n_add (instrumentation for tiny problems). */
long long oracle_gemm_full(PROBLEM_ARGS, double* out, int nthreads, int count_ops,
                           long long* n_mul, long long* n_add) {
    oracle_problem p = make_problem(M, N, K, alpha, A, lda, opA, B, ldb, opB, ab_dtype,
                                    beta, C, ldc, c_dtype, bias, bias_dtype, act,
                                    scale_a, scale_b);
    p.count_ops = count_ops;
    attach_thread_state(&p);
    int* rows = (int*)malloc(sizeof(int) * (size_t)(M > 0 ? M : 1));
    int* cols = (int*)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
    if (!rows || !cols) { free(rows); free(cols); return -1; }
    for (int i = 0; i < M; ++i) rows[i] = i;
    for (int j = 0; j < N; ++j) cols[j] = j;
    long long r = run_positions(&p, rows, M, cols, N, out, nthreads, n_mul, n_add);
    free(rows); free(cols);
    return r;
}

/* Decoders over arrays, for the exhaustive pins. */
void oracle_decode_bf16_array(const uint16_t* in, double* out, long long n) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_decode_bf16(in[i]);
}
void oracle_decode_e4m3_array(const uint8_t* in, double* out, long long n) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_decode_e4m3(in[i]);
}
void oracle_decode_f16_array(const uint16_t* in, double* out, long long n) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_decode_f16(in[i]);
}
void oracle_decode_e5m2_array(const uint8_t* in, double* out, long long n) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_decode_e5m2(in[i]);
}
void oracle_decode_e8m0_array(const uint8_t* in, double* out, long long n) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_decode_e8m0(in[i]);
}
void oracle_decode_ue4m3_array(const uint8_t* in, double* out, long long n) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_decode_ue4m3(in[i]);
}
void oracle_decode_e2m1_array(const uint8_t* in, double* out, long long n) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_decode_e2m1(in[i]);
}
void oracle_act_array(int act, const double* in, double* out, long long n) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_act(act, in[i]);
}
