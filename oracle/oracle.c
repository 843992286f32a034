/*
 * CPU oracle for the tensor-core GEMM / implicit-GEMM convolution hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline / reference arm may load this library.  The
 * product path (the CUDA library under implicit_gemm_conv_tcgen05_gb300/) never
 * calls it, shares no code with it, and fails loudly when its own extension is
 * missing.
 *
 * Everything here is the plain definition of what the path computes, written
 * out with no blocking, fusion or reordering beyond splitting output rows over
 * threads (each output element is still computed by one thread, in k order).
 *
 * Pages cited (by title and section):
 *  [P1] "TVM在CUDA GPU上跑GEMM的全套张量化实现：WMMA/DP4A/IMMA + TensorIR调度 +
 *       INT8/FP16多精度支持" -- §2.3 (multi-precision: C = (A_q - zp_A)(B_q - zp_B),
 *       four-term fusion quantize/dequantize), §4.1 (GEMM compute definition
 *       C[i,j] = sum_k A[i,k] * B[k,j], fp16 operands).
 *  [P3] "如何使用 TensorCores 优化卷积" (TVM tutorial "How to optimize convolution
 *       using TensorCores") -- section "准备和算法" (the Apad zero-padded input
 *       and the Conv reduction over ic, kh, kw with operands cast to float32).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - "B column-major": B is stored as Bt, N x K row-major (K contiguous), so
 *    C[i,j] = sum_k A[i,k] * Bt[j,k].  C is M x N row-major.
 *  - fp16 GEMM / conv reference values are computed in double: every fp16
 *    product is exact in double and the sum's rounding error is ~1e-16
 *    relative, far below the acceptance bound 2e-3 * sum_k |a_ik * b_kj|.
 *  - Requantisation: fp32(C32) (round to nearest even), one fp32 multiply by
 *    the fp32 scale (round to nearest even, no fused multiply-add), round to
 *    the nearest integer with ties to even, clamp to [-128, 127].  A NaN
 *    product maps to 0.
 *  - Convolution is cross-correlation (no kernel flip) with symmetric zero
 *    padding: input row = p*stride_h + r - pad_h, column = q*stride_w + s -
 *    pad_w, zero outside [0,H) x [0,W).
 *
 * Parity pins (checked by the CPU test suite, not by this file): identity and
 * permutation matrices, small-integer exactness, the zero-point expansion
 * identity, hand-computed requantisation cases, delta-kernel convolutions,
 * brute-force im2col on tiny shapes, numpy's IEEE conversions for the three
 * number-format helpers, and float64 library matmul / conv2d on tiny shapes.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -pthread -shared -fPIC
 * (-ffp-contract=off keeps the requantisation multiply a plain fp32 multiply).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#if defined(__FLT_EVAL_METHOD__) && __FLT_EVAL_METHOD__ != 0
#error "the oracle needs float arithmetic evaluated in float (FLT_EVAL_METHOD == 0)"
#endif

/* ------------------------------------------------------------------------ */
/* number formats (IEEE 754 binary16 / binary32), written from the standard  */
/* ------------------------------------------------------------------------ */

/* binary16 bits -> exact double value. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                   /* zero / subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x400), e - 25);       /* 1.m * 2^(e-15) */
    return sign ? -v : v;
}

/* binary32 value -> binary16 bits, round to nearest, ties to even.
 * Overflow gives +-inf, NaN gives a quiet NaN, subnormal results are kept. */
uint16_t oracle_f32_to_f16_rne(float f)
{
    uint32_t x;
    memcpy(&x, &f, 4);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ax = x & 0x7fffffffu;
    if (ax >= 0x7f800000u)                            /* inf or NaN */
        return (uint16_t)(sign | 0x7c00u | (ax > 0x7f800000u ? 0x200u : 0u));
    if (ax >= 0x477ff000u)                            /* >= 65520: rounds to inf */
        return (uint16_t)(sign | 0x7c00u);
    int e = (int)(ax >> 23) - 127;                    /* unbiased exponent */
    if (e >= -14) {                                   /* normal binary16 result */
        uint32_t mant = ax & 0x7fffffu;
        uint32_t h = ((uint32_t)(e + 15) << 10) | (mant >> 13);
        uint32_t rem = mant & 0x1fffu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u)))
            h += 1;                                   /* a carry into the exponent is correct */
        return (uint16_t)(sign | h);
    }
    /* subnormal binary16 result: q = |f| / 2^-24 rounded to nearest even */
    int shift = -(e + 1);                             /* |f| = sig * 2^(e-23); q = sig >> shift */
    if (shift > 24)
        return sign;                                  /* |f| < 2^-25 (float subnormals included) */
    uint32_t sig = (ax & 0x7fffffu) | 0x800000u;
    uint32_t q = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u)))
        q += 1;                                       /* q == 0x400 encodes the smallest normal */
    return (uint16_t)(sign | q);
}

/* Array form of oracle_f32_to_f16_rne. */
void oracle_f32_to_f16_rne_array(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_f16_rne(in[i]);
}

/* bfloat16 bits (the top half of a binary32) -> exact double value. */
double oracle_bf16_to_f64(uint16_t h)
{
    uint32_t x = (uint32_t)h << 16;
    float f;
    memcpy(&f, &x, 4);
    return (double)f;
}

/* binary32 value -> bfloat16 bits, round to nearest, ties to even on the 16
 * dropped bits; NaN stays a (quiet) NaN, overflow rounds to +-inf. */
uint16_t oracle_f32_to_bf16_rne(float f)
{
    uint32_t x;
    memcpy(&x, &f, 4);
    if ((x & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((x >> 16) | 0x0040u);
    uint32_t hi = x >> 16;
    uint32_t rem = x & 0xffffu;
    if (rem > 0x8000u || (rem == 0x8000u && (hi & 1u)))
        hi += 1;                                      /* carries into the exponent correctly */
    return (uint16_t)hi;
}

void oracle_f32_to_bf16_rne_array(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_bf16_rne(in[i]);
}

/* int32 -> binary32, round to nearest, ties to even. */
float oracle_i32_to_f32_rne(int32_t v)
{
    int64_t s = v;
    int neg = s < 0;
    uint64_t u = (uint64_t)(neg ? -s : s);
    if (u < (1u << 24))
        return neg ? -(float)u : (float)u;            /* exactly representable */
    int len = 0;
    while ((u >> len) != 0)
        ++len;                                        /* bit length, 25..32 */
    int shift = len - 24;
    uint64_t q = u >> shift;
    uint64_t rem = u & ((1ull << shift) - 1ull);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1ull)))
        q += 1;
    if (q == (1ull << 24)) {
        q >>= 1;
        shift += 1;
    }
    float r = ldexpf((float)q, shift);                /* q < 2^24: exact */
    return neg ? -r : r;
}

/* Requantisation of one int32 accumulator with an fp32 scale ([P1] §2.3's
 * dequantise/requantise step; precision and rounding as read above). */
int8_t oracle_requant(int32_t c32, float scale)
{
    float v = oracle_i32_to_f32_rne(c32);
    float p = v * scale;                              /* one fp32 multiply, RNE */
    if (p != p)
        return 0;
    if (p >= 127.0f)
        return 127;
    if (p <= -128.0f)
        return -128;
    double d = (double)p;                             /* |p| < 128: exact in double */
    double fl = floor(d);
    double frac = d - fl;
    long r = (long)fl;
    if (frac > 0.5 || (frac == 0.5 && (r & 1L)))
        r += 1;                                       /* ties to even */
    if (r > 127)
        r = 127;
    if (r < -128)
        r = -128;
    return (int8_t)r;
}

/* Dequantised float output of the int8 GEMM ([P1] §2.3's dequantize(C) +
 * add_bias; order and precision as read above): each step one fp32 operation
 * rounded to nearest even, a NULL pointer skips its step. */
float oracle_dequant(int32_t c32, const float *s_row, const float *s_col, const float *bias)
{
    float t = oracle_i32_to_f32_rne(c32);
    if (s_row)
        t = t * *s_row;
    if (s_col)
        t = t * *s_col;
    if (bias)
        t = t + *bias;
    return t;
}

/* Y[i,j] = oracle_dequant(C32[i,j], s_row[i], s_col[j], bias[j]) over an M x N matrix. */
void oracle_dequant_matrix(int64_t M, int64_t N, const int32_t *C32, const float *s_row,
                           const float *s_col, const float *bias, float *Y)
{
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            Y[i * N + j] = oracle_dequant(C32[i * N + j], s_row ? s_row + i : NULL,
                                          s_col ? s_col + j : NULL, bias ? bias + j : NULL);
}

/* ------------------------------------------------------------------------ */
/* threading: rows [0, rows) split into contiguous blocks                     */
/* ------------------------------------------------------------------------ */

typedef void (*row_fn)(void *ctx, int64_t row);

struct worker {
    pthread_t tid;
    row_fn fn;
    void *ctx;
    int64_t begin, end;
};

static void *worker_main(void *arg)
{
    struct worker *w = (struct worker *)arg;
    for (int64_t r = w->begin; r < w->end; ++r)
        w->fn(w->ctx, r);
    return NULL;
}

int oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void parallel_rows(int64_t rows, int nthreads, row_fn fn, void *ctx)
{
    if (nthreads <= 0)
        nthreads = oracle_default_threads();
    if (nthreads > rows)
        nthreads = (int)(rows > 0 ? rows : 1);
    if (nthreads <= 1) {
        for (int64_t r = 0; r < rows; ++r)
            fn(ctx, r);
        return;
    }
    struct worker *ws = (struct worker *)calloc((size_t)nthreads, sizeof(struct worker));
    int64_t per = (rows + nthreads - 1) / nthreads;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        ws[t].fn = fn;
        ws[t].ctx = ctx;
        ws[t].begin = (int64_t)t * per;
        ws[t].end = ws[t].begin + per < rows ? ws[t].begin + per : rows;
        if (ws[t].begin >= ws[t].end)
            break;
        if (pthread_create(&ws[t].tid, NULL, worker_main, &ws[t]) != 0) {
            worker_main(&ws[t]);                      /* run inline if no thread */
            ws[t].end = -1;
        }
        started = t + 1;
    }
    for (int t = 0; t < started; ++t)
        if (ws[t].end != -1)
            pthread_join(ws[t].tid, NULL);
    free(ws);
}

/* ------------------------------------------------------------------------ */
/* FP16 GEMM: ref[i,j] = sum_k A[i,k] * Bt[j,k] in double ([P1] §4.1)       */
/*            sabs[i,j] = sum_k |A[i,k] * Bt[j,k]|                           */
/* ------------------------------------------------------------------------ */

struct gemm_f16_ctx {
    int64_t N, K;
    const uint16_t *A;
    int64_t lda;
    const double *Bd;                                 /* Bt converted to double, N x K */
    double *ref, *sabs;
    int64_t ldr;
};

static void gemm_f16_row(void *p, int64_t i)
{
    struct gemm_f16_ctx *c = (struct gemm_f16_ctx *)p;
    double *a = (double *)malloc(sizeof(double) * (size_t)(c->K > 0 ? c->K : 1));
    for (int64_t k = 0; k < c->K; ++k)
        a[k] = oracle_f16_to_f64(c->A[i * c->lda + k]);
    for (int64_t j = 0; j < c->N; ++j) {
        const double *b = c->Bd + j * c->K;
        double s = 0.0, sa = 0.0;
        for (int64_t k = 0; k < c->K; ++k) {
            double prod = a[k] * b[k];
            s += prod;
            sa += fabs(prod);
        }
        c->ref[i * c->ldr + j] = s;
        if (c->sabs)
            c->sabs[i * c->ldr + j] = sa;
    }
    free(a);
}

/* A: M x K fp16 bits (row stride lda); Bt: N x K fp16 bits (row stride ldb).
 * ref / sabs: M x N doubles (row stride N).  Returns 0, or -1 on bad args. */
int oracle_gemm_f16(int64_t M, int64_t N, int64_t K,
                    const uint16_t *A, int64_t lda,
                    const uint16_t *Bt, int64_t ldb,
                    double *ref, double *sabs, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || !ref)
        return -1;
    double *Bd = (double *)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!Bd)
        return -1;
    for (int64_t j = 0; j < N; ++j)
        for (int64_t k = 0; k < K; ++k)
            Bd[j * K + k] = oracle_f16_to_f64(Bt[j * ldb + k]);
    struct gemm_f16_ctx c = {N, K, A, lda, Bd, ref, sabs, N};
    parallel_rows(M, nthreads, gemm_f16_row, &c);
    free(Bd);
    return 0;
}

/* BF16 GEMM ([P1] §3.3's f16 -> bf16 swap of the same definition):
 * ref[i,j] = sum_k A[i,k] * Bt[j,k] in double from bf16 operands, sabs likewise. */
int oracle_gemm_bf16(int64_t M, int64_t N, int64_t K,
                     const uint16_t *A, int64_t lda,
                     const uint16_t *Bt, int64_t ldb,
                     double *ref, double *sabs, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K || !ref)
        return -1;
    double *Ad = (double *)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    double *Bd = (double *)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!Ad || !Bd) {
        free(Ad);
        free(Bd);
        return -1;
    }
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k)
            Ad[i * K + k] = oracle_bf16_to_f64(A[i * lda + k]);
    for (int64_t j = 0; j < N; ++j)
        for (int64_t k = 0; k < K; ++k)
            Bd[j * K + k] = oracle_bf16_to_f64(Bt[j * ldb + k]);
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0, sa = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double prod = Ad[i * K + k] * Bd[j * K + k];
                acc += prod;
                sa += fabs(prod);
            }
            ref[i * N + j] = acc;
            if (sabs)
                sabs[i * N + j] = sa;
        }
    (void)nthreads;
    free(Ad);
    free(Bd);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* INT8 GEMM with zero points ([P1] §2.3):                                    */
/*   C32[i,j] = sum_k (A_q[i,k] - zA_i) * (B_q[k,j] - zB_j)   (int64, direct) */
/*   C8[i,j]  = requant(C32[i,j], scale_j)                                    */
/* ------------------------------------------------------------------------ */

struct gemm_s8_ctx {
    int64_t N, K;
    const uint8_t *A;
    int a_signed;
    int64_t lda;
    const uint8_t *Bt;
    int b_signed;
    int64_t ldb;
    int32_t zA;
    const int32_t *zA_row;
    int32_t zB;
    const int32_t *zB_col;
    int32_t *C32;
    int64_t ldc32;
    int8_t *C8;
    int64_t ldc8;
    float scale;
    const float *scale_col;
    int64_t *C64;                                     /* optional exact values, M x N */
    volatile int overflow;
};

static inline int64_t q_value(uint8_t byte, int is_signed)
{
    return is_signed ? (int64_t)(int8_t)byte : (int64_t)byte;
}

static void gemm_s8_row(void *p, int64_t i)
{
    struct gemm_s8_ctx *c = (struct gemm_s8_ctx *)p;
    int64_t za = c->zA_row ? c->zA_row[i] : c->zA;
    for (int64_t j = 0; j < c->N; ++j) {
        int64_t zb = c->zB_col ? c->zB_col[j] : c->zB;
        int64_t s = 0;
        for (int64_t k = 0; k < c->K; ++k) {
            int64_t a = q_value(c->A[i * c->lda + k], c->a_signed) - za;
            int64_t b = q_value(c->Bt[j * c->ldb + k], c->b_signed) - zb;
            s += a * b;
        }
        if (c->C64)
            c->C64[i * c->N + j] = s;
        if (s > INT32_MAX || s < INT32_MIN)
            c->overflow = 1;
        /* the result as an int32 (two's complement wrap when it does not fit) */
        int32_t s32 = (int32_t)(uint32_t)(uint64_t)s;
        if (c->C32)
            c->C32[i * c->ldc32 + j] = s32;
        if (c->C8) {
            float sc = c->scale_col ? c->scale_col[j] : c->scale;
            c->C8[i * c->ldc8 + j] = oracle_requant(s32, sc);
        }
    }
}

/* A: M x K bytes (u8 or s8), Bt: N x K bytes (u8 or s8), i.e. B column-major.
 * zA_row (len M) / zB_col (len N) / scale_col (len N) override the per-tensor
 * values when non-null.  C32 / C8 / C64 are optional outputs.
 * Returns 0, 1 if some exact result does not fit int32, or -1 on bad args. */
int oracle_gemm_s8_zp(int64_t M, int64_t N, int64_t K,
                      const uint8_t *A, int a_signed, int64_t lda,
                      const uint8_t *Bt, int b_signed, int64_t ldb,
                      int32_t zA, const int32_t *zA_row,
                      int32_t zB, const int32_t *zB_col,
                      int32_t *C32, int64_t ldc32,
                      int8_t *C8, int64_t ldc8,
                      float scale, const float *scale_col,
                      int64_t *C64, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < K)
        return -1;
    if (C32 && ldc32 < N)
        return -1;
    if (C8 && ldc8 < N)
        return -1;
    struct gemm_s8_ctx c = {N, K, A, a_signed, lda, Bt, b_signed, ldb, zA, zA_row, zB, zB_col,
                            C32, ldc32, C8, ldc8, scale, scale_col, C64, 0};
    parallel_rows(M, nthreads, gemm_s8_row, &c);
    return c.overflow ? 1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Convolution ([P3] "准备和算法"):                                            */
/*   y[n,p,q,k] = sum_r sum_s sum_c xpad(n, p*sh + r - ph, q*sw + s - pw, c)  */
/*                                  * w[k,r,s,c]                              */
/* x NHWC, w KRSC, y NPQK; xpad is x with zeros outside [0,H) x [0,W).        */
/* ------------------------------------------------------------------------ */

struct conv_ctx {
    int N, H, W, C, K, R, S, ph, pw, sh, sw, P, Q;
    const double *xd, *wd;
    double *ref, *sabs;
};

static void conv_row(void *p, int64_t m)
{
    struct conv_ctx *c = (struct conv_ctx *)p;
    int64_t pq = (int64_t)c->P * c->Q;
    int n = (int)(m / pq);
    int pp = (int)((m % pq) / c->Q);
    int q = (int)(m % c->Q);
    for (int k = 0; k < c->K; ++k) {
        double s = 0.0, sa = 0.0;
        for (int r = 0; r < c->R; ++r) {
            int h = pp * c->sh + r - c->ph;
            if (h < 0 || h >= c->H)
                continue;                             /* zero padding */
            for (int ss = 0; ss < c->S; ++ss) {
                int w = q * c->sw + ss - c->pw;
                if (w < 0 || w >= c->W)
                    continue;
                const double *xv = c->xd + (((int64_t)n * c->H + h) * c->W + w) * c->C;
                const double *wv = c->wd + (((int64_t)k * c->R + r) * c->S + ss) * c->C;
                for (int ch = 0; ch < c->C; ++ch) {
                    double prod = xv[ch] * wv[ch];
                    s += prod;
                    sa += fabs(prod);
                }
            }
        }
        c->ref[m * c->K + k] = s;
        if (c->sabs)
            c->sabs[m * c->K + k] = sa;
    }
}

/* Output spatial size along one axis; -1 if the window does not fit. */
int oracle_conv_out_dim(int in, int filt, int pad, int stride)
{
    if (stride <= 0 || in + 2 * pad < filt)
        return -1;
    return (in + 2 * pad - filt) / stride + 1;
}

/* x: N*H*W*C fp16 bits; w: K*R*S*C fp16 bits; ref / sabs: N*P*Q*K doubles. */
int oracle_conv2d_nhwc_f16(int N, int H, int W, int C, int K, int R, int S,
                           int pad_h, int pad_w, int stride_h, int stride_w,
                           const uint16_t *x, const uint16_t *w,
                           double *ref, double *sabs, int nthreads)
{
    if (N < 0 || H <= 0 || W <= 0 || C <= 0 || K <= 0 || R <= 0 || S <= 0 ||
        pad_h < 0 || pad_w < 0 || !ref)
        return -1;
    int P = oracle_conv_out_dim(H, R, pad_h, stride_h);
    int Q = oracle_conv_out_dim(W, S, pad_w, stride_w);
    if (P <= 0 || Q <= 0)
        return -1;
    int64_t nx = (int64_t)N * H * W * C, nw = (int64_t)K * R * S * C;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(nx > 0 ? nx : 1));
    double *wd = (double *)malloc(sizeof(double) * (size_t)nw);
    if (!xd || !wd) {
        free(xd);
        free(wd);
        return -1;
    }
    for (int64_t i = 0; i < nx; ++i)
        xd[i] = oracle_f16_to_f64(x[i]);
    for (int64_t i = 0; i < nw; ++i)
        wd[i] = oracle_f16_to_f64(w[i]);
    struct conv_ctx c = {N, H, W, C, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q, xd, wd, ref, sabs};
    parallel_rows((int64_t)N * P * Q, nthreads, conv_row, &c);
    free(xd);
    free(wd);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* INT8 convolution with zero points ([P1] §2.2-2.3 with [P3]'s padding):      */
/*   y32[n,p,q,k] = sum_{r,s,c} (xpad - zX) * (w[k,r,s,c] - zW_k)              */
/* xpad = x inside the image and zX outside, so a padded tap adds nothing.     */
/* ------------------------------------------------------------------------ */

struct conv_s8_ctx {
    int N, H, W, C, K, R, S, ph, pw, sh, sw, P, Q;
    const uint8_t *x;
    int x_signed;
    int32_t zX;
    const uint8_t *w;
    int w_signed;
    int32_t zW;
    const int32_t *zW_k;
    int32_t *y32;
    int8_t *y8;
    float scale;
    const float *scale_k;
    volatile int overflow;
};

static void conv_s8_row(void *p, int64_t m)
{
    struct conv_s8_ctx *c = (struct conv_s8_ctx *)p;
    int64_t pq = (int64_t)c->P * c->Q;
    int n = (int)(m / pq);
    int pp = (int)((m % pq) / c->Q);
    int q = (int)(m % c->Q);
    for (int k = 0; k < c->K; ++k) {
        int64_t zw = c->zW_k ? c->zW_k[k] : c->zW;
        int64_t s = 0;
        for (int r = 0; r < c->R; ++r) {
            int h = pp * c->sh + r - c->ph;
            if (h < 0 || h >= c->H)
                continue;                             /* padded tap: (zX - zX) * (...) = 0 */
            for (int ss = 0; ss < c->S; ++ss) {
                int w = q * c->sw + ss - c->pw;
                if (w < 0 || w >= c->W)
                    continue;
                const uint8_t *xv = c->x + (((int64_t)n * c->H + h) * c->W + w) * c->C;
                const uint8_t *wv = c->w + (((int64_t)k * c->R + r) * c->S + ss) * c->C;
                for (int ch = 0; ch < c->C; ++ch)
                    s += (q_value(xv[ch], c->x_signed) - c->zX) * (q_value(wv[ch], c->w_signed) - zw);
            }
        }
        if (s > INT32_MAX || s < INT32_MIN)
            c->overflow = 1;
        int32_t s32 = (int32_t)(uint32_t)(uint64_t)s;
        if (c->y32)
            c->y32[m * c->K + k] = s32;
        if (c->y8)
            c->y8[m * c->K + k] = oracle_requant(s32, c->scale_k ? c->scale_k[k] : c->scale);
    }
}

/* x: N*H*W*C bytes; w: K*R*S*C bytes; y32 / y8: N*P*Q*K (optional).
 * Returns 0, 1 if some exact result does not fit int32, or -1 on bad args. */
int oracle_conv2d_nhwc_s8_zp(int N, int H, int W, int C, int K, int R, int S,
                             int pad_h, int pad_w, int stride_h, int stride_w,
                             const uint8_t *x, int x_signed, int32_t zX,
                             const uint8_t *w, int w_signed, int32_t zW, const int32_t *zW_k,
                             int32_t *y32, int8_t *y8, float scale, const float *scale_k,
                             int nthreads)
{
    if (N < 0 || H <= 0 || W <= 0 || C <= 0 || K <= 0 || R <= 0 || S <= 0 ||
        pad_h < 0 || pad_w < 0)
        return -1;
    int P = oracle_conv_out_dim(H, R, pad_h, stride_h);
    int Q = oracle_conv_out_dim(W, S, pad_w, stride_w);
    if (P <= 0 || Q <= 0)
        return -1;
    struct conv_s8_ctx c = {N, H, W, C, K, R, S, pad_h, pad_w, stride_h, stride_w, P, Q,
                            x, x_signed, zX, w, w_signed, zW, zW_k, y32, y8, scale, scale_k, 0};
    parallel_rows((int64_t)N * P * Q, nthreads, conv_s8_row, &c);
    return c.overflow ? 1 : 0;
}
