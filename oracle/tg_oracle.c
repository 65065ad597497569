/*
 * tg_oracle.c -- plain, slow, obviously correct CPU oracle for C = A x B.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  The product path (the
 * CUDA library under tiled_gemm_tg_gb300/) never calls it and shares no code,
 * header, table or helper with it.
 *
 * What it computes, and where the pages define it:
 *   - The product is the plain definition  C[i,j] = sum_k A[i,k] * B[k,j]
 *     over row-major operands, written out as the triple loop of
 *     "TileLang实战：用Python DSL自动生成高性能GPU计算内核" (gsyq.cn), §3.1,
 *     which the same page's §3.2 checks against a NumPy dot product.
 *   - Inputs are fp16 (or fp32 for the small example) and the pages accumulate
 *     in fp32 ("企业官网建设流程全解析" (cf-1.com), §3.3: accum_dtype float32).
 *     The 8-bit variant takes FP8 E4M3 inputs (the pages discuss 8-bit
 *     quantised GEMMs in "TileLang：GPU异构计算的声明式分块编程范式"
 *     (kwkr.cn), §5.5, with INT8, which GB300's tensor cores do not offer
 *     through tcgen05); they are decoded exactly like fp16.
 *     The oracle is stricter than that: every fp16 input is decoded exactly to
 *     binary64 from the IEEE-754 binary16 bit layout, every product of two
 *     fp16 values is exact in binary64, and the sum runs in binary64 in
 *     ascending k.  Its own error is therefore far below any kernel's.
 *   - Alongside C it returns S[i,j] = sum_k |A[i,k] * B[k,j]|, the scale that
 *     the acceptance bound  |C_gpu - C| <= 2e-3 * S + 1e-5 (+ 1e-2 |C| for an
 *     fp16 output; the 1e-2 relative threshold is the one in §3.3 "第四步" of
 *     the gsyq.cn/news/429607 article) is written against.
 *   - An fp64 -> fp16 round-to-nearest-even encoder, written from the
 *     binary16 definition, converts oracle results for bitwise comparison
 *     with an fp16 kernel output.  It converts directly from binary64, so no
 *     intermediate fp32 rounding (double rounding) can occur.
 *
 * Pins (tests/test_oracle.py): the decoder over all 65536 bit patterns
 * against NumPy's binary16 conversion; the encoder against NumPy on random
 * values and against hand-built ties; the product against a hand-computed
 * 4x4 integer example (tests/golden), the 8x8 all-ones example of the
 * TileLang实战 page §6.2, closed forms (identity, all-ones, diagonal), the
 * transpose invariant (AB)^T = B^T A^T bitwise, and NumPy fp64 matmul on
 * exactly representable inputs.  The E4M3 decoder is pinned over all 256
 * patterns against PyTorch's float8_e4m3fn conversion and by the format's
 * defining values (448, 2^-6, 2^-9, the two NaNs, no infinities); an E4M3
 * product of small integers equals NumPy's and the fp16 product.  Attention
 * is pinned against SciPy's softmax of NumPy's logits, by closed forms
 * (identical keys give the mean of V exactly, a dominant key gives its V row
 * exactly, V of ones gives ones), by invariants (a joint permutation of keys
 * and values, a shift shared by all keys, row independence, strided views),
 * and by the page's own blockwise running-max recurrence run in fp64.  The fused epilogue is pinned by the block
 * identity alpha*AB + beta*D + 1 bias^T = [alpha*A | beta*I | 1] [B; D; bias^T]
 * evaluated by NumPy, by x * Phi(x) against SciPy's normal distribution
 * function, and by the odd-part identities f(x) - f(-x) = x of ReLU and GELU.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define TGO_F16 1
#define TGO_F32 2
#define TGO_E4M3 3

/* ---- binary16 decode (IEEE-754: 1 sign, 5 exponent bits biased by 15,
 *      10 fraction bits) ------------------------------------------------- */
double tgo_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        /* zero and subnormals: 2^-14 * (f / 1024) = f * 2^-24 */
        v = ldexp((double)f, -24);
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        /* normals: 2^(e-15) * (1 + f/1024) = (1024 + f) * 2^(e-25) */
        v = ldexp((double)(1024 + f), e - 25);
    }
    return sign ? -v : v;
}

/* ---- binary64 -> binary16, round to nearest, ties to even -------------- */
uint16_t tgo_f64_to_f16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7c00u);
    /* 65504 is the largest finite half; the midpoint to the next binade
     * value 65536 is 65520, and a tie there goes to the even significand
     * (65536), which overflows.  So everything >= 65520 becomes infinity. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: values are integer multiples of 2^-24.
         * Scaling by 2^24 is exact; nearbyint() rounds ties to even under the
         * default rounding mode.  A result of 1024 is the smallest normal,
         * whose bit pattern 0x0400 is exactly 1024. */
        double q = nearbyint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)q);
    }
    int e2;
    (void)frexp(a, &e2);            /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;                 /* a in [2^E, 2^(E+1)), E in [-14, 15] */
    double q = nearbyint(ldexp(a, 10 - E)); /* significand scaled to [1024, 2048] */
    uint32_t mant = (uint32_t)q;
    if (mant == 2048u) {            /* rounding carried into the next binade */
        mant = 1024u;
        E += 1;
    }
    if (E > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)(((uint32_t)(E + 15) << 10) | (mant - 1024u)));
}

/* ---- FP8 E4M3 decode (the OCP 8-bit floating-point format's E4M3: 1 sign,
 *      4 exponent bits biased by 7, 3 fraction bits; no infinities, and the
 *      two patterns S.1111.111 are NaN, so the largest finite value is
 *      1.75 * 2^8 = 448) ---------------------------------------------------- */
double tgo_e4m3_to_f64(uint8_t q)
{
    int sign = (q >> 7) & 1;
    int e = (q >> 3) & 0xf;
    int f = q & 0x7;
    double v;
    if (e == 0xf && f == 0x7) {
        v = NAN;
    } else if (e == 0) {
        /* zero and subnormals: 2^-6 * (f / 8) = f * 2^-9 */
        v = ldexp((double)f, -9);
    } else {
        /* normals: 2^(e-7) * (1 + f/8) = (8 + f) * 2^(e-10) */
        v = ldexp((double)(8 + f), e - 10);
    }
    return sign ? -v : v;
}

void tgo_e4m3_to_f64_n(const uint8_t* src, double* dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = tgo_e4m3_to_f64(src[i]);
}

/* Bulk helpers so the Python side need not loop element by element. */
void tgo_f16_to_f64_n(const uint16_t* src, double* dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = tgo_f16_to_f64(src[i]);
}

void tgo_f64_to_f16_n(const double* src, uint16_t* dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) dst[i] = tgo_f64_to_f16(src[i]);
}

static double load_elem(const void* p, int64_t idx, int dtype)
{
    if (dtype == TGO_F16) return tgo_f16_to_f64(((const uint16_t*)p)[idx]);
    if (dtype == TGO_E4M3) return tgo_e4m3_to_f64(((const uint8_t*)p)[idx]);
    return (double)(((const float*)p)[idx]);
}

static int dtype_ok(int dtype)
{
    return dtype == TGO_F16 || dtype == TGO_F32 || dtype == TGO_E4M3;
}

int tgo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Full product.  A is M x K with row stride lda, B is K x N with row stride
 * ldb (both row-major, element type in_dtype); C and S are dense M x N fp64.
 * Rows of C are independent, so they are spread over threads; within a row
 * the sum runs in ascending k exactly as the definition reads.
 * Returns 0, or -1 on a bad argument or failed allocation.
 */
int tgo_gemm(int64_t M, int64_t N, int64_t K,
             const void* A, int64_t lda, const void* B, int64_t ldb,
             int in_dtype, double* C, double* S, int nthreads)
{
    if (M < 0 || N < 0 || K < 0) return -1;
    if (!dtype_ok(in_dtype)) return -1;
    if (M == 0 || N == 0) return 0;
    if (K > 0 && (lda < K || ldb < N || !A || !B)) return -1;

    /* Decode B once; A is decoded one element at a time inside the loop. */
    double* Bd = NULL;
    if (K > 0) {
        Bd = (double*)malloc(sizeof(double) * (size_t)K * (size_t)N);
        if (!Bd) return -1;
        for (int64_t k = 0; k < K; ++k)
            for (int64_t j = 0; j < N; ++j)
                Bd[k * N + j] = load_elem(B, k * ldb + j, in_dtype);
    }
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t i = 0; i < M; ++i) {
        double* c = C + i * N;
        double* s = S + i * N;
        for (int64_t j = 0; j < N; ++j) { c[j] = 0.0; s[j] = 0.0; }
        for (int64_t k = 0; k < K; ++k) {
            double a = load_elem(A, i * lda + k, in_dtype);
            const double* b = Bd + k * N;
            for (int64_t j = 0; j < N; ++j) {
                double p = a * b[j];
                c[j] += p;
                s[j] += fabs(p);
            }
        }
    }
    (void)nthreads;
    free(Bd);
    return 0;
}

/*
 * Selected elements only: for each t < n, C[t] and S[t] for output element
 * (rows[t], cols[t]), by the same definition (ascending k, fp64).  This is
 * what lets the tests check a full-size product element by element without
 * computing all of it.
 */
int tgo_gemm_at(int64_t M, int64_t N, int64_t K,
                const void* A, int64_t lda, const void* B, int64_t ldb,
                int in_dtype, int64_t n, const int64_t* rows,
                const int64_t* cols, double* C, double* S, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || n < 0) return -1;
    if (!dtype_ok(in_dtype)) return -1;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads)
#endif
    for (int64_t t = 0; t < n; ++t) {
        int64_t i = rows[t], j = cols[t];
        double c = 0.0, s = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = load_elem(A, i * lda + k, in_dtype) * load_elem(B, k * ldb + j, in_dtype);
            c += p;
            s += fabs(p);
        }
        C[t] = c;
        S[t] = s;
    }
    (void)nthreads;
    return 0;
}

/*
 * Fused epilogue, applied to a product computed above:
 *     out[i,j] = act(alpha * C[i,j] + beta * Cin[i,j] + bias[j])
 * with act = identity (0), ReLU max(x, 0) (1), or GELU (2) in its defining
 * form x * Phi(x) = 0.5 * x * (1 + erf(x / sqrt(2))), Phi the standard
 * normal distribution function.  This is the multi-operator fusion that
 * "企业官网建设流程全解析" (cf-1.com), §6.2, lists as the next direction after
 * the plain GEMM kernel (merging operators into one kernel to save launches
 * and memory round trips).  The pages give no formula for it, so the terms
 * are the usual GEMM epilogue ones with their textbook definitions, applied
 * in the order written.  C is dense M x N fp64 (the oracle's product); Cin is
 * M x N of element type cin_dtype with row stride ldcin (may be NULL when
 * beta == 0, and is then never read); bias holds N fp32 values (or NULL).
 * Everything is evaluated in fp64.  Returns 0, or -1 on a bad argument.
 */
int tgo_epilogue(int64_t M, int64_t N, const double* C, double alpha, double beta,
                 const void* Cin, int64_t ldcin, int cin_dtype, const float* bias, int act,
                 double* out)
{
    if (M < 0 || N < 0 || act < 0 || act > 2) return -1;
    if (beta != 0.0 && (!Cin || ldcin < N || (cin_dtype != TGO_F16 && cin_dtype != TGO_F32)))
        return -1;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double y = alpha * C[i * N + j];
            if (beta != 0.0) y += beta * load_elem(Cin, i * ldcin + j, cin_dtype);
            if (bias) y += (double)bias[j];
            if (act == 1) y = y > 0.0 ? y : 0.0;
            else if (act == 2) y = 0.5 * y * (1.0 + erf(y / sqrt(2.0)));
            out[i * N + j] = y;
        }
    }
    return 0;
}

/*
 * Attention forward, by its definition:
 *     O[i,c] = sum_j w_ij V[j,c],  w_ij = exp(s_ij - m_i) / sum_j' exp(s_ij' - m_i),
 *     s_ij = scale * sum_d Q[i,d] K[j,d],  m_i = max_j s_ij.
 * This is the softmax(Q K^T) V that "TileLang实战：用Python DSL自动生成高性能GPU
 * 计算内核" (gsyq.cn), §4.1, states and its §4.2 computes blockwise with a
 * running maximum M and normaliser L; the blockwise recurrence reaches the
 * same value up to rounding, so the oracle is the definition.  The page's
 * kernel applies no 1/sqrt(d) factor: `scale` is 1 for it.  Subtracting m_i
 * is the usual overflow guard and cancels exactly in the ratio.
 * Q is Nq x d (row stride ldq), K is Nk x d (ldk), V is Nk x dv (ldv), all of
 * element type in_dtype.  O and E are dense Nq x dv fp64 with
 * E[i,c] = sum_j w_ij |V[j,c]| (the scale the acceptance bound is written
 * against), and G[i] = |scale| * max_j sum_d |Q[i,d] K[j,d]| (the largest
 * logit magnitude a row's dot products can reach).  Everything in fp64.
 * Returns 0, or -1 on a bad argument or failed allocation.
 */
int tgo_attention(int64_t Nq, int64_t Nk, int64_t d, int64_t dv, const void* Q, int64_t ldq,
                  const void* K, int64_t ldk, const void* V, int64_t ldv, int in_dtype,
                  double scale, double* O, double* E, double* G, int nthreads)
{
    if (Nq < 0 || Nk < 1 || d < 1 || dv < 1 || !dtype_ok(in_dtype)) return -1;
    if (ldq < d || ldk < d || ldv < dv || !Q || !K || !V) return -1;
    double* Kd = (double*)malloc(sizeof(double) * (size_t)Nk * (size_t)d);
    double* Vd = (double*)malloc(sizeof(double) * (size_t)Nk * (size_t)dv);
    if (!Kd || !Vd) {
        free(Kd);
        free(Vd);
        return -1;
    }
    for (int64_t j = 0; j < Nk; ++j) {
        for (int64_t c = 0; c < d; ++c) Kd[j * d + c] = load_elem(K, j * ldk + c, in_dtype);
        for (int64_t c = 0; c < dv; ++c) Vd[j * dv + c] = load_elem(V, j * ldv + c, in_dtype);
    }
    int rc = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t i = 0; i < Nq; ++i) {
        double* s = (double*)malloc(sizeof(double) * (size_t)Nk);
        double* q = (double*)malloc(sizeof(double) * (size_t)d);
        if (!s || !q) {
            free(s);
            free(q);
            rc = -1;
            continue;
        }
        for (int64_t c = 0; c < d; ++c) q[c] = load_elem(Q, i * ldq + c, in_dtype);
        double m = -INFINITY, g = 0.0;
        for (int64_t j = 0; j < Nk; ++j) {
            double acc = 0.0, mag = 0.0;
            for (int64_t c = 0; c < d; ++c) {
                acc += q[c] * Kd[j * d + c];
                mag += fabs(q[c] * Kd[j * d + c]);
            }
            s[j] = scale * acc;
            if (s[j] > m) m = s[j];
            if (mag > g) g = mag;
        }
        double l = 0.0;
        for (int64_t j = 0; j < Nk; ++j) {
            s[j] = exp(s[j] - m); /* now the unnormalised weight */
            l += s[j];
        }
        for (int64_t c = 0; c < dv; ++c) {
            double o = 0.0, e = 0.0;
            for (int64_t j = 0; j < Nk; ++j) {
                o += s[j] * Vd[j * dv + c];
                e += s[j] * fabs(Vd[j * dv + c]);
            }
            O[i * dv + c] = o / l;
            E[i * dv + c] = e / l;
        }
        G[i] = fabs(scale) * g;
        free(s);
        free(q);
    }
    (void)nthreads;
    free(Kd);
    free(Vd);
    return rc;
}
