/*
 * CPU oracle for the general matrix multiply  D = alpha * (A @ B) + beta * C.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously-correct
 * statement of what the GPU library computes.  Only the tests, the smoke check
 * and the benchmark's CPU-baseline leg may load it; the library never does, and
 * it shares no code with the CUDA path.
 *
 * What it follows:
 *  - The operation D = alpha * (A @ B) + beta * C with scale operands U/V and
 *    the rule that C is not read when beta == 0: "InternLM Lmdeploy Gemm
 *    Interface", sections Description / Signature / Usage Examples.
 *  - The definition C = alpha*A*B + beta*C with A M x K and B K x N:
 *    DeepGEMM kernel-set blog, section 1.1.
 *  - U/V are group-wise scales that advance at K-group boundaries:
 *    "InternLM Lmdeploy Gemm MainloopSm80V2", section Description (GroupIter).
 *    Asymmetric int4 weights add a zero point z per (K-group, column) that
 *    advances the same way: b-hat = RN_A((q - z) * v).
 *  - FP8 (E4M3 / E5M2) operands, among the quantised inputs the DeepGEMM
 *    kernel-set blog targets (sections 1.2 and 6.3): decoded exactly like the
 *    16-bit ones; every product of two of them is exact in double.
 *  - The fused epilogue of the DeepGEMM kernel-set blog, section 6.1: a bias
 *    per output column, then ReLU or GELU, applied to alpha*(A@B) + beta*C.
 *    GELU is the exact form x * Phi(x) = x/2 * (1 + erf(x / sqrt 2)); ReLU maps
 *    x < 0 to 0 and keeps NaN.
 *
 * Arithmetic: every operand element is decoded exactly to double; a scaled
 * operand is formed as the exact product with its group scale and rounded once
 * (round-to-nearest-even) to the MMA input type; every product of two such
 * values is exact in double and the K-sum is accumulated in double in
 * ascending k.  The result is the exact real value up to ~1e-12 relative
 * error, which is what the fp32-accumulating GPU path must approach.
 *
 * Alongside ref[i][j] it returns bound[i][j] = |alpha| * sum_k |a_ik * b_kj|
 * + |beta * c_ij| (+ |bias_j|), the scale against which the GPU tolerance is
 * stated; after GELU it is multiplied by 1.129, the largest slope of x*Phi(x)
 * (reached at x = sqrt 2: Phi(sqrt 2) + sqrt 2 * phi(sqrt 2) = 1.1289...), so
 * an error in the pre-activation value stays covered.  ReLU's slope is at most 1.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC gemm_oracle.c -o liboracle.so -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_S4 = 3, OR_S8 = 4, OR_E4M3 = 5, OR_E5M2 = 6 };

/* ---- storage formats ---------------------------------------------------- */

/* Exact value of an 8-bit float (the FP8 inputs of the DeepGEMM kernel-set
 * blog, sections 1.2 and 6.3): sign, ebits exponent bits, mbits mantissa bits.
 * E4M3 (bias 7) has no infinities; only exponent and mantissa all ones is NaN,
 * so its largest value is 1.75 * 2^8 = 448.  E5M2 (bias 15) follows IEEE 754:
 * exponent all ones is infinity (mantissa 0) or NaN.  Exponent 0 holds the
 * subnormals m * 2^(1 - bias - mbits). */
static double decode_fp8(int type, uint32_t bits)
{
    const int e4 = (type == OR_E4M3);
    const int mbits = e4 ? 3 : 2, ebits = e4 ? 4 : 5;
    const int bias = (1 << (ebits - 1)) - 1;
    const uint32_t sign = (bits >> 7) & 1u;
    const uint32_t e = (bits >> mbits) & ((1u << ebits) - 1u);
    const uint32_t m = bits & ((1u << mbits) - 1u);
    const uint32_t emax = (1u << ebits) - 1u;
    double v;
    if (e4 && e == emax && m == (1u << mbits) - 1u)
        v = NAN;
    else if (!e4 && e == emax)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, 1 - bias - mbits);
    else
        v = ldexp((double)((1u << mbits) + m), (int)e - bias - mbits);
    return sign ? -v : v;
}

/* Exact value of a stored fp16 / bf16 / fp32 bit pattern (IEEE 754 binary16,
 * the bfloat16 truncation of binary32, binary32), or of an 8-bit float. */
double oracle_decode(int type, uint32_t bits)
{
    if (type == OR_F32) {
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    if (type == OR_E4M3 || type == OR_E5M2)
        return decode_fp8(type, bits & 0xFFu);
    int mbits = (type == OR_F16) ? 10 : 7;
    int ebits = (type == OR_F16) ? 5 : 8;
    int bias = (1 << (ebits - 1)) - 1;
    uint32_t sign = (bits >> 15) & 1u;
    uint32_t e = (bits >> mbits) & ((1u << ebits) - 1u);
    uint32_t m = bits & ((1u << mbits) - 1u);
    double v;
    if (e == 0)                       /* zero / subnormal: m * 2^(1 - bias - mbits) */
        v = ldexp((double)m, 1 - bias - mbits);
    else if (e == (1u << ebits) - 1u) /* inf / nan */
        v = m ? NAN : INFINITY;
    else                              /* (2^mbits + m) * 2^(e - bias - mbits) */
        v = ldexp((double)((1u << mbits) + m), (int)e - bias - mbits);
    return sign ? -v : v;
}

/* Round a double to the nearest fp16 / bf16 value, ties to even, overflow to
 * infinity, with gradual underflow.  Returns the bit pattern. */
uint32_t oracle_encode_rn(int type, double x)
{
    if (type == OR_F32) {
        float f = (float)x;          /* C conversion rounds to nearest-even */
        uint32_t b;
        memcpy(&b, &f, sizeof b);
        return b;
    }
    int p = (type == OR_F16) ? 11 : 8;         /* significand bits incl. hidden */
    int emin = (type == OR_F16) ? -14 : -126;  /* exponent of smallest normal   */
    int emax = (type == OR_F16) ? 15 : 127;
    int bias = -emin + 1;
    uint32_t sign = signbit(x) ? 1u : 0u;
    if (isnan(x))
        return (type == OR_F16) ? 0x7E00u : 0x7FC0u;
    double a = fabs(x);
    uint32_t all_ones_exp = (uint32_t)(2 * emax + 1); /* 31 for fp16, 255 for bf16 */
    uint32_t inf = (sign << 15) | (all_ones_exp << (p - 1));
    if (isinf(a))
        return inf;
    if (a == 0.0)
        return sign << 15;
    int e2;
    (void)frexp(a, &e2);
    int E = e2 - 1;                          /* a in [2^E, 2^(E+1)) */
    int qexp = (E < emin ? emin : E) - (p - 1);
    double r = rint(ldexp(a, -qexp));        /* exact scaling, then RN-even */
    if (E < emin) {
        /* subnormal field; r == 2^(p-1) carries into the exponent field and
         * yields the smallest normal number, which is the right encoding */
        return (sign << 15) | (uint32_t)r;
    }
    if (r >= ldexp(1.0, p)) {                 /* rounded up to the next binade */
        r = ldexp(1.0, p - 1);
        E += 1;
    }
    if (E > emax)
        return inf;
    uint32_t field = (uint32_t)(E + bias);
    return (sign << 15) | (field << (p - 1)) | ((uint32_t)r - (1u << (p - 1)));
}

/* Unit in the last place of the fp16 / bf16 / fp32 grid at |x|: the spacing
 * between the two representable values around |x| (the subnormal spacing
 * below the smallest normal). */
double oracle_ulp(int type, double x)
{
    int p = (type == OR_F16) ? 11 : (type == OR_BF16 ? 8 : 24);
    int emin = (type == OR_F16) ? -14 : -126;
    double a = fabs(x);
    int E = emin;
    if (a > 0 && isfinite(a)) {
        int e2;
        (void)frexp(a, &e2);
        E = e2 - 1;
        if (E < emin)
            E = emin;
    }
    return ldexp(1.0, E - (p - 1));
}

/* ---- the problem -------------------------------------------------------- */

typedef struct {
    int64_t M, N, K;
    int a_type;                 /* OR_F16 / OR_BF16 / OR_E4M3 / OR_E5M2          */
    const void* A; int64_t lda; /* M x K row-major, lda in elements              */
    int b_type;                 /* OR_F16 / OR_BF16 / OR_S4 / OR_E4M3 / OR_E5M2  */
    const void* B; int64_t ldb; /* N x K, K contiguous; S4: bytes per row        */
    int u_type; const void* U; int64_t ldu; int64_t ga; /* [K/ga][M] or U == 0  */
    int v_type; const void* V; int64_t ldv; int64_t gb; /* [K/gb][N] or V == 0  */
    int c_type; const void* C; int64_t ldc;             /* M x N row-major      */
    double alpha, beta;
    int epilogue;               /* bit 0: + bias[j]; bit 1: ReLU; bit 2: GELU     */
    int bias_type; const void* bias;                    /* N values (bit 0)     */
    const void* Z; int64_t ldz; /* int4 B with V: zero points [K/gb][N], one per
                                   byte (low nibble, two's complement), or 0   */
} oracle_gemm_t;

static uint32_t load_bits(int type, const void* p, int64_t idx)
{
    if (type == OR_F32)
        return ((const uint32_t*)p)[idx];
    if (type == OR_E4M3 || type == OR_E5M2)
        return ((const uint8_t*)p)[idx];
    return ((const uint16_t*)p)[idx];
}

/* a-hat[i][k]: A's stored value, or RN_A(a * u[k/ga][i]) when U is given. */
static double a_hat(const oracle_gemm_t* P, int64_t i, int64_t k)
{
    double a = oracle_decode(P->a_type, load_bits(P->a_type, P->A, i * P->lda + k));
    if (!P->U)
        return a;
    double u = oracle_decode(P->u_type, load_bits(P->u_type, P->U, (k / P->ga) * P->ldu + i));
    return oracle_decode(P->a_type, oracle_encode_rn(P->a_type, a * u));
}

/* Signed nibble k of row n of a packed int4 matrix: byte k/2, low nibble for
 * even k, high nibble for odd k, two's complement. */
int oracle_int4_at(const uint8_t* B, int64_t ldb, int64_t n, int64_t k)
{
    uint8_t byte = B[n * ldb + k / 2];
    int nib = (k & 1) ? (byte >> 4) : (byte & 0xF);
    return nib >= 8 ? nib - 16 : nib;
}

/* Zero point of K-group g, column j: the two's-complement value of the low
 * nibble of byte [g][j] (a 4-bit zero point stored one per byte). */
int oracle_zero_at(const uint8_t* Z, int64_t ldz, int64_t g, int64_t j)
{
    int nib = Z[g * ldz + j] & 0xF;
    return nib >= 8 ? nib - 16 : nib;
}

/* b-hat[k][j]: B's stored value (B is stored N x K), or the dequantised value.
 * 16-bit B with V: RN_B(b * v).  int4 B: RN_A((q - z) * v), with z = 0 unless
 * zero points are given (asymmetric quantisation), or q without V. */
static double b_hat(const oracle_gemm_t* P, int64_t k, int64_t j)
{
    double v = 1.0;
    if (P->V)
        v = oracle_decode(P->v_type, load_bits(P->v_type, P->V, (k / P->gb) * P->ldv + j));
    if (P->b_type == OR_S4) {
        int q = oracle_int4_at((const uint8_t*)P->B, P->ldb, j, k);
        if (!P->V)
            return (double)q;
        if (P->Z)
            q -= oracle_zero_at((const uint8_t*)P->Z, P->ldz, k / P->gb, j);
        return oracle_decode(P->a_type, oracle_encode_rn(P->a_type, (double)q * v));
    }
    double b = oracle_decode(P->b_type, load_bits(P->b_type, P->B, j * P->ldb + k));
    if (!P->V)
        return b;
    return oracle_decode(P->b_type, oracle_encode_rn(P->b_type, b * v));
}

static int check(const oracle_gemm_t* P)
{
    if (!P || P->M < 0 || P->N < 0 || P->K < 0 || !P->A || !P->B)
        return 1;
    if (P->U && (P->ga <= 0 || P->K % P->ga))
        return 1;
    if (P->V && (P->gb <= 0 || P->K % P->gb))
        return 1;
    if (P->Z && (!P->V || P->b_type != OR_S4))
        return 1;
    if (P->beta != 0.0 && !P->C)
        return 1;
    if ((P->epilogue & 1) && !P->bias)
        return 1;
    if ((P->epilogue & 2) && (P->epilogue & 4))
        return 1;
    return 0;
}

static void finish(const oracle_gemm_t* P, int64_t i, int64_t j, double s, double sabs,
                   double* ref, double* bound)
{
    double r = P->alpha * s, b = fabs(P->alpha) * sabs;
    if (P->beta != 0.0) {   /* C is not read when beta == 0 */
        double c = oracle_decode(P->c_type, load_bits(P->c_type, P->C, i * P->ldc + j));
        r += P->beta * c;
        b += fabs(P->beta * c);
    }
    if (P->epilogue & 1) {
        double bj = oracle_decode(P->bias_type, load_bits(P->bias_type, P->bias, j));
        r += bj;
        b += fabs(bj);
    }
    if (P->epilogue & 2)
        r = r < 0.0 ? 0.0 : r;
    if (P->epilogue & 4) {
        r = 0.5 * r * (1.0 + erf(r / sqrt(2.0)));
        b *= 1.129;
    }
    *ref = r;
    *bound = b;
}

/* Full result: ref and bound are M x N row-major.  Rows are independent and
 * split across OpenMP threads; each (i, j) is a plain ascending-k sum. */
int oracle_gemm(const oracle_gemm_t* P, double* ref, double* bound)
{
    if (check(P) || !ref || !bound)
        return 1;
    const int64_t M = P->M, N = P->N, K = P->K;
    double* bh = (double*)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!bh)
        return 2;
    /* the operand B-hat, decoded (and dequantised) once, stored [j][k] */
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j)
        for (int64_t k = 0; k < K; ++k)
            bh[j * K + k] = b_hat(P, k, j);
    int err = 0;
#pragma omp parallel
    {
        double* ah = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!ah) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < M; ++i) {
                for (int64_t k = 0; k < K; ++k)
                    ah[k] = a_hat(P, i, k);
                for (int64_t j = 0; j < N; ++j) {
                    const double* bj = bh + j * K;
                    double s = 0.0, sabs = 0.0;
                    for (int64_t k = 0; k < K; ++k) {
                        double t = ah[k] * bj[k];
                        s += t;
                        sabs += fabs(t);
                    }
                    finish(P, i, j, s, sabs, &ref[i * N + j], &bound[i * N + j]);
                }
            }
            free(ah);
        }
    }
    free(bh);
    return err;
}

/* Selected entries (ii[t], jj[t]) only, each computed on its own from the
 * stored bits: the check for problems too large to evaluate in full. */
int oracle_gemm_entries(const oracle_gemm_t* P, const int64_t* ii, const int64_t* jj, int64_t n,
                        double* ref, double* bound)
{
    if (check(P) || (n > 0 && (!ii || !jj || !ref || !bound)))
        return 1;
    for (int64_t t = 0; t < n; ++t)
        if (ii[t] < 0 || ii[t] >= P->M || jj[t] < 0 || jj[t] >= P->N)
            return 1;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < n; ++t) {
        double s = 0.0, sabs = 0.0;
        for (int64_t k = 0; k < P->K; ++k) {
            double x = a_hat(P, ii[t], k) * b_hat(P, k, jj[t]);
            s += x;
            sabs += fabs(x);
        }
        finish(P, ii[t], jj[t], s, sabs, &ref[t], &bound[t]);
    }
    return 0;
}

/* Number of threads an OpenMP region in this library runs with. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
