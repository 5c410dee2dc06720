/*
 * CPU oracle for the fused cascaded (back-to-back) GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (patent "数据处理方法、装置、设备及介质", Alibaba 2023):
 *   - a GEMM multiplies two input matrices into one output matrix
 *     (Detailed description, terms: "通用矩阵乘法 gemm", para. 30);
 *   - cascaded operators feed the output of operator 1 directly to operator 2,
 *     and a chain of three operators is fused the same way (para. 31, 41);
 *   - the rearrangement between the operators is a pure permutation of the
 *     result into the operand layout; the number of elements per thread does
 *     not change (para. 70, 79), so it does not change any value.
 * Hence the fused chain computes exactly
 *     P1 = A.W1,  P2 = round(P1).W2,  ...,  Out = round_out(P_last)
 * with the intermediate rounded to the second operator's operand data type
 * (fp16 / tf32 / fp64 are the types the patent names, para. 28).
 *
 * Rounding placement mirrors the fused kernel: every product is accumulated
 * (here exactly, in fp64, k ascending), rounded once to the accumulator type
 * (fp32, or nothing for fp64), then to the operand type for an intermediate,
 * or to the output type for the last product.
 *
 * The rounding routine is written from the definition of a binary
 * floating-point format (IEEE 754-2008 section 3.3: precision p, exponent
 * range [emin, emax], gradual underflow), not from any GPU header.
 *
 * Pins (see tests/test_oracle.py): identity, permutation and diagonal
 * matrices, associativity on exact integer inputs, brute force over tiny
 * shapes, every fp16 / bf16 bit pattern round-tripped, and random / edge fp32
 * values compared with numpy's float16 cast and torch's bfloat16 cast.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Rounding kinds (the same small integers are used by oracle/__init__.py). */
enum {
    ORC_NONE = 0, /* keep the fp64 value                                  */
    ORC_F32 = 1,  /* binary32, round to nearest, ties to even             */
    ORC_F16 = 2,  /* binary16, round to nearest, ties to even             */
    ORC_BF16 = 3, /* bfloat16 (8 exponent bits, 7 fraction bits), RNE     */
    ORC_TF32 = 4, /* tf32 (8 exponent bits, 10 fraction bits), ties away  */
    ORC_TF32_RNE = 5 /* tf32, ties to even (alternative reading)          */
};

/*
 * Round x to the binary format with `p` fraction bits and normal exponents in
 * [emin, emax].  Values below 2^emin use the fixed subnormal spacing
 * 2^(emin - p).  A magnitude that rounds above the largest finite value
 * becomes infinity.  NaN, infinities and zeros pass through.
 */
static double round_binary(double x, int p, int emin, int emax, int ties_away)
{
    if (x != x || x == 0.0 || isinf(x))
        return x;
    double ax = fabs(x);
    int e2;
    (void)frexp(ax, &e2); /* ax = f * 2^e2 with f in [0.5, 1) */
    int E = e2 - 1;       /* floor(log2(ax)) */
    if (E < emin)
        E = emin;
    double q = ldexp(1.0, E - p); /* spacing of representable values here */
    double t = ax / q;            /* exact: division by a power of two    */
    double fl = floor(t);
    double fr = t - fl;           /* exact */
    int up;
    if (fr > 0.5)
        up = 1;
    else if (fr < 0.5)
        up = 0;
    else
        up = ties_away ? 1 : (fmod(fl, 2.0) != 0.0);
    double r = (fl + (up ? 1.0 : 0.0)) * q;
    double maxv = ldexp(2.0 - ldexp(1.0, -p), emax);
    if (r > maxv)
        r = INFINITY;
    return copysign(r, x);
}

double oracle_round1(int kind, double x)
{
    switch (kind) {
    case ORC_NONE: return x;
    case ORC_F32: return round_binary(x, 23, -126, 127, 0);
    case ORC_F16: return round_binary(x, 10, -14, 15, 0);
    case ORC_BF16: return round_binary(x, 7, -126, 127, 0);
    case ORC_TF32: return round_binary(x, 10, -126, 127, 1);
    case ORC_TF32_RNE: return round_binary(x, 10, -126, 127, 0);
    default: return NAN;
    }
}

/* Element-wise rounding of an array, exposed for the tests. */
void oracle_round(int kind, const double *x, double *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        y[i] = oracle_round1(kind, x[i]);
}

/*
 * The cascaded chain, row by row.
 *   A      : [batch][M][K]            (fp64 copies of the stored inputs)
 *   W[s]   : [batch][Kin_s][N[s]]     Kin_0 = K, Kin_s = N[s-1]
 *   out    : [batch][M][N[n_stages-1]]
 * acc_kind rounds each finished product (ORC_F32, or ORC_NONE for fp64);
 * interm_kind then rounds every intermediate to GEMM(s+1)'s operand type;
 * out_kind rounds the last product after acc_kind.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_chain(int n_stages, int64_t batch, int64_t M, int64_t K, const int64_t *N,
                 const double *A, const double *const *W, int acc_kind, int interm_kind,
                 int out_kind, double *out, int n_threads)
{
    if (n_stages < 1 || n_stages > 8 || batch < 0 || M < 0 || K < 1)
        return -1;
    int64_t width = K;
    for (int s = 0; s < n_stages; ++s) {
        if (N[s] < 1)
            return -1;
        if (N[s] > width)
            width = N[s];
    }
    const int64_t n_last = N[n_stages - 1];
    const int64_t rows = batch * M;
#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int failed = 0;
#pragma omp parallel
    {
        double *cur = (double *)malloc(sizeof(double) * (size_t)width);
        double *nxt = (double *)malloc(sizeof(double) * (size_t)width);
        if (!cur || !nxt) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(static)
            for (int64_t r = 0; r < rows; ++r) {
                const int64_t b = r / M;
                int64_t kin = K;
                memcpy(cur, A + r * K, sizeof(double) * (size_t)K);
                for (int s = 0; s < n_stages; ++s) {
                    const int64_t n_out = N[s];
                    const double *w = W[s] + b * kin * n_out;
                    for (int64_t n = 0; n < n_out; ++n) {
                        double acc = 0.0;
                        for (int64_t k = 0; k < kin; ++k)
                            acc += cur[k] * w[k * n_out + n];
                        nxt[n] = oracle_round1(acc_kind, acc);
                    }
                    const int last = (s == n_stages - 1);
                    for (int64_t n = 0; n < n_out; ++n)
                        cur[n] = oracle_round1(last ? out_kind : interm_kind, nxt[n]);
                    kin = n_out;
                }
                memcpy(out + r * n_last, cur, sizeof(double) * (size_t)n_last);
            }
        }
        free(cur);
        free(nxt);
    }
    return failed ? -1 : 0;
}

/* Threads the OpenMP runtime will use by default (reported by the benchmark). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
