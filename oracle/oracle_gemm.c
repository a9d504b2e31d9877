/*
 * CPU oracle for the dense product C = A*B with fp16/bf16 inputs.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no header, helper, table or constant
 * with the GPU library; its only contact with the GPU path is that both are
 * fed the same seeded input bytes.
 *
 * What it computes (issue "Stream-k matmul implementation very slow" on the
 * triton tracker, issue body: every schedule "generates the right output"
 * up to rounding; the HF post "naive vs persistent matmul": each tile is the
 * sum-reduction over K of row tiles of A times column tiles of B).  All
 * schedules reach the plain product, so the oracle is that definition:
 *
 *     C64[i][j] = sum_{k=0..K-1} double(A[i][k]) * double(B[k][j])
 *
 * summed in ascending k in IEEE double.  Each product of two fp16 values (11
 * significant bits each) or two bf16 values (8 bits each) is exact in double,
 * so the only rounding is in the running sum, and an integer-valued sum below
 * 2^53 is exact.  The output is rounded once, directly from double to the
 * 16-bit type (round to nearest, ties to even; overflow to infinity;
 * subnormals kept).  It never passes through fp32, so there is no double
 * rounding.  It also returns S[i][j] = sum_k |A[i][k]| * |B[k][j]|, which
 * enters the acceptance bound.
 *
 * Blocking: the outer (i, j) loops are cut into blocks that OpenMP threads
 * take in parallel, and four neighbouring columns j share each pass over k.
 * Each output element keeps its own accumulator summed in plain k order, so
 * the blocking changes no result bit.
 *
 * Type codes: 0 = IEEE binary16, 1 = bfloat16.
 * Layout codes: 0 = row-major, 1 = column-major.
 *   A is M x K: row-major A[i*K + k], column-major A[k*M + i].
 *   B is K x N: row-major B[k*N + j], column-major B[j*K + k].
 *   C is M x N row-major.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_F16 0
#define ORC_BF16 1

/* ---- 16-bit float formats, from the IEEE 754 binary16 definition and the
 *      bfloat16 definition (the top half of an IEEE binary32). ---- */

/* significand bits p (with the hidden bit) and the smallest normal exponent */
static void fmt_params(int dtype, int *p, int *emin, int *emax, int *ebits) {
    if (dtype == ORC_F16) { *p = 11; *emin = -14; *emax = 15; *ebits = 5; }
    else { *p = 8; *emin = -126; *emax = 127; *ebits = 8; }
}

/* exact value of a 16-bit pattern */
static double decode16(int dtype, uint16_t h) {
    int p, emin, emax, ebits;
    fmt_params(dtype, &p, &emin, &emax, &ebits);
    int mbits = p - 1;
    int sign = (h >> 15) & 1;
    int efield = (h >> mbits) & ((1 << ebits) - 1);
    int mant = h & ((1 << mbits) - 1);
    double v;
    if (efield == 0) {
        /* subnormal: mant * 2^(emin - mbits) */
        v = ldexp((double)mant, emin - mbits);
    } else if (efield == (1 << ebits) - 1) {
        v = mant ? NAN : INFINITY;
    } else {
        int e = efield - emax; /* bias == emax for both formats */
        v = ldexp((double)((1 << mbits) + mant), e - mbits);
    }
    return sign ? -v : v;
}

/* round a non-negative double n (an exact multiple of 1/2^m for small m) to
 * the nearest integer, ties to the even neighbour */
static double round_half_even(double n) {
    double fl = floor(n);
    double d = n - fl; /* exact: n and fl share an exponent range */
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* double -> 16-bit pattern, one rounding, to nearest with ties to even */
static uint16_t encode16(int dtype, double x) {
    int p, emin, emax, ebits;
    fmt_params(dtype, &p, &emin, &emax, &ebits);
    int mbits = p - 1;
    uint16_t inf_bits = (uint16_t)(((1 << ebits) - 1) << mbits);
    if (isnan(x)) return (uint16_t)(inf_bits | (1u << (mbits - 1)));
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    /* the largest finite value is (2 - 2^(1-p)) * 2^emax; anything at or
     * above the midpoint to 2^(emax+1) rounds to infinity (the tie goes up
     * because the largest finite significand is odd) */
    double overflow_at = ldexp(2.0 - ldexp(1.0, -p), emax);
    if (a >= overflow_at) return (uint16_t)(sign | inf_bits);
    if (a < ldexp(1.0, emin)) {
        /* subnormal range: fixed quantum 2^(emin - mbits); a carry out of
         * the mantissa lands exactly on the smallest normal pattern */
        double n = round_half_even(ldexp(a, mbits - emin));
        return (uint16_t)(sign | (uint16_t)n);
    }
    int E;
    (void)frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1;      /* a in [2^e, 2^(e+1)) */
    double n = round_half_even(ldexp(a, mbits - e)); /* in [2^mbits, 2^p] */
    if (n == ldexp(1.0, p)) { n = ldexp(1.0, mbits); e += 1; }
    if (e > emax) return (uint16_t)(sign | inf_bits);
    uint16_t efield = (uint16_t)(e + emax);
    uint16_t mant = (uint16_t)(n - ldexp(1.0, mbits));
    return (uint16_t)(sign | (efield << mbits) | mant);
}

/* ---- exported element helpers ---- */

int oracle_decode(int dtype, const uint16_t *bits, int64_t n, double *out) {
    if (dtype != ORC_F16 && dtype != ORC_BF16) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = decode16(dtype, bits[i]);
    return 0;
}

int oracle_round(int dtype, const double *x, int64_t n, uint16_t *out) {
    if (dtype != ORC_F16 && dtype != ORC_BF16) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = encode16(dtype, x[i]);
    return 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- the product ---- */

static int check_args(int64_t M, int64_t N, int64_t K, int dtype, int la, int lb) {
    if (M < 0 || N < 0 || K < 0) return -1;
    if (dtype != ORC_F16 && dtype != ORC_BF16) return -1;
    if ((la != 0 && la != 1) || (lb != 0 && lb != 1)) return -1;
    return 0;
}

/*
 * Full product.  C64 (M*N doubles) is required; S (M*N doubles, the sum of
 * |a||b|) and Cout (M*N rounded patterns) may be NULL.  Rows of A and columns
 * of B are decoded once into double panels with k contiguous, then every
 * C[i][j] is a dot product over k in ascending order.
 * Returns 0, or -1 on bad arguments, -2 if a panel cannot be allocated.
 */
int oracle_gemm(int64_t M, int64_t N, int64_t K, int dtype, int layout_a, int layout_b,
                const uint16_t *A, const uint16_t *B,
                double *C64, double *S, uint16_t *Cout) {
    if (check_args(M, N, K, dtype, layout_a, layout_b)) return -1;
    if (M == 0 || N == 0) return 0;
    size_t kk = (size_t)(K > 0 ? K : 1);
    double *Ad = (double *)malloc(sizeof(double) * (size_t)M * kk);
    double *Bt = (double *)malloc(sizeof(double) * (size_t)N * kk);
    if (!Ad || !Bt) { free(Ad); free(Bt); return -2; }

    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k) {
            uint16_t h = layout_a == 0 ? A[i * K + k] : A[k * M + i];
            Ad[i * K + k] = decode16(dtype, h);
        }
    #pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < N; ++j)
        for (int64_t k = 0; k < K; ++k) {
            uint16_t h = layout_b == 0 ? B[k * N + j] : B[j * K + k];
            Bt[j * K + k] = decode16(dtype, h);
        }

    const int64_t BI = 32, BJ = 64;
    int64_t nbi = (M + BI - 1) / BI, nbj = (N + BJ - 1) / BJ;
    #pragma omp parallel for schedule(dynamic, 1) collapse(2)
    for (int64_t bi = 0; bi < nbi; ++bi)
        for (int64_t bj = 0; bj < nbj; ++bj) {
            int64_t i1 = bi * BI + BI < M ? bi * BI + BI : M;
            int64_t j1 = bj * BJ + BJ < N ? bj * BJ + BJ : N;
            for (int64_t i = bi * BI; i < i1; ++i) {
                const double *a = Ad + i * K;
                int64_t j = bj * BJ;
                for (; j + 4 <= j1; j += 4) {
                    const double *b0 = Bt + (j + 0) * K, *b1 = Bt + (j + 1) * K;
                    const double *b2 = Bt + (j + 2) * K, *b3 = Bt + (j + 3) * K;
                    double c0 = 0, c1 = 0, c2 = 0, c3 = 0;
                    for (int64_t k = 0; k < K; ++k) {
                        double av = a[k];
                        c0 += av * b0[k]; c1 += av * b1[k];
                        c2 += av * b2[k]; c3 += av * b3[k];
                    }
                    C64[i * N + j + 0] = c0; C64[i * N + j + 1] = c1;
                    C64[i * N + j + 2] = c2; C64[i * N + j + 3] = c3;
                    if (S) {
                        double s0 = 0, s1 = 0, s2 = 0, s3 = 0;
                        for (int64_t k = 0; k < K; ++k) {
                            double av = fabs(a[k]);
                            s0 += av * fabs(b0[k]); s1 += av * fabs(b1[k]);
                            s2 += av * fabs(b2[k]); s3 += av * fabs(b3[k]);
                        }
                        S[i * N + j + 0] = s0; S[i * N + j + 1] = s1;
                        S[i * N + j + 2] = s2; S[i * N + j + 3] = s3;
                    }
                }
                for (; j < j1; ++j) {
                    const double *b = Bt + j * K;
                    double c = 0, s = 0;
                    for (int64_t k = 0; k < K; ++k) c += a[k] * b[k];
                    C64[i * N + j] = c;
                    if (S) {
                        for (int64_t k = 0; k < K; ++k) s += fabs(a[k]) * fabs(b[k]);
                        S[i * N + j] = s;
                    }
                }
            }
        }
    if (Cout) {
        #pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < M * N; ++t) Cout[t] = encode16(dtype, C64[t]);
    }
    free(Ad);
    free(Bt);
    return 0;
}

/*
 * Selected entries only: for each e < n, C64[e] and S[e] (S may be NULL) for
 * the element (rows[e], cols[e]), read straight from the 16-bit inputs.  Used
 * on products too large for the full oracle.  Returns 0, -1 on bad arguments,
 * -3 if an index is out of range.
 */
int oracle_gemm_entries(int64_t M, int64_t N, int64_t K, int dtype, int layout_a, int layout_b,
                        const uint16_t *A, const uint16_t *B, int64_t n,
                        const int64_t *rows, const int64_t *cols, double *C64, double *S) {
    if (check_args(M, N, K, dtype, layout_a, layout_b)) return -1;
    for (int64_t e = 0; e < n; ++e)
        if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N) return -3;
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t e = 0; e < n; ++e) {
        int64_t i = rows[e], j = cols[e];
        double c = 0, s = 0;
        for (int64_t k = 0; k < K; ++k) {
            double a = decode16(dtype, layout_a == 0 ? A[i * K + k] : A[k * M + i]);
            double b = decode16(dtype, layout_b == 0 ? B[k * N + j] : B[j * K + k]);
            c += a * b;
            s += fabs(a) * fabs(b);
        }
        C64[e] = c;
        if (S) S[e] = s;
    }
    return 0;
}
