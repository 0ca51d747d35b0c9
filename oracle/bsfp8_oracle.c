/*
 * bsfp8_oracle.c -- plain, slow, obviously correct CPU reference for the
 * block-scaled E4M3 GEMM and its grouped variant.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library (block_scaled_fp8_sm_gb300/)
 * may include, link, load or call this file.  Only the tests, the smoke check
 * in __graft_entry__.py and the CPU-baseline leg of bench.py use it.  It
 * shares no code, header, table or constant with the CUDA path.
 *
 * What it computes (FP8 GEMM library article, hncyxsy.com/news/241433,
 * section 2.2 "scale granularity": one fp32 scale per 32x32 block of A and of B,
 * applied during accumulation; section 6 "usage example": A is [M,K], B is
 * [N,K], scale_a is [M/32,K/32], scale_b is [N/32,K/32]):
 *
 *   C[m,n] = sum_{kb} sA[m/32][kb] * sB[n/32][kb] * sum_{k in kb} A[m,k] * B[n,k]
 *
 * with kb running over blocks of 32 consecutive k.  A and B hold E4M3 codes
 * (article section 2.1: 4 exponent bits, 3 mantissa bits, largest value 448).
 *
 * Arithmetic:
 *   - E4M3 codes are decoded through a 256-entry table built from the bit-field
 *     definition (bias 7, subnormals m*2^-9, S.1111.111 is NaN, no infinity).
 *   - Each 32-term inner sum is formed in fp64 and is EXACT: every product of
 *     two E4M3 values is an integer multiple of 2^-18 with at most 8 significant
 *     bits and magnitude below 2^18, so a sum of 32 of them needs at most 41
 *     bits.
 *   - sA*sB is exact in fp64 (two 24-bit significands).  The scaled block sum is
 *     then rounded once and accumulated in fp64, kb ascending.
 *   - T[m,n] = sum_kb |sA*sB| * sum_k |A*B| (the magnitude sum used by the
 *     acceptance bound) is accumulated the same way.
 *
 * Compile without -ffast-math and with -ffp-contract=off (the build script
 * does): the kb accumulation order is part of the definition above.
 *
 * Pins: every function here is checked in tests/test_oracle_pins.py against
 * facts fixed independently of this file (the format definition, the pages'
 * worked rounding example, exact rational brute force, identity / one-hot
 * operands, per-tensor and per-channel closed forms, the block rescaling
 * invariant, and operand-swap symmetry).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---------------------------------------------------------------- E4M3 ---- */

/* Value of one E4M3 code, straight from the bit fields. */
static double e4m3_value(unsigned code) {
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double v;
    if (e == 15u && m == 7u) return NAN;              /* S.1111.111: NaN */
    if (e == 0u) v = ldexp((double)m, -9);            /* (m/8) * 2^(1-7) */
    else v = ldexp((double)(8u + m), (int)e - 10);    /* (1+m/8) * 2^(e-7) */
    return s ? -v : v;
}

void oracle_e4m3_table(double *out256) {
    for (unsigned c = 0; c < 256u; ++c) out256[c] = e4m3_value(c);
}

/* Round x to the nearest E4M3 value, ties to the even code (the even mantissa),
 * saturating to +-448; NaN maps to 0x7F.  Written as a search over the 127
 * non-negative finite codes, the plainest statement of "nearest". */
unsigned oracle_e4m3_quantize_one(double x) {
    if (isnan(x)) return 0x7Fu;
    unsigned sign = signbit(x) ? 0x80u : 0u;
    double a = fabs(x);
    unsigned best = 0u;
    double best_d = INFINITY;
    for (unsigned c = 0; c <= 0x7Eu; ++c) {
        double d = fabs(e4m3_value(c) - a);
        if (d < best_d || (d == best_d && (c & 1u) == 0u)) {
            best = c;
            best_d = d;
        }
    }
    return sign | best;   /* a > 448 lands on 0x7E: saturation */
}

void oracle_e4m3_quantize(const double *x, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)oracle_e4m3_quantize_one(x[i]);
}

/* ---------------------------------------------------------------- bf16 ---- */

/* Round x to bf16 (1 sign, 8 exponent bits with bias 127, 7 stored mantissa
 * bits), nearest with ties to even; overflow past the largest finite value
 * rounds to infinity as IEEE round-to-nearest does.  Returns the 16-bit
 * pattern. */
uint16_t oracle_bf16_rne_one(double x) {
    if (isnan(x)) return 0x7FC0u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);                 /* a = f * 2^e, f in [0.5,1) */
    int ue = e - 1;                     /* unbiased exponent: a in [2^ue, 2^(ue+1)) */
    if (ue < -126) ue = -126;           /* subnormal range keeps spacing 2^-133 */
    double ulp = ldexp(1.0, ue - 7);
    double q = a / ulp;                 /* exact: power-of-two scaling */
    double r = nearbyint(q);            /* default mode: to nearest, ties to even */
    double v = r * ulp;
    if (v >= ldexp(1.0, 128)) return sign | 0x7F80u;   /* infinity */
    /* encode v */
    if (v < ldexp(1.0, -126)) {         /* subnormal (or zero after rounding) */
        uint16_t mant = (uint16_t)(v / ldexp(1.0, -133));
        return sign | mant;
    }
    int ve;
    double vf = frexp(v, &ve);          /* v = vf * 2^ve */
    unsigned biased = (unsigned)(ve - 1 + 127);
    unsigned mant = (unsigned)((vf * 2.0 - 1.0) * 128.0);
    return (uint16_t)(sign | (biased << 7) | mant);
}

void oracle_bf16_rne(const double *x, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_rne_one(x[i]);
}

double oracle_bf16_value(uint16_t bits) {
    unsigned s = bits >> 15, e = (bits >> 7) & 0xFFu, m = bits & 0x7Fu;
    double v;
    if (e == 0xFFu) v = m ? NAN : INFINITY;
    else if (e == 0u) v = ldexp((double)m, -133);
    else v = ldexp((double)(128u + m), (int)e - 134);
    return s ? -v : v;
}

/* ---------------------------------------------------------------- GEMM ---- */

typedef struct {
    const uint8_t *A; const float *sA; const uint8_t *B; const float *sB;
    int64_t M, N, K;
    const int64_t *ms, *ns;   /* sampled mode when non-NULL */
    int64_t count;
    double *C, *T;
    const double *tab;
    int64_t begin, end;       /* rows (full mode) or samples (sampled mode) */
    int mutation;
} job_t;

/* One output element, following the definition term by term. */
static void element(const job_t *j, int64_t m, int64_t n, double *c_out, double *t_out) {
    const int64_t KB = j->K / 32;
    const uint8_t *a = j->A + m * j->K;
    const uint8_t *b = j->B + n * j->K;
    double acc = 0.0, mag = 0.0;
    for (int64_t kb = 0; kb < KB; ++kb) {
        double s = 0.0, sabs = 0.0;
        for (int64_t k = kb * 32; k < kb * 32 + 32; ++k) {
            double p = j->tab[a[k]] * j->tab[b[k]];
            s += p;
            sabs += fabs(p);
        }
        int64_t ra = m / 32, rb = n / 32;
        /* Planted mistakes, used only by the tests that show the pins catch
         * them (mutation 0 is the oracle proper). */
        if (j->mutation == 1) rb = m / 32;                      /* wrong scale index */
        double sc = (double)j->sA[ra * KB + kb] * (double)j->sB[rb * KB + kb];
        if (j->mutation == 2 && kb == KB - 1) continue;          /* dropped term */
        if (j->mutation == 3) sc = (double)j->sA[ra * KB + kb]; /* missing B scale */
        acc += sc * s;
        mag += fabs(sc) * sabs;
    }
    *c_out = acc;
    *t_out = mag;
}

static void *worker(void *arg) {
    job_t *j = (job_t *)arg;
    if (j->ms) {
        for (int64_t i = j->begin; i < j->end; ++i)
            element(j, j->ms[i], j->ns[i], &j->C[i], &j->T[i]);
    } else {
        for (int64_t m = j->begin; m < j->end; ++m)
            for (int64_t n = 0; n < j->N; ++n)
                element(j, m, n, &j->C[m * j->N + n], &j->T[m * j->N + n]);
    }
    return NULL;
}

static int run(job_t proto, int64_t units, int nthreads) {
    double tab[256];
    oracle_e4m3_table(tab);
    proto.tab = tab;
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if ((int64_t)nthreads > units) nthreads = units > 0 ? (int)units : 1;
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    if (!th || !jobs) { free(th); free(jobs); return -1; }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].begin = units * t / nthreads;
        jobs[t].end = units * (t + 1) / nthreads;
    }
    int rc = 0;
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, worker, &jobs[t]) != 0) { rc = -2; break; }
        started = t;
    }
    worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    if (rc != 0) {   /* a thread could not start: finish its share here */
        for (int t = started + 1; t < nthreads; ++t) worker(&jobs[t]);
        rc = 0;
    }
    free(th);
    free(jobs);
    return rc;
}

/* Full C (M x N, row-major) and T.  sA is [ceil(M/32), K/32], sB is
 * [ceil(N/32), K/32], both row-major fp32.  K must be a multiple of 32.
 * Returns 0, or -1 on a bad argument. */
int oracle_gemm(const uint8_t *A, const float *sA, const uint8_t *B, const float *sB,
                int64_t M, int64_t N, int64_t K, double *C, double *T,
                int nthreads, int mutation) {
    if (M < 0 || N < 0 || K < 0 || (K % 32) != 0) return -1;
    if (M == 0 || N == 0) return 0;
    job_t p;
    memset(&p, 0, sizeof p);
    p.A = A; p.sA = sA; p.B = B; p.sB = sB; p.M = M; p.N = N; p.K = K;
    p.C = C; p.T = T; p.mutation = mutation;
    return run(p, M, nthreads);
}

/* The same definition evaluated only at (ms[i], ns[i]) for i < count. */
int oracle_gemm_sampled(const uint8_t *A, const float *sA, const uint8_t *B, const float *sB,
                        int64_t M, int64_t N, int64_t K,
                        const int64_t *ms, const int64_t *ns, int64_t count,
                        double *C, double *T, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || (K % 32) != 0 || count < 0) return -1;
    for (int64_t i = 0; i < count; ++i)
        if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) return -1;
    if (count == 0) return 0;
    job_t p;
    memset(&p, 0, sizeof p);
    p.A = A; p.sA = sA; p.B = B; p.sB = sB; p.M = M; p.N = N; p.K = K;
    p.ms = ms; p.ns = ns; p.count = count; p.C = C; p.T = T;
    return run(p, count, nthreads);
}

/* ------------------------------------------------- block quantization ---- */

/* Activation quantization to the operand format above (FP8 GEMM library
 * article, hncyxsy.com/news/241433, section 2.1: E4M3 with largest value 448;
 * section 2.2: one scale per 32x32 block).  For each 32x32 block of the bf16
 * matrix x [M, K] (row-major; the last row block may be partial):
 *
 *   s = amax / 448, an fp32 division (s = 1 when the block is all zero),
 *   q = E4M3(x / s), the division in fp32, then nearest-even and saturating
 *       through the search above.
 *
 * The quotient is an fp32 value, so the code decision is taken in fp32 as the
 * stated recipe reads; the search then sees it exactly (fp32 -> fp64 is exact).
 * q is [M, K] codes, s is [ceil(M/32), K/32] fp32, both row-major.
 * Returns 0, or -1 on a bad argument. */
static float bf16_bits_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

int oracle_quantize_blocks(const uint16_t *x, int64_t M, int64_t K, uint8_t *q, float *s) {
    if (M < 0 || K < 0 || (K % 32) != 0) return -1;
    const int64_t MB = (M + 31) / 32, KB = K / 32;
    for (int64_t mb = 0; mb < MB; ++mb) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            const int64_t r1 = (mb * 32 + 32 < M) ? mb * 32 + 32 : M;
            float amax = 0.0f;
            for (int64_t r = mb * 32; r < r1; ++r)
                for (int64_t c = kb * 32; c < kb * 32 + 32; ++c) {
                    const float a = fabsf(bf16_bits_to_float(x[r * K + c]));
                    if (a > amax) amax = a;
                }
            const float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
            s[mb * KB + kb] = sc;
            for (int64_t r = mb * 32; r < r1; ++r)
                for (int64_t c = kb * 32; c < kb * 32 + 32; ++c) {
                    const float t = bf16_bits_to_float(x[r * K + c]) / sc;
                    q[r * K + c] = (uint8_t)oracle_e4m3_quantize_one((double)t);
                }
        }
    }
    return 0;
}

/* ------------------------------------------ per-token x per-channel ---- */

/* Scales that do not vary along K (FP8 GEMM library article, section 2.2:
 * per-tensor, per-channel and per-token granularities; section 2.3: such
 * scales are applied in the GEMM's epilogue):
 *
 *   C[m,n] = sA[m] * sB[n] * sum_k A[m,k] * B[n,k]
 *
 * with sA [M] (per token / row of A) and sB [N] (per output channel / row of
 * B) fp32; a per-tensor scale is the constant vector.  The K sum is EXACT in
 * fp64 for K <= 2^15: each product is a multiple of 2^-18 below 2^18, so the
 * sum needs at most 51 bits.  It is then multiplied once by sA*sB (exact in
 * fp64).  T = |sA*sB| * sum_k |A*B|.  Returns 0, or -1 on a bad argument. */
int oracle_gemm_rowcol(const uint8_t *A, const float *sA, const uint8_t *B, const float *sB,
                       int64_t M, int64_t N, int64_t K, double *C, double *T) {
    if (M < 0 || N < 0 || K < 0 || K > (int64_t)1 << 15) return -1;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double p = e4m3_value(A[m * K + k]) * e4m3_value(B[n * K + k]);
                acc += p;
                mag += fabs(p);
            }
            const double s = (double)sA[m] * (double)sB[n];
            C[m * N + n] = s * acc;
            T[m * N + n] = fabs(s) * mag;
        }
    }
    return 0;
}

/* --------------------------------------------------- GEMM + residual ---- */

/* The block-scaled GEMM above followed by a bf16 residual added to each
 * output element (FP8 GEMM library article, hncyxsy.com/news/241433, section
 * 2.3: element-wise tail work belongs in the GEMM's epilogue instead of a
 * separate pass; section 5, pitfall 4, names the residual / LayerNorm fusion):
 *
 *   C[m,n] = sum_kb sA[m/32][kb] * sB[n/32][kb] * sum_{k in kb} A[m,k] * B[n,k]  +  R[m,n]
 *
 * R is bf16 [M, N] row-major, given as its 16-bit patterns; its value is exact
 * in fp64, and the GEMM value is the one oracle_gemm returns, so the sum is
 * the only extra rounding.  T is the GEMM's magnitude sum, unchanged.
 * `mutation` plants a known mistake for the pin tests only (0: none; 4: the
 * residual is left out; 5: the residual of column (n+1) mod N is added). */
static double residual_term(const uint16_t *R, int64_t N, int64_t m, int64_t n, int mutation) {
    if (mutation == 4) return 0.0;
    if (mutation == 5) n = (n + 1) % N;
    return oracle_bf16_value(R[m * N + n]);
}

int oracle_gemm_residual(const uint8_t *A, const float *sA, const uint8_t *B, const float *sB,
                         const uint16_t *R, int64_t M, int64_t N, int64_t K, double *C, double *T,
                         int nthreads, int mutation) {
    const int rc = oracle_gemm(A, sA, B, sB, M, N, K, C, T, nthreads, 0);
    if (rc != 0) return rc;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            C[m * N + n] += residual_term(R, N, m, n, mutation);
    return 0;
}

/* The same at the sampled coordinates (ms[i], ns[i]) for i < count. */
int oracle_gemm_residual_sampled(const uint8_t *A, const float *sA, const uint8_t *B, const float *sB,
                                 const uint16_t *R, int64_t M, int64_t N, int64_t K,
                                 const int64_t *ms, const int64_t *ns, int64_t count,
                                 double *C, double *T, int nthreads) {
    const int rc = oracle_gemm_sampled(A, sA, B, sB, M, N, K, ms, ns, count, C, T, nthreads);
    if (rc != 0) return rc;
    for (int64_t i = 0; i < count; ++i) C[i] += residual_term(R, N, ms[i], ns[i], 0);
    return 0;
}

/* ------------------------------------------------ per-token A scales ---- */

/* Per-token scales for A (FP8 GEMM library article, hncyxsy.com/news/241433,
 * section 2.2: per-token scales for activations, the finer alternative to
 * 32x32 blocks; here one scale per row of A per 32-K block, B keeping its
 * 32x32 blocks):
 *
 *   C[m,n] = sum_kb sA[m][kb] * sB[n/32][kb] * sum_{k in kb} A[m,k] * B[n,k]
 *
 * sA is [M, K/32] row-major, sB [ceil(N/32), K/32].  The same arithmetic as
 * oracle_gemm (exact 32-term sums in fp64, the exact product of the two fp32
 * scales, fp64 accumulation in ascending kb); only the A scale's row index
 * differs.  `mutation` 6 (pin tests only) reads the A scale of row
 * 32*(m/32) instead of m. */
int oracle_gemm_pertoken(const uint8_t *A, const float *sA, const uint8_t *B, const float *sB,
                         int64_t M, int64_t N, int64_t K, double *C, double *T, int mutation) {
    if (M < 0 || N < 0 || K < 0 || (K % 32) != 0) return -1;
    double tab[256];
    oracle_e4m3_table(tab);
    const int64_t KB = K / 32;
    for (int64_t m = 0; m < M; ++m) {
        const int64_t ra = mutation == 6 ? 32 * (m / 32) : m;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, mag = 0.0;
            for (int64_t kb = 0; kb < KB; ++kb) {
                double s = 0.0, sabs = 0.0;
                for (int64_t k = kb * 32; k < kb * 32 + 32; ++k) {
                    const double p = tab[A[m * K + k]] * tab[B[n * K + k]];
                    s += p;
                    sabs += fabs(p);
                }
                const double sc = (double)sA[ra * KB + kb] * (double)sB[(n / 32) * KB + kb];
                acc += sc * s;
                mag += fabs(sc) * sabs;
            }
            C[m * N + n] = acc;
            T[m * N + n] = mag;
        }
    }
    return 0;
}
