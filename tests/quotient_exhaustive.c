/* Exhaustive check of the block quantizer's scale and reciprocal quotient.
 *
 * The quantizer codes q = E4M3(x / s) with s = RN(amax / 448) for a block whose
 * largest magnitude is amax (FP8 GEMM library article, hncyxsy.com/news/241433,
 * sections 2.1-2.2).  Its kernel divides nowhere in the common case; both
 * steps use Markstein's correction (P. Markstein, IBM J. Res. Develop. 34(1),
 * 1990), emulated here operation by operation in IEEE fp32 with fused
 * multiply-adds:
 *   scale:    y = RN(amax r448), r448 = RN(1/448);
 *             s = RN(y + r448 RN(amax - 448 y))
 *   quotient: for finite s >= 2^T, nr = -RN(1/s), y' = RN(x nr),
 *             e = RN(y' s + x), n = RN(y' + e nr), code = E4M3(n) ^ 0x80
 *             (n is the negated quotient; flipping the code's sign bit gives
 *             the code of -n); smaller or non-finite scales divide.
 * x and amax are bf16 values, so the input space is small enough to
 * enumerate: every positive finite bf16 amax, every bf16 x with |x| <= amax,
 * both signs.  The scale is compared with RN(amax/448), -n with RN(x/s), and
 * the code with E4M3(RN(x/s)) (nearest, ties to the even code, saturating at
 * 448, written as a search over the codes).
 *
 * usage: quotient_exhaustive T_log2 amax_bits_lo amax_bits_hi nthreads
 * prints: pairs quotient_mismatches big_quotient_mismatches code_mismatches
 *         scale_mismatches
 * where big_quotient_mismatches counts those with |x/s| >= 2^-10.
 * Build with -ffp-contract=off so that no other product is fused. */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float from_bits(uint32_t u) {
    float x;
    memcpy(&x, &u, sizeof x);
    return x;
}
static uint32_t to_bits(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    return u;
}

/* E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; 0x7F/0xFF are NaN. */
static double e4m3_value(unsigned c) {
    const unsigned e = (c >> 3) & 15u, m = c & 7u;
    const double v = e == 0u ? ldexp((double)m, -9) : ldexp((double)(8u + m), (int)e - 10);
    return (c & 0x80u) ? -v : v;
}
static unsigned e4m3_code(float x) {
    if (isnan(x)) return 0x7Fu;
    const double a = fabs((double)x);
    unsigned best = 0u;
    double best_d = INFINITY;
    for (unsigned c = 0; c <= 0x7Eu; ++c) {
        const double d = fabs(e4m3_value(c) - a);
        if (d < best_d || (d == best_d && (c & 1u) == 0u)) {
            best = c;
            best_d = d;
        }
    }
    return (signbit(x) ? 0x80u : 0u) | best;
}

struct job {
    float threshold;
    uint32_t lo, hi, tid, nthreads;
    long long pairs, bad_q, bad_big, bad_code, bad_scale;
};

static float block_scale(float amax) {
    const float r448 = 1.0f / 448.0f;
    const float y = amax * r448;
    return fmaf(fmaf(-y, 448.0f, amax), r448, y);
}

static void *run(void *arg) {
    struct job *j = (struct job *)arg;
    for (uint32_t ab = j->lo + j->tid; ab <= j->hi; ab += j->nthreads) {
        const float amax = from_bits(ab << 16);
        const float s = block_scale(amax);
        if (to_bits(s) != to_bits(amax / 448.0f)) ++j->bad_scale;
        if (!(s >= j->threshold && s <= 3.40282347e38f)) continue;   /* the division branch */
        const float nr = -(1.0f / s);
        for (uint32_t xb = 0; xb <= ab; ++xb) {
            for (int neg = 0; neg < 2; ++neg) {
                const float x = from_bits((xb << 16) | (neg ? 0x80000000u : 0u));
                const float y = x * nr;          /* -RN(x r) */
                const float e = fmaf(y, s, x);   /* x - y s  */
                const float n = fmaf(e, nr, y);  /* -q       */
                const float t = x / s;
                ++j->pairs;
                /* equal bits give equal codes: the code search below is
                 * symmetric in the sign, so E4M3(n) ^ 0x80 == E4M3(-n) */
                if (to_bits(-n) == to_bits(t)) continue;
                ++j->bad_q;
                if (fabsf(t) >= 0x1p-10f) ++j->bad_big;
                if ((e4m3_code(n) ^ 0x80u) != e4m3_code(t)) ++j->bad_code;
            }
        }
    }
    return NULL;
}

int main(int argc, char **argv) {
    if (argc != 5) {
        fprintf(stderr, "usage: %s T_log2 amax_bits_lo amax_bits_hi nthreads\n", argv[0]);
        return 2;
    }
    const float threshold = ldexpf(1.0f, atoi(argv[1]));
    const uint32_t lo = (uint32_t)strtoul(argv[2], NULL, 0), hi = (uint32_t)strtoul(argv[3], NULL, 0);
    int nt = atoi(argv[4]);
    if (nt < 1) nt = 1;
    if (nt > 256) nt = 256;
    if (lo < 1u || hi > 0x7F7Fu || lo > hi) return 2;   /* positive finite bf16 only */
    struct job jobs[256];
    pthread_t th[256];
    for (int t = 0; t < nt; ++t) {
        jobs[t] = (struct job){threshold, lo, hi, (uint32_t)t, (uint32_t)nt, 0, 0, 0, 0, 0};
        if (pthread_create(&th[t], NULL, run, &jobs[t]) != 0) return 3;
    }
    long long pairs = 0, bad_q = 0, bad_big = 0, bad_code = 0, bad_scale = 0;
    for (int t = 0; t < nt; ++t) {
        pthread_join(th[t], NULL);
        pairs += jobs[t].pairs;
        bad_q += jobs[t].bad_q;
        bad_big += jobs[t].bad_big;
        bad_code += jobs[t].bad_code;
        bad_scale += jobs[t].bad_scale;
    }
    printf("%lld %lld %lld %lld %lld\n", pairs, bad_q, bad_big, bad_code, bad_scale);
    return 0;
}
