/*
 * CPU oracle for the ragged MXFP8 weight-gradient grouped GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it. It shares no code, header, table or constant generator with the
 * CUDA library.
 *
 * What it computes (plain definition, fp64, no blocking or fusion):
 *   "Ragged MXFP8 Weight Gradients: A FlyDSL Grouped GEMM on MI355X", section 1:
 *     wgrad dW[g] = dY[g]^T X[g]; the per-expert offsets cut the contraction
 *     (token) axis; A = dY^T [N,M] and B = X^T [K,M] are token-contiguous E4M3
 *     with one E8M0 scale per 32 tokens (planes [N,M/32] and [K,M/32]);
 *     offs records where each expert's run of tokens ends.
 *   Same page, section 5.5: the output is narrowed to bf16 with
 *     round-to-nearest-even.
 *   "Group-GEMM in XLA", Part 3, "Contracting": group g contracts only over
 *     [prefix_exclusive[g], prefix_inclusive[g]) of the contracted axis and
 *     writes out[g].
 *
 *   out[g,n,k] = bf16_rne( sum_{t in [lo_g, hi_g)}
 *                   (e4m3(A[n,t]) * e8m0(sA[n,t/32])) * (e4m3(B[k,t]) * e8m0(sB[k,t/32])) )
 *   lo_0 = 0, lo_g = offs[g-1], hi_g = offs[g].
 *
 * Each product is exact in fp64 (4-bit significands times powers of two), the
 * sum runs in token order in fp64, and the fp64 sum is rounded to bf16 in one
 * step (no intermediate fp32).
 *
 * The tokenwise quantiser follows the same page, section 1 (one E8M0 scale per
 * 32 elements along the token axis) with the scale rule 2^ceil(log2(amax/448)),
 * read exactly as: e = the smallest integer with amax <= 448 * 2^e, clamped to
 * [-127, 127]; elements are x * 2^-e rounded to E4M3 (nearest-even, saturating).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- decoding */

/* OCP E4M3 ("E4M3FN"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; largest finite value 448. */
double oracle_dec_e4m3(uint8_t b) {
    int s = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);            /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10);  /* (1 + m/8) * 2^(e-7)   */
    return s ? -v : v;
}

/* E8M0: an unsigned biased exponent, value 2^(b-127); 0xFF is NaN. */
double oracle_dec_e8m0(uint8_t b) {
    if (b == 0xFF) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* ------------------------------------------------------------- rounding */

/* Round an integer-valued double r to even if it lies exactly halfway. r is
 * the exact quotient x/q; return nearest integer, ties to even. */
static double round_half_even(double r) {
    double f = floor(r);
    double d = r - f; /* exact: r and f share the binade scale */
    if (d > 0.5) return f + 1.0;
    if (d < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* fp64 -> bf16 bits, round to nearest even, directly from the fp64 value.
 * bf16: 8 exponent bits (bias 127), 7 stored mantissa bits; the quantum in the
 * binade [2^E, 2^(E+1)) is 2^(E-7), and 2^-133 below the normal range. */
uint16_t oracle_bf16_rne(double x) {
    if (isnan(x)) return 0x7FC0;
    int neg = signbit(x) ? 1 : 0;
    double ax = fabs(x);
    uint16_t sign = neg ? 0x8000 : 0;
    if (isinf(ax)) return sign | 0x7F80;
    if (ax == 0.0) return sign;
    int ex;
    (void)frexp(ax, &ex);          /* ax = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;                /* ax in [2^E, 2^(E+1)) */
    if (E < -126) E = -126;        /* subnormal range shares the 2^-133 quantum */
    double q = ldexp(1.0, E - 7);
    double r = round_half_even(ax / q); /* ax/q is exact (power-of-two divisor) */
    double v = r * q;
    if (v > 3.3895313892515355e38) return sign | 0x7F80; /* above max finite bf16 */
    /* v is exactly representable in bf16, hence in fp32: take the top half. */
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

/* fp64 -> E4M3 bits, nearest-even, saturating to +-448. Used by the quantiser
 * on y = x * 2^-e, which is computed exactly in fp64. */
static uint8_t e4m3_rne_satfinite(double y) {
    if (isnan(y)) return 0x7F;
    int neg = signbit(y) ? 1 : 0;
    double ay = fabs(y);
    uint8_t sign = neg ? 0x80 : 0;
    if (ay >= 448.0) return sign | 0x7E; /* satfinite */
    if (ay == 0.0) return sign;
    int ex;
    (void)frexp(ay, &ex);
    int E = ex - 1;               /* ay in [2^E, 2^(E+1)) */
    if (E < -6) E = -6;           /* subnormals: quantum 2^-9 */
    double q = ldexp(1.0, E - 3);
    double r = round_half_even(ay / q);
    double v = r * q;
    if (v > 448.0) v = 448.0;     /* cannot happen below 448, kept for clarity */
    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -6)) {      /* subnormal: v = m * 2^-9 */
        int m = (int)(v / ldexp(1.0, -9));
        return sign | (uint8_t)m;
    }
    int ev;
    double fv = frexp(v, &ev);    /* v = fv * 2^ev, fv in [0.5,1) */
    int Ev = ev - 1;              /* v = (1 + m/8) * 2^Ev */
    int m = (int)((fv * 2.0 - 1.0) * 8.0);
    return sign | (uint8_t)(((Ev + 7) << 3) | m);
}

/* ------------------------------------------------------------- threading */

typedef void (*range_fn)(void* ctx, int64_t lo, int64_t hi);
typedef struct { range_fn fn; void* ctx; int64_t lo, hi; } range_job;

static void* range_thunk(void* p) {
    range_job* j = (range_job*)p;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

/* Split [0, n) into nthreads contiguous parts, one pthread each. */
static void parallel_for(int64_t n, int nthreads, range_fn fn, void* ctx) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    if (nthreads == 1) { fn(ctx, 0, n); return; }
    pthread_t th[256];
    range_job jobs[256];
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].fn = fn; jobs[i].ctx = ctx;
        jobs[i].lo = n * i / nthreads;
        jobs[i].hi = n * (i + 1) / nthreads;
        pthread_create(&th[i], NULL, range_thunk, &jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------- wgrad */

/* Validate the offsets as the definition needs them: non-decreasing, within
 * [0, M], multiples of 32 (the scale block). Returns 0 or -1. */
static int check_offs(const int32_t* offs, int E, int64_t M) {
    int64_t prev = 0;
    for (int g = 0; g < E; ++g) {
        int64_t o = offs[g];
        if (o < prev || o > M || (o % 32) != 0) return -1;
        prev = o;
    }
    return 0;
}

typedef struct {
    const uint8_t *A, *sA, *B, *sB;
    int N, K;
    int64_t M, lo, hi;
    const double *lutA;     /* e4m3 decode table */
    const double *lutS;     /* e8m0 decode table */
    uint16_t* out;          /* [N,K] slab of this expert */
    double* acc;            /* optional [N,K] fp64 sums */
    double* absacc;         /* optional [N,K] sum of |a*b| */
} wgrad_ctx;

static void wgrad_rows(void* p, int64_t n0, int64_t n1) {
    wgrad_ctx* c = (wgrad_ctx*)p;
    int64_t sM = c->M / 32;
    for (int64_t n = n0; n < n1; ++n) {
        const uint8_t* a = c->A + n * c->M;
        const uint8_t* sa = c->sA + n * sM;
        for (int64_t k = 0; k < c->K; ++k) {
            const uint8_t* b = c->B + k * c->M;
            const uint8_t* sb = c->sB + k * sM;
            double acc = 0.0, aacc = 0.0;
            for (int64_t t = c->lo; t < c->hi; ++t) {
                double av = c->lutA[a[t]] * c->lutS[sa[t / 32]];
                double bv = c->lutA[b[t]] * c->lutS[sb[t / 32]];
                double pr = av * bv;
                acc += pr;
                aacc += fabs(pr);
            }
            int64_t o = n * c->K + k;
            c->out[o] = oracle_bf16_rne(acc);
            if (c->acc) c->acc[o] = acc;
            if (c->absacc) c->absacc[o] = aacc;
        }
    }
}

static void fill_luts(double* lutA, double* lutS) {
    for (int i = 0; i < 256; ++i) {
        lutA[i] = oracle_dec_e4m3((uint8_t)i);
        lutS[i] = oracle_dec_e8m0((uint8_t)i);
    }
}

/* Full output. out: bf16 bits [E,N,K]; acc/absacc: optional fp64 [E,N,K].
 * Returns 0, or -1 on invalid arguments (nothing written). */
int oracle_wgrad(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                 const int32_t* offs, int E, int N, int K, int64_t M,
                 uint16_t* out, double* acc, double* absacc, int nthreads) {
    if (E < 0 || N < 0 || K < 0 || M < 0 || (M % 32) != 0) return -1;
    if (E > 0 && !offs) return -1;
    if (check_offs(offs, E, M) != 0) return -1;
    double lutA[256], lutS[256];
    fill_luts(lutA, lutS);
    for (int g = 0; g < E; ++g) {
        wgrad_ctx c;
        c.A = A; c.sA = sA; c.B = B; c.sB = sB;
        c.N = N; c.K = K; c.M = M;
        c.lo = g == 0 ? 0 : offs[g - 1];
        c.hi = offs[g];
        c.lutA = lutA; c.lutS = lutS;
        int64_t slab = (int64_t)g * N * K;
        c.out = out + slab;
        c.acc = acc ? acc + slab : NULL;
        c.absacc = absacc ? absacc + slab : NULL;
        parallel_for(N, nthreads, wgrad_rows, &c);
    }
    return 0;
}

typedef struct {
    const uint8_t *A, *sA, *B, *sB;
    const int32_t* offs;
    int64_t M;
    const int32_t *pg, *pn, *pk;
    const double *lutA, *lutS;
    uint16_t* out;
    double *acc, *absacc;
} points_ctx;

static void wgrad_points_range(void* p, int64_t i0, int64_t i1) {
    points_ctx* c = (points_ctx*)p;
    int64_t sM = c->M / 32;
    for (int64_t i = i0; i < i1; ++i) {
        int g = c->pg[i];
        int64_t n = c->pn[i], k = c->pk[i];
        int64_t lo = g == 0 ? 0 : c->offs[g - 1];
        int64_t hi = c->offs[g];
        const uint8_t* a = c->A + n * c->M;
        const uint8_t* sa = c->sA + n * sM;
        const uint8_t* b = c->B + k * c->M;
        const uint8_t* sb = c->sB + k * sM;
        double acc = 0.0, aacc = 0.0;
        for (int64_t t = lo; t < hi; ++t) {
            double pr = (c->lutA[a[t]] * c->lutS[sa[t / 32]]) * (c->lutA[b[t]] * c->lutS[sb[t / 32]]);
            acc += pr;
            aacc += fabs(pr);
        }
        c->out[i] = oracle_bf16_rne(acc);
        if (c->acc) c->acc[i] = acc;
        if (c->absacc) c->absacc[i] = aacc;
    }
}

/* Selected output elements (g[i], n[i], k[i]), i < P, by the same definition. */
int oracle_wgrad_points(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                        const int32_t* offs, int E, int N, int K, int64_t M,
                        const int32_t* pg, const int32_t* pn, const int32_t* pk, int64_t P,
                        uint16_t* out, double* acc, double* absacc, int nthreads) {
    if (E < 0 || N < 0 || K < 0 || M < 0 || (M % 32) != 0 || P < 0) return -1;
    if (check_offs(offs, E, M) != 0) return -1;
    for (int64_t i = 0; i < P; ++i)
        if (pg[i] < 0 || pg[i] >= E || pn[i] < 0 || pn[i] >= N || pk[i] < 0 || pk[i] >= K) return -1;
    double lutA[256], lutS[256];
    fill_luts(lutA, lutS);
    points_ctx c;
    c.A = A; c.sA = sA; c.B = B; c.sB = sB; c.offs = offs; c.M = M;
    c.pg = pg; c.pn = pn; c.pk = pk;
    c.lutA = lutA; c.lutS = lutS;
    c.out = out; c.acc = acc; c.absacc = absacc;
    parallel_for(P, nthreads, wgrad_points_range, &c);
    return 0;
}

/* ------------------------------------------------------------- grouped GEMM */

/* The non-contracting ragged dot ("Group-GEMM in XLA", Part 1, "The Ragged-Dot
 * Operation"), in MXFP8: the rows of X are cut into E contiguous groups by
 * offs (inclusive ends), and every row t of group g multiplies the weights of
 * expert g:
 *   out[t][n] = bf16_rne( sum_k x(t,k) w(g,n,k) ),
 *   x(t,k) = e4m3(X[t][k]) 2^(sX[t][k/32] - 127),  w likewise from W[g][n][k],
 * both operands quantised along the contracted axis k. Rows at or past
 * offs[E-1] belong to no group and are zero. offs need not be multiples of
 * 32 (the scale blocks run along k, not t). */
static int check_row_offs(const int32_t* offs, int E, int64_t M) {
    int64_t prev = 0;
    for (int g = 0; g < E; ++g) {
        int64_t o = offs[g];
        if (o < prev || o > M) return -1;
        prev = o;
    }
    return 0;
}

typedef struct {
    const uint8_t *X, *sX, *W, *sW;
    const int32_t* offs;
    int E, N, K;
    int64_t M;
    const double *lutA, *lutS;
    uint16_t* out;
    double *acc, *absacc;
    const int64_t *pt, *pn; /* points (NULL: every element) */
} gemm_ctx;

static int group_of_row(const int32_t* offs, int E, int64_t t) {
    for (int g = 0; g < E; ++g)
        if (t < offs[g]) return g;
    return -1; /* past the last group */
}

static void gemm_element(const gemm_ctx* c, int64_t t, int64_t n, int64_t o) {
    int g = group_of_row(c->offs, c->E, t);
    double acc = 0.0, aacc = 0.0;
    if (g >= 0) {
        int64_t sK = c->K / 32;
        const uint8_t* x = c->X + t * c->K;
        const uint8_t* sx = c->sX + t * sK;
        const uint8_t* w = c->W + ((int64_t)g * c->N + n) * c->K;
        const uint8_t* sw = c->sW + ((int64_t)g * c->N + n) * sK;
        for (int64_t k = 0; k < c->K; ++k) {
            double pr = (c->lutA[x[k]] * c->lutS[sx[k / 32]]) * (c->lutA[w[k]] * c->lutS[sw[k / 32]]);
            acc += pr;
            aacc += fabs(pr);
        }
    }
    c->out[o] = oracle_bf16_rne(acc);
    if (c->acc) c->acc[o] = acc;
    if (c->absacc) c->absacc[o] = aacc;
}

static void gemm_rows(void* p, int64_t t0, int64_t t1) {
    gemm_ctx* c = (gemm_ctx*)p;
    for (int64_t t = t0; t < t1; ++t)
        for (int64_t n = 0; n < c->N; ++n) gemm_element(c, t, n, t * c->N + n);
}

static void gemm_points(void* p, int64_t i0, int64_t i1) {
    gemm_ctx* c = (gemm_ctx*)p;
    for (int64_t i = i0; i < i1; ++i) gemm_element(c, c->pt[i], c->pn[i], i);
}

/* Full output out [M][N] bf16 bits (acc/absacc optional fp64 [M][N]); with
 * pt/pn (P points) only those elements, out[i] for (pt[i], pn[i]). Returns 0,
 * or -1 on invalid arguments (nothing written). */
int oracle_grouped_gemm(const uint8_t* X, const uint8_t* sX, const uint8_t* W, const uint8_t* sW,
                        const int32_t* offs, int E, int64_t M, int N, int K,
                        const int64_t* pt, const int64_t* pn, int64_t P,
                        uint16_t* out, double* acc, double* absacc, int nthreads) {
    if (E < 1 || M < 0 || N < 0 || K < 32 || (K % 32) != 0 || !offs) return -1;
    if (check_row_offs(offs, E, M) != 0) return -1;
    if (pt) {
        for (int64_t i = 0; i < P; ++i)
            if (pt[i] < 0 || pt[i] >= M || pn[i] < 0 || pn[i] >= N) return -1;
    }
    double lutA[256], lutS[256];
    fill_luts(lutA, lutS);
    gemm_ctx c;
    c.X = X; c.sX = sX; c.W = W; c.sW = sW; c.offs = offs;
    c.E = E; c.N = N; c.K = K; c.M = M;
    c.lutA = lutA; c.lutS = lutS;
    c.out = out; c.acc = acc; c.absacc = absacc;
    c.pt = pt; c.pn = pn;
    if (pt) parallel_for(P, nthreads, gemm_points, &c);
    else parallel_for(M, nthreads, gemm_rows, &c);
    return 0;
}

/* ------------------------------------------------------------- quantiser */

typedef struct {
    const float* x;
    int64_t M;
    uint8_t *q, *s;
} quant_ctx;

static void quant_rows(void* p, int64_t r0, int64_t r1) {
    quant_ctx* c = (quant_ctx*)p;
    int64_t nb = c->M / 32;
    for (int64_t r = r0; r < r1; ++r) {
        const float* xr = c->x + r * c->M;
        for (int64_t bI = 0; bI < nb; ++bI) {
            const float* xb = xr + bI * 32;
            uint8_t* qb = c->q + r * c->M + bI * 32;
            double amax = 0.0;
            int finite = 1;
            for (int i = 0; i < 32; ++i) {
                double v = fabs((double)xb[i]);
                if (!isfinite(v)) finite = 0;
                else if (v > amax) amax = v;
            }
            if (!finite) {       /* reading: a non-finite block gets NaN scale and NaN data */
                c->s[r * nb + bI] = 0xFF;
                memset(qb, 0x7F, 32);
                continue;
            }
            int e;
            if (amax == 0.0) {
                e = -127;
            } else {
                /* smallest integer e with amax <= 448 * 2^e */
                int ex;
                double f = frexp(amax, &ex);     /* amax = f * 2^ex, f in [0.5,1) */
                /* 448 = 0.875 * 2^9: f <= 0.875 -> e = ex - 9, else ex - 8 */
                e = (f <= 0.875) ? ex - 9 : ex - 8;
                if (e < -127) e = -127;
                if (e > 127) e = 127;
            }
            c->s[r * nb + bI] = (uint8_t)(e + 127);
            double inv = ldexp(1.0, -e);
            for (int i = 0; i < 32; ++i) qb[i] = e4m3_rne_satfinite((double)xb[i] * inv);
        }
    }
}

/* x: fp32 [R,M] token-contiguous -> q: E4M3 [R,M], s: E8M0 [R,M/32]. */
int oracle_quantize_tokenwise(const float* x, int64_t R, int64_t M, uint8_t* q, uint8_t* s, int nthreads) {
    if (R < 0 || M < 0 || (M % 32) != 0) return -1;
    quant_ctx c;
    c.x = x; c.M = M; c.q = q; c.s = s;
    parallel_for(R, nthreads, quant_rows, &c);
    return 0;
}
