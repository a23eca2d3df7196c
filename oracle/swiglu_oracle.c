/*
 * Plain CPU oracle for the fused SwiGLU up-projection.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or load
 * this file: only the tests, the smoke check and the bench's CPU-baseline leg
 * use it. It shares no code, header or constant with the CUDA library.
 *
 * What it computes ("Tile-Level Activation Overlap for Efficient LLM
 * Inference", Section 1 Introduction, the gated-MLP definition; restated in
 * the technical summary's problem statement): for every output row m and
 * column n,
 *
 *     Gate[m,n] = sum_k A[m,k] * W1[k,n]
 *     Up[m,n]   = sum_k A[m,k] * W2[k,n]
 *     Y[m,n]    = SiLU(Gate[m,n]) * Up[m,n],   SiLU(x) = x / (1 + e^-x)
 *
 * A [M,K], W1 [K,N], W2 [K,N] and Y [M,N] are row-major arrays of BF16 bit
 * patterns (or, in oracle_swiglu_up_fp8, FP8 E4M3 bytes for the inputs with
 * per-tensor scales; Y stays BF16). Every BF16 x BF16 product is exact in binary64, the K-term sums
 * run in binary64 in increasing k, SiLU and the final product are evaluated
 * in binary64, and the result is rounded ONCE to BF16 with
 * round-to-nearest-even, straight from the double (going through binary32
 * first could round twice).
 *
 * oracle_matmul computes the plain product C = A x B the same way (one
 * binary64 sum per element, one BF16 rounding): the down-projection
 * out = Y x W3 that completes the gated MLP.
 *
 * The loops are the definition written out: no blocking, no reordering of
 * the k sum, no fusion beyond the definition. Rows are split across threads;
 * each output element is computed by exactly one thread in the fixed order
 * above, so the result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* BF16 bit pattern -> binary64. A BF16 value is the upper half of a binary32
 * pattern, so the conversion is exact. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* binary64 -> BF16 bit pattern, round to nearest, ties to even.
 * BF16: 1 sign bit, 8 exponent bits (bias 127), 7 stored significand bits.
 * For |x| in [2^E, 2^(E+1)) with E >= -126 the spacing of BF16 values is
 * 2^(E-7); below 2^-126 (subnormals) it is fixed at 2^-133. Dividing |x| by
 * the spacing is an exact power-of-two scaling, nearbyint() rounds the
 * quotient to the nearest integer with ties to even (default rounding mode),
 * and multiplying back is exact. Results at or above 2^128 overflow to
 * infinity. */
uint16_t oracle_double_to_bf16(double x)
{
    if (isnan(x))
        return (uint16_t)0x7FC0;
    uint16_t sign = signbit(x) ? (uint16_t)0x8000 : (uint16_t)0;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    int e;
    (void)frexp(a, &e);          /* a = f * 2^e with f in [0.5, 1) */
    int E = e - 1;               /* a in [2^E, 2^(E+1)) */
    if (E < -126)
        E = -126;
    double spacing = ldexp(1.0, E - 7);
    double r = nearbyint(a / spacing);
    double v = r * spacing;
    if (v >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80);
    float f = (float)v;          /* v is a BF16 value: exact in binary32 */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

/* FP8 E4M3 bit pattern -> binary64 (exact): 1 sign bit, 4 exponent bits with
 * bias 7, 3 stored significand bits; exponent field 0 holds subnormals
 * (significand * 2^-9); the pattern S.1111.111 is NaN and there is no
 * infinity, so the largest finite magnitude is 1.75 * 2^8 = 448. */
double oracle_e4m3_to_double(uint8_t b)
{
    const int sign = (b >> 7) & 1;
    const int e = (b >> 3) & 0xF;
    const int m = b & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* SiLU (Swish with beta = 1): x * sigmoid(x) = x / (1 + e^-x). For x far
 * below zero e^-x overflows to +inf and the quotient is -0, the limit. */
double oracle_silu(double x)
{
    return x / (1.0 + exp(-x));
}

typedef struct {
    const uint16_t *A, *W1, *W2;        /* BF16 inputs, or NULL when FP8 */
    const uint8_t *A8, *W18, *W28;      /* FP8 E4M3 inputs, or NULL when BF16 */
    double scale_gate, scale_up;        /* FP8: s_a * s_w1 and s_a * s_w2; BF16: 1 */
    int plain;                          /* 1: out = A x W1 alone (no W2, no SiLU) */
    int64_t M, N, K;
    int64_t n0, n1;        /* output columns [n0, n1) */
    const int64_t *rows;   /* NULL: rows 0..nrows-1 */
    int64_t nrows;
    uint16_t *Y;           /* [nrows, n1-n0] bf16 bits, may be NULL */
    double *Yd;            /* [nrows, n1-n0] unrounded SiLU(g)*u, may be NULL */
    double *G, *U;         /* [nrows, n1-n0], may be NULL */
    int64_t r_begin, r_end;
    int status;
} job_t;

static void *run_rows(void *arg)
{
    job_t *j = (job_t *)arg;
    const int64_t N = j->N, K = j->K, n0 = j->n0, n1 = j->n1, W = n1 - n0;
    double *g = (double *)malloc((size_t)W * sizeof(double));
    double *u = (double *)malloc((size_t)W * sizeof(double));
    if (!g || !u) {
        free(g);
        free(u);
        j->status = 1;
        return NULL;
    }
    for (int64_t r = j->r_begin; r < j->r_end; ++r) {
        const int64_t m = j->rows ? j->rows[r] : r;
        for (int64_t i = 0; i < W; ++i) {
            g[i] = 0.0;
            u[i] = 0.0;
        }
        /* Gate = A x W1 and Up = A x W2, summed over k in increasing order. */
        if (j->A) {
            const uint16_t *a_row = j->A + m * K;
            for (int64_t k = 0; k < K; ++k) {
                const double a = oracle_bf16_to_double(a_row[k]);
                const uint16_t *w1 = j->W1 + k * N + n0;
                for (int64_t i = 0; i < W; ++i)
                    g[i] += a * oracle_bf16_to_double(w1[i]);
                if (j->plain)
                    continue;
                const uint16_t *w2 = j->W2 + k * N + n0;
                for (int64_t i = 0; i < W; ++i)
                    u[i] += a * oracle_bf16_to_double(w2[i]);
            }
        } else {
            /* FP8: the sums of the raw E4M3 values, then the per-tensor
             * scales (A = s_a * A8, W1 = s_w1 * W1_8, W2 = s_w2 * W2_8). */
            const uint8_t *a_row = j->A8 + m * K;
            for (int64_t k = 0; k < K; ++k) {
                const double a = oracle_e4m3_to_double(a_row[k]);
                const uint8_t *w1 = j->W18 + k * N + n0;
                const uint8_t *w2 = j->W28 + k * N + n0;
                for (int64_t i = 0; i < W; ++i) {
                    g[i] += a * oracle_e4m3_to_double(w1[i]);
                    u[i] += a * oracle_e4m3_to_double(w2[i]);
                }
            }
            for (int64_t i = 0; i < W; ++i) {
                g[i] *= j->scale_gate;
                u[i] *= j->scale_up;
            }
        }
        /* Y = SiLU(Gate) (.) Up (or, plain, the sum itself), rounded once
         * to BF16. */
        for (int64_t i = 0; i < W; ++i) {
            const double y = j->plain ? g[i] : oracle_silu(g[i]) * u[i];
            if (j->Y)
                j->Y[r * W + i] = oracle_double_to_bf16(y);
            if (j->Yd)
                j->Yd[r * W + i] = y;
            if (j->G)
                j->G[r * W + i] = g[i];
            if (j->U)
                j->U[r * W + i] = u[i];
        }
    }
    free(g);
    free(u);
    return NULL;
}

static int run_jobs(const job_t *proto, int64_t nrows, int nthreads)
{
    if (nthreads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = c > 0 ? (int)c : 1;
    }
    if (nthreads > nrows)
        nthreads = (int)nrows;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    char *created = (char *)calloc((size_t)nthreads, 1);
    if (!jobs || !tids || !created) {
        free(jobs);
        free(tids);
        free(created);
        return 1;
    }
    int status = 0;
    for (int t = 0; t < nthreads; ++t) {
        job_t *j = &jobs[t];
        *j = *proto;
        j->r_begin = nrows * t / nthreads;
        j->r_end = nrows * (t + 1) / nthreads;
        if (pthread_create(&tids[t], NULL, run_rows, j) == 0)
            created[t] = 1;
        else
            run_rows(j);   /* no thread available: run it here */
    }
    for (int t = 0; t < nthreads; ++t) {
        if (created[t])
            pthread_join(tids[t], NULL);
        status |= jobs[t].status;
    }
    free(jobs);
    free(tids);
    free(created);
    return status;
}

static int check_rows(int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                      int64_t n0, int64_t n1)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0)
        return 1;
    if (n0 < 0 || n1 > N || n0 > n1)
        return 1;
    if (!rows && nrows > M)
        return 1;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M)
            return 1;
    return 0;
}

/*
 * Computes the rows listed in `rows` (or rows 0..nrows-1 when rows is NULL)
 * and the columns [n0, n1) of Y = SiLU(A x W1) (.) (A x W2). Outputs are
 * [nrows, n1-n0], indexed by position in the row list and by n - n0. Any of
 * Y, Yd, G, U may be NULL. nthreads <= 0 uses every online core. Returns 0 on
 * success, 1 on bad arguments or allocation failure.
 */
int oracle_swiglu_up(const uint16_t *A, const uint16_t *W1, const uint16_t *W2,
                     int64_t M, int64_t N, int64_t K,
                     const int64_t *rows, int64_t nrows, int64_t n0, int64_t n1,
                     uint16_t *Y, double *Yd, double *G, double *U,
                     int nthreads)
{
    if (!A || !W1 || !W2 || check_rows(M, N, K, rows, nrows, n0, n1))
        return 1;
    if (nrows == 0 || n1 == n0)
        return 0;
    job_t proto;
    memset(&proto, 0, sizeof proto);
    proto.A = A; proto.W1 = W1; proto.W2 = W2;
    proto.scale_gate = 1.0; proto.scale_up = 1.0;
    proto.M = M; proto.N = N; proto.K = K;
    proto.n0 = n0; proto.n1 = n1;
    proto.rows = rows; proto.nrows = nrows;
    proto.Y = Y; proto.Yd = Yd; proto.G = G; proto.U = U;
    return run_jobs(&proto, nrows, nthreads);
}

/*
 * The same with FP8 E4M3 inputs and per-tensor scales: the inputs stand for
 * A = s_a * A8, W1 = s_w1 * W1_8, W2 = s_w2 * W2_8 (A8 [M,K], W1_8/W2_8
 * [K,N], row-major bytes). Gate = s_a*s_w1 * sum_k A8 W1_8 and Up likewise:
 * the E4M3 products and sums are exact in binary64, then scaled, then SiLU,
 * the product and one rounding to BF16 as in oracle_swiglu_up.
 */
int oracle_swiglu_up_fp8(const uint8_t *A8, const uint8_t *W18, const uint8_t *W28,
                         int64_t M, int64_t N, int64_t K,
                         double s_a, double s_w1, double s_w2,
                         const int64_t *rows, int64_t nrows, int64_t n0, int64_t n1,
                         uint16_t *Y, double *Yd, double *G, double *U,
                         int nthreads)
{
    if (!A8 || !W18 || !W28 || check_rows(M, N, K, rows, nrows, n0, n1))
        return 1;
    if (nrows == 0 || n1 == n0)
        return 0;
    job_t proto;
    memset(&proto, 0, sizeof proto);
    proto.A8 = A8; proto.W18 = W18; proto.W28 = W28;
    proto.scale_gate = s_a * s_w1;
    proto.scale_up = s_a * s_w2;
    proto.M = M; proto.N = N; proto.K = K;
    proto.n0 = n0; proto.n1 = n1;
    proto.rows = rows; proto.nrows = nrows;
    proto.Y = Y; proto.Yd = Yd; proto.G = G; proto.U = U;
    return run_jobs(&proto, nrows, nthreads);
}

/*
 * Plain product C = A x B of BF16 bit patterns, A [M,K] and B [K,N]
 * row-major: every product exact in binary64, the sum in increasing k, one
 * BF16 round-to-nearest-even at the end. This is the down-projection that
 * completes the gated MLP whose share of run time the paper measures
 * ("Tile-Level Activation Overlap for Efficient LLM Inference", Section 1
 * Introduction, Figure 1): out = Y x W3 with Y the BF16 output of the
 * fused up-projection, W3 [N, H]. The paper defines only Gate, Up and Y;
 * the down-projection is the usual completion of that MLP. Rows and
 * columns as in oracle_swiglu_up; C_d (may be NULL) receives the unrounded
 * binary64 sums.
 */
int oracle_matmul(const uint16_t *A, const uint16_t *B, int64_t M, int64_t N, int64_t K,
                  const int64_t *rows, int64_t nrows, int64_t n0, int64_t n1,
                  uint16_t *C, double *C_d, int nthreads)
{
    if (!A || !B || check_rows(M, N, K, rows, nrows, n0, n1))
        return 1;
    if (nrows == 0 || n1 == n0)
        return 0;
    job_t proto;
    memset(&proto, 0, sizeof proto);
    proto.A = A; proto.W1 = B; proto.W2 = NULL;
    proto.plain = 1;
    proto.scale_gate = 1.0; proto.scale_up = 1.0;
    proto.M = M; proto.N = N; proto.K = K;
    proto.n0 = n0; proto.n1 = n1;
    proto.rows = rows; proto.nrows = nrows;
    proto.Y = C; proto.Yd = C_d;
    return run_jobs(&proto, nrows, nthreads);
}
