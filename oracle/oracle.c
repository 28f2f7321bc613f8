/*
 * oracle.c -- plain CPU definition of what the streamed tiled linear operator
 * computes.  TEST INFRASTRUCTURE ONLY: it is called by the test-suite, by the
 * smoke check and by the benchmark's CPU-baseline leg, never by the library.
 * It shares no code, header or helper with the CUDA path.
 *
 * What is computed (the definition, written out):
 *   The operator is Y = X.W with X [T,K] and W [K,M]
 *   (pwwt.cn/news/5430303, "关键技术一: Memory-centric tiling", 核心思想).
 *   Splitting W along its output dimension into tiles W_1..W_N and computing
 *   Y_i = X.W_i gives column blocks of the same Y, with no cross-tile term
 *   (same section, and aicassindra tm_zero_infinity, "Memory-centric tiling:
 *   operators bigger than the device").  Tiling therefore changes only the
 *   schedule, and the oracle is the untiled product.
 *   The backward pass costs twice the forward FLOPs (tm_zero_infinity, "The
 *   FLOPs-per-byte test every tier must pass": forward 2P, backward 4P per
 *   token).  The pages do not write the two backward products out; they are
 *   the standard gradients of a linear map for a loss L with dY = dL/dY:
 *       dX[t,k] = sum_m dY[t,m] * W[k,m]
 *       dW[k,m] = sum_t X[t,k]  * dY[t,m]
 *
 * Precision: inputs are bf16 bit patterns (uint16), widened exactly to fp32.
 * Each output element is a single fp32 accumulator that starts at +0.0f and
 * adds the products in ascending order of the summation index.  A product of
 * two bf16 values has at most 16 significant bits, so it is exact in fp32;
 * only the additions round.  Outputs stay fp32 and are not rounded to bf16.
 * Build with -ffp-contract=off so that the result is identical on every host.
 *
 * Chains of operators (Y_l = X_l.W_l, X_{l+1} = Y_l; with two operators, the
 * FFN's two matrices, tm_zero_infinity, "Memory-centric tiling: operators
 * bigger than the device") pass activations and gradients between the
 * operators in bf16: X_{l+1} = bf16(Y_l) and, in the backward, the dY of
 * operator l is bf16(dX of operator l+1).  oracle_round_bf16 is that
 * rounding, round to nearest with ties to even; the chain itself is composed
 * from the single-operator functions in oracle.py.
 *
 * Layouts: row-major.  X [T,K] (ld K), W [K,M] (ld M), dY [T,M] (ld M),
 * Y [T,M], dX [T,K], dW [K,M].  The sampled functions also read W stored
 * tile by tile: M/C column blocks of C columns, block j held as its own
 * row-major [K][C] array, blocks one after another.  C = M is the plain
 * row-major layout.
 */
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static float bf16_to_f32(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Y[t,m] = sum_{k=0..K-1} X[t,k] * W[k,m].  The loop over m is innermost so
 * that W is read row by row; each Y[t,m] still receives its K products in
 * ascending k, one fp32 add each. */
void oracle_forward(int64_t T, int64_t K, int64_t M,
                    const uint16_t *X, const uint16_t *W, float *Y)
{
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; ++t) {
        float *yrow = Y + t * M;
        for (int64_t m = 0; m < M; ++m) yrow[m] = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float x = bf16_to_f32(X[t * K + k]);
            const uint16_t *wrow = W + k * M;
            for (int64_t m = 0; m < M; ++m)
                yrow[m] = yrow[m] + x * bf16_to_f32(wrow[m]);
        }
    }
}

/* dX[t,k] = sum_{m=0..M-1} dY[t,m] * W[k,m]: a dot product of row t of dY
 * with row k of W, summed in ascending m. */
void oracle_backward_dx(int64_t T, int64_t K, int64_t M,
                        const uint16_t *dY, const uint16_t *W, float *dX)
{
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; ++t) {
        const uint16_t *dyrow = dY + t * M;
        for (int64_t k = 0; k < K; ++k) {
            const uint16_t *wrow = W + k * M;
            float acc = 0.0f;
            for (int64_t m = 0; m < M; ++m)
                acc = acc + bf16_to_f32(dyrow[m]) * bf16_to_f32(wrow[m]);
            dX[t * K + k] = acc;
        }
    }
}

/* dW[k,m] = sum_{t=0..T-1} X[t,k] * dY[t,m].  The loop over m is innermost;
 * each dW[k,m] receives its T products in ascending t. */
void oracle_backward_dw(int64_t T, int64_t K, int64_t M,
                        const uint16_t *X, const uint16_t *dY, float *dW)
{
    int64_t k;
#pragma omp parallel for schedule(static)
    for (k = 0; k < K; ++k) {
        float *dwrow = dW + k * M;
        for (int64_t m = 0; m < M; ++m) dwrow[m] = 0.0f;
        for (int64_t t = 0; t < T; ++t) {
            float x = bf16_to_f32(X[t * K + k]);
            const uint16_t *dyrow = dY + t * M;
            for (int64_t m = 0; m < M; ++m)
                dwrow[m] = dwrow[m] + x * bf16_to_f32(dyrow[m]);
        }
    }
}

/* Element W[k,m] of a [K,M] matrix stored as M/C column blocks of C columns,
 * each block row-major [K][C] (C = M: plain row-major). */
static uint16_t w_at(const uint16_t *W, int64_t K, int64_t C, int64_t k, int64_t m)
{
    int64_t blk = m / C, col = m - blk * C;
    return W[blk * K * C + k * C + col];
}

/* The same three definitions, evaluated only at n chosen entries (row[i],
 * col[i]).  Each entry is summed in the same ascending order as above, so a
 * sampled value equals the full-tensor value bit for bit.  wcols is the
 * block width C of W's storage (see w_at). */
void oracle_sample_y(int64_t T, int64_t K, int64_t M, int64_t wcols,
                     const uint16_t *X, const uint16_t *W, int64_t n,
                     const int64_t *row, const int64_t *col, float *out)
{
    int64_t i;
    (void)T; (void)M;
#pragma omp parallel for schedule(dynamic, 16)
    for (i = 0; i < n; ++i) {
        int64_t t = row[i], m = col[i];
        float acc = 0.0f;
        for (int64_t k = 0; k < K; ++k)
            acc = acc + bf16_to_f32(X[t * K + k]) * bf16_to_f32(w_at(W, K, wcols, k, m));
        out[i] = acc;
    }
}

void oracle_sample_dx(int64_t T, int64_t K, int64_t M, int64_t wcols,
                      const uint16_t *dY, const uint16_t *W, int64_t n,
                      const int64_t *row, const int64_t *col, float *out)
{
    int64_t i;
    (void)T;
#pragma omp parallel for schedule(dynamic, 16)
    for (i = 0; i < n; ++i) {
        int64_t t = row[i], k = col[i];
        float acc = 0.0f;
        for (int64_t m = 0; m < M; ++m)
            acc = acc + bf16_to_f32(dY[t * M + m]) * bf16_to_f32(w_at(W, K, wcols, k, m));
        out[i] = acc;
    }
}

void oracle_sample_dw(int64_t T, int64_t K, int64_t M,
                      const uint16_t *X, const uint16_t *dY, int64_t n,
                      const int64_t *row, const int64_t *col, float *out)
{
    int64_t i;
#pragma omp parallel for schedule(dynamic, 16)
    for (i = 0; i < n; ++i) {
        int64_t k = row[i], m = col[i];
        float acc = 0.0f;
        for (int64_t t = 0; t < T; ++t)
            acc = acc + bf16_to_f32(X[t * K + k]) * bf16_to_f32(dY[t * M + m]);
        out[i] = acc;
    }
}

/* bf16 keeps the sign, the 8 exponent bits and the top 7 fraction bits of an
 * fp32 value.  Rounding to nearest, ties to even, on the bit pattern u: the
 * dropped low 16 bits are compared with half (0x8000); adding 0x7FFF plus the
 * lowest kept bit carries into the kept bits exactly when they exceed half,
 * or equal it with an odd kept part.  A carry out of the fraction bumps the
 * exponent, which is the correct next value (up to infinity).  NaN is kept
 * NaN (quiet bit set) instead of being rounded. */
static uint16_t f32_to_bf16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* out[i] = bf16 bits of in[i] rounded to nearest even, i < n. */
void oracle_round_bf16(int64_t n, const float *in, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}
