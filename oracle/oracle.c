/*
 * CPU oracle for the drafter's decode GEMM and reduce + residual + RMSNorm.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct
 * definition that the CUDA path is compared against. Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it; the library never does.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * Sources (the vLLM API pages for the DSpark drafter):
 *  - "drafter/linears" module text and DraftGemm docstring: out[M,N] = x[M,K] @
 *    weight[N,K]^T with BF16 operands, FP32 accumulation and one BF16 rounding,
 *    cuBLAS's arithmetic with the order of the additions left free. The oracle takes the plainest
 *    reading of that: the dot product in FP64 (every BF16 x BF16 product is exact
 *    in FP64), rounded once to BF16 with round-to-nearest-even.
 *  - "drafter/comm" module text, ArNorm docstring and ArNorm.kernel: the TP BF16
 *    partial rows are summed in FP32 in rank order 0..TP-1 starting from slot 0,
 *    rounded once to BF16; the residual is added in FP32 and rounded once to BF16
 *    (that is the new residual); RMSNorm of the new residual is
 *    x * rsqrt(sum(x^2) / 7168 + eps) * gamma, rounded once to BF16.
 *  - "cutedsl/common/twoshot" reduce: the same rank-order FP32 sum, one rounding.
 *
 * Every BF16 value crosses this interface as its 16-bit pattern (uint16_t).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fno-fast-math -shared -fPIC.
 * -ffp-contract=off keeps a*b+c as two roundings on every target (aarch64 GCC
 * would otherwise fuse them), so results are the same on x86_64 and Arm hosts.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- BF16 <-> binary64 ------------------------------------------------------ */

/* A BF16 pattern is the upper half of a binary32 pattern, so widening is exact. */
double oracle_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a binary64 value to the nearest BF16 value, ties to even (IEEE 754
 * roundTiesToEven onto the BF16 grid: 8 significant bits, binary32's exponent
 * range, subnormals down to 2^-133). Done in one step from the double, never via
 * binary32, so there is no double rounding.
 *
 * Method: find the spacing u of the BF16 grid around |v| (2^(e-7) for |v| in
 * [2^e, 2^(e+1)), fixed at 2^-133 below 2^-126), scale |v| by 1/u (exact: a power
 * of two), round that to an integer with ties to even, scale back (exact).
 * A result of 2^128 or more is beyond the largest finite BF16 and becomes Inf.
 * NaN becomes the quiet NaN 0x7FC0 with the input's sign.
 */
uint16_t oracle_bf16_from_f64(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(v);
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    int e2;
    (void)frexp(a, &e2);              /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;                   /* a in [2^e, 2^(e+1)) */
    if (e < -126)
        e = -126;                     /* subnormal BF16: fixed spacing 2^-133 */
    double u = ldexp(1.0, e - 7);
    double q = a / u;                 /* exact: division by a power of two */
    double r = floor(q);              /* q < 2^9, so q - r is exact */
    double d = q - r;
    if (d > 0.5 || (d == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    double res = r * u;               /* exact: at most 9 significant bits */
    if (res >= 0x1p128)
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)res;             /* exact: every BF16 value is a binary32 value */
    uint32_t bits;
    memcpy(&bits, &f, sizeof bits);
    return (uint16_t)(sign | (uint16_t)((bits >> 16) & 0x7FFFu));
}

/* Element-wise oracle_bf16_from_f64 over an array (the same rule, no shortcuts). */
void oracle_bf16_from_f64_array(const double *v, uint16_t *out, long n)
{
    for (long i = 0; i < n; ++i)
        out[i] = oracle_bf16_from_f64(v[i]);
}

static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ---- decode GEMM ------------------------------------------------------------ */

/*
 * out[m, n] = BF16( sum_k x[m, k] * W[n, k] ), the sum taken in binary64 in k order.
 * x is [M, K] row-major, W is [N, K] row-major (each weight row is one output
 * column), out is [M, N] row-major.
 *
 * cols == NULL: every n in 0..N-1. Otherwise only the n listed in cols[0..ncols)
 * are computed, and out is [M, ncols] (column j holds output column cols[j]):
 * this is how a full-size problem is checked on sampled outputs.
 * threads <= 0 leaves OpenMP's default; the loop over output columns is split
 * across threads, which does not change any single output's arithmetic.
 */
void oracle_decode_gemm(const uint16_t *x, const uint16_t *W, uint16_t *out,
                        int M, int N, int K, const int *cols, int ncols, int threads)
{
    int count = cols ? ncols : N;
#ifdef _OPENMP
    if (threads > 0)
        omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 4)
#endif
    for (int j = 0; j < count; ++j) {
        int n = cols ? cols[j] : j;
        const uint16_t *w = W + (size_t)n * (size_t)K;
        for (int m = 0; m < M; ++m) {
            const uint16_t *xr = x + (size_t)m * (size_t)K;
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += oracle_bf16_to_f64(xr[k]) * oracle_bf16_to_f64(w[k]);
            out[(size_t)m * (size_t)count + (size_t)j] = oracle_bf16_from_f64(acc);
        }
    }
}

/*
 * The unrounded binary64 sums behind oracle_decode_gemm, and beside each the sum
 * of the absolute values of its terms (sum_k |x[m,k] * W[n,k]|), for the output
 * columns in cols[0..ncols). Both are [M, ncols] row-major. The second array is
 * the scale an FP32 accumulation's rounding error is proportional to; the tests
 * use it to tell a cancelled (near-zero) output from a resolvable one.
 */
void oracle_decode_gemm_f64(const uint16_t *x, const uint16_t *W, double *sum,
                            double *abs_sum, int M, int N, int K, const int *cols,
                            int ncols, int threads)
{
    (void)N;
#ifdef _OPENMP
    if (threads > 0)
        omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 4)
#endif
    for (int j = 0; j < ncols; ++j) {
        const uint16_t *w = W + (size_t)cols[j] * (size_t)K;
        for (int m = 0; m < M; ++m) {
            const uint16_t *xr = x + (size_t)m * (size_t)K;
            double acc = 0.0, mag = 0.0;
            for (int k = 0; k < K; ++k) {
                double t = oracle_bf16_to_f64(xr[k]) * oracle_bf16_to_f64(w[k]);
                acc += t;
                mag += fabs(t);
            }
            sum[(size_t)m * (size_t)ncols + (size_t)j] = acc;
            abs_sum[(size_t)m * (size_t)ncols + (size_t)j] = mag;
        }
    }
}

/*
 * The lm_head logits of "drafter/linears", draft_logits: the vocab-shard GEMM,
 * then the slice to the first n_out (org_vocab_size) columns, then, if
 * soft_cap > 0, tanh(logits / soft_cap) * soft_cap, then logits * scale.
 * Reading: the three element-wise steps act on the exact binary64 dot product and
 * the result is rounded once to BF16 (the pages apply them to BF16 tensors one
 * PyTorch op at a time; a fused epilogue rounds once). tanh is libm's binary64
 * tanh, a library step. out is [M, n_out] row-major; W rows n_out.. are unused.
 */
void oracle_decode_gemm_logits(const uint16_t *x, const uint16_t *W, uint16_t *out, int M,
                               int N, int K, int n_out, double soft_cap, double scale,
                               int threads)
{
    (void)N;
#ifdef _OPENMP
    if (threads > 0)
        omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 4)
#endif
    for (int n = 0; n < n_out; ++n) {
        const uint16_t *w = W + (size_t)n * (size_t)K;
        for (int m = 0; m < M; ++m) {
            const uint16_t *xr = x + (size_t)m * (size_t)K;
            double acc = 0.0;
            for (int k = 0; k < K; ++k)
                acc += oracle_bf16_to_f64(xr[k]) * oracle_bf16_to_f64(w[k]);
            double v = acc;
            if (soft_cap > 0.0)
                v = tanh(v / soft_cap) * soft_cap;
            v = v * scale;
            out[(size_t)m * (size_t)n_out + (size_t)n] = oracle_bf16_from_f64(v);
        }
    }
}

/* ---- reduce + residual ------------------------------------------------------ */

/*
 * For every row m < M and column c < width:
 *   s = p[0][m][c];  s = s + p[r][m][c] for r = 1..TP-1   (binary32 adds, RNE)
 *   a = BF16(s)
 *   h = residual ? BF16(a + residual[m][c]) (one binary32 add) : a
 *   residual_out[m][c] = h
 * partials is [TP, M, width]; residual (may be NULL) and residual_out are
 * [M, width]. The sum starts from slot 0, not from 0.0f: an all-(-0) column
 * stays -0. Only additions appear, so contraction cannot change anything.
 */
void oracle_reduce_residual(const uint16_t *partials, int TP, const uint16_t *residual,
                            uint16_t *residual_out, int M, int width)
{
    size_t slot = (size_t)M * (size_t)width;
    for (int m = 0; m < M; ++m) {
        for (int c = 0; c < width; ++c) {
            size_t i = (size_t)m * (size_t)width + (size_t)c;
            float s = bf16_to_f32(partials[i]);
            for (int r = 1; r < TP; ++r) {
                volatile float t = s + bf16_to_f32(partials[(size_t)r * slot + i]);
                s = t;
            }
            uint16_t a = oracle_bf16_from_f64((double)s);
            uint16_t h = a;
            if (residual) {
                volatile float t = bf16_to_f32(a) + bf16_to_f32(residual[i]);
                h = oracle_bf16_from_f64((double)t);
            }
            residual_out[i] = h;
        }
    }
}

/* ---- RMSNorm ------------------------------------------------------------------ */

/*
 * out[m][c] = BF16( h[m][c] * rstd_m * gamma[c] ),
 * rstd_m = 1 / sqrt( sum_c h[m][c]^2 / width + eps ), all in binary64.
 * The pages fix the formula (sum of squares over the 7168 columns, divided by
 * 7168, plus eps, reciprocal square root, times the value, times gamma) and one
 * rounding at the end; the oracle evaluates it in binary64. eps arrives as the
 * binary32 the library receives and is widened exactly.
 * h is [M, width], gamma [width], out [M, width].
 */
void oracle_rmsnorm(const uint16_t *h, const uint16_t *gamma, uint16_t *out,
                    int M, int width, float eps)
{
    for (int m = 0; m < M; ++m) {
        const uint16_t *row = h + (size_t)m * (size_t)width;
        double ss = 0.0;
        for (int c = 0; c < width; ++c) {
            double v = oracle_bf16_to_f64(row[c]);
            ss += v * v;
        }
        double rstd = 1.0 / sqrt(ss / (double)width + (double)eps);
        for (int c = 0; c < width; ++c) {
            double v = oracle_bf16_to_f64(row[c]);
            double g = oracle_bf16_to_f64(gamma[c]);
            out[(size_t)m * (size_t)width + (size_t)c] = oracle_bf16_from_f64(v * rstd * g);
        }
    }
}

/*
 * Diagnostic only: the same RMSNorm with the binary32 steps the ArNorm kernel
 * lists, in the plainest order: sum of squares as a sequential fma chain in
 * column order, rstd = 1 / sqrtf(sum / width + eps), (v * rstd) * gamma in
 * binary32, then one BF16 rounding. Used to show that a binary32 evaluation sits
 * within one BF16 ulp of the binary64 oracle; never a parity reference itself.
 */
void oracle_rmsnorm_f32_steps(const uint16_t *h, const uint16_t *gamma, uint16_t *out,
                              int M, int width, float eps)
{
    for (int m = 0; m < M; ++m) {
        const uint16_t *row = h + (size_t)m * (size_t)width;
        float ss = 0.0f;
        for (int c = 0; c < width; ++c) {
            float v = bf16_to_f32(row[c]);
            ss = fmaf(v, v, ss);
        }
        volatile float mean = ss / (float)width;
        volatile float arg = mean + eps;
        float rstd = 1.0f / sqrtf(arg);
        for (int c = 0; c < width; ++c) {
            volatile float t = bf16_to_f32(row[c]) * rstd;
            volatile float y = t * bf16_to_f32(gamma[c]);
            out[(size_t)m * (size_t)width + (size_t)c] = oracle_bf16_from_f64((double)y);
        }
    }
}

/* ---- gather ------------------------------------------------------------------ */

/*
 * out[m][r * S + j] = shards[r][m][j]: every rank's [M, S] shard placed at
 * columns r*S .. r*S + S - 1 of the gathered [M, TP * S] rows ("drafter/comm",
 * Gather docstring and module text: rank r's shard starts at column r*S; gather_context
 * and gather_logits build [M, TP * S] from [M, S] shards). A byte move: the
 * values are copied unchanged (no sentinel cleaning -- the local slots have no
 * sentinel). shards is [TP, M, S], out is [M, TP * S].
 */
void oracle_gather_shards(const uint16_t *shards, int TP, int M, int S, uint16_t *out)
{
    for (int r = 0; r < TP; ++r)
        for (int m = 0; m < M; ++m)
            for (int j = 0; j < S; ++j)
                out[(size_t)m * (size_t)TP * (size_t)S + (size_t)r * (size_t)S + (size_t)j] =
                    shards[((size_t)r * (size_t)M + (size_t)m) * (size_t)S + (size_t)j];
}

/* Threads OpenMP would use for the GEMM loop (reported beside CPU timings). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
