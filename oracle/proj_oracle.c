/*
 * Oracle for the dense projection: test infrastructure only.
 *
 * Only tests, the smoke check and the benchmark's CPU-baseline leg may load
 * this library.  It shares no code with the CUDA path.
 *
 * What it computes (muse_bf16_proj guide, ch. 1, §1.1 "What is computed"):
 *     ref[i, n] = sum over k of x[i, k] * W[n, k]          (out = x @ W.T)
 * for x in bf16 [m, K] and W in bf16 [N, K] (router: W in float32).
 *
 * Precision (guide ch. 1, §1.5 "What counts as correct": the judge compares
 * against an FP64 reference): every operand is widened exactly to double,
 * each product is exact in double (bf16 x bf16 has 16 significant bits,
 * bf16 x fp32 has 32), and the sum runs in double in ascending k.  The only
 * rounding is that of the running double sum.
 *
 * Rows computed: the caller passes n_rows <= N; rows n < n_rows of W are used
 * (the unpooler computes only its first 1024 rows at <= 8 tokens, guide
 * ch. 1, §1.1).  Output ref is double [m, n_rows], row-major.
 *
 * Parallelism: OpenMP over (i, n) pairs when built with -fopenmp.  Each
 * output is still one sequential ascending-k sum, so the result does not
 * depend on the thread count.
 */
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> double, exact: bf16 is the high half of a float32. */
static double bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_threads(void)
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

/* x: bf16 bits [m, K]; W: bf16 bits [N, K] (only the first n_rows rows read). */
void oracle_proj_bf16(const uint16_t *x, const uint16_t *W, int64_t m,
                      int64_t n_rows, int64_t K, double *ref)
{
    int64_t total = m * n_rows;
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < total; ++t) {
        int64_t i = t / n_rows, n = t % n_rows, k;
        const uint16_t *xi = x + i * K;
        const uint16_t *wn = W + n * K;
        double acc = 0.0;
        for (k = 0; k < K; ++k)
            acc += bf16_to_double(xi[k]) * bf16_to_double(wn[k]);
        ref[t] = acc;
    }
}

/* Router form: x bf16 bits [m, K]; W float32 [N, K]. */
void oracle_proj_f32w(const uint16_t *x, const float *W, int64_t m,
                      int64_t n_rows, int64_t K, double *ref)
{
    int64_t total = m * n_rows;
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < total; ++t) {
        int64_t i = t / n_rows, n = t % n_rows, k;
        const uint16_t *xi = x + i * K;
        const float *wn = W + n * K;
        double acc = 0.0;
        for (k = 0; k < K; ++k)
            acc += bf16_to_double(xi[k]) * (double)wn[k];
        ref[t] = acc;
    }
}

/*
 * Selected outputs only (for full-size parity checks): for each j < count,
 * ref[j] = dot(x[rows_i[j]], W[rows_n[j]]), same definition as above.
 * w_is_f32 selects the router form.
 */
void oracle_proj_entries(const uint16_t *x, const void *W, int w_is_f32,
                         int64_t K, const int64_t *rows_i,
                         const int64_t *rows_n, int64_t count, double *ref)
{
    int64_t j;
#pragma omp parallel for schedule(static)
    for (j = 0; j < count; ++j) {
        const uint16_t *xi = x + rows_i[j] * K;
        double acc = 0.0;
        int64_t k;
        if (w_is_f32) {
            const float *wn = (const float *)W + rows_n[j] * K;
            for (k = 0; k < K; ++k)
                acc += bf16_to_double(xi[k]) * (double)wn[k];
        } else {
            const uint16_t *wn = (const uint16_t *)W + rows_n[j] * K;
            for (k = 0; k < K; ++k)
                acc += bf16_to_double(xi[k]) * bf16_to_double(wn[k]);
        }
        ref[j] = acc;
    }
}
