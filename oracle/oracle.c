/*
 * oracle.c -- CPU oracle for the warp-specialized pipeline operators.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA path and never includes anything
 * from the package.
 *
 * What it computes (plain definitions, no blocking, no fusion):
 *
 *  - GEMM + bias + ReLU.  "pwwt.cn news/4436243", section 4.1 (the SGEMM
 *    test bench): inputs A[M,K] and B[K,N], output C[M,N] = A*B + bias,
 *    then ReLU.  Here C[m,n] = max(0, bias[n] + sum_k A[m,k] * B[k,n]),
 *    evaluated in IEEE binary64 over the exact values the GPU receives
 *    (fp32 inputs, or bf16 inputs widened exactly to fp32 by the caller).
 *    The k-sum runs in increasing k; the bias is added once to the finished
 *    sum; ReLU is applied last.
 *
 *  - Staged copy.  "Producer-Consumer Warp Specialization for TMA
 *    Operations", the double-buffered load/store example: the data that
 *    goes in through the staging buffers comes out unchanged, so the
 *    oracle is memcpy.
 *
 * All arrays are contiguous row-major, owned by the caller.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int oracle_has_openmp(void)
{
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}

/* Full product.  C is an M x N array of doubles.  Rows are independent, so
 * they are shared out over nthreads (<= 0 means the OpenMP default); each
 * row is the same sequential i-k-j loop regardless of the thread count. */
void oracle_gemm_bias_relu(const float *A, const float *B, const float *bias,
                           double *C, int64_t M, int64_t N, int64_t K,
                           int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    #pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t m = 0; m < M; ++m) {
        double *c = C + m * N;
        for (int64_t n = 0; n < N; ++n) c[n] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = (double)A[m * K + k];
            const float *b = B + k * N;
            for (int64_t n = 0; n < N; ++n) c[n] += a * (double)b[n];
        }
        for (int64_t n = 0; n < N; ++n) {
            const double v = c[n] + (double)bias[n];
            c[n] = v > 0.0 ? v : 0.0;
        }
    }
}

/* Selected output elements (m_idx[p], n_idx[p]) of the same product, for
 * checking large problems element by element.  Same summation order as the
 * full product above. */
void oracle_gemm_bias_relu_points(const float *A, const float *B,
                                  const float *bias, int64_t M, int64_t N,
                                  int64_t K, const int64_t *m_idx,
                                  const int64_t *n_idx, int64_t npts,
                                  double *out, int nthreads)
{
    (void)M;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    #pragma omp parallel for schedule(static) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (int64_t p = 0; p < npts; ++p) {
        const int64_t m = m_idx[p], n = n_idx[p];
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
            s += (double)A[m * K + k] * (double)B[k * N + n];
        const double v = s + (double)bias[n];
        out[p] = v > 0.0 ? v : 0.0;
    }
}

/* The staged copy's result: the bytes of src, unchanged. */
void oracle_copy(const void *src, void *dst, size_t bytes)
{
    memcpy(dst, src, bytes);
}

/* The same copy cut into nthreads contiguous pieces, one per thread; used
 * only to time the copy on all host cores. */
void oracle_copy_parallel(const void *src, void *dst, size_t bytes,
                          int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    const size_t piece = (bytes + (size_t)nthreads - 1) / (size_t)nthreads;
    #pragma omp parallel for schedule(static) num_threads(nthreads)
    for (int t = 0; t < nthreads; ++t) {
        const size_t lo = (size_t)t * piece;
        if (lo < bytes) {
            const size_t len = (bytes - lo < piece) ? bytes - lo : piece;
            memcpy((char *)dst + lo, (const char *)src + lo, len);
        }
    }
#else
    (void)nthreads;
    memcpy(dst, src, bytes);
#endif
}
