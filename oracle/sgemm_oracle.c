/*
 * CPU oracle for single-precision GEMM.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg load
 * this file's library.  The CUDA product path never calls it, and the two
 * share no code, header, table or helper: this file includes nothing but the
 * C standard library (and OpenMP for the parallel sweep over columns).
 *
 * What it computes is the plain definition of the operation, in double:
 *
 *     Cref[i,j] = alpha * sum_{p=0}^{k-1} opA[i,p] * opB[p,j]  +  beta * Cin[i,j]
 *     den [i,j] = sum_{p=0}^{k-1} |alpha * opA[i,p] * opB[p,j]|  +  |beta * Cin[i,j]|
 *
 * with column-major storage and leading dimensions:
 *     opA[i,p] = A[i + p*lda]  if transa is 'N'/'n',  else A[p + i*lda]
 *     opB[p,j] = B[p + j*ldb]  if transb is 'N'/'n',  else B[j + p*ldb]
 *
 * Sources for the definition:
 *   - "Optimizing SGEMM on NVIDIA Turing GPUs" (README): SGEMM on column-major
 *     matrices with A and B not transposed is the primary case.
 *   - "HPC - Lecture 13 - MatMat GPU", section "Kernel 1: Global Memory
 *     Access": the kernel starts its sum from the existing C entry and adds
 *     the dot product of row i of A with column j of B (C += A*B); the
 *     host wrapper matmatgpu1 addresses strided arrays through lda/ldb/ldc.
 *   - "V3. Vectorized and double buffer" (Explore-GPU-performance wiki),
 *     section 2: the kernel overwrites C with A*B (no accumulate).
 *   The BLAS form alpha*A*B + beta*C covers both readings: (1,1) for the
 *   lecture's kernels and (1,0) for the wiki's.
 *
 * Readings where the pages are silent:
 *   - beta == 0 means Cin is not read at all (a NaN in Cin does not
 *     propagate); alpha == 0 or k == 0 means A and B are not read.
 *   - Every product of two fp32 values is exact in double (24+24 bits < 53),
 *     so the only rounding is in the running sum, in increasing p.  The
 *     library is compiled with -ffp-contract=off so x86 and Arm hosts agree.
 *
 * Loop orders: oracle_sgemm_full / oracle_sgemm_entries take one dot product
 * per entry (the "ijk" order).  oracle_sgemm_ikj is the second brute-force
 * order the lecture lists among its CPU routines (matmatikj): rows outer,
 * the reduction index in the middle, columns inner.  It exists only so the
 * tests can check the first order against an independently indexed loop.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int is_notrans(char t) { return t == 'N' || t == 'n'; }

static int valid_trans(char t)
{
    return t == 'N' || t == 'n' || t == 'T' || t == 't' || t == 'C' || t == 'c';
}

/* Element (i,p) of op(A): A is m x k after the optional transpose. */
static double op_a(char transa, const float *A, int64_t lda, int64_t i, int64_t p)
{
    return is_notrans(transa) ? (double)A[i + p * lda] : (double)A[p + i * lda];
}

/* Element (p,j) of op(B): B is k x n after the optional transpose. */
static double op_b(char transb, const float *B, int64_t ldb, int64_t p, int64_t j)
{
    return is_notrans(transb) ? (double)B[p + j * ldb] : (double)B[j + p * ldb];
}

/* One output entry and its error denominator, straight from the definition. */
static void one_entry(char transa, char transb, int64_t k, float alpha,
                      const float *A, int64_t lda, const float *B, int64_t ldb,
                      float beta, const float *C, int64_t ldc, int64_t i, int64_t j,
                      double *cref, double *den)
{
    double a = (double)alpha, b = (double)beta;
    double sum = 0.0, abs_sum = 0.0;
    if (a != 0.0) {
        for (int64_t p = 0; p < k; ++p) {
            double prod = op_a(transa, A, lda, i, p) * op_b(transb, B, ldb, p, j);
            sum += prod;
            abs_sum += fabs(a * prod);
        }
    }
    double c_term = 0.0;
    if (b != 0.0)
        c_term = b * (double)C[i + j * ldc];
    *cref = a * sum + c_term;
    *den = abs_sum + fabs(c_term);
}

static int check_args(char transa, char transb, int64_t m, int64_t n, int64_t k)
{
    if (!valid_trans(transa) || !valid_trans(transb))
        return -1;
    if (m < 0 || n < 0 || k < 0)
        return -2;
    return 0;
}

/* Every entry of the m x n result; cref/den are column-major with ld = m. */
int oracle_sgemm_full(char transa, char transb, int64_t m, int64_t n, int64_t k,
                      float alpha, const float *A, int64_t lda, const float *B, int64_t ldb,
                      float beta, const float *C, int64_t ldc, double *cref, double *den,
                      int nthreads)
{
    int rc = check_args(transa, transb, m, n, k);
    if (rc)
        return rc;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t j = 0; j < n; ++j)
        for (int64_t i = 0; i < m; ++i)
            one_entry(transa, transb, k, alpha, A, lda, B, ldb, beta, C, ldc, i, j,
                      &cref[i + j * m], &den[i + j * m]);
    (void)nthreads;
    return 0;
}

/* Only the listed entries (ii[e], jj[e]); used for the configurations whose full
 * product is too large to evaluate on the CPU. */
int oracle_sgemm_entries(char transa, char transb, int64_t m, int64_t n, int64_t k,
                         float alpha, const float *A, int64_t lda, const float *B, int64_t ldb,
                         float beta, const float *C, int64_t ldc, int64_t count,
                         const int64_t *ii, const int64_t *jj, double *cref, double *den,
                         int nthreads)
{
    int rc = check_args(transa, transb, m, n, k);
    if (rc)
        return rc;
    for (int64_t e = 0; e < count; ++e)
        if (ii[e] < 0 || ii[e] >= m || jj[e] < 0 || jj[e] >= n)
            return -3;
#ifdef _OPENMP
    if (nthreads <= 0)
        nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 16) num_threads(nthreads)
#endif
    for (int64_t e = 0; e < count; ++e)
        one_entry(transa, transb, k, alpha, A, lda, B, ldb, beta, C, ldc, ii[e], jj[e],
                  &cref[e], &den[e]);
    (void)nthreads;
    return 0;
}

/* Second loop order (rows, then the reduction index, then columns), full result
 * only, single-threaded; cref is column-major with ld = m.  It accumulates the
 * scaled products into a zeroed result and adds the beta term at the end. */
int oracle_sgemm_ikj(char transa, char transb, int64_t m, int64_t n, int64_t k,
                     float alpha, const float *A, int64_t lda, const float *B, int64_t ldb,
                     float beta, const float *C, int64_t ldc, double *cref)
{
    int rc = check_args(transa, transb, m, n, k);
    if (rc)
        return rc;
    double a = (double)alpha, b = (double)beta;
    for (int64_t j = 0; j < n; ++j)
        for (int64_t i = 0; i < m; ++i)
            cref[i + j * m] = 0.0;
    if (a != 0.0) {
        for (int64_t i = 0; i < m; ++i)
            for (int64_t p = 0; p < k; ++p) {
                double aip = op_a(transa, A, lda, i, p);
                for (int64_t j = 0; j < n; ++j)
                    cref[i + j * m] += aip * op_b(transb, B, ldb, p, j);
            }
    }
    for (int64_t j = 0; j < n; ++j)
        for (int64_t i = 0; i < m; ++i) {
            double s = a * cref[i + j * m];
            if (b != 0.0)
                s += b * (double)C[i + j * ldc];
            cref[i + j * m] = s;
        }
    return 0;
}

/* Threads an OpenMP region would use by default (reported beside timings). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
