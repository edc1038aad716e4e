// The host co-worker of the hybrid CPU + GPU column split: a blocked FP32 GEMM
// on the host cores with OpenMP.
//
// "HPC - Lecture 13 - MatMat GPU", section "the hybrid function matmatgpu3":
// the columns of C are divided between the GPU and the CPU in the ratio Q : 1 of
// their speeds, the kernel is launched (asynchronously), and the host cores
// compute their share with the lecture's blocked, multithreaded product
// (matmatthreadomp) while the GPU computes its own.  This file is that host
// share, written for this library: C is cut into MB x NB blocks, one OpenMP
// task each; a block's K is walked in chunks of KC, each chunk of op(A) and
// op(B) packed contiguously (so transposed operands cost nothing extra in the
// inner loop), and a 16 x 4 register micro-tile runs the FMAs.  The block's
// sums live in a small buffer between chunks, so every output is one FP32
// fused multiply-add chain in increasing p, whatever the blocking or the
// number of threads -- deterministic.
#include "host_sgemm.h"

#include <omp.h>

#include <algorithm>
#include <vector>

namespace pg {
namespace {

constexpr int MB = 128;  // rows of a C block (a multiple of the micro-tile's 16)
constexpr int NB = 32;   // columns of a C block (a multiple of 4)
constexpr int KC = 256;  // K per packed chunk
constexpr int MR = 16, NR = 4;

bool notrans(char t) { return t == 'N' || t == 'n'; }

// acc[j][i] (the block buffer, column j of NB, rows of MB) += sum over the
// chunk's kc values of ap[p][i] * bp[p][j], one FMA per (p, i, j) in increasing p.
inline void micro_tile(const float* __restrict__ ap, const float* __restrict__ bp, int kc,
                       float* __restrict__ ct) {
    float acc[NR][MR];
#pragma GCC unroll 4
    for (int j = 0; j < NR; ++j)
#pragma GCC unroll 16
        for (int i = 0; i < MR; ++i) acc[j][i] = ct[j * MB + i];
    for (int p = 0; p < kc; ++p) {
        const float* a = ap + p * MB;
        const float* b = bp + p * NB;
#pragma GCC unroll 4
        for (int j = 0; j < NR; ++j) {
            const float bj = b[j];
#pragma GCC unroll 16
            for (int i = 0; i < MR; ++i) acc[j][i] = __builtin_fmaf(a[i], bj, acc[j][i]);
        }
    }
#pragma GCC unroll 4
    for (int j = 0; j < NR; ++j)
#pragma GCC unroll 16
        for (int i = 0; i < MR; ++i) ct[j * MB + i] = acc[j][i];
}

}  // namespace

void host_sgemm(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha, const float* A,
                int64_t lda, const float* B, int64_t ldb, float beta, float* C, int64_t ldc, int threads) {
    if (m <= 0 || n <= 0) return;
    const bool product = k > 0 && alpha != 0.0f;
    const int64_t mb_count = (m + MB - 1) / MB, nb_count = (n + NB - 1) / NB;
    const int nthreads = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
    {
        std::vector<float> apack(static_cast<size_t>(KC) * MB), bpack(static_cast<size_t>(KC) * NB),
            ctile(static_cast<size_t>(NB) * MB);
#pragma omp for collapse(2) schedule(dynamic, 1)
        for (int64_t jb = 0; jb < nb_count; ++jb) {
            for (int64_t ib = 0; ib < mb_count; ++ib) {
                const int64_t i0 = ib * MB, j0 = jb * NB;
                const int mb = static_cast<int>(std::min<int64_t>(MB, m - i0));
                const int nb = static_cast<int>(std::min<int64_t>(NB, n - j0));
                std::fill(ctile.begin(), ctile.end(), 0.0f);
                for (int64_t p0 = 0; product && p0 < k; p0 += KC) {
                    const int kc = static_cast<int>(std::min<int64_t>(KC, k - p0));
                    // ap[p][i] = op(A)(i0 + i, p0 + p), rows past m zero
                    for (int p = 0; p < kc; ++p) {
                        float* dst = apack.data() + p * MB;
                        if (notrans(transa)) {
                            const float* src = A + (p0 + p) * lda + i0;
                            for (int i = 0; i < mb; ++i) dst[i] = src[i];
                        } else {
                            const float* src = A + i0 * lda + (p0 + p);
                            for (int i = 0; i < mb; ++i) dst[i] = src[i * lda];
                        }
                        for (int i = mb; i < MB; ++i) dst[i] = 0.0f;
                    }
                    // bp[p][j] = op(B)(p0 + p, j0 + j), columns past n zero
                    for (int p = 0; p < kc; ++p) {
                        float* dst = bpack.data() + p * NB;
                        if (notrans(transb)) {
                            const float* src = B + j0 * ldb + (p0 + p);
                            for (int j = 0; j < nb; ++j) dst[j] = src[j * ldb];
                        } else {
                            const float* src = B + (p0 + p) * ldb + j0;
                            for (int j = 0; j < nb; ++j) dst[j] = src[j];
                        }
                        for (int j = nb; j < NB; ++j) dst[j] = 0.0f;
                    }
                    for (int jr = 0; jr < nb; jr += NR)
                        for (int ir = 0; ir < mb; ir += MR)
                            micro_tile(apack.data() + ir, bpack.data() + jr, kc, ctile.data() + jr * MB + ir);
                }
                for (int j = 0; j < nb; ++j) {
                    float* c = C + (j0 + j) * ldc + i0;
                    const float* t = ctile.data() + j * MB;
                    for (int i = 0; i < mb; ++i) {
                        float o = alpha * t[i];
                        if (beta != 0.0f) o = __builtin_fmaf(beta, c[i], o);
                        c[i] = o;
                    }
                }
            }
        }
    }
}

}  // namespace pg
