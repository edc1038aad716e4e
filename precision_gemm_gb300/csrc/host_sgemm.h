// The host co-worker of the hybrid CPU + GPU column split (plain C++, no CUDA).
#pragma once

#include <cstdint>

namespace pg {

// C = alpha * op(A) * op(B) + beta * C on host arrays, column-major with
// leading dimensions, op(X) = X for 'N'/'n', X^T for 'T'/'t'/'C'/'c'; every
// output is one FP32 fused multiply-add chain over p = 0 .. k-1 in increasing
// order, then alpha and beta (C is not read when beta == 0; A and B are not
// read when k == 0 or alpha == 0).  Runs on the host cores with OpenMP,
// `threads` of them (0: OpenMP's default); deterministic whatever the thread
// count.  Arguments are assumed valid (the C ABI checks them first).
void host_sgemm(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha, const float* A,
                int64_t lda, const float* B, int64_t ldb, float beta, float* C, int64_t ldc, int threads);

}  // namespace pg
