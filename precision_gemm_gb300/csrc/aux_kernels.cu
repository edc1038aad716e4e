// Memory-bound helper kernels around the GEMM kernels:
//   * operand preparation: copy an operand into the layout the GEMM kernels
//     read through TMA (16-byte aligned base, leading dimension a multiple of 4,
//     A M-major and B K-major), transposing it when trans = 'T', and for 3xTF32
//     splitting every value into a TF32 "big" part and its exact remainder;
//   * the split-K reduction C = alpha * sum_s P[s] + beta * C, slices summed in
//     increasing s (deterministic);
//   * C = beta * C for calls with k == 0 or alpha == 0.
// All are bound by HBM bandwidth: grids are sized as a multiple of the SM count
// and every warp touches 128 contiguous bytes per access where the layout allows.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace pg {
namespace {

// x = big + small with big holding x's leading 11 significant bits (the TF32
// format: 8-bit exponent, 10 stored mantissa bits), rounded to nearest with
// ties away from zero by adding half a TF32 unit to the magnitude bits before
// clearing the low 13 bits.  small = x - big is exact in FP32 (|small| is at
// most half a TF32 unit of x).  Non-finite inputs pass through as big with a
// zero remainder; a finite value whose rounding would overflow is truncated.
__device__ __forceinline__ void split_tf32(float x, float& big, float& small) {
    const uint32_t u = __float_as_uint(x);
    if (!isfinite(x)) {
        big = x;
        small = 0.0f;
        return;
    }
    float b = __uint_as_float((u + 0x1000u) & 0xFFFFE000u);
    if (!isfinite(b)) b = __uint_as_float(u & 0xFFFFE000u);
    big = b;
    small = x - b;
}

// dst(r, c) = src(r, c), r < rows, c < cols; one warp row-stride per column.
template <bool SPLIT>
__global__ void __launch_bounds__(256) prep_copy_kernel(const float* __restrict__ src, int64_t lds,
                                                        int64_t rows, int64_t cols, float* __restrict__ dst,
                                                        float* __restrict__ dst_small, int64_t ldd) {
    for (int64_t c = blockIdx.y; c < cols; c += gridDim.y) {
        const float* s = src + c * lds;
        float* d = dst + c * ldd;
        float* ds = SPLIT ? dst_small + c * ldd : nullptr;
        for (int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; r < rows;
             r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            const float x = s[r];
            if (SPLIT) {
                float b, sm;
                split_tf32(x, b, sm);
                d[r] = b;
                ds[r] = sm;
            } else {
                d[r] = x;
            }
        }
    }
}

// dst(r, c) = src(c, r): 32 x 32 tiles through shared memory so that both the
// read (along c) and the write (along r) are coalesced.
template <bool SPLIT>
__global__ void __launch_bounds__(256) prep_transpose_kernel(const float* __restrict__ src, int64_t lds,
                                                             int64_t rows, int64_t cols,
                                                             float* __restrict__ dst,
                                                             float* __restrict__ dst_small, int64_t ldd) {
    __shared__ float tile[32][33];
    const int64_t tiles_r = (rows + 31) / 32;
    const int64_t tiles_c = (cols + 31) / 32;
    for (int64_t t = blockIdx.x; t < tiles_r * tiles_c; t += gridDim.x) {
        const int64_t r0 = (t % tiles_r) * 32;
        const int64_t c0 = (t / tiles_r) * 32;
        // src(c, r) lives at src[c + r * lds]: contiguous along c.
        for (int y = threadIdx.y; y < 32; y += blockDim.y) {
            const int64_t r = r0 + y, c = c0 + threadIdx.x;
            if (r < rows && c < cols) tile[y][threadIdx.x] = src[c + r * lds];
        }
        __syncthreads();
        for (int y = threadIdx.y; y < 32; y += blockDim.y) {
            const int64_t c = c0 + y, r = r0 + threadIdx.x;
            if (r < rows && c < cols) {
                const float x = tile[threadIdx.x][y];
                if (SPLIT) {
                    float b, sm;
                    split_tf32(x, b, sm);
                    dst[r + c * ldd] = b;
                    dst_small[r + c * ldd] = sm;
                } else {
                    dst[r + c * ldd] = x;
                }
            }
        }
        __syncthreads();
    }
}

// C = alpha * sum_{s < split} P[s] + beta * C over the m x n output.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const GemmParams p) {
    for (int64_t j = blockIdx.y; j < p.n; j += gridDim.y) {
        const float* pj = p.P + j * p.ldp;
        float* cj = p.C + j * p.ldc;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < p.m;
             i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
            float acc = 0.0f;
            for (int s = 0; s < p.split; ++s) acc += pj[s * p.p_stride + i];
            float o = p.alpha * acc;
            if (p.beta != 0.0f) o = fmaf(p.beta, cj[i], o);
            cj[i] = o;
        }
    }
}

__global__ void __launch_bounds__(256) scale_kernel(float* __restrict__ C, int64_t ldc, int64_t m, int64_t n,
                                                    float beta) {
    for (int64_t j = blockIdx.y; j < n; j += gridDim.y) {
        float* cj = C + j * ldc;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < m;
             i += static_cast<int64_t>(gridDim.x) * blockDim.x)
            cj[i] = (beta == 0.0f) ? 0.0f : beta * cj[i];
    }
}

// Column-sweep grid: x covers rows (256 threads each), y covers columns; the
// total is a multiple of the SM count, capped so each CTA loops a few times.
dim3 column_grid(int64_t rows, int64_t cols, int num_sms) {
    const int64_t bx = (rows + 255) / 256;
    const int64_t bx_c = bx < 8 ? bx : 8;
    int64_t by = (static_cast<int64_t>(num_sms) * 8 + bx_c - 1) / bx_c;
    if (by > cols) by = cols;
    if (by > 65535) by = 65535;
    if (by < 1) by = 1;
    return dim3(static_cast<unsigned>(bx_c < 1 ? 1 : bx_c), static_cast<unsigned>(by));
}

}  // namespace

cudaError_t launch_prep(const float* src, int64_t lds, bool transposed, int64_t rows, int64_t cols, float* dst,
                        float* dst_small, int64_t ldd, int num_sms, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    if (transposed) {
        const int64_t tiles = ((rows + 31) / 32) * ((cols + 31) / 32);
        int64_t g = static_cast<int64_t>(num_sms) * 8;
        if (g > tiles) g = tiles;
        const dim3 block(32, 8);
        if (dst_small)
            prep_transpose_kernel<true><<<static_cast<unsigned>(g), block, 0, stream>>>(src, lds, rows, cols, dst,
                                                                                        dst_small, ldd);
        else
            prep_transpose_kernel<false><<<static_cast<unsigned>(g), block, 0, stream>>>(src, lds, rows, cols,
                                                                                         dst, nullptr, ldd);
    } else {
        const dim3 grid = column_grid(rows, cols, num_sms);
        if (dst_small)
            prep_copy_kernel<true><<<grid, 256, 0, stream>>>(src, lds, rows, cols, dst, dst_small, ldd);
        else
            prep_copy_kernel<false><<<grid, 256, 0, stream>>>(src, lds, rows, cols, dst, nullptr, ldd);
    }
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const GemmParams& p, int num_sms, cudaStream_t stream) {
    splitk_reduce_kernel<<<column_grid(p.m, p.n, num_sms), 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_scale(float* C, int64_t ldc, int64_t m, int64_t n, float beta, int num_sms,
                         cudaStream_t stream) {
    scale_kernel<<<column_grid(m, n, num_sms), 256, 0, stream>>>(C, ldc, m, n, beta);
    return cudaGetLastError();
}

}  // namespace pg
