// Memory-bound helper kernels around the GEMM kernels:
//   * operand preparation: copy an operand into the layout the GEMM kernels
//     read through TMA (16-byte aligned base, leading dimension a multiple of 4,
//     A M-major and B K-major), transposing it when trans = 'T', and for 3xTF32
//     splitting every value into a TF32 "big" part and its exact remainder;
//   * the split-K reduction C = alpha * sum_s P[s] + beta * C, slices summed in
//     a fixed order (increasing s; with many slices, four contiguous groups in
//     increasing s, then the groups in order) -- deterministic;
//   * C = beta * C for calls with k == 0 or alpha == 0.
// All are bound by HBM bandwidth: grids are sized as a multiple of the SM count
// and every warp touches 128 contiguous bytes per access where the layout allows.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"  // split_tf32

namespace pg {
namespace {

// Column sweep over a column-major rows x cols matrix: a CTA of 256 threads
// covers TX = 2^tx_shift consecutive rows (32 <= TX <= 256, the smallest power of
// two >= rows) of 256 / TX columns, so a narrow matrix keeps every lane busy and
// every warp still touches 128 contiguous bytes.  A thread issues kU loads before
// any store -- kU of its columns, or, when it owns fewer than kU columns, kU of
// its rows (by_rows) -- because a thread whose loads wait on its own earlier
// stores keeps a single load in flight.
constexpr int kU = 8;

struct Sweep {
    int tx, ty;        // this thread's row / column offset inside the CTA's block
    int TX, TY;        // rows and columns one CTA covers per step
    int64_t rstep;     // row distance between a thread's consecutive rows
    int64_t cstep;     // column distance between a thread's consecutive columns
};

__device__ __forceinline__ Sweep sweep_setup(int tx_shift) {
    Sweep w;
    w.TX = 1 << tx_shift;
    w.TY = 256 >> tx_shift;
    w.tx = threadIdx.x & (w.TX - 1);
    w.ty = threadIdx.x >> tx_shift;
    w.rstep = static_cast<int64_t>(gridDim.x) * w.TX;
    w.cstep = static_cast<int64_t>(gridDim.y) * w.TY;
    return w;
}

// Visit every (r, c) of the sweep in batches of up to kU positions of one thread:
// f_load(batch index, r, c) for the whole batch, then f_store(batch index, r, c).
template <class Load, class Store>
__device__ __forceinline__ void sweep_batches(const Sweep& w, int64_t rows, int64_t cols, bool by_rows,
                                              Load&& f_load, Store&& f_store) {
    const int64_t r_first = static_cast<int64_t>(blockIdx.x) * w.TX + w.tx;
    const int64_t c_first = static_cast<int64_t>(blockIdx.y) * w.TY + w.ty;
    if (by_rows) {
        for (int64_t c = c_first; c < cols; c += w.cstep) {
            for (int64_t r0 = r_first; r0 < rows; r0 += kU * w.rstep) {
                const int64_t left = (rows - r0 + w.rstep - 1) / w.rstep;
                const int nu = left < kU ? static_cast<int>(left) : kU;
#pragma unroll
                for (int u = 0; u < kU; ++u)
                    if (u < nu) f_load(u, r0 + u * w.rstep, c);
#pragma unroll
                for (int u = 0; u < kU; ++u)
                    if (u < nu) f_store(u, r0 + u * w.rstep, c);
            }
        }
    } else {
        for (int64_t r = r_first; r < rows; r += w.rstep) {
            for (int64_t c0 = c_first; c0 < cols; c0 += kU * w.cstep) {
                const int64_t left = (cols - c0 + w.cstep - 1) / w.cstep;
                const int nu = left < kU ? static_cast<int>(left) : kU;
#pragma unroll
                for (int u = 0; u < kU; ++u)
                    if (u < nu) f_load(u, r, c0 + u * w.cstep);
#pragma unroll
                for (int u = 0; u < kU; ++u)
                    if (u < nu) f_store(u, r, c0 + u * w.cstep);
            }
        }
    }
}

// dst(r, c) = src(r, c), r < rows, c < cols (and the TF32 split when SPLIT).
template <bool SPLIT>
__global__ void __launch_bounds__(256, SPLIT ? 3 : 4)
    prep_copy_kernel(const float* __restrict__ src, int64_t lds, int64_t rows, int64_t cols,
                     float* __restrict__ dst, float* __restrict__ dst_small, int64_t ldd, int tx_shift,
                     int by_rows, int wait_last) {
    // Launched after the other operand's pass (independent data): with wait_last
    // the two passes overlap and this one waits for the other only before it
    // retires, so that the GEMM, which waits for this pass, also finds the other
    // one complete.
    if (!wait_last) pdl_wait();
    if (threadIdx.x == 0) pdl_trigger();  // the GEMM may be scheduled; it waits for this pass
    const Sweep w = sweep_setup(tx_shift);
    float x[kU];
    sweep_batches(
        w, rows, cols, by_rows != 0, [&](int u, int64_t r, int64_t c) { x[u] = src[c * lds + r]; },
        [&](int u, int64_t r, int64_t c) {
            if (SPLIT) {
                float b, sm;
                split_tf32(x[u], b, sm);
                dst[c * ldd + r] = b;
                dst_small[c * ldd + r] = sm;
            } else {
                dst[c * ldd + r] = x[u];
            }
        });
    if (wait_last) pdl_wait();
}

// prep_copy_kernel for a 16-byte aligned src with lds % 4 == 0 (dst is 256-byte
// aligned with ldd = round_up(rows, 4)): a thread moves 4 consecutive rows of one
// column as one float4, kU chunks loaded before any is stored, so that small
// operands (a few MB, where the scalar sweep is bound by DRAM latency) move with
// many loads in flight.  A column's last chunk, when rows % 4 != 0, is read and
// written element by element.
template <bool SPLIT>
__global__ void __launch_bounds__(256) prep_copy_vec_kernel(const float* __restrict__ src, int64_t lds, int64_t rows,
                                                            int64_t cols, float* __restrict__ dst,
                                                            float* __restrict__ dst_small, int64_t ldd,
                                                            int wait_last) {
    if (!wait_last) pdl_wait();  // as in prep_copy_kernel
    if (threadIdx.x == 0) pdl_trigger();
    const int64_t rq = (rows + 3) / 4;  // chunks per column
    const int64_t total = rq * cols;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t0 < total; t0 += kU * stride) {
        float4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t t = t0 + u * stride;
            if (t < total) {
                const int64_t c = t / rq, r = (t - c * rq) * 4;
                const float* s = src + c * lds + r;
                if (r + 4 <= rows) {
                    v[u] = *reinterpret_cast<const float4*>(s);
                } else {
                    v[u] = make_float4(s[0], r + 1 < rows ? s[1] : 0.0f, r + 2 < rows ? s[2] : 0.0f, 0.0f);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int64_t t = t0 + u * stride;
            if (t < total) {
                const int64_t c = t / rq, r = (t - c * rq) * 4;
                const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                float b[4], sm[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (SPLIT) {
                        split_tf32(x[e], b[e], sm[e]);
                    } else {
                        b[e] = x[e];
                    }
                }
                float* d = dst + c * ldd + r;
                float* ds = SPLIT ? dst_small + c * ldd + r : nullptr;
                if (r + 4 <= rows) {
                    *reinterpret_cast<float4*>(d) = make_float4(b[0], b[1], b[2], b[3]);
                    if (SPLIT) *reinterpret_cast<float4*>(ds) = make_float4(sm[0], sm[1], sm[2], sm[3]);
                } else {
                    for (int e = 0; e < 4 && r + e < rows; ++e) {
                        d[e] = b[e];
                        if (SPLIT) ds[e] = sm[e];
                    }
                }
            }
        }
    }
    if (wait_last) pdl_wait();
}

// dst(r, c) = src(c, r): 32 x 32 tiles through shared memory so that both the
// read (along c) and the write (along r) are coalesced.
template <bool SPLIT>
__global__ void __launch_bounds__(256) prep_transpose_kernel(const float* __restrict__ src, int64_t lds,
                                                             int64_t rows, int64_t cols,
                                                             float* __restrict__ dst,
                                                             float* __restrict__ dst_small, int64_t ldd,
                                                             int wait_last) {
    __shared__ float tile[32][33];
    if (!wait_last) pdl_wait();  // as in prep_copy_kernel
    if (threadIdx.x == 0 && threadIdx.y == 0) pdl_trigger();
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
    if (wait_last) pdl_wait();
}

// Loads of the split-K reductions run up to kS slices ahead of the additions.
constexpr int kS = 8;

// C = alpha * sum_{s < split} P[s] + beta * C over the m x n output, every output
// summing its slices in increasing s.  A thread takes 4 consecutive rows of one
// column.  The slices' float4s of P (16-byte aligned: ldp % 4 == 0 and P starts
// on 256 bytes) are loaded before the first addition -- up to kS per batch -- so
// that even a thread with one output keeps several loads in flight.  C is read
// and written as a float4 when it is 16-byte aligned with ldc % 4 == 0 and the
// chunk is whole, else element by element.  Rows from m up to ldp of P are
// loaded with the chunk but never stored.
__global__ void __launch_bounds__(256) splitk_reduce_vec_kernel(const GemmParams p) {
    pdl_wait();  // the GEMM's partial sums
    const int64_t rq = (p.m + 3) / 4;
    const int64_t total = rq * p.n;
    const int64_t st4 = p.p_stride / 4;
    for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t c = t / rq, r = (t - c * rq) * 4;
        const float4* ps = reinterpret_cast<const float4*>(p.P + c * p.ldp + r);
        float* dst = p.C + c * p.ldc + r;
        const bool whole = r + 4 <= p.m;
        const bool vec = whole && p.c_vec;
        float4 cin = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (p.beta != 0.0f) {
            if (vec) {
                cin = *reinterpret_cast<const float4*>(dst);
            } else {
                cin.x = dst[0];
                if (r + 1 < p.m) cin.y = dst[1];
                if (r + 2 < p.m) cin.z = dst[2];
                if (r + 3 < p.m) cin.w = dst[3];
            }
        }
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int s = 0; s < p.split; s += kS) {
            float4 v[kS];
#pragma unroll
            for (int j = 0; j < kS; ++j)
                if (s + j < p.split) v[j] = ps[(s + j) * st4];
#pragma unroll
            for (int j = 0; j < kS; ++j) {
                if (s + j < p.split) {
                    acc.x += v[j].x;
                    acc.y += v[j].y;
                    acc.z += v[j].z;
                    acc.w += v[j].w;
                }
            }
        }
        float o[4] = {p.alpha * acc.x, p.alpha * acc.y, p.alpha * acc.z, p.alpha * acc.w};
        if (p.beta != 0.0f) {
            o[0] = fmaf(p.beta, cin.x, o[0]);
            o[1] = fmaf(p.beta, cin.y, o[1]);
            o[2] = fmaf(p.beta, cin.z, o[2]);
            o[3] = fmaf(p.beta, cin.w, o[3]);
        }
        if (vec) {
            *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
            for (int e = 0; e < 4 && r + e < p.m; ++e) dst[e] = o[e];
        }
    }
}

// The same reduction when there are many slices and few outputs (a 128 x 128
// result split 152 or 304 ways): a thread summing all S slices of its outputs
// would wait out S/kS DRAM latencies in turn, so kG threads share each group of
// four rows.  A CTA covers 64 rows of one column as 16 float4 quads x kG groups:
// thread (g, q) sums the contiguous slices [g*S/kG, (g+1)*S/kG) of quad q in
// increasing order (kS float4 loads in flight), and the kG partial sums are then
// added in increasing g -- a fixed association, so the result does not depend
// on scheduling.  P is 16-byte aligned with ldp % 4 == 0, so every quad that
// starts below m can be loaded whole.  Dependent-launched (the earlier form,
// four groups of scalar rows, ran longer and lost 3 % that way; this one gains:
// 128 x 128 x 262144 FFMA 0.160 -> 0.156 ms, 256 x 256 x 65536 TF32 0.049 ->
// 0.046, against the earlier form launched the ordinary way).
constexpr int kG = 16;

__global__ void __launch_bounds__(256) splitk_reduce_grouped_kernel(const GemmParams p) {
    __shared__ float4 part[kG][16];
    pdl_wait();  // the GEMM's partial sums
    const int q = threadIdx.x & 15;
    const int g = threadIdx.x >> 4;
    const int s0 = (g * p.split) / kG, s1 = ((g + 1) * p.split) / kG;
    const int64_t st4 = p.p_stride / 4;
    for (int64_t c = blockIdx.y; c < p.n; c += gridDim.y) {
        for (int64_t r0 = static_cast<int64_t>(blockIdx.x) * 64; r0 < p.m; r0 += static_cast<int64_t>(gridDim.x) * 64) {
            const int64_t r = r0 + 4 * q;
            float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (r < p.m) {
                const float4* ps = reinterpret_cast<const float4*>(p.P + c * p.ldp + r);
                int s = s0;
                for (; s + kS <= s1; s += kS) {
                    float4 v[kS];
#pragma unroll
                    for (int u = 0; u < kS; ++u) v[u] = ps[(s + u) * st4];
#pragma unroll
                    for (int u = 0; u < kS; ++u) {
                        acc.x += v[u].x;
                        acc.y += v[u].y;
                        acc.z += v[u].z;
                        acc.w += v[u].w;
                    }
                }
                for (; s < s1; ++s) {
                    const float4 v = ps[s * st4];
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
            }
            part[g][q] = acc;
            __syncthreads();
            if (g == 0 && r < p.m) {
                float4 sum = part[0][q];
#pragma unroll
                for (int h = 1; h < kG; ++h) {
                    const float4 v = part[h][q];
                    sum.x += v.x;
                    sum.y += v.y;
                    sum.z += v.z;
                    sum.w += v.w;
                }
                float o[4] = {p.alpha * sum.x, p.alpha * sum.y, p.alpha * sum.z, p.alpha * sum.w};
                float* dst = p.C + c * p.ldc + r;
                const bool whole = r + 4 <= p.m;
                if (p.beta != 0.0f) {
                    if (whole && p.c_vec) {
                        const float4 cv = *reinterpret_cast<const float4*>(dst);
                        o[0] = fmaf(p.beta, cv.x, o[0]);
                        o[1] = fmaf(p.beta, cv.y, o[1]);
                        o[2] = fmaf(p.beta, cv.z, o[2]);
                        o[3] = fmaf(p.beta, cv.w, o[3]);
                    } else {
                        for (int e = 0; e < 4 && r + e < p.m; ++e) o[e] = fmaf(p.beta, dst[e], o[e]);
                    }
                }
                if (whole && p.c_vec) {
                    *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
                } else {
                    for (int e = 0; e < 4 && r + e < p.m; ++e) dst[e] = o[e];
                }
            }
            __syncthreads();
        }
    }
}

// Stream-K fix-up (the FFMA and the single-SM tensor-core stream-K kernels):
// C = alpha * sum_j P[t][j] + beta * C per 128 x BN tile t, the segments j of t
// added in increasing order -- increasing k, so deterministic.  A thread takes 4 consecutive rows of one column of a tile
// (one float4 of each partial block), all of its segments' loads issued before
// the additions; C is read and written as a float4 when it is 16-byte aligned
// with ldc % 4 == 0 and the 4 rows lie inside C.
template <int BN>
__global__ void __launch_bounds__(256) streamk_fixup_kernel(const GemmParams p, int G) {
    pdl_wait();  // the stream-K kernel's partial blocks
    constexpr int BM = kBM;
    constexpr int RQ = BM / 4;       // float4 chunks per tile column
    constexpr int CH = RQ * BN;      // per tile
    constexpr int kMaxSeg = 8;       // loads in flight per batch
    const int64_t T = p.sk_iters;
    const int kb = p.kb_total;
    const int64_t total = static_cast<int64_t>(p.tiles_m) * p.tiles_n * CH;
    for (int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; q < total;
         q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(q / CH);
        const int r = static_cast<int>(q - static_cast<int64_t>(t) * CH);
        const int col = r / RQ, row4 = (r - col * RQ) * 4;
        int tmi, tni;
        tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tmi, tni);
        const int64_t i = static_cast<int64_t>(tmi) * BM + row4;
        const int64_t jc = static_cast<int64_t>(tni) * BN + col;
        if (i >= p.m || jc >= p.n) continue;
        const int64_t first = static_cast<int64_t>(t) * kb;
        const int nseg = sk_cta_of(first + kb - 1, G, T) - sk_cta_of(first, G, T) + 1;
        const float4* src = reinterpret_cast<const float4*>(p.sk_P + static_cast<int64_t>(t) * p.sk_maxseg * (BM * BN) +
                                                            col * BM + row4);
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int j0 = 0; j0 < nseg; j0 += kMaxSeg) {
            float4 v[kMaxSeg];
#pragma unroll
            for (int u = 0; u < kMaxSeg; ++u)
                if (j0 + u < nseg) v[u] = __ldcg(src + static_cast<int64_t>(j0 + u) * (BM * BN / 4));
#pragma unroll
            for (int u = 0; u < kMaxSeg; ++u) {
                if (j0 + u < nseg) {
                    acc.x += v[u].x;
                    acc.y += v[u].y;
                    acc.z += v[u].z;
                    acc.w += v[u].w;
                }
            }
        }
        float* dst = p.C + jc * p.ldc + i;
        const bool vec = p.c_vec && i + 3 < p.m;
        float o[4] = {p.alpha * acc.x, p.alpha * acc.y, p.alpha * acc.z, p.alpha * acc.w};
        if (p.beta != 0.0f) {
            float cin[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (vec) {
                const float4 cv = *reinterpret_cast<const float4*>(dst);
                cin[0] = cv.x;
                cin[1] = cv.y;
                cin[2] = cv.z;
                cin[3] = cv.w;
            } else {
                for (int e = 0; e < 4 && i + e < p.m; ++e) cin[e] = dst[e];
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = fmaf(p.beta, cin[e], o[e]);
        }
        if (vec) {
            *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
            for (int e = 0; e < 4 && i + e < p.m; ++e) dst[e] = o[e];
        }
    }
}

// C = beta * C (beta = 0 writes zeros without reading C).
__global__ void __launch_bounds__(256, 4) scale_kernel(float* __restrict__ C, int64_t ldc, int64_t m, int64_t n,
                                                       float beta, int tx_shift, int by_rows) {
    const Sweep w = sweep_setup(tx_shift);
    float x[kU];
    sweep_batches(
        w, m, n, by_rows != 0,
        [&](int u, int64_t r, int64_t c) { x[u] = beta != 0.0f ? C[c * ldc + r] : 0.0f; },
        [&](int u, int64_t r, int64_t c) { C[c * ldc + r] = (beta == 0.0f) ? 0.0f : beta * x[u]; });
}

// Grid of the column sweep: about 8 CTAs per SM; y spans column groups of
// 256 / TX columns first, x then spans row blocks.  *by_rows tells the kernel
// to batch a thread's rows when it owns fewer than kU columns.
dim3 sweep_grid(int64_t rows, int64_t cols, int num_sms, int* tx_shift, int* by_rows) {
    int sh = 5;
    while (sh < 8 && (int64_t(1) << sh) < rows) ++sh;
    *tx_shift = sh;
    const int64_t TX = int64_t(1) << sh, TY = 256 >> sh;
    const int64_t target = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
    const int64_t col_groups = (cols + TY - 1) / TY;
    const int64_t row_blocks = (rows + TX - 1) / TX;
    int64_t by = col_groups < target ? col_groups : target;
    if (by > 65535) by = 65535;
    if (by < 1) by = 1;
    int64_t bx = (target + by - 1) / by;
    if (bx > row_blocks) bx = row_blocks;
    if (bx > 65535) bx = 65535;
    if (bx < 1) bx = 1;
    const int64_t cols_per_thread = (cols + by * TY - 1) / (by * TY);
    const int64_t rows_per_thread = (rows + bx * TX - 1) / (bx * TX);
    *by_rows = (cols_per_thread < kU && rows_per_thread > cols_per_thread) ? 1 : 0;
    return dim3(static_cast<unsigned>(bx), static_cast<unsigned>(by));
}

}  // namespace

cudaError_t launch_prep(const float* src, int64_t lds, bool transposed, int64_t rows, int64_t cols, float* dst,
                        float* dst_small, int64_t ldd, int num_sms, cudaStream_t stream, bool after_previous) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const bool dep = PG_PDL_PREP && after_previous;
    const int wl = (dep && PG_PREP_OVERLAP) ? 1 : 0;
    if (transposed) {
        const int64_t tiles = ((rows + 31) / 32) * ((cols + 31) / 32);
        int64_t g = static_cast<int64_t>(num_sms) * 8;
        if (g > tiles) g = tiles;
        const dim3 block(32, 8);
        if (dst_small)
            return launch_kernel(dep, prep_transpose_kernel<true>, dim3(static_cast<unsigned>(g)), block, 0, stream,
                                 src, lds, rows, cols, dst, dst_small, ldd, wl);
        return launch_kernel(dep, prep_transpose_kernel<false>, dim3(static_cast<unsigned>(g)), block, 0, stream, src,
                             lds, rows, cols, dst, static_cast<float*>(nullptr), ldd, wl);
    } else if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0 && lds % 4 == 0 &&
               (reinterpret_cast<uintptr_t>(dst) & 15u) == 0 && ldd % 4 == 0 &&
               (dst_small == nullptr || (reinterpret_cast<uintptr_t>(dst_small) & 15u) == 0)) {
        const int64_t chunks = (rows + 3) / 4 * cols;
        int64_t g = (chunks + 255) / 256;
        const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
        if (g > cap) g = cap;
        if (dst_small)
            return launch_kernel(dep, prep_copy_vec_kernel<true>, dim3(static_cast<unsigned>(g)), dim3(256), 0,
                                 stream, src, lds, rows, cols, dst, dst_small, ldd, wl);
        return launch_kernel(dep, prep_copy_vec_kernel<false>, dim3(static_cast<unsigned>(g)), dim3(256), 0, stream,
                             src, lds, rows, cols, dst, static_cast<float*>(nullptr), ldd, wl);
    }
    int sh = 8, by_rows = 0;
    const dim3 grid = sweep_grid(rows, cols, num_sms, &sh, &by_rows);
    if (dst_small)
        return launch_kernel(dep, prep_copy_kernel<true>, grid, dim3(256), 0, stream, src, lds, rows, cols, dst,
                             dst_small, ldd, sh, by_rows, wl);
    return launch_kernel(dep, prep_copy_kernel<false>, grid, dim3(256), 0, stream, src, lds, rows, cols, dst,
                         static_cast<float*>(nullptr), ldd, sh, by_rows, wl);
}

cudaError_t launch_splitk_reduce(const GemmParams& p, int num_sms, cudaStream_t stream) {
    // the grouped form from 32 slices on (each of the kG groups then sums two or more)
    if (p.split >= 32 && p.ldp % 4 == 0 && (reinterpret_cast<uintptr_t>(p.P) & 15u) == 0) {
        const int64_t row_blocks = (p.m + 63) / 64;
        const int64_t target = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
        int64_t by = p.n < 65535 ? p.n : 65535;
        int64_t bx = (target + by - 1) / by;
        if (bx > row_blocks) bx = row_blocks;
        if (bx < 1) bx = 1;
        return launch_after_previous(splitk_reduce_grouped_kernel,
                                     dim3(static_cast<unsigned>(bx), static_cast<unsigned>(by)), dim3(256), 0, stream, p);
    }
    // the partial sums' layout: ldp a multiple of 4, P 16-byte aligned (the workspace regions start on 256 bytes)
    if (p.ldp % 4 != 0 || (reinterpret_cast<uintptr_t>(p.P) & 15u) != 0) return cudaErrorInvalidValue;
    const int64_t chunks = (p.m + 3) / 4 * p.n;
    int64_t g = (chunks + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
    if (g > cap) g = cap;
    return launch_after_previous(splitk_reduce_vec_kernel, dim3(static_cast<unsigned>(g)), dim3(256), 0, stream, p);
}

cudaError_t launch_streamk_fixup(const GemmParams& p, int bn, int ctas, int num_sms, cudaStream_t stream) {
    const int64_t chunks = static_cast<int64_t>(p.tiles_m) * p.tiles_n * (kBM / 4) * bn;
    int64_t g = (chunks + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
    if (g > cap) g = cap;
    switch (bn) {
        case 64:
            return launch_after_previous(streamk_fixup_kernel<64>, dim3(static_cast<unsigned>(g)), dim3(256), 0, stream,
                                         p, ctas);
        case 128:
            return launch_after_previous(streamk_fixup_kernel<128>, dim3(static_cast<unsigned>(g)), dim3(256), 0,
                                         stream, p, ctas);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_scale(float* C, int64_t ldc, int64_t m, int64_t n, float beta, int num_sms,
                         cudaStream_t stream) {
    int sh = 8, by_rows = 0;
    const dim3 grid = sweep_grid(m, n, num_sms, &sh, &by_rows);
    scale_kernel<<<grid, 256, 0, stream>>>(C, ldc, m, n, beta, sh, by_rows);
    return cudaGetLastError();
}

}  // namespace pg
