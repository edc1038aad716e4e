// Declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>  // CUtensorMap (header only; the driver is reached at run time)
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>

namespace pg {

// Programmatic dependent launch for a kernel that consumes the previous
// kernel's output in the same call (the split-K reduction, the stream-K
// fix-up): the GPU may start scheduling it once every CTA of the previous
// kernel has issued its trigger (pdl_trigger, after the main loop) while that
// kernel finishes; the kernel itself waits (pdl_wait: griddepcontrol.wait) for
// that kernel's completion and memory before it touches global memory.
// Measured on GB300 (L2 flushed, against ordinary launches): FFMA 256^3
// 0.0160 -> 0.0140 ms, row-major 1024^3 0.0580 -> 0.0540, 8192 x 64 x 8192
// TF32 0.0632 -> 0.0611 and 3xTF32 0.0826 -> 0.0806, 1000 x 1300 x 4000 TF32
// 0.0375 -> 0.0345.
#ifndef PG_PDL
#define PG_PDL 1
#endif
// The same for a GEMM kernel right after an operand copy or split of the same
// call (no memset between them), and for the second of two such passes
// (GB300, L2 flushed, against ordinary launches of the whole chain: the ragged
// 3000 x 1500 x 777 problem with lda = 3013 TF32 0.0314 -> 0.0274 ms, 3xTF32
// 1536^2 x 1024 on SM pairs 0.0539 -> 0.0467, 8192 x 64 x 8192 3xTF32 0.0826 ->
// 0.0765, 333 x 444 x 555 FFMA 0.0334 -> 0.0262).
#ifndef PG_PDL_PREP
#define PG_PDL_PREP 1
#endif
// The second of two operand passes (A's, then B's: disjoint data) runs alongside
// the first and waits for it only before it retires; the GEMM, which waits for
// the second pass, then finds both complete.  GB300, L2 flushed, 3xTF32 on SM
// pairs (both operands split): row-major 2048^3 0.0856 -> 0.0816 ms, 1536^2 x
// 1024 0.0467 -> 0.0447, the ragged 3000 x 1500 x 777 0.0549 -> 0.0543, 4096^3
// 0.475 -> 0.471; 8192^3 and 6144^3 within 1 %.
#ifndef PG_PREP_OVERLAP
#define PG_PREP_OVERLAP 1
#endif
template <typename... Params, typename... Args>
cudaError_t launch_kernel(bool after_previous, void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = after_previous ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}
template <typename... Params, typename... Args>
cudaError_t launch_after_previous(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                  Args... args) {
    return launch_kernel(PG_PDL != 0, kern, grid, block, smem, st, args...);
}

// Raise a kernel's dynamic shared-memory limit to `bytes` once per device:
// the attribute stays set for the process, and setting it on every launch cost
// a driver call per call.  `done` holds one bit per device ordinal (a static of
// the launcher instantiation that owns the kernel).
inline cudaError_t set_smem_limit_once(std::atomic<uint64_t>& done, const void* kern, int bytes) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    const uint64_t bit = uint64_t(1) << dev;
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Tile geometry common to every GEMM kernel: BM rows of C per CTA.
constexpr int kBM = 128;
// FFMA kernel: K block staged per ring slot.
constexpr int kFfmaBK = 32;

// Parameters every GEMM kernel receives (by value, in the kernel's param space).
struct GemmParams {
    int64_t m, n, k;
    float alpha, beta;
    float* C;            // final output (split == 1)
    int64_t ldc;
    float* P;            // partial sums [split][n][ldp] (split > 1)
    int64_t ldp;         // multiple of 4
    int64_t p_stride;    // elements between two slices of P (= ldp * n)
    int32_t tiles_m, tiles_n;
    int32_t kb_total;        // K blocks in total
    int32_t kb_per_split;    // K blocks per slice
    int32_t split;           // number of slices
    int32_t group_m;         // rasterisation: tile rows per group
    int32_t c_vec;           // C 16-byte aligned and ldc % 4 == 0
    int32_t c_tma;           // FFMA: whole-tile CTAs store C through the tensor map tmC (beta = 0, split 1)
    int32_t after_prep;      // host side: launch the GEMM dependent on the operand pass right before it
    int32_t debug_flags;
    int32_t a3d;             // tcgen05 kernels: A tensor map is 3-D {32, k, m/32} (one box per 128 rows)
    int32_t a_kmajor;        // tcgen05 kernels: A is read K-major (transa = 'T'), else M-major
    int32_t b_mnmajor;       // tcgen05 kernels: B is read N-major (transb = 'T'), else K-major
    int32_t b3d;             // tcgen05 kernels, N-major B: tensor map 3-D {32, k, n/32}
    int32_t b_presplit;      // single-SM 3xTF32, BN <= 128: B's TF32 parts come split (tmB big, tmBs small)
    // Last-wave split (SM-pair kernel, split == 1): tiles [tail_first, tiles) each
    // run as tail_split K slices of tail_kb blocks; every slice stores its partial
    // 256 x BN block in tail_P ([tail tile][slice][column][row]), and per epilogue
    // warp region a counter in tail_cnt (zeroed before the launch) finds the last
    // slice to finish, which sums the partials in slice order and writes C.
    int32_t tail_first;
    int32_t tail_split;      // 1: no tail split
    int32_t tail_kb;
    float* tail_P;
    int* tail_cnt;
    // FFMA stream-K: the CTAs share the sk_iters = tiles x kb_total (tile,
    // k-block) iterations in equal contiguous ranges; segment j of tile t stores
    // its partial block at sk_P + (t * sk_maxseg + j) * BM * BN ([column][row]).
    int64_t sk_iters;
    int32_t sk_maxseg;
    float* sk_P;
    uint64_t timeout_ns;     // limit of every bounded wait
    int* status;             // per-device status word
};

// Device status values written by kernels (match SGEMM_ERR_* of the ABI).
constexpr int kStatusTimeout = 4;

// ---- launchers (each lives beside its kernel) -------------------------------

// FFMA kernel: tile 128 x bn, bn in {64, 128, 256}.
int ffma_threads(int bn);
int ffma_stages(int bn);
int ffma_ctas_per_sm(int bn);
size_t ffma_smem_bytes(int bn);
cudaError_t launch_ffma(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, const GemmParams& p,
                        int bn, dim3 grid, cudaStream_t stream);
// FFMA stream-K (bn in {64, 128}): `ctas` co-resident CTAs share the product's
// (tile, k-block) iterations; then the fix-up kernel adds each tile's partial
// blocks in order and applies alpha/beta.  Two launches.
cudaError_t launch_ffma_sk(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int bn, int ctas,
                           int num_sms, cudaStream_t stream);

// tcgen05 kernel: tile 128 x bn, bn in {64, 128, 256}; split3 selects 3xTF32,
// whose TF32 split this kernel does itself in shared memory (it serves the
// narrow shapes, m <= 128 or n <= 64, where a split pre-pass would cost more
// HBM traffic than the product).
int tc_bk(bool split3);
int tc_stages(int bn, bool split3);
int tc_threads(int bn, bool split3);
size_t tc_smem_bytes(int bn, bool split3);
// tmBs: B's remainders when p.b_presplit (otherwise unused; pass tmB).
cudaError_t launch_tc(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmBs, const GemmParams& p,
                      int bn, bool split3, dim3 grid, cudaStream_t stream);

// The same kernel in stream-K form (3xTF32, bn = 128): `ctas` CTAs share
// the (tile, k-block) iterations in equal ranges, storing partial blocks to
// p.sk_P; launch_streamk_fixup then sums them.
cudaError_t launch_tc_sk(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmBs, const GemmParams& p,
                         int bn, int ctas, cudaStream_t stream);

// tcgen05 kernel on SM pairs (cta_group::2, persistent, double-buffered TMEM):
// pair tile 256 x bn, bn in {128, 256}; launches min(units, resident pairs) pairs.
int tc2_bk(bool split3);
int tc2_threads();
int tc2_epilogue_warps();  // per CTA
int tc2_stages(int bn, bool split3);
size_t tc2_smem_bytes(int bn, bool split3);
cudaError_t launch_tc2(const CUtensorMap& tmA, const CUtensorMap& tmAs, const CUtensorMap& tmB,
                       const CUtensorMap& tmBs, const GemmParams& p, int bn, bool split3, int units, int num_sms,
                       cudaStream_t stream, int* pairs_launched);

// Operand preparation: dst(r, c) = src(r, c) (or src(c, r) when transposed) for
// r < rows, c < cols, dst with leading dimension ldd.  With dst_small != null
// the value is split into a TF32 "big" part (dst) and the exact remainder
// (dst_small), the operands of the SM-pair kernel's 3xTF32 mode.
cudaError_t launch_prep(const float* src, int64_t lds, bool transposed, int64_t rows,
                        int64_t cols, float* dst, float* dst_small, int64_t ldd,
                        int num_sms, cudaStream_t stream, bool after_previous);

// C = alpha * sum_s P[s] + beta * C, slices summed in increasing s.
cudaError_t launch_splitk_reduce(const GemmParams& p, int num_sms, cudaStream_t stream);

// Stream-K fix-up: C = alpha * sum_j P[t][j] + beta * C per 128 x bn tile t
// (bn in {64, 128}), the partial blocks p.sk_P + (t * sk_maxseg + j) * 128 * bn
// ([column][row]) of its segments j added in increasing order; `ctas` is the
// stream-K grid, whose ranges give each tile's number of segments.
cudaError_t launch_streamk_fixup(const GemmParams& p, int bn, int ctas, int num_sms, cudaStream_t stream);

// C = beta * C (beta == 0 writes zeros without reading C).
cudaError_t launch_scale(float* C, int64_t ldc, int64_t m, int64_t n, float beta, int num_sms,
                         cudaStream_t stream);

}  // namespace pg
