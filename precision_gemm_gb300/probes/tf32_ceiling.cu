// TF32 tensor-core throughput with the operands already in shared memory: the
// practical ceiling of the tcgen05 path.
//
// One CTA per SM fills an A tile (128 x 32) and a B tile (N x 32) in shared
// memory once, then one thread issues a long stream of
// tcgen05.mma.cta_group::1.kind::tf32 (M = 128, N, K = 8) into a TMEM
// accumulator -- no TMA, no epilogue in the timed work -- for N = 64, 128 and
// 256.  A second kernel does the same on SM pairs (clusters of two CTAs, each
// holding 128 rows of A and N/2 rows of B): one thread of the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256, N, K = 8), the instruction of the SM-pair
// GEMM.  Prints one JSON line: TFLOP/s over all SMs and dense flops per clock
// per SM (against the device's reported maximum SM clock) for each case.  Used
// to put the TF32 and 3xTF32 GEMMs' rates in context next to the TF32 peak
// derived from the measured bf16 peak.
#include <cuda_runtime.h>

#include <cstdio>

#include "../csrc/ptx.cuh"

namespace {

constexpr int kSmemBytes = 120 * 1024;  // one CTA per SM (TMEM is allocated per CTA)

// SM clock cycles and global-timer nanoseconds, read together by the issuing
// thread of block 0 around its MMA stream: their ratio is the SM clock the
// stream actually ran at.
__device__ __forceinline__ void stamp(unsigned long long* out) {
    unsigned long long c, g;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g));
    out[0] = c;
    out[1] = g;
}

template <int N>
__global__ void __launch_bounds__(128, 1) tf32_mma_stream(int iters, float* sink, int* status,
                                                          unsigned long long* clk) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = pg::align_smem_1024(smem_raw);
    float* tiles = reinterpret_cast<float*>(smem);  // A: 128 rows x 32, then B: N rows x 32 (K-major)
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + (128 + N) * 32 * 4);
    uint32_t* holder = reinterpret_cast<uint32_t*>(bar + 1);
    for (int i = threadIdx.x; i < (128 + N) * 32; i += blockDim.x) tiles[i] = 1.0f / static_cast<float>(1 + (i & 63));
    if (threadIdx.x == 0) {
        pg::mbar_init(pg::smem_u32(bar), 1);
        pg::fence_mbar_init();
    }
    pg::fence_proxy_async_smem();  // the tensor core reads the tiles written above
    if (threadIdx.x < 32) {
        pg::tmem_alloc(pg::smem_u32(holder), N);
        pg::tmem_relinquish();
    }
    pg::tc_fence_before_sync();
    __syncthreads();
    pg::tc_fence_after_sync();
    const uint32_t tmem = *holder;
    if (threadIdx.x == 0) {
        const uint32_t a = pg::smem_u32(smem), b = a + 128 * 32 * 4;
        const uint32_t idesc = pg::idesc_tf32(128, N, false, false);
        uint32_t acc = 0;
        if (blockIdx.x == 0) stamp(clk);
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                pg::mma_tf32(tmem, pg::operand_desc<32>(a, kk, true), pg::operand_desc<32>(b, kk, true), idesc, acc);
                acc = 1;
            }
        }
        pg::mma_commit(pg::smem_u32(bar));
        if (!pg::mbar_wait_bounded(pg::smem_u32(bar), 0, 4000000000ull, nullptr)) atomicExch(status, 1);
        if (blockIdx.x == 0) stamp(clk + 2);
    }
    __syncthreads();
    pg::tc_fence_after_sync();
    if (threadIdx.x < 32) {  // read the accumulator back so the work is observable
        uint32_t v[32];
        pg::tmem_ld_32x32b_x32(tmem, v);
        pg::tmem_wait_ld();
        if (threadIdx.x == 0) sink[blockIdx.x] = __uint_as_float(v[0]);
    }
    pg::tc_fence_before_sync();
    __syncthreads();
    if (threadIdx.x < 32) {
        pg::tc_fence_after_sync();
        pg::tmem_dealloc(tmem, N);
    }
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The SM-pair form: each CTA holds A rows [128 r, 128 r + 128) and B rows
// [r N/2, (r + 1) N/2) at the same shared-memory offsets; the even CTA issues.
template <int N>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    tf32_mma_stream_pair(int iters, float* sink, int* status, unsigned long long* clk) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = pg::align_smem_1024(smem_raw);
    float* tiles = reinterpret_cast<float*>(smem);  // A: 128 rows x 32, then B: N/2 rows x 32 (K-major)
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + (128 + N / 2) * 32 * 4);
    uint32_t* holder = reinterpret_cast<uint32_t*>(bar + 1);
    const uint32_t rank = cluster_rank();
    for (int i = threadIdx.x; i < (128 + N / 2) * 32; i += blockDim.x)
        tiles[i] = 1.0f / static_cast<float>(1 + (i & 63));
    if (threadIdx.x == 0) {
        pg::mbar_init(pg::smem_u32(bar), 1);
        pg::fence_mbar_init();
    }
    pg::fence_proxy_async_smem();
    if (threadIdx.x < 32) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(pg::smem_u32(holder)),
                     "r"(N)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    pg::tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    pg::tc_fence_after_sync();
    const uint32_t tmem = *holder;
    if (rank == 0 && threadIdx.x == 0) {
        const uint32_t a = pg::smem_u32(smem), b = a + 128 * 32 * 4;
        const uint32_t idesc = pg::idesc_tf32(256, N, false, false);
        uint32_t acc = 0;
        if (blockIdx.x == 0) stamp(clk);
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                asm volatile(
                    "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                    "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
                    "l"(pg::operand_desc<32>(a, kk, true)), "l"(pg::operand_desc<32>(b, kk, true)), "r"(idesc),
                    "r"(acc)
                    : "memory");
                acc = 1;
            }
        }
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         pg::smem_u32(bar))
                     : "memory");
        if (!pg::mbar_wait_bounded(pg::smem_u32(bar), 0, 4000000000ull, nullptr)) atomicExch(status, 1);
        if (blockIdx.x == 0) stamp(clk + 2);
    }
    pg::tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // the pair's MMAs are complete before either CTA reads or frees TMEM
    pg::tc_fence_after_sync();
    if (threadIdx.x < 32) {
        uint32_t v[32];
        pg::tmem_ld_32x32b_x32(tmem, v);
        pg::tmem_wait_ld();
        if (threadIdx.x == 0) sink[blockIdx.x] = __uint_as_float(v[0]);
    }
    pg::tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    if (threadIdx.x < 32) {
        pg::tc_fence_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(N) : "memory");
    }
}

template <int N, bool PAIR>
bool run(int sms, int clk_khz, bool first) {
    auto kern = PAIR ? tf32_mma_stream_pair<N> : tf32_mma_stream<N>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess) return false;
    float* sink = nullptr;
    int* status = nullptr;
    unsigned long long* clk = nullptr;
    if (cudaMalloc(&sink, sms * sizeof(float)) != cudaSuccess || cudaMalloc(&status, sizeof(int)) != cudaSuccess ||
        cudaMalloc(&clk, 4 * sizeof(unsigned long long)) != cudaSuccess)
        return false;
    cudaMemset(status, 0, sizeof(int));
    const int iters = 1 << 15;
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    for (int pass = 0; pass < 2; ++pass) {  // pass 0 warms up
        cudaEventRecord(e0);
        kern<<<PAIR ? sms & ~1 : sms, 128, kSmemBytes>>>(pass ? iters : 256, sink, status, clk);
        cudaEventRecord(e1);
        if (cudaEventSynchronize(e1) != cudaSuccess) return false;
    }
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    int st = 0;
    unsigned long long c[4] = {0, 0, 0, 0};
    cudaMemcpy(&st, status, sizeof(int), cudaMemcpyDeviceToHost);
    cudaMemcpy(c, clk, sizeof(c), cudaMemcpyDeviceToHost);
    const double run_mhz = c[3] > c[1] ? static_cast<double>(c[2] - c[0]) / static_cast<double>(c[3] - c[1]) * 1e3 : 0.0;
    // per SM: 128 rows of the product and N columns per MMA in both forms
    const int used = PAIR ? sms & ~1 : sms;
    const double flops = 2.0 * 128.0 * N * 8.0 * 4.0 * iters * used;
    printf("%s{\"form\": \"%s\", \"n\": %d, \"ms\": %.4f, \"tflops\": %.2f, \"flops_per_clk_per_sm\": %.1f, "
           "\"sm_mhz_in_kernel\": %.0f, \"timed_out\": %d}",
           first ? "" : ", ", PAIR ? "cta_group::2 (M=256)" : "cta_group::1 (M=128)", N, ms,
           flops / (ms * 1e-3) / 1e12, flops / (ms * 1e-3) / used / (clk_khz * 1e3), run_mhz, st);
    cudaFree(sink);
    cudaFree(status);
    cudaFree(clk);
    return cudaGetLastError() == cudaSuccess;
}

}  // namespace

int main() {
    int sms = 0, clk_khz = 0, major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess) return 1;
    cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, 0);
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, 0);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, 0);
    if (major != 10 || minor != 3) {
        printf("{\"error\": \"needs compute capability 10.3, found %d.%d\"}\n", major, minor);
        return 1;
    }
    printf("{\"probe\": \"tcgen05 kind::tf32, K=8, operands resident in shared memory\", \"sms\": %d, "
           "\"max_sm_mhz\": %d, \"runs\": [",
           sms, clk_khz / 1000);
    const bool ok = run<64, false>(sms, clk_khz, true) && run<128, false>(sms, clk_khz, false) &&
                    run<256, false>(sms, clk_khz, false) && run<128, true>(sms, clk_khz, false) &&
                    run<256, true>(sms, clk_khz, false);
    printf("]}\n");
    return ok ? 0 : 1;
}
