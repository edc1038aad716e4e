// Register-only FP32 FMA throughput: the practical ceiling of the CUDA-core path.
//
// Every thread runs long independent streams of fused multiply-adds on 32
// accumulators held in registers (no memory traffic in the timed loop), with
// scalar FFMA and with the packed two-lane fma.rn.f32x2, at several CTAs per SM.
// Prints one JSON line: TFLOP/s and FMAs per clock per SM (against the device's
// reported maximum SM clock) for each variant.  Used to put the FFMA GEMM's
// fraction of the nominal peak (SMs x 128 lanes x 2 x clock) in context.
#include <cuda_runtime.h>

#include <cstdio>

template <bool PACKED>
__global__ void __launch_bounds__(256) fma_stream(float* out, int iters, float x, float y) {
    float2 acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = make_float2(threadIdx.x * 1e-7f + i, i * 1e-3f);
    const float2 a = make_float2(x, y), b = make_float2(y, x);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (PACKED) {
                acc[i] = __ffma2_rn(a, b, acc[i]);
            } else {
                acc[i].x = fmaf(a.x, b.x, acc[i].x);
                acc[i].y = fmaf(a.y, b.y, acc[i].y);
            }
        }
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s += acc[i].x + acc[i].y;
    if (s == 12345.678f) out[threadIdx.x] = s;  // keeps the arithmetic live
}

int main() {
    int sms = 0, clk_khz = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess) return 1;
    cudaDeviceGetAttribute(&clk_khz, cudaDevAttrClockRate, 0);
    float* out = nullptr;
    if (cudaMalloc(&out, 1024 * sizeof(float)) != cudaSuccess) return 1;
    const int iters = 100000;
    printf("{\"sms\": %d, \"max_sm_mhz\": %d, \"runs\": [", sms, clk_khz / 1000);
    bool first = true;
    for (int packed = 0; packed < 2; ++packed) {
        for (int ctas : {2, 4, 8}) {
            const dim3 grid(sms * ctas), block(256);
            cudaEvent_t e0, e1;
            cudaEventCreate(&e0);
            cudaEventCreate(&e1);
            for (int pass = 0; pass < 2; ++pass) {  // pass 0 warms up
                cudaEventRecord(e0);
                if (packed) fma_stream<true><<<grid, block>>>(out, pass ? iters : 1000, 1.0001f, 0.9999f);
                else fma_stream<false><<<grid, block>>>(out, pass ? iters : 1000, 1.0001f, 0.9999f);
                cudaEventRecord(e1);
                cudaEventSynchronize(e1);
            }
            float ms = 0.f;
            cudaEventElapsedTime(&ms, e0, e1);
            const double fmas = 32.0 * iters * 256.0 * grid.x;
            printf("%s{\"op\": \"%s\", \"ctas_per_sm\": %d, \"ms\": %.3f, \"tflops\": %.2f, \"fma_per_clk_per_sm\": %.1f}",
                   first ? "" : ", ", packed ? "fma.rn.f32x2" : "fma.rn.f32", ctas, ms,
                   2.0 * fmas / (ms * 1e-3) / 1e12, fmas / (ms * 1e-3) / sms / (clk_khz * 1e3));
            first = false;
            cudaEventDestroy(e0);
            cudaEventDestroy(e1);
        }
    }
    const cudaError_t err = cudaGetLastError();
    printf("], \"error\": \"%s\"}\n", cudaGetErrorString(err));
    cudaFree(out);
    return err == cudaSuccess ? 0 : 1;
}
