// Exact-FP32 GEMM on the CUDA cores (FFMA), sm_103a.
//
// One CTA computes a 128 x BN tile of C from column-major A (m x k, M-major)
// and B (k x n, K-major), both read through TMA.  Prior art on the pages --
// register tiles of C per thread, shared-memory staging of A and B tiles,
// float4 accesses and double buffering ("Optimizing SGEMM on NVIDIA Turing
// GPUs", kernels 2-10; "V3. Vectorized and double buffer", sections 1-2) -- is
// kept where it still holds on Blackwell and replaced where it does not:
//
//   * thread 0 issues TMA tile loads PD k-blocks ahead into a STAGES-deep ring
//     of shared-memory slots, each guarded by a "full" mbarrier (TMA bytes
//     landed) and an "empty" mbarrier (every warp is done with the slot); this
//     replaces the pages' register prefetch + ping-pong buffers and their
//     __syncthreads.  The loader is a consumer thread rather than a warp of its
//     own so that the warps split evenly over the SM's four sub-partitions and
//     each thread keeps 128 registers for its 8 x 8 tile;
//   * the A tile lands as BK rows of 128 floats (k-major rows of m, the layout
//     the wiki builds by hand with its transposed As[k][m] store); the B tile
//     lands as BN rows of 32 floats (128 B) with the 128-byte TMA swizzle, so a
//     quarter-warp reading one 16-byte chunk from 8 different rows hits 8
//     different bank groups (no bank conflicts, the wiki's V3.1/V3.2 goal);
//   * each thread owns an 8 x 8 register tile: rows {4tm..4tm+3} and
//     {64+4tm..64+4tm+3}, columns {tn + (BN/8)*jj}, held as 4 x 8 register
//     pairs (two rows of one column).  Per pair of k values it reads 8 float2
//     of B (two k values of one column each) and, per k, 2 float4 of A, then
//     issues 32 packed two-lane FMAs (fma.rn.f32x2, sm_100 and later: the A
//     pair of two rows times the broadcast B value of the column), which halves
//     the FMA instructions that compete for issue slots;
//   * the epilogue stages the tile in the free ring as [column][row], then each
//     warp computes alpha*acc + beta*C for whole columns and stores float4s
//     (scalar stores at ragged edges or when C / ldc is not 16-byte aligned);
//     with split-K it writes raw partial sums instead.  A last-wave K slice's
//     CTA keeps the per-thread epilogue (its warps finish one by one).
//
// Tile shapes: 128 x 128 (256 threads, 3 slots, two CTAs per SM) is the default;
// 128 x 64 (128 threads, 3 slots, three CTAs per SM) serves n <= 64 and tiny
// products, and 128 x 256 (512 threads, 4 slots) stays selectable.
// Measured on GB300 at 8192^3: 128 x 128 with float2 B reads and PD = 1 runs at
// 62.7 TFLOP/s against 58.7 for 128 x 256 with float4 B reads.
//
// Every mbarrier wait is bounded (see ptx.cuh); a CTA whose wait expires marks
// the device status word, waits (bounded) for its own TMA copies and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace pg {
namespace {

// Columns per thread for the 128-wide tile (a compile-time tunable, 8 or 16).
#ifndef PG_FFMA_JJ128
#define PG_FFMA_JJ128 8
#endif
// Slot waits of the consumer warps: 1 = lane 0 polls, then every lane acquires
// (mbar_wait_warp); 0 = every lane polls.  Measured on GB300: the one-lane poll
// takes the barrier's polling off the shared-memory banks but runs 0.7 % slower
// (8192^3 17.24 -> 17.35 ms, 16384^3 137.2 -> 138.3 ms), so all lanes poll.
#ifndef PG_FFMA_WARP_WAIT
#define PG_FFMA_WARP_WAIT 0
#endif

template <int BN, int JJ>
struct FfmaCfg {
    static constexpr int BM = kBM;
    static constexpr int BK = kFfmaBK;
    static constexpr int TGN = BN / JJ;                   // thread columns (JJ columns per thread)
    static constexpr int THREADS = 16 * TGN;              // 16 thread rows x TGN
    static constexpr int CWARPS = THREADS / 32;
    static constexpr int STAGES = (BN == 256) ? 4 : 3;
    // While k-block `it` is computed, thread 0 issues k-block it + PD into slot
    // (it + PD) % STAGES, whose previous contents (k-block it + PD - STAGES) every
    // warp released STAGES - PD iterations ago; with a spare slot (PD = STAGES-2)
    // the loader waits only if some warp trails by two whole k-blocks.
    static constexpr int PD = STAGES - 2;
    // 128 x 64 tiles run three CTAs per SM (12 warps; 74.8 KB of shared memory
    // and up to 170 registers each): against two CTAs with four slots, 8192 x 64 x
    // 8192 0.1686 -> 0.1604 ms, 16384 x 64 x 16384 0.627 -> 0.603, 8192 x 32 x
    // 8192 0.169 -> 0.158 (2048 x 64 x 16384 0.0887 -> 0.0908).
    static constexpr int CTAS_PER_SM = (BN == 256) ? 1 : (BN == 64 ? 3 : 2);
    static constexpr int A_BYTES = BM * BK * 4;           // 16 KiB
    static constexpr int B_BYTES = BN * BK * 4;           // BN rows of 128 B
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int BAR_BYTES = 2 * STAGES * 8 + 16;
    static constexpr size_t SMEM = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + BAR_BYTES;
    static_assert(TGN % 8 == 0, "column stride must keep (row % 8) fixed per thread");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "128B-swizzle slots need 1 KiB alignment");
};

// Epilogue of a CTA that computed its tile (or K slice) alone, through shared
// memory.  Each thread's register tile holds four rows of eight columns spread
// over the tile, so storing it straight from registers makes every warp
// instruction write eight 64-byte pieces of eight columns.  Instead the tile is
// written to a [column][row] block in the ring (free once every warp has left
// the k loop) and each warp then moves whole columns, lane l taking rows
// 4l..4l+3: one instruction per 512-byte column segment of C (or of the K
// slice's partial block), and the same for the reads of C when beta != 0.
// Measured on GB300 (L2 flushed): 16384^2 x 64 0.792 -> 0.679 ms, 16384^2 x 128
// 1.314 -> 1.193, 8192^2 x 64 0.206 -> 0.177, row-major 1024^3 0.060 -> 0.056.
// The column stride BM + 4 puts the eight consecutive columns that a quarter
// warp writes in eight different 16-byte bank groups.  Must be called by every
// thread of the CTA (it holds a block barrier).
template <int BN, int JJ>
__device__ __forceinline__ void ffma_epilogue_staged(const float2 (&acc)[4][JJ], uint8_t* smem, int warp, int lane,
                                                     int tm, int tn, int64_t m0, int64_t n0, int slice,
                                                     const GemmParams& p) {
    using Cfg = FfmaCfg<BN, JJ>;
    constexpr int CS = Cfg::BM + 4;
    constexpr int NC = BN / Cfg::CWARPS;  // columns per warp
    static_assert(Cfg::BM == 128, "one float4 of rows per lane");
    static_assert(BN * CS * 4 <= Cfg::STAGES * Cfg::STAGE_BYTES, "the staging block must fit in the ring");
    float* Cs = reinterpret_cast<float*>(smem);
#pragma unroll
    for (int jj = 0; jj < JJ; ++jj)
#pragma unroll
        for (int h = 0; h < 2; ++h)
            *reinterpret_cast<float4*>(Cs + (tn + Cfg::TGN * jj) * CS + 64 * h + 4 * tm) =
                make_float4(acc[2 * h][jj].x, acc[2 * h][jj].y, acc[2 * h + 1][jj].x, acc[2 * h + 1][jj].y);
    __syncthreads();

    const int64_t i = m0 + 4 * lane;
    if (i >= p.m) return;
    const bool rows4 = i + 3 < p.m;
    const float alpha = p.alpha, beta = p.beta;
    const bool read_c = p.split == 1 && beta != 0.0f;
    // Warp w takes columns w, w + CWARPS, ...  All reads of C are issued before
    // the first store: interleaved, each read would be ordered after the
    // previous store (the compiler cannot rule out aliasing) and wait out the
    // full DRAM latency.
    float4 cin[NC];
    if (read_c) {
#pragma unroll
        for (int q = 0; q < NC; ++q) {
            const int64_t j = n0 + warp + Cfg::CWARPS * q;
            float4 c = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (j < p.n) {
                const float* src = p.C + j * p.ldc + i;
                if (p.c_vec && rows4) {
                    c = *reinterpret_cast<const float4*>(src);
                } else {
                    c.x = src[0];
                    if (i + 1 < p.m) c.y = src[1];
                    if (i + 2 < p.m) c.z = src[2];
                    if (i + 3 < p.m) c.w = src[3];
                }
            }
            cin[q] = c;
        }
    }
#pragma unroll
    for (int q = 0; q < NC; ++q) {
        const int c = warp + Cfg::CWARPS * q;
        const int64_t j = n0 + c;
        if (j >= p.n) break;
        const float4 v = *reinterpret_cast<const float4*>(Cs + c * CS + 4 * lane);
        if (p.split > 1) {
            float* dst = p.P + slice * p.p_stride + j * p.ldp + i;
            if (rows4) {
                *reinterpret_cast<float4*>(dst) = v;
            } else {
                dst[0] = v.x;
                if (i + 1 < p.m) dst[1] = v.y;
                if (i + 2 < p.m) dst[2] = v.z;
            }
        } else {
            float4 o = make_float4(alpha * v.x, alpha * v.y, alpha * v.z, alpha * v.w);
            if (read_c) {
                o.x = fmaf(beta, cin[q].x, o.x);
                o.y = fmaf(beta, cin[q].y, o.y);
                o.z = fmaf(beta, cin[q].z, o.z);
                o.w = fmaf(beta, cin[q].w, o.w);
            }
            float* dst = p.C + j * p.ldc + i;
            if (p.c_vec && rows4) {
                *reinterpret_cast<float4*>(dst) = o;
            } else {
                dst[0] = o.x;
                if (i + 1 < p.m) dst[1] = o.y;
                if (i + 2 < p.m) dst[2] = o.z;
                if (i + 3 < p.m) dst[3] = o.w;
            }
        }
    }
}

// The same epilogue when beta = 0, C is 16-byte aligned with ldc % 4 == 0 and K
// is not split: the tile, scaled by alpha, goes to the ring as four boxes of 32
// rows x BN columns in the 128-byte TMA swizzle (box b holds rows 32b..32b+31,
// column c at bytes 128c of the box, 16-byte chunk q of the column's 128 bytes
// at chunk q ^ (c % 8) -- so the eight consecutive columns a quarter warp
// writes land in eight bank groups), and one thread stores the boxes with TMA.
// Whole 128-byte lines reach L2 and no thread issues a global store (against the
// thread stores of whole columns, L2 flushed: 16384^2 x 64 0.670 -> 0.654 ms,
// 16384^2 x 128 1.197 -> 1.141, 8192^2 x 64 0.175 -> 0.170).  Columns
// beyond n are dropped by the copy.  Only boxes wholly inside m go by TMA: a
// bulk store of the box that m cuts also wrote rows past m (into the ld gap of
// C) on GB300, so the threads store that box's rows below m themselves.  Must
// be called by every thread of the CTA.
template <int BN, int JJ>
__device__ __forceinline__ void ffma_epilogue_tma(const float2 (&acc)[4][JJ], uint8_t* smem, int tm, int tn,
                                                  int64_t m0, int64_t n0, const CUtensorMap* tmC,
                                                  const GemmParams& p) {
    using Cfg = FfmaCfg<BN, JJ>;
    constexpr int BOX = BN * 128;
    static_assert(Cfg::BM == 128 && BOX % 1024 == 0, "four 1 KiB-aligned boxes of 32 rows");
    static_assert(4 * BOX <= Cfg::STAGES * Cfg::STAGE_BYTES, "the boxes must fit in the ring");
    const float alpha = p.alpha;
#pragma unroll
    for (int jj = 0; jj < JJ; ++jj)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int c = tn + Cfg::TGN * jj;
            const int r = 64 * h + 4 * tm;
            const int q = (r & 31) >> 2;
            *reinterpret_cast<float4*>(smem + (r >> 5) * BOX + c * 128 + ((q ^ (c & 7)) << 4)) =
                make_float4(alpha * acc[2 * h][jj].x, alpha * acc[2 * h][jj].y, alpha * acc[2 * h + 1][jj].x,
                            alpha * acc[2 * h + 1][jj].y);
        }
    fence_proxy_async_smem();  // the generic-proxy writes above, before the bulk copy reads them
    __syncthreads();
    const int64_t rows = p.m - m0;
    const int whole = rows >= 128 ? 4 : static_cast<int>(rows >> 5);  // boxes wholly inside m
    if (threadIdx.x == 0) {
        for (int b = 0; b < whole; ++b)
            tma_store_2d(tmC, smem_u32(smem + b * BOX), static_cast<int32_t>(m0 + 32 * b), static_cast<int32_t>(n0));
        bulk_commit();
    }
    if (whole < 4 && 32 * whole < rows) {
        // the box that m cuts: 8 chunks of 4 rows per column, consecutive threads
        // taking consecutive chunks of a column
        const int b = whole;
        for (int u = threadIdx.x; u < 8 * BN; u += Cfg::THREADS) {
            const int c = u >> 3, q = u & 7;
            const int64_t i = m0 + 32 * b + 4 * q, j = n0 + c;
            if (j >= p.n || i >= p.m) continue;
            const float4 v = *reinterpret_cast<const float4*>(smem + b * BOX + c * 128 + ((q ^ (c & 7)) << 4));
            float* dst = p.C + j * p.ldc + i;
            if (i + 3 < p.m) {
                *reinterpret_cast<float4*>(dst) = v;
            } else {
                dst[0] = v.x;
                if (i + 1 < p.m) dst[1] = v.y;
                if (i + 2 < p.m) dst[2] = v.z;
            }
        }
    }
    if (threadIdx.x == 0) bulk_wait_read();  // the ring must outlive the copy's reads
}

// One k-block of the thread's 8 x JJ register tile from the ring slot at `slot`
// (the stream-K kernel's form of the data-parallel kernel's inner loop): per
// pair of k values JJ float2 of B (two k values of one column each), per k 2
// float4 of A, then the packed two-lane FMAs.
template <int BN, int JJ>
__device__ __forceinline__ void ffma_kblock(float2 (&acc)[4][JJ], const uint8_t* slot, int tm, int tn,
                                            uint32_t bchunk_xor) {
    using Cfg = FfmaCfg<BN, JJ>;
    const float* As = reinterpret_cast<const float*>(slot);
    const uint8_t* Bs = slot + Cfg::A_BYTES + tn * 128;
#pragma unroll
    for (int g2 = 0; g2 < Cfg::BK / 2; ++g2) {
        float2 b[JJ];
        const uint32_t off2 = (((static_cast<uint32_t>(g2 >> 1)) ^ bchunk_xor) << 4) + ((g2 & 1) << 3);
#pragma unroll
        for (int jj = 0; jj < JJ; ++jj) b[jj] = *reinterpret_cast<const float2*>(Bs + jj * (Cfg::TGN * 128) + off2);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const float* arow = As + (2 * g2 + kk) * Cfg::BM;
            const float4 a0 = *reinterpret_cast<const float4*>(arow + 4 * tm);
            const float4 a1 = *reinterpret_cast<const float4*>(arow + 64 + 4 * tm);
            const float2 a[4] = {make_float2(a0.x, a0.y), make_float2(a0.z, a0.w), make_float2(a1.x, a1.y),
                                 make_float2(a1.z, a1.w)};
#pragma unroll
            for (int jj = 0; jj < JJ; ++jj) {
                const float bv = kk == 0 ? b[jj].x : b[jj].y;
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[r][jj] = __ffma2_rn(a[r], make_float2(bv, bv), acc[r][jj]);
            }
        }
    }
}

template <int BN, int JJ>
__global__ void __launch_bounds__(FfmaCfg<BN, JJ>::THREADS, FfmaCfg<BN, JJ>::CTAS_PER_SM)
    ffma_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
    if (PG_PDL_EARLY && threadIdx.x == 0) pdl_trigger();
    using Cfg = FfmaCfg<BN, JJ>;
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem_1024(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::STAGE_BYTES);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * S);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + S);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Block -> (tile, K slice).  With the last-wave split, blocks from tail_first
    // on take the last partial wave's tiles, tail_split K slices each.
    int tile = blockIdx.x, slice = blockIdx.y, kb0, nkb;
    const bool tail = p.tail_split > 1 && tile >= p.tail_first;
    if (tail) {
        const int v = tile - p.tail_first;
        tile = p.tail_first + v / p.tail_split;
        slice = v % p.tail_split;
        kb0 = slice * p.tail_kb;
        nkb = min(kb0 + p.tail_kb, p.kb_total) - kb0;
    } else {
        kb0 = slice * p.kb_per_split;
        nkb = min(kb0 + p.kb_per_split, p.kb_total) - kb0;
    }
    int tile_m, tile_n;
    tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, tile_m, tile_n);
    const int64_t m0 = static_cast<int64_t>(tile_m) * Cfg::BM;
    const int64_t n0 = static_cast<int64_t>(tile_n) * BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, Cfg::CWARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();  // launched right after an operand pass: its output, before any copy

    // Thread 0 is also the loader: it issues k-block `it` into slot it % S once
    // every warp has released that slot's previous contents (k-block it - S).
    const bool loader = (threadIdx.x == 0) && !(p.debug_flags & 1);
    int issued = 0;
    auto issue = [&](int it) -> bool {
        const int s = it % S;
        if (!mbar_wait_bounded(empty0 + 8 * s, ((it / S) & 1) ^ 1, p.timeout_ns, abort_flag)) {
            raise_abort(abort_flag, p.status);
            return false;
        }
        const uint32_t full = full0 + 8 * s;
        mbar_arrive_expect_tx(full, Cfg::STAGE_BYTES);
        const int32_t kc = (kb0 + it) * Cfg::BK;
        const uint32_t slot = smem_u32(smem + s * Cfg::STAGE_BYTES);
        tma_load_2d(slot, &tmA, static_cast<int32_t>(m0), kc, full);
        tma_load_2d(slot + Cfg::A_BYTES, &tmB, kc, static_cast<int32_t>(n0), full);
        issued = it + 1;
        return true;
    };
    if (loader) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        for (int it = 0; it < min(Cfg::PD, nkb); ++it)
            if (!issue(it)) break;
    }

    // ---------------- consumers ----------------
    const int wm = warp & 3;
    const int wn = warp >> 2;
    const int tm = 4 * wm + (lane >> 3);   // 0..15
    const int tn = 8 * wn + (lane & 7);    // 0..TGN-1
    const uint32_t bchunk_xor = static_cast<uint32_t>(tn & 7);

    // acc[r][jj] holds rows (2r, 2r+1) of the thread's 8 rows {4tm..4tm+3, 64+4tm..64+4tm+3}
    // in column jj, as a register pair (the operand shape of the packed FP32 FMA).
    float2 acc[4][JJ];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int j = 0; j < JJ; ++j) acc[r][j] = make_float2(0.0f, 0.0f);

    bool ok = true;
    for (int it = 0; it < nkb; ++it) {
        const int s = it % S;
        const uint32_t ph = (it / S) & 1;
        if (loader && issued == it + Cfg::PD && issued < nkb && !*abort_flag) issue(issued);
        // Every lane waits, then the warp agrees on the outcome so that a lane whose
        // limit expired a moment earlier cannot leave the others at __syncwarp.
        const bool landed = PG_FFMA_WARP_WAIT
                                 ? mbar_wait_warp(full0 + 8 * s, ph, p.timeout_ns, abort_flag)
                                 : __all_sync(0xffffffffu, mbar_wait_bounded(full0 + 8 * s, ph, p.timeout_ns,
                                                                              abort_flag));
        if (!landed) {
            if (lane == 0) raise_abort(abort_flag, p.status);
            ok = false;
            break;
        }
        const float* As = reinterpret_cast<const float*>(smem + s * Cfg::STAGE_BYTES);
        const uint8_t* Bs = smem + s * Cfg::STAGE_BYTES + Cfg::A_BYTES + tn * 128;
#pragma unroll
        for (int g2 = 0; g2 < Cfg::BK / 2; ++g2) {
            float2 b[JJ];
            const uint32_t off2 = (((static_cast<uint32_t>(g2 >> 1)) ^ bchunk_xor) << 4) + ((g2 & 1) << 3);
#pragma unroll
            for (int jj = 0; jj < JJ; ++jj)
                b[jj] = *reinterpret_cast<const float2*>(Bs + jj * (Cfg::TGN * 128) + off2);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const float* arow = As + (2 * g2 + kk) * Cfg::BM;
                const float4 a0 = *reinterpret_cast<const float4*>(arow + 4 * tm);
                const float4 a1 = *reinterpret_cast<const float4*>(arow + 64 + 4 * tm);
                const float2 a[4] = {make_float2(a0.x, a0.y), make_float2(a0.z, a0.w), make_float2(a1.x, a1.y),
                                     make_float2(a1.z, a1.w)};
#pragma unroll
                for (int jj = 0; jj < JJ; ++jj) {
                    const float bv = kk == 0 ? b[jj].x : b[jj].y;
#pragma unroll
                    for (int r = 0; r < 4; ++r) acc[r][jj] = __ffma2_rn(a[r], make_float2(bv, bv), acc[r][jj]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
    }
    // the main loop is done: a dependent reduction may be scheduled now
    if (!PG_PDL_EARLY && threadIdx.x == 0) pdl_trigger();
    if (loader) {
        // The last (up to S) slots issued may still be landing after an abort; do
        // not let the CTA retire while a copy into its shared memory is in flight.
        for (int it = max(0, issued - S); it < issued; ++it)
            mbar_wait_bounded(full0 + 8 * (it % S), (it / S) & 1, p.timeout_ns, nullptr);
    }
    if (!tail) {
        // No warp has returned (a failed wait only leaves the k loop), so all of
        // them meet here; past this barrier no warp reads the ring any more.
        __syncthreads();
        if (!ok || *abort_flag) return;
        if (p.c_tma)
            ffma_epilogue_tma<BN, JJ>(acc, smem, tm, tn, m0, n0, &tmC, p);
        else
            ffma_epilogue_staged<BN, JJ>(acc, smem, warp, lane, tm, tn, m0, n0, slice, p);
        return;
    }
    if (!ok || *abort_flag) return;

    // ---------------- last-wave fix-up ----------------
    // A tail slice stores its partial block ([column][row], BM x BN floats), and
    // each warp counts itself in for the outputs it holds (a warp of every slice
    // holds the same ones); the warp that arrives last adds the blocks in slice
    // order (0, 1, ...: the same association whichever slice is last, so the
    // result is deterministic) and runs the epilogue below on the sum.  No
    // block-wide barrier: a warp that gave up on a wait has already returned.
    if (tail) {
        const int tt = tile - p.tail_first;
        float* part0 = p.tail_P + static_cast<int64_t>(tt) * p.tail_split * (Cfg::BM * BN);
#pragma unroll
        for (int jj = 0; jj < JJ; ++jj)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float* d = part0 + static_cast<int64_t>(slice) * (Cfg::BM * BN) + (tn + Cfg::TGN * jj) * Cfg::BM +
                           64 * h + 4 * tm;
                *reinterpret_cast<float4*>(d) =
                    make_float4(acc[2 * h][jj].x, acc[2 * h][jj].y, acc[2 * h + 1][jj].x, acc[2 * h + 1][jj].y);
            }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(p.tail_cnt + tt * Cfg::CWARPS + warp, 1) == p.tail_split - 1;
        if (!__shfl_sync(0xffffffffu, last, 0)) return;
        __threadfence();
        // All slices' blocks, this one's included, are read back from L2 (the
        // thread's own stores are ordered before its loads), so the accumulators
        // need not stay live beside the sums.
#pragma unroll
        for (int jj = 0; jj < JJ; ++jj)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float* src = part0 + (tn + Cfg::TGN * jj) * Cfg::BM + 64 * h + 4 * tm;
                float4 sum = __ldcg(reinterpret_cast<const float4*>(src));
                for (int sl = 1; sl < p.tail_split; ++sl) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(src + sl * (Cfg::BM * BN)));
                    sum.x += v.x;
                    sum.y += v.y;
                    sum.z += v.z;
                    sum.w += v.w;
                }
                acc[2 * h][jj] = make_float2(sum.x, sum.y);
                acc[2 * h + 1][jj] = make_float2(sum.z, sum.w);
            }
    }

    // ---------------- epilogue ----------------
    // C is read ahead of the stores, G columns of the thread's tile at a time:
    // interleaved with the stores, each load would wait for the previous store
    // (the compiler cannot rule out that they alias) at full DRAM latency.
    const float alpha = p.alpha, beta = p.beta;
    const bool read_c = p.split == 1 && beta != 0.0f;
    constexpr int G = JJ < 4 ? JJ : 4;
#pragma unroll
    for (int j0 = 0; j0 < JJ; j0 += G) {
        float4 cfr[G][2];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int64_t j = n0 + tn + Cfg::TGN * (j0 + g);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t i = m0 + 64 * h + 4 * tm;
                const float* src = p.C + j * p.ldc + i;
                float4 c = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (read_c && j < p.n && i < p.m) {
                    if (p.c_vec && i + 3 < p.m) {
                        c = *reinterpret_cast<const float4*>(src);
                    } else {
                        c.x = src[0];
                        if (i + 1 < p.m) c.y = src[1];
                        if (i + 2 < p.m) c.z = src[2];
                        if (i + 3 < p.m) c.w = src[3];
                    }
                }
                cfr[g][h] = c;
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int jj = j0 + g;
            const int64_t j = n0 + tn + Cfg::TGN * jj;
            if (j >= p.n) continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t i = m0 + 64 * h + 4 * tm;
                if (i >= p.m) continue;
                const float v[4] = {acc[2 * h][jj].x, acc[2 * h][jj].y, acc[2 * h + 1][jj].x, acc[2 * h + 1][jj].y};
                if (p.split > 1) {
                    float* dst = p.P + slice * p.p_stride + j * p.ldp + i;
                    if (i + 3 < p.m) {
                        *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
                    } else {
                        for (int e = 0; e < 4; ++e)
                            if (i + e < p.m) dst[e] = v[e];
                    }
                } else {
                    float* dst = p.C + j * p.ldc + i;
                    const float4 c = cfr[g][h];
                    float4 o = make_float4(alpha * v[0], alpha * v[1], alpha * v[2], alpha * v[3]);
                    if (read_c) {
                        o.x = fmaf(beta, c.x, o.x);
                        o.y = fmaf(beta, c.y, o.y);
                        o.z = fmaf(beta, c.z, o.z);
                        o.w = fmaf(beta, c.w, o.w);
                    }
                    if (p.c_vec && i + 3 < p.m) {
                        *reinterpret_cast<float4*>(dst) = o;
                    } else {
                        dst[0] = o.x;
                        if (i + 1 < p.m) dst[1] = o.y;
                        if (i + 2 < p.m) dst[2] = o.z;
                        if (i + 3 < p.m) dst[3] = o.w;
                    }
                }
            }
        }
    }
}

// ---------------- stream-K ----------------
//
// For products whose tiles fill less than one wave of CTA slots (the pages'
// "tail" share of the gap, "V3. Vectorized and double buffer", section 4),
// every one of G co-resident CTAs takes the same share of all (tile, k-block)
// iterations: CTA c runs the contiguous range [c T / G, (c + 1) T / G) of the
// T = tiles x k-blocks iterations in tile-major order, crossing tile boundaries.
// Its loader streams the whole range through the ring without a break; at the
// end of each tile segment the consumers store the segment's accumulators as
// a raw 128 x BN partial block and start the next segment from zero.  Segment j
// of tile t (the j-th CTA touching t) goes to slot t * maxseg + j.  A second
// kernel then adds each tile's partial blocks in segment order -- increasing k,
// whichever CTA finished first, so the result is deterministic -- and applies
// alpha and beta.

// At most this many tile segments per CTA (the planner keeps to it).
constexpr int kSkMaxSegs = 8;

template <int BN, int JJ>
__global__ void __launch_bounds__(FfmaCfg<BN, JJ>::THREADS, FfmaCfg<BN, JJ>::CTAS_PER_SM)
    ffma_sk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmParams p) {
    if (PG_PDL_EARLY && threadIdx.x == 0) pdl_trigger();
    using Cfg = FfmaCfg<BN, JJ>;
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem_1024(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::STAGE_BYTES);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * S);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + S);
    // This CTA's tile segments, built once by thread 0: tile, partial-block slot
    // (t * maxseg + j), k-blocks, first k-block, and the tile's origin in C.
    __shared__ int seg_slot[kSkMaxSegs], seg_len[kSkMaxSegs], seg_k0[kSkMaxSegs], seg_m0[kSkMaxSegs],
        seg_n0[kSkMaxSegs];
    __shared__ int n_segs, n_its, ld_seg, ld_kb;  // ld_*: the loader's position (thread 0 only)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, Cfg::CWARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
        const int G = gridDim.x, c = blockIdx.x;
        const int64_t T = p.sk_iters;
        const int kb = p.kb_total;
        const int64_t it0 = static_cast<int64_t>(c) * T / G, it1 = static_cast<int64_t>(c + 1) * T / G;
        int ns = 0;
        for (int64_t it = it0; it < it1 && ns < kSkMaxSegs; ++ns) {
            const int tile = static_cast<int>(it / kb);
            const int k0 = static_cast<int>(it - static_cast<int64_t>(tile) * kb);
            const int len = static_cast<int>(min(static_cast<int64_t>(kb - k0), it1 - it));
            int tm_, tn_;
            tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, tm_, tn_);
            seg_slot[ns] = tile * p.sk_maxseg + (c - sk_cta_of(static_cast<int64_t>(tile) * kb, G, T));
            seg_len[ns] = len;
            seg_k0[ns] = k0;
            seg_m0[ns] = tm_ * Cfg::BM;
            seg_n0[ns] = tn_ * BN;
            it += len;
        }
        n_segs = ns;
        n_its = static_cast<int>(it1 - it0);
        // The planner keeps every CTA within kSkMaxSegs segments; were the range
        // longer, this CTA would leave part of it undone: report a failure
        // instead of a wrong C.
        int64_t covered = 0;
        for (int q = 0; q < ns; ++q) covered += seg_len[q];
        if (covered != it1 - it0) {
            n_its = 0;
            raise_abort(abort_flag, p.status);
        }
        ld_seg = 0;
        ld_kb = 0;
    }
    __syncthreads();
    pdl_wait();  // launched right after an operand pass: its output, before any copy
    const int n_it = n_its;

    // Thread 0 is also the loader, PD k-blocks ahead of the consumers.
    const bool loader = (threadIdx.x == 0) && !(p.debug_flags & 1);
    int issued = 0;
    auto issue = [&](int g) -> bool {
        const int s = g % S;
        if (!mbar_wait_bounded(empty0 + 8 * s, ((g / S) & 1) ^ 1, p.timeout_ns, abort_flag)) {
            raise_abort(abort_flag, p.status);
            return false;
        }
        const int sg = ld_seg, kq = ld_kb;
        const uint32_t full = full0 + 8 * s;
        mbar_arrive_expect_tx(full, Cfg::STAGE_BYTES);
        const int32_t kc = (seg_k0[sg] + kq) * Cfg::BK;
        const uint32_t slot = smem_u32(smem + s * Cfg::STAGE_BYTES);
        tma_load_2d(slot, &tmA, seg_m0[sg], kc, full);
        tma_load_2d(slot + Cfg::A_BYTES, &tmB, kc, seg_n0[sg], full);
        if (kq + 1 == seg_len[sg]) {
            ld_seg = sg + 1;
            ld_kb = 0;
        } else {
            ld_kb = kq + 1;
        }
        issued = g + 1;
        return true;
    };
    if (loader) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        for (int g = 0; g < min(Cfg::PD, n_it); ++g)
            if (!issue(g)) break;
    }

    const int wm = warp & 3;
    const int wn = warp >> 2;
    const int tm = 4 * wm + (lane >> 3);
    const int tn = 8 * wn + (lane & 7);
    const uint32_t bchunk_xor = static_cast<uint32_t>(tn & 7);
    float2 acc[4][JJ];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int j = 0; j < JJ; ++j) acc[r][j] = make_float2(0.0f, 0.0f);

    int seg = 0, left = seg_len[0];  // the segment being computed and its k-blocks still to come
    for (int g = 0; g < n_it; ++g) {
        const int s = g % S;
        if (loader && issued == g + Cfg::PD && issued < n_it && !*abort_flag) issue(issued);
        const bool landed = PG_FFMA_WARP_WAIT
                                 ? mbar_wait_warp(full0 + 8 * s, (g / S) & 1, p.timeout_ns, abort_flag)
                                 : __all_sync(0xffffffffu, mbar_wait_bounded(full0 + 8 * s, (g / S) & 1,
                                                                              p.timeout_ns, abort_flag));
        if (!landed) {
            if (lane == 0) raise_abort(abort_flag, p.status);
            break;
        }
        ffma_kblock<BN, JJ>(acc, smem + s * Cfg::STAGE_BYTES, tm, tn, bchunk_xor);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        if (--left == 0) {  // the segment's last k-block: store its partial block, start the next from zero
            float* part = p.sk_P + static_cast<int64_t>(seg_slot[seg]) * (Cfg::BM * BN) + 4 * tm;
#pragma unroll
            for (int jj = 0; jj < JJ; ++jj)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    *reinterpret_cast<float4*>(part + (tn + Cfg::TGN * jj) * Cfg::BM + 64 * h) =
                        make_float4(acc[2 * h][jj].x, acc[2 * h][jj].y, acc[2 * h + 1][jj].x, acc[2 * h + 1][jj].y);
                    acc[2 * h][jj] = make_float2(0.0f, 0.0f);
                    acc[2 * h + 1][jj] = make_float2(0.0f, 0.0f);
                }
            if (++seg < n_segs) left = seg_len[seg];
        }
    }
    // the main loop is done: the fix-up may be scheduled now
    if (!PG_PDL_EARLY && threadIdx.x == 0) pdl_trigger();
    if (loader) {
        for (int g = max(0, issued - S); g < issued; ++g)
            mbar_wait_bounded(full0 + 8 * (g % S), (g / S) & 1, p.timeout_ns, nullptr);
    }
}

template <int BN, int JJ>
cudaError_t launch_sk_impl(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int ctas,
                           int num_sms, cudaStream_t stream) {
    using Cfg = FfmaCfg<BN, JJ>;
    auto kern = ffma_sk_kernel<BN, JJ>;
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = set_smem_limit_once(smem_set, reinterpret_cast<const void*>(kern), static_cast<int>(Cfg::SMEM));
    if (e != cudaSuccess) return e;
    if ((e = launch_kernel(p.after_prep != 0, kern, dim3(ctas), dim3(Cfg::THREADS), Cfg::SMEM, stream, tmA, tmB, p)) !=
        cudaSuccess)
        return e;
    return launch_streamk_fixup(p, BN, ctas, num_sms, stream);
}

template <int BN, int JJ>
cudaError_t launch_impl(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, const GemmParams& p,
                        dim3 grid, cudaStream_t stream) {
    using Cfg = FfmaCfg<BN, JJ>;
    auto kern = ffma_gemm_kernel<BN, JJ>;
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = set_smem_limit_once(smem_set, reinterpret_cast<const void*>(kern), static_cast<int>(Cfg::SMEM));
    if (e != cudaSuccess) return e;
    return launch_kernel(p.after_prep != 0, kern, grid, dim3(Cfg::THREADS), Cfg::SMEM, stream, tmA, tmB, tmC, p);
}

using Cfg64 = FfmaCfg<64, 8>;
using Cfg128 = FfmaCfg<128, PG_FFMA_JJ128>;
using Cfg256 = FfmaCfg<256, 8>;

}  // namespace

int ffma_threads(int bn) { return bn == 64 ? Cfg64::THREADS : bn == 128 ? Cfg128::THREADS : Cfg256::THREADS; }
int ffma_stages(int bn) { return bn == 64 ? Cfg64::STAGES : bn == 128 ? Cfg128::STAGES : Cfg256::STAGES; }
int ffma_ctas_per_sm(int bn) {
    return bn == 64 ? Cfg64::CTAS_PER_SM : bn == 128 ? Cfg128::CTAS_PER_SM : Cfg256::CTAS_PER_SM;
}
size_t ffma_smem_bytes(int bn) { return bn == 64 ? Cfg64::SMEM : bn == 128 ? Cfg128::SMEM : Cfg256::SMEM; }

cudaError_t launch_ffma_sk(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmParams& p, int bn, int ctas,
                           int num_sms, cudaStream_t stream) {
    switch (bn) {
        case 64: return launch_sk_impl<64, 8>(tmA, tmB, p, ctas, num_sms, stream);
        case 128: return launch_sk_impl<128, PG_FFMA_JJ128>(tmA, tmB, p, ctas, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_ffma(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, const GemmParams& p,
                        int bn, dim3 grid, cudaStream_t stream) {
    switch (bn) {
        case 64: return launch_impl<64, 8>(tmA, tmB, tmC, p, grid, stream);
        case 128: return launch_impl<128, PG_FFMA_JJ128>(tmA, tmB, tmC, p, grid, stream);
        case 256: return launch_impl<256, 8>(tmA, tmB, tmC, p, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pg
