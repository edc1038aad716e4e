// Tensor-core GEMM on SM pairs (tcgen05 cta_group::2, sm_103a): TF32 and 3xTF32.
//
// A cluster of two CTAs on two SMs computes a 256 x BN tile of C per work unit:
// CTA r of the pair stages rows [128r, 128r + 128) of the A tile and columns
// [r*BN/2, (r+1)*BN/2) of the B tile, and one thread of CTA 0 issues
// tcgen05.mma.cta_group::2 (M = 256, N = BN, K = 8), which reads both CTAs'
// shared memory and leaves rows 128r.. of the product in CTA r's tensor memory.
// Each SM therefore stages 128 + BN/2 operand rows per k-step instead of
// 128 + BN, which is what bounds the single-SM kernel (its operand feed, not the
// tensor pipe, is the limit measured with ncu).
//
// The kernel is persistent: each pair walks work units (tile, K slice) with a
// static stride, and the accumulator is double-buffered in TMEM (2 x BN columns)
// so the epilogue of one unit overlaps the MMAs of the next.  When the tiles fill
// whole waves of pairs plus a partial last wave, the last wave's tiles are cut
// into K slices that occupy the otherwise idle pairs; each slice leaves a
// partial block in global memory and the last slice of a region to finish adds
// them in slice order (deterministic) and writes C.
//
// Warp roles, in both CTAs of the pair (320 threads each):
//   warp 0      TMA loader: this CTA's A rows and B columns for every k-block,
//               completing on CTA 0's "full" barrier of the ring slot
//   warp 1      TMEM allocation (pair-wide); in CTA 0 one thread issues the MMAs
//   warps 2-9   epilogue: TMEM -> registers -> alpha/beta -> C rows of this CTA;
//               a warp may read only TMEM lane quarter (warp % 4), so two warps
//               share each quarter and take alternate 32-column chunks (with one
//               warp per quarter the epilogue is issue-bound when K is short)
// Barriers: full[s] (CTA 0: expect-tx for both CTAs' bytes), empty[s] (both CTAs;
// the MMA completion is multicast), acc_full[b] (both CTAs; multicast),
// acc_empty[b] (CTA 0; arrived by the 16 epilogue warps of the pair).
//
// 3xTF32: A and B arrive split by a pre-pass into TF32 "big" parts and exact
// remainders (four tensor maps); each ring slot holds all four tiles at BK 16 and
// the MMA thread issues small*big, big*small, big*big per k-step.  (Splitting in
// shared memory instead, as the single-SM kernel does for its narrow shapes,
// measured 2.3x slower here: the transform's latency joins every slot's round trip.)
//
// Shared-memory layouts are those of the single-SM kernel (tc_kernel.cu): A
// M-major in the 128-byte swizzle with 32-byte atoms, B K-major in the 128-byte
// (BK 32) or 64-byte (BK 16) swizzle.  In the pair the descriptors name
// offsets that are valid in both CTAs (the slots sit at the same offsets).
//
// Every wait is bounded.  After an expired wait a CTA raises its abort flag and
// the status word, lets the MMAs it issued finish (bounded), and meets its peer
// at the final cluster barrier before TMEM is released; a peer whose waits
// then expire in turn leaves the same way.
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace pg {
namespace {

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

// Arrive on a barrier of another CTA of the cluster, without release semantics:
// for signals that publish no memory writes.  The epilogue frees a TMEM
// accumulator buffer with it once tcgen05.wait::ld has returned (the buffer is
// no longer read); a release arrive would first wait for all of the warp's
// outstanding stores of C to be performed.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA tile load into this CTA's shared memory that completes on the mbarrier at
// `bar_cluster` (CTA 0 of the pair).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at offset `bar` in both CTAs of the pair once the MMAs
// issued so far have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(static_cast<uint16_t>(3))
        : "memory");
}

// Arrive on this CTA's barrier `bar` once the MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_pair_local(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

template <int BN, bool SPLIT3>
struct Tc2Cfg {
    static constexpr int BM = kBM;               // rows per CTA (256 per pair)
// Shared-memory budget of the operand ring (a compile-time tunable; one more slot
// than the default measured no faster: the feed rate, not latency, bounds TF32).
#ifndef PG_TC2_RING_BYTES
#define PG_TC2_RING_BYTES (200 * 1024)
#endif
    static constexpr int BK = SPLIT3 ? 16 : 32;
    static constexpr int OPS = SPLIT3 ? 2 : 1;
    static constexpr int BNH = BN / 2;           // B columns staged per CTA
    static constexpr int A_BYTES = BM * BK * 4;
    static constexpr int B_BYTES = BNH * BK * 4;
    static constexpr int A_BOX_BYTES = 32 * BK * 4;
    static constexpr int STAGE_BYTES = OPS * (A_BYTES + B_BYTES);
    static constexpr int STAGES_RAW = (PG_TC2_RING_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 16 ? 16 : STAGES_RAW;
// Epilogue warps (a compile-time tunable: 4 or 8).
#ifndef PG_TC2_EPI_WARPS
#define PG_TC2_EPI_WARPS 8
#endif
    static constexpr int EPI_WARPS = PG_TC2_EPI_WARPS;
    static_assert(EPI_WARPS == 4 || EPI_WARPS == 8, "epilogue warps");
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int BAR_BYTES = (2 * STAGES + 5) * 8 + 16;
    static constexpr size_t SMEM = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + BAR_BYTES;
    // Accumulator buffers in TMEM: two (epilogue of one unit overlaps the MMAs of
    // the next) up to BN = 256; the 512-wide tile takes all 512 columns, one buffer.
    static constexpr int NBUF = BN == 512 ? 1 : 2;
    static constexpr uint32_t TMEM_COLS = NBUF * BN;
    // MMAs per k-step: one of N = BN, or two of N = 256 for the 512-wide tile (each
    // CTA then stages its B columns as two halves of 128, one per MMA)
    static constexpr int NMMA = BN == 512 ? 2 : 1;
    static constexpr int MMA_N = BN / NMMA;
    static_assert(BN == 128 || BN == 256 || (BN == 512 && !SPLIT3), "BN");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "slots need 1 KiB alignment");
    static_assert(STAGES >= 3, "ring too shallow");
};

template <int BN, bool SPLIT3>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Tc2Cfg<BN, SPLIT3>::THREADS, 1)
    tc2_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAs,
                    const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmBs,
                    const GemmParams p) {
    if (PG_PDL_EARLY && threadIdx.x == 0) pdl_trigger();
    using Cfg = Tc2Cfg<BN, SPLIT3>;
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem_1024(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::STAGE_BYTES);
    // [0,S) full, [S,2S) empty, 2S..2S+1 acc_full, 2S+2..2S+3 acc_empty, 2S+4 mma_done
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + S);
    const uint32_t acc_full0 = smem_u32(bars + 2 * S);
    const uint32_t acc_empty0 = smem_u32(bars + 2 * S + 2);
    const uint32_t mma_done = smem_u32(bars + 2 * S + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1;
    const int pairs = gridDim.x >> 1;
    const int tiles = p.tiles_m * p.tiles_n;
    const bool tail_on = p.tail_split > 1;
    const int units = tail_on ? p.tail_first + (tiles - p.tail_first) * p.tail_split : tiles * p.split;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full0 + 8 * b, 1);
            mbar_init(acc_empty0 + 8 * b, 2 * Cfg::EPI_WARPS);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(Cfg::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers and TMEM exist before any cross-CTA traffic
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    pdl_wait();  // launched right after an operand pass: its output, before any copy

    // Work unit -> (pair tile t, K slice, k-block range).
    auto unit_geometry = [&](int u, int64_t& m0, int64_t& n0, int& slice, int& kb0, int& nkb, int& t) {
        if (tail_on) {
            if (u < p.tail_first) {
                t = u;
                slice = 0;
                kb0 = 0;
                nkb = p.kb_total;
            } else {
                const int v = u - p.tail_first;
                t = p.tail_first + v / p.tail_split;
                slice = v % p.tail_split;
                kb0 = slice * p.tail_kb;
                nkb = min(kb0 + p.tail_kb, p.kb_total) - kb0;
            }
        } else {
            t = u % tiles;
            slice = u / tiles;
            kb0 = slice * p.kb_per_split;
            nkb = min(kb0 + p.kb_per_split, p.kb_total) - kb0;
        }
        int tm, tn;
        tile_coords(t, p.tiles_m, p.tiles_n, p.group_m, tm, tn);
        m0 = static_cast<int64_t>(tm) * (2 * Cfg::BM);
        n0 = static_cast<int64_t>(tn) * BN;
    };

    if (warp == 0) {
        // ---------------- TMA loader (both CTAs) ----------------
        if (lane == 0 && !(p.debug_flags & 1)) {
            prefetch_tmap(&tmA);
            prefetch_tmap(&tmB);
            if (SPLIT3) {
                prefetch_tmap(&tmAs);
                prefetch_tmap(&tmBs);
            }
            const uint32_t full_leader0 = map_to_rank(full0, 0);
            int it = 0;
            bool ok = true;
            for (int u = pair; u < units && ok; u += pairs) {
                int64_t m0, n0;
                int slice, kb0, nkb, t;
                unit_geometry(u, m0, n0, slice, kb0, nkb, t);
                const int32_t ma = static_cast<int32_t>(m0 + Cfg::BM * rank);
                const int32_t nb = static_cast<int32_t>(n0 + Cfg::BNH * rank);
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = it % S;
                    if (!mbar_wait_bounded(empty0 + 8 * s, ((it / S) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                        raise_abort(abort_flag, p.status);
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(full0 + 8 * s, 2 * Cfg::STAGE_BYTES);
                    const uint32_t bar = full_leader0 + 8 * s;
                    const int32_t kc = (kb0 + kb) * Cfg::BK;
                    const uint32_t slot = smem_u32(smem + s * Cfg::STAGE_BYTES);
                    // A K-major (transa 'T'): one box of 128 rows x BK.  A M-major: one 3-D
                    // box {32 rows, BK, 4 row groups} when m % 32 == 0, else four 2-D boxes
                    // of 32 rows (both land as 4 x [BK][32] row groups).  B K-major: one box
                    // of BN/2 columns; B N-major (transb 'T'): BN/64 groups of 32 columns.
                    auto load_a = [&](uint32_t dst, const CUtensorMap* map) {
                        if (p.a_kmajor) {
                            tma_load_2d_pair(dst, map, kc, ma, bar);
                        } else if (p.a3d) {
                            tma_load_3d_pair(dst, map, 0, kc, ma / 32, bar);
                        } else {
#pragma unroll
                            for (int g = 0; g < 4; ++g)
                                tma_load_2d_pair(dst + g * Cfg::A_BOX_BYTES, map, ma + 32 * g, kc, bar);
                        }
                    };
                    auto load_b = [&](uint32_t dst, const CUtensorMap* map) {
                        if (Cfg::NMMA == 2) {
                            // two halves of 128 columns: n0 + 256 j + 128 rank + [0, 128)
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const int32_t nj = static_cast<int32_t>(n0) + 256 * j + 128 * static_cast<int32_t>(rank);
                                const uint32_t dj = dst + j * (Cfg::B_BYTES / 2);
                                if (!p.b_mnmajor) {
                                    tma_load_2d_pair(dj, map, kc, nj, bar);
                                } else if (p.b3d) {
                                    tma_load_3d_pair(dj, map, 0, kc, nj / 32, bar);
                                } else {
#pragma unroll
                                    for (int g = 0; g < 4; ++g)
                                        tma_load_2d_pair(dj + g * Cfg::A_BOX_BYTES, map, nj + 32 * g, kc, bar);
                                }
                            }
                        } else if (!p.b_mnmajor) {
                            tma_load_2d_pair(dst, map, kc, nb, bar);
                        } else if (p.b3d) {
                            tma_load_3d_pair(dst, map, 0, kc, nb / 32, bar);
                        } else {
#pragma unroll
                            for (int g = 0; g < Cfg::BNH / 32; ++g)
                                tma_load_2d_pair(dst + g * Cfg::A_BOX_BYTES, map, nb + 32 * g, kc, bar);
                        }
                    };
                    load_a(slot, &tmA);
                    uint32_t b_slot = slot + Cfg::A_BYTES;
                    if (SPLIT3) {
                        load_a(slot + Cfg::A_BYTES, &tmAs);
                        b_slot = slot + 2 * Cfg::A_BYTES;
                        load_b(b_slot + Cfg::B_BYTES, &tmBs);
                    }
                    load_b(b_slot, &tmB);
                }
            }
            // every copy of the main loop is issued: a dependent reduction may be
            // scheduled now
            if (!PG_PDL_EARLY) pdl_trigger();
            if (leader) {
                // Let every copy of the pair land before the CTAs may retire (CTA 0's
                // full barriers count both CTAs' bytes).
                for (int j = max(0, it - S); j < it; ++j)
                    mbar_wait_bounded(full0 + 8 * (j % S), (j / S) & 1, p.timeout_ns, nullptr);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer (CTA 0 of the pair) ----------------
        if (leader && lane == 0) {
            int lu = 0;
            bool ok = true;
            const uint32_t idesc = idesc_tf32(2 * Cfg::BM, Cfg::MMA_N, !p.a_kmajor, p.b_mnmajor != 0);
            // Descriptors of slot 0's tiles, built once; a slot and a k-step only move
            // the start address field (bits 0-13, in 16-byte units; shared addresses
            // stay below 256 KiB, so the field does not overflow).
            const bool a_k = p.a_kmajor != 0, b_k = p.b_mnmajor == 0;
            const uint32_t slot0 = smem_u32(smem);
            const uint64_t a_desc0 = operand_desc<Cfg::BK>(slot0, 0, a_k);
            const uint64_t as_desc0 = operand_desc<Cfg::BK>(slot0 + Cfg::A_BYTES, 0, a_k);
            const uint64_t b_desc0 = operand_desc<Cfg::BK>(slot0 + Cfg::OPS * Cfg::A_BYTES, 0, b_k);
            const uint64_t bs_desc0 = operand_desc<Cfg::BK>(slot0 + Cfg::OPS * Cfg::A_BYTES + Cfg::B_BYTES, 0, b_k);
            const uint32_t a_kstep = a_k ? 2 : 64, b_kstep = b_k ? 2 : 64;  // 32 B or 1 KiB per k-step
            int s = 0;  // ring slot
            uint32_t phase = 0;
            for (int u = pair; u < units && ok; u += pairs, ++lu) {
                int64_t m0, n0;
                int slice, kb0, nkb, t;
                unit_geometry(u, m0, n0, slice, kb0, nkb, t);
                const int buf = lu % Cfg::NBUF;
                if (!mbar_wait_bounded(acc_empty0 + 8 * buf, ((lu / Cfg::NBUF) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                    raise_abort(abort_flag, p.status);
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d = tmem + buf * BN;
                uint32_t accumulate = 0;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait_bounded(full0 + 8 * s, phase, p.timeout_ns, abort_flag)) {
                        raise_abort(abort_flag, p.status);
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t off = static_cast<uint32_t>(s * Cfg::STAGE_BYTES) >> 4;
#pragma unroll
                    for (int kk = 0; kk < Cfg::BK / 8; ++kk) {
                        const uint64_t ad = a_desc0 + (off + kk * a_kstep);
                        const uint64_t bd = b_desc0 + (off + kk * b_kstep);
                        if (SPLIT3) {
                            const uint64_t asd = as_desc0 + (off + kk * a_kstep);
                            const uint64_t bsd = bs_desc0 + (off + kk * b_kstep);
                            mma_tf32_pair(d, asd, bd, idesc, accumulate);
                            accumulate = 1;
                            mma_tf32_pair(d, ad, bsd, idesc, 1);
                            mma_tf32_pair(d, ad, bd, idesc, 1);
                        } else {
#pragma unroll
                            for (int j = 0; j < Cfg::NMMA; ++j)  // B half j: 128 rows = 16 KiB further
                                mma_tf32_pair(d + j * Cfg::MMA_N, ad, bd + j * 1024, idesc, accumulate);
                            accumulate = 1;
                        }
                    }
                    mma_commit_pair(empty0 + 8 * s);  // both CTAs' slot s reusable after these MMAs
                    if (++s == S) {
                        s = 0;
                        phase ^= 1;
                    }
                }
                if (ok) mma_commit_pair(acc_full0 + 8 * buf);  // unit's accumulator complete
            }
            mma_commit_pair_local(mma_done);  // every MMA issued here has completed
            mbar_wait_bounded(mma_done, 0, p.timeout_ns, nullptr);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..9, both CTAs) ----------------
        const int q = warp & 3;            // TMEM lane quarter this warp may access
        constexpr int kGroups = Cfg::EPI_WARPS / 4;  // warps sharing a lane quarter
        const int half = (warp - 2) >> 2;            // which of their 32-column chunks it takes
        const uint32_t acc_empty_leader0 = map_to_rank(acc_empty0, 0);
        const float alpha = p.alpha, beta = p.beta;
        int lu = 0;
        for (int u = pair; u < units; u += pairs, ++lu) {
            int64_t m0, n0;
            int slice, kb0, nkb, tile;
            unit_geometry(u, m0, n0, slice, kb0, nkb, tile);
            const bool tail = tail_on && tile >= p.tail_first;
            const int64_t i_loc = Cfg::BM * rank + 32 * q + lane;  // row inside the 256-row tile
            // this slice's partial block of a last-wave tile: [column][row], 256 rows
            float* tpart = tail ? p.tail_P + (static_cast<int64_t>(tile - p.tail_first) * p.tail_split + slice) *
                                                 (2 * Cfg::BM) * BN
                                : nullptr;
            const int buf = lu % Cfg::NBUF;
            const bool ready = __all_sync(
                0xffffffffu, mbar_wait_bounded(acc_full0 + 8 * buf, (lu / Cfg::NBUF) & 1, p.timeout_ns, abort_flag));
            if (!ready) {
                if (lane == 0) raise_abort(abort_flag, p.status);
                break;
            }
            tc_fence_after_sync();
            const int64_t i = m0 + Cfg::BM * rank + 32 * q + lane;
            const bool row_ok = i < p.m;
            // all 32 rows of this warp inside C: chunks that are also whole in n take
            // the short path below (no predicates, pointer stepping)
            const bool rows_whole = m0 + Cfg::BM * rank + 32 * q + 32 <= p.m;
            const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16) + buf * BN;
#pragma unroll 1
            for (int c = half; c < BN / 32; c += kGroups) {
                const int64_t jb = n0 + 32 * c;
                if (jb >= p.n) break;  // uniform across the warp
                const bool full = p.n - jb >= 32;
                if (full && rows_whole && !tail && p.split == 1) {
                    // C(i, jb + t) for t < 32, all inside C; reads of C first (when beta != 0)
                    float* d = p.C + jb * p.ldc + i;
                    const int64_t ldc = p.ldc;
                    uint32_t v[32];
                    if (beta == 0.0f) {
                        tmem_ld_32x32b_x32(lane_base + 32 * c, v);
                        tmem_wait_ld();
                        if (alpha == 1.0f) {
#pragma unroll
                            for (int t = 0; t < 32; ++t, d += ldc) *d = __uint_as_float(v[t]);
                        } else {
#pragma unroll
                            for (int t = 0; t < 32; ++t, d += ldc) *d = alpha * __uint_as_float(v[t]);
                        }
                    } else {
                        float cv[32];
                        const float* s = d;
#pragma unroll
                        for (int t = 0; t < 32; ++t, s += ldc) cv[t] = *s;
                        tmem_ld_32x32b_x32(lane_base + 32 * c, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int t = 0; t < 32; ++t, d += ldc) *d = fmaf(beta, cv[t], alpha * __uint_as_float(v[t]));
                    }
                    continue;
                }
                const int jn = full ? 32 : static_cast<int>(p.n - jb);
                // All 32 loads of C are issued before the tensor-memory read and
                // before any store: interleaved with the stores, each load would wait
                // for the previous store (the compiler cannot rule out that they
                // alias) and the epilogue would run at DRAM latency.
                float* dst = p.C + jb * p.ldc + i;
                const bool read_c = row_ok && p.split == 1 && !tail && beta != 0.0f;
                float cv[32];
#pragma unroll
                for (int t = 0; t < 32; ++t) cv[t] = (read_c && t < jn) ? dst[t * p.ldc] : 0.0f;
                uint32_t v[32];
                tmem_ld_32x32b_x32(lane_base + 32 * c, v);
                tmem_wait_ld();
                if (!row_ok) continue;
                if (tail) {
                    float* part = tpart + (32 * c) * (2 * Cfg::BM) + i_loc;
#pragma unroll
                    for (int t = 0; t < 32; ++t) part[t * (2 * Cfg::BM)] = __uint_as_float(v[t]);
                } else if (p.split > 1) {
                    float* part = p.P + slice * p.p_stride + jb * p.ldp + i;
#pragma unroll
                    for (int t = 0; t < 32; ++t)
                        if (t < jn) part[t * p.ldp] = __uint_as_float(v[t]);
                } else {
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        if (t < jn) {
                            float o = alpha * __uint_as_float(v[t]);
                            if (beta != 0.0f) o = fmaf(beta, cv[t], o);
                            dst[t * p.ldc] = o;
                        }
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote_relaxed(acc_empty_leader0 + 8 * buf);  // buffer free for the next unit
            if (tail) {
                // Publish this slice's partials; the last slice of this warp's region
                // to arrive sums all of them in slice order and writes C.
                __threadfence();
                __syncwarp();
                int arrived = 0;
                const int region = (tile - p.tail_first) * (2 * Cfg::EPI_WARPS) + static_cast<int>(rank) * Cfg::EPI_WARPS +
                                   (warp - 2);
                if (lane == 0) arrived = atomicAdd(p.tail_cnt + region, 1);
                arrived = __shfl_sync(0xffffffffu, arrived, 0);
                if (arrived == p.tail_split - 1) {
                    __threadfence();
                    const float* tile0 = p.tail_P + static_cast<int64_t>(tile - p.tail_first) * p.tail_split *
                                                        (2 * Cfg::BM) * BN;
#pragma unroll 1
                    for (int c = half; c < BN / 32; c += kGroups) {
                        const int64_t jb = n0 + 32 * c;
                        if (jb >= p.n) break;
                        if (!row_ok) continue;
                        const int jn = (p.n - jb < 32) ? static_cast<int>(p.n - jb) : 32;
                        float* dst = p.C + jb * p.ldc + i;
                        float acc[32], cv[32];
#pragma unroll
                        for (int t = 0; t < 32; ++t) {
                            acc[t] = 0.0f;
                            cv[t] = (beta != 0.0f && t < jn) ? dst[t * p.ldc] : 0.0f;
                        }
                        for (int j = 0; j < p.tail_split; ++j) {
                            const float* src = tile0 + static_cast<int64_t>(j) * (2 * Cfg::BM) * BN +
                                               (32 * c) * (2 * Cfg::BM) + i_loc;
                            float pv[32];
#pragma unroll
                            for (int t = 0; t < 32; ++t) pv[t] = __ldcg(src + t * (2 * Cfg::BM));
#pragma unroll
                            for (int t = 0; t < 32; ++t) acc[t] += pv[t];
                        }
#pragma unroll
                        for (int t = 0; t < 32; ++t) {
                            if (t < jn) {
                                float o = alpha * acc[t];
                                if (beta != 0.0f) o = fmaf(beta, cv[t], o);
                                dst[t * p.ldc] = o;
                            }
                        }
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();  // no CTA leaves while its peer may still read its shared memory or barriers
    if (warp == 1) {
        tc_fence_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Cfg::TMEM_COLS)
                     : "memory");
    }
}

template <int BN, bool SPLIT3>
struct Launcher {
    static cudaError_t run(const CUtensorMap& a, const CUtensorMap& as, const CUtensorMap& b, const CUtensorMap& bs,
                           const GemmParams& p, int units, int num_sms, cudaStream_t st, int* pairs_out) {
        using Cfg = Tc2Cfg<BN, SPLIT3>;
        auto kern = tc2_gemm_kernel<BN, SPLIT3>;
        static std::atomic<uint64_t> smem_set{0};
        cudaError_t e =
            set_smem_limit_once(smem_set, reinterpret_cast<const void*>(kern), static_cast<int>(Cfg::SMEM));
        if (e != cudaSuccess) return e;
        // Pairs that can be resident at once (clusters must fit inside GPCs), asked
        // once per device so a call captured into a CUDA graph only launches.
        static int cached[64] = {0};
        int dev = 0;
        cudaGetDevice(&dev);
        int max_clusters = (dev >= 0 && dev < 64) ? cached[dev] : 0;
        if (max_clusters <= 0) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2, 1, 1);
            cfg.blockDim = dim3(Cfg::THREADS, 1, 1);
            cfg.dynamicSmemBytes = Cfg::SMEM;
            e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
            if (e != cudaSuccess || max_clusters <= 0) {
                cudaGetLastError();
                max_clusters = num_sms / 2;
            }
            if (dev >= 0 && dev < 64) cached[dev] = max_clusters;
        }
        int pairs = units < max_clusters ? units : max_clusters;
        if (pairs < 1) pairs = 1;
        *pairs_out = pairs;
        return launch_kernel(p.after_prep != 0, kern, dim3(2 * pairs), dim3(Cfg::THREADS), Cfg::SMEM, st, a, as, b, bs,
                             p);
    }
};

}  // namespace

int tc2_bk(bool split3) { return split3 ? Tc2Cfg<256, true>::BK : Tc2Cfg<256, false>::BK; }

int tc2_threads() { return Tc2Cfg<256, false>::THREADS; }

int tc2_epilogue_warps() { return Tc2Cfg<256, false>::EPI_WARPS; }

int tc2_stages(int bn, bool split3) {
    if (split3) return bn == 128 ? Tc2Cfg<128, true>::STAGES : Tc2Cfg<256, true>::STAGES;
    if (bn == 512) return Tc2Cfg<512, false>::STAGES;
    return bn == 128 ? Tc2Cfg<128, false>::STAGES : Tc2Cfg<256, false>::STAGES;
}

size_t tc2_smem_bytes(int bn, bool split3) {
    if (split3) return bn == 128 ? Tc2Cfg<128, true>::SMEM : Tc2Cfg<256, true>::SMEM;
    if (bn == 512) return Tc2Cfg<512, false>::SMEM;
    return bn == 128 ? Tc2Cfg<128, false>::SMEM : Tc2Cfg<256, false>::SMEM;
}

cudaError_t launch_tc2(const CUtensorMap& tmA, const CUtensorMap& tmAs, const CUtensorMap& tmB,
                       const CUtensorMap& tmBs, const GemmParams& p, int bn, bool split3, int units, int num_sms,
                       cudaStream_t stream, int* pairs_launched) {
    if (bn == 128)
        return split3 ? Launcher<128, true>::run(tmA, tmAs, tmB, tmBs, p, units, num_sms, stream, pairs_launched)
                      : Launcher<128, false>::run(tmA, tmAs, tmB, tmBs, p, units, num_sms, stream, pairs_launched);
    if (bn == 256)
        return split3 ? Launcher<256, true>::run(tmA, tmAs, tmB, tmBs, p, units, num_sms, stream, pairs_launched)
                      : Launcher<256, false>::run(tmA, tmAs, tmB, tmBs, p, units, num_sms, stream, pairs_launched);
    if (bn == 512 && !split3)
        return Launcher<512, false>::run(tmA, tmAs, tmB, tmBs, p, units, num_sms, stream, pairs_launched);
    return cudaErrorInvalidValue;
}

}  // namespace pg
