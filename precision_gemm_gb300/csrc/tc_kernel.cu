// Tensor-core GEMM (tcgen05, sm_103a): TF32 and 3xTF32 modes.
//
// One CTA computes a 128 x BN tile of C with the fifth-generation tensor cores:
// operands are staged in shared memory by TMA, one elected thread issues
// tcgen05.mma (M = 128, N = BN, K = 8 per instruction) into an FP32 accumulator
// held in tensor memory (TMEM), and four epilogue warps read the accumulator
// back with tcgen05.ld and apply alpha/beta.  The pages' tensor-core prior art
// ("cuda-kernel-opt": asynchronous loads, consumer warps decoupled from each
// other, accumulators tuned per warp) is superseded here: a single issuing
// thread replaces per-warp MMA fragments, so the pages' per-warp "shift"
// barriers have nothing left to order.
//
// Warp roles (192 threads; 320 or 448 in 3xTF32):
//   warp 0      TMA loader (one thread): A as one box (K-major, or M-major as one
//               3-D box of four 32-row groups) or four 32-row boxes; B likewise
//   warp 1      allocates TMEM; one thread issues the MMAs; frees TMEM at exit
//   warps 2-5   epilogue; warp w may access TMEM lanes 32*(w%4) .. +31
//   warps 6-13  3xTF32 only: split each landed slot into TF32 parts, in one or
//               two groups of four (warp w handles the A rows of TMEM lane
//               quarter w % 4)
//
// Shared-memory operand layouts (canonical tcgen05 layouts, 1 KiB aligned):
//   A (column-major, M-major): per 32-row group of M a box of BK rows of k,
//     each row 32 floats = 128 B, in the 128-byte swizzle with 32-byte atoms
//     (TMA SWIZZLE_128B_ATOM_32B; descriptor layout 1) -- the form tcgen05 takes
//     for an M-major TF32 operand (measured: the plain 128-byte swizzle reads as
//     zeros for M-major TF32).  Leading byte offset (between 32-row groups of M)
//     = 128*BK, stride byte offset (between 4-row atoms of k) = 512.  The k-step
//     kk (8 values, two atoms) starts at +1024*kk.
//   B (column-major, K-major): BN rows of BK floats; BK = 32 -> 128-byte rows
//     with the 128-byte swizzle (8-row groups of 1024 B); BK = 16 -> 64-byte
//     rows with the 64-byte swizzle (groups of 512 B).  The k-step kk starts at
//     +32*kk bytes inside the swizzle atom.
//
// 3xTF32 (SPLIT3): TMA brings the FP32 tiles of A and B into the ring's slots
// as for TF32 (A M-major without swizzle: the tensor core does not read it from
// shared memory).  Groups of four transform warps then split every value into its TF32
// "big" part and the exact remainder ("small"):
//   A  each thread takes one row of the 128 (its warp's TMEM lane quarter),
//      reads the row's BK values and writes big and small with tcgen05.st into a
//      TMEM operand stage (lane = row, one value per column: big in 32 columns,
//      small in the next 32), from which the MMAs read A;
//   B  split in place in the slot; for BN <= 128 the remainders go to the space
//      the sub-slot keeps free right in front of B (layout [A][B small][B]), for
//      BN = 256 to a slot of a second, short ring of B remainders.
// They then fence their writes for the tensor core and arrive on the slot's
// "ready" barrier, which the MMA thread waits for.  Per k-step it issues, for
// BN <= 128, big * [small | big] as one MMA of N = 2 BN into accumulator
// columns [0, 2 BN) and small * big into columns [BN, 2 BN) -- two MMAs where
// three would do the same products, and the 64-wide tile's N = 128 MMA runs at
// the full rate where N = 64 runs at two thirds of it; the epilogue adds the
// two halves.  For BN = 256 it issues small*big, big*small, big*big into one
// accumulator.  (The small*small term is below FP32 resolution and dropped.)
// It then releases the slot and the remainder slot with its TMEM stage.
// 3xTF32 thus reads each operand byte from
// DRAM once, like TF32 (these shapes are HBM-bound), and A's parts never pass
// through shared memory (a split in place for A as well, the earlier form of
// this kernel, measured 3-7 % slower on the narrow shapes).  Two groups of
// transform warps take alternate k-blocks.
//
// Every wait is bounded; on expiry the CTA records the status, lets its
// in-flight TMA copies and MMAs finish (bounded), frees TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace pg {
namespace {

// Transform warp groups of the 3xTF32 kernel (a compile-time tunable, 1 or 2).
#ifndef PG_TC_XF_GROUPS
#define PG_TC_XF_GROUPS 2
#endif

// K-blocks of BK per ring slot for the 64-wide TF32 tile (a compile-time
// tunable, 1 or 2).  Its MMAs are short (48 cycles for 128 x 64 x 8), so the
// issuing thread's per-slot work -- a barrier wait and a commit -- drains the
// tensor pipe unless each slot carries more MMAs.  The fused 3xTF32 form issues
// 112 cycles of MMAs per k-step and does better with one k-block per slot, which
// leaves room for seven slots and six TMEM operand stages (8192 x 64 x 8192:
// 0.087 -> 0.083 ms against two k-blocks per slot with three of each).
#ifndef PG_TC_KPS
#define PG_TC_KPS 2
#endif

template <int BN, bool SPLIT3>
struct TcCfg {
    static constexpr int BM = kBM;
    static constexpr int BK = 32;
    static constexpr int A_BYTES = BM * BK * 4;  // A tile of a slot
    static constexpr int B_BYTES = BN * BK * 4;  // B tile of a slot
    static constexpr int A_BOX_BYTES = 32 * BK * 4;
    static constexpr int KPS = (BN == 64 && !SPLIT3) ? PG_TC_KPS : 1;  // k-blocks per slot
    // 3xTF32 with BN <= 128 ("fused"): a k-block's sub-slot is [A][B small][B],
    // the B remainders written by the transform warps right in front of the
    // split B, so that one N = 2 BN operand covers both.  BN = 256 keeps its
    // remainders in a second, short ring.
    static constexpr bool FUSED = SPLIT3 && BN <= 128;
    static constexpr int B_OFF = A_BYTES + (FUSED ? B_BYTES : 0);   // B in a sub-slot
    static constexpr int SUB_BYTES = B_OFF + B_BYTES;               // one k-block's sub-slot
    static constexpr int LOAD_BYTES = A_BYTES + B_BYTES;            // what TMA brings per k-block
    static constexpr int STAGE_BYTES = KPS * SUB_BYTES;             // one ring slot
    static constexpr int SMALL_BYTES = KPS * B_BYTES;               // B remainders of one slot
    static constexpr int RING_BYTES = (FUSED || KPS == 2 ? 224 : 200) * 1024;
    // TMEM: the accumulator in columns [0, ACC_COLS) (fused 3xTF32: [0, 2 BN),
    // the big * small products in the first BN and big * big + small * big in the
    // second); with SPLIT3 the A operand stages at columns A_TMEM_COL +
    // A_STAGE_COLS j, 64 per k-block (32 big, then 32 small), all 512 columns
    // allocated
    static constexpr int ACC_COLS = FUSED ? 2 * BN : BN;
    static constexpr uint32_t A_TMEM_COL = FUSED ? ACC_COLS : 256;
    static constexpr uint32_t A_STAGE_COLS = 64 * KPS;
    // 3xTF32: remainder slots, each with a TMEM stage of A's parts.  Fused (BN <=
    // 128): as many TMEM stages as fit beside the accumulator, at most one per
    // ring slot, so that the transform warps can run that far ahead of the MMAs.
    // BN = 256: one slot, which also holds B's remainders (a second ring).
    static constexpr int SMALL_RING_BYTES = FUSED ? 0 : (SPLIT3 ? KPS * B_BYTES : 0);
    static constexpr int STAGES_RAW = (RING_BYTES - SMALL_RING_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr int TMEM_STAGES_FIT = static_cast<int>((512 - A_TMEM_COL) / A_STAGE_COLS);
    static constexpr int SMALL_STAGES =
        !SPLIT3 ? 0 : (!FUSED ? 1 : (TMEM_STAGES_FIT < STAGES ? TMEM_STAGES_FIT : STAGES));
    // 3xTF32 transform: groups of four warps (one per TMEM lane quarter), group g
    // taking k-blocks g, g + XF_GROUPS, ... so that one group's per-k-block
    // latencies (barrier waits, fences) overlap another group's arithmetic.  A
    // group waits on barrier phases out of step with the other groups, so the
    // phase it waits for must be at most one ahead of the barrier's current
    // phase; see the transform loop for why XF_GROUPS <= SMALL_STAGES <= STAGES
    // guarantees it.
    static constexpr int XF_GROUPS = !SPLIT3 ? 0 : (PG_TC_XF_GROUPS < SMALL_STAGES ? PG_TC_XF_GROUPS : SMALL_STAGES);
    static constexpr int XF_WARPS = 4 * XF_GROUPS;      // transform warps
    static constexpr int THREADS = 192 + 32 * XF_WARPS;
    static constexpr int BAR_BYTES = (3 * STAGES + SMALL_STAGES + 1) * 8 + 16;
    static constexpr size_t SMEM = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES +
                                   static_cast<size_t>(SMALL_RING_BYTES) + BAR_BYTES;
    static constexpr uint32_t TMEM_COLS = SPLIT3 ? 512 : BN;  // power of two >= 32
    static_assert(!SPLIT3 || A_TMEM_COL + A_STAGE_COLS * SMALL_STAGES <= 512, "TMEM operand stages");
    static_assert(!SPLIT3 || ACC_COLS <= static_cast<int>(A_TMEM_COL), "accumulator below the operand stages");
    static_assert(KPS == 1 || KPS == 2, "k-blocks per slot");
    static_assert(STAGES >= 2 && (STAGES >= 3 || !SPLIT3), "ring too shallow");
    static_assert(!SPLIT3 || (XF_GROUPS >= 1 && XF_GROUPS <= SMALL_STAGES && SMALL_STAGES <= STAGES),
                  "transform groups may run ahead of a barrier by at most one phase");
    static_assert(SMEM <= 232448, "over the 227 KiB of dynamic shared memory per CTA");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "slots need 1 KiB alignment");
    static_assert(BN == 64 || BN == 128 || BN == 256, "BN");
};

// At most this many tile segments per stream-K CTA (the planner keeps to it).
constexpr int kTcSkMaxSegs = 8;

// SK: stream-K (3xTF32 with BN <= 128; the planner takes it for BN = 128).  The
// grid's CTAs share the T = tiles x k-blocks (tile, k-block) iterations in equal
// contiguous ranges [c T / G, (c + 1) T / G), crossing tile boundaries; the
// accumulator is drained into a partial block at the end of each tile segment
// (slot t * sk_maxseg + j for the j-th CTA touching tile t) and restarted for the
// next, and a fix-up kernel adds each tile's blocks in k order.  The MMA thread
// waits for the epilogue warps to have drained the accumulator (acc_empty)
// before the next segment's first MMA.
template <int BN, bool SPLIT3, bool SK>
__global__ void __launch_bounds__(TcCfg<BN, SPLIT3>::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmBs, const GemmParams p) {
    if (PG_PDL_EARLY && threadIdx.x == 0) pdl_trigger();
    using Cfg = TcCfg<BN, SPLIT3>;
    static_assert(!SK || (SPLIT3 && Cfg::FUSED && Cfg::KPS == 1), "stream-K: fused 3xTF32, one k-block per slot");
    constexpr int S = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_smem_1024(smem_raw);
    constexpr int SS = Cfg::SMALL_STAGES;
    uint8_t* small_ring = smem + S * Cfg::STAGE_BYTES;  // 3xTF32 with BN = 256: B remainders, SS slots
    uint64_t* bars = reinterpret_cast<uint64_t*>(small_ring + Cfg::SMALL_RING_BYTES);
    // [0,S) full, [S,2S) empty, 2S accum, [2S+1, 3S+1) ready, [3S+1, 3S+1+SS) small_empty
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 3 * S + 1 + SS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + S);
    const uint32_t accum_bar = smem_u32(bars + 2 * S);
    const uint32_t ready0 = smem_u32(bars + 2 * S + 1);
    const uint32_t small_empty0 = smem_u32(bars + 3 * S + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Stream-K: this CTA's tile segments (partial-block slot, k-blocks, first
    // k-block, tile origin), built by thread 0; the barriers of the accumulator's
    // hand-back (acc_empty) and of the last MMA (done).
    __shared__ int seg_slot[SK ? kTcSkMaxSegs : 1], seg_len[SK ? kTcSkMaxSegs : 1], seg_k0[SK ? kTcSkMaxSegs : 1],
        seg_m0[SK ? kTcSkMaxSegs : 1], seg_n0[SK ? kTcSkMaxSegs : 1];
    __shared__ int sk_nsegs, sk_nits;
    __shared__ __align__(8) uint64_t sk_bars[2];
    const uint32_t acc_empty_bar = smem_u32(&sk_bars[0]);
    const uint32_t done_bar = smem_u32(&sk_bars[1]);

    int tile_m = 0, tile_n = 0;
    if (!SK) tile_coords(blockIdx.x, p.tiles_m, p.tiles_n, p.group_m, tile_m, tile_n);
    const int64_t m0 = static_cast<int64_t>(tile_m) * Cfg::BM;
    const int64_t n0 = static_cast<int64_t>(tile_n) * BN;
    const int slice = SK ? 0 : blockIdx.y;
    const int kb0 = slice * p.kb_per_split;
    const int nkb = min(kb0 + p.kb_per_split, p.kb_total) - kb0;
    constexpr int KPS = Cfg::KPS;
    // B arrives split (big through tmB, remainders through tmBs into the space in
    // front of B): the transform warps split A only.
    const bool b_presplit = Cfg::FUSED && p.b_presplit != 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
            if (SPLIT3) mbar_init(ready0 + 8 * s, 4);  // the four warps of one transform group
        }
        for (int j = 0; j < SS; ++j) mbar_init(small_empty0 + 8 * j, 1);
        mbar_init(accum_bar, 1);
        *abort_flag = 0;
        if (SK) {
            mbar_init(acc_empty_bar, 4);  // the four epilogue warps
            mbar_init(done_bar, 1);
            const int G = gridDim.x, c = blockIdx.x;
            const int64_t T = p.sk_iters;
            const int kb = p.kb_total;
            const int64_t it0 = static_cast<int64_t>(c) * T / G, it1 = static_cast<int64_t>(c + 1) * T / G;
            int ns = 0;
            int64_t covered = 0;
            for (int64_t it = it0; it < it1 && ns < kTcSkMaxSegs; ++ns) {
                const int tile = static_cast<int>(it / kb);
                const int k0 = static_cast<int>(it - static_cast<int64_t>(tile) * kb);
                const int len = static_cast<int>(min(static_cast<int64_t>(kb - k0), it1 - it));
                int tm_, tn_;
                tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, tm_, tn_);
                seg_slot[SK ? ns : 0] = tile * p.sk_maxseg + (c - sk_cta_of(static_cast<int64_t>(tile) * kb, G, T));
                seg_len[SK ? ns : 0] = len;
                seg_k0[SK ? ns : 0] = k0;
                seg_m0[SK ? ns : 0] = tm_ * Cfg::BM;
                seg_n0[SK ? ns : 0] = tn_ * BN;
                it += len;
                covered += len;
            }
            sk_nsegs = ns;
            sk_nits = static_cast<int>(it1 - it0);
            // the planner keeps every CTA within kTcSkMaxSegs segments; were the
            // range longer, report a failure rather than leave part of it undone
            if (covered != it1 - it0) {
                sk_nits = 0;
                raise_abort(abort_flag, p.status);
            }
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    pdl_wait();  // launched right after an operand pass: its output, before any copy
    // ring slots' worth of k-blocks; the last may hold fewer
    const int nst = SK ? sk_nits : (nkb + KPS - 1) / KPS;

    if (warp == 0) {
        // ---------------- TMA loader ----------------
        if (lane == 0) {
            prefetch_tmap(&tmA);
            prefetch_tmap(&tmB);
            if (b_presplit) prefetch_tmap(&tmBs);
            int issued = 0;
            int ld_seg = 0, ld_kq = 0;  // stream-K: the loader's segment and k-block in it
            if (!(p.debug_flags & 1)) {
                for (int it = 0; it < nst; ++it) {
                    const int s = it % S;
                    const int64_t lm0 = SK ? seg_m0[SK ? ld_seg : 0] : m0;
                    const int64_t ln0 = SK ? seg_n0[SK ? ld_seg : 0] : n0;
                    const int lkb0 = SK ? seg_k0[SK ? ld_seg : 0] + ld_kq : kb0 + it * KPS;
                    if (SK && ++ld_kq == seg_len[SK ? ld_seg : 0]) {
                        ld_kq = 0;
                        ++ld_seg;
                    }
                    if (!mbar_wait_bounded(empty0 + 8 * s, ((it / S) & 1) ^ 1, p.timeout_ns, abort_flag)) {
                        raise_abort(abort_flag, p.status);
                        break;
                    }
                    const uint32_t full = full0 + 8 * s;
                    const int nsub = SK ? 1 : min(KPS, nkb - it * KPS);  // stream-K: one k-block per slot
                    mbar_arrive_expect_tx(full, nsub * (Cfg::LOAD_BYTES + (b_presplit ? Cfg::B_BYTES : 0)));
                    for (int u = 0; u < nsub; ++u) {
                        const int32_t kc = (lkb0 + u) * Cfg::BK;
                        const uint32_t slot = smem_u32(smem + s * Cfg::STAGE_BYTES + u * Cfg::SUB_BYTES);
                        // A K-major (transa 'T'): one box of 128 rows x BK.  A M-major: one 3-D
                        // box {32 rows, BK, 4 row groups} when m % 32 == 0, else four 2-D boxes
                        // of 32 rows (both land as 4 x [BK][32] row groups).
                        auto load_a = [&](uint32_t dst, const CUtensorMap* map) {
                            if (p.a_kmajor) {
                                tma_load_2d(dst, map, kc, static_cast<int32_t>(lm0), full);
                            } else if (p.a3d) {
                                tma_load_3d(dst, map, 0, kc, static_cast<int32_t>(lm0 / 32), full);
                            } else {
#pragma unroll
                                for (int g = 0; g < 4; ++g)
                                    tma_load_2d(dst + g * Cfg::A_BOX_BYTES, map, static_cast<int32_t>(lm0 + 32 * g),
                                                kc, full);
                            }
                        };
                        // B K-major: one box of BN columns x BK.  B N-major (transb 'T'): BN/32
                        // groups of 32 columns, as one 3-D box or as 2-D boxes.
                        auto load_b = [&](uint32_t dst, const CUtensorMap* map) {
                            if (!p.b_mnmajor) {
                                tma_load_2d(dst, map, kc, static_cast<int32_t>(ln0), full);
                            } else if (p.b3d) {
                                tma_load_3d(dst, map, 0, kc, static_cast<int32_t>(ln0 / 32), full);
                            } else {
#pragma unroll
                                for (int g = 0; g < BN / 32; ++g)
                                    tma_load_2d(dst + g * Cfg::A_BOX_BYTES, map, static_cast<int32_t>(ln0 + 32 * g),
                                                kc, full);
                            }
                        };
                        load_a(slot, &tmA);
                        load_b(slot + Cfg::B_OFF, &tmB);
                        if (b_presplit) load_b(slot + Cfg::A_BYTES, &tmBs);
                    }
                    issued = it + 1;
                }
            }
            // every copy of the main loop is issued: a dependent reduction or fix-up
            // may be scheduled now
            if (!PG_PDL_EARLY) pdl_trigger();
            // Let every copy this CTA issued land before it may retire.
            for (int it = max(0, issued - S); it < issued; ++it)
                mbar_wait_bounded(full0 + 8 * (it % S), (it / S) & 1, p.timeout_ns, nullptr);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            uint32_t accumulate = 0;
            // A from TMEM (3xTF32) is K-major by construction
            const uint32_t idesc = idesc_tf32(Cfg::BM, BN, !SPLIT3 && !p.a_kmajor, p.b_mnmajor != 0);
            const uint32_t idesc2 = idesc_tf32(Cfg::BM, 2 * BN, false, p.b_mnmajor != 0);  // fused: N = 2 BN
            // The 48-cycle MMAs of the 64-wide tile leave the issuing thread little
            // time per instruction, so descriptors are not rebuilt per MMA: those of
            // slot 0 are built once, and a slot, a k-block in it and a k-step only
            // move the start address field (bits 0-13, in 16-byte units; shared
            // addresses stay below 256 KiB, so the field does not overflow).
            const bool a_k = p.a_kmajor != 0, b_k = p.b_mnmajor == 0;
            const uint64_t a_desc0 = operand_desc<Cfg::BK>(smem_u32(smem), 0, a_k);
            const uint64_t b_desc0 = operand_desc<Cfg::BK>(smem_u32(smem) + Cfg::B_OFF, 0, b_k);
            // B remainders: in front of B in the sub-slot (fused), else in the second ring
            const uint64_t bs_desc0 =
                operand_desc<Cfg::BK>(Cfg::FUSED ? smem_u32(smem) + Cfg::A_BYTES : smem_u32(small_ring), 0, b_k);
            const uint32_t a_kstep = a_k ? 2 : 64, b_kstep = b_k ? 2 : 64;  // 32 B or 1 KiB per k-step
            int s = 0, j = 0;  // ring slot, remainder slot and TMEM stage (3xTF32)
            uint32_t phase = 0;
            int seg = 0, seg_left = SK ? seg_len[0] : 0;  // stream-K: the segment and its k-blocks to come
            for (int it = 0; it < nst; ++it) {
                // 3xTF32: the transform warps have split the slot
                if (!mbar_wait_bounded((SPLIT3 ? ready0 : full0) + 8 * s, phase, p.timeout_ns, abort_flag)) {
                    raise_abort(abort_flag, p.status);
                    break;
                }
                if (SK && seg > 0 && seg_left == seg_len[SK ? seg : 0]) {
                    // the segment's first k-block: the epilogue warps must have drained
                    // the previous segment's sums out of the accumulator
                    if (!mbar_wait_bounded(acc_empty_bar, (seg - 1) & 1, p.timeout_ns, abort_flag)) {
                        raise_abort(abort_flag, p.status);
                        break;
                    }
                    accumulate = 0;
                }
                tc_fence_after_sync();
                const int nsub = SK ? 1 : min(KPS, nkb - it * KPS);  // stream-K: one k-block per slot
                for (int u = 0; u < nsub; ++u) {
                    const uint32_t off = static_cast<uint32_t>(s * Cfg::STAGE_BYTES + u * Cfg::SUB_BYTES) >> 4;
                    const uint32_t soff =
                        Cfg::FUSED ? off : static_cast<uint32_t>(j * Cfg::SMALL_BYTES + u * Cfg::B_BYTES) >> 4;
                    // lane 0, A's big parts of this k-block
                    const uint32_t ta_big = tmem + Cfg::A_TMEM_COL + Cfg::A_STAGE_COLS * j + 64 * u;
#pragma unroll
                    for (int kk = 0; kk < Cfg::BK / 8; ++kk) {
                        const uint64_t bd = b_desc0 + (off + kk * b_kstep);
                        if (Cfg::FUSED) {
                            // big * [small | big] into columns [0, 2 BN), then small * big
                            // into [BN, 2 BN): two MMAs per k-step instead of three
                            const uint64_t bsd = bs_desc0 + (soff + kk * b_kstep);
                            const uint32_t tab = ta_big + 8 * kk;  // k-step kk: columns 8kk .. 8kk+7
                            mma_tf32_tmem_a(tmem, tab, bsd, idesc2, accumulate);
                            accumulate = 1;
                            mma_tf32_tmem_a(tmem + BN, tab + 32, bd, idesc, 1);
                        } else if (SPLIT3) {
                            const uint64_t bsd = bs_desc0 + (soff + kk * b_kstep);
                            const uint32_t tab = ta_big + 8 * kk;  // k-step kk: columns 8kk .. 8kk+7
                            mma_tf32_tmem_a(tmem, tab + 32, bd, idesc, accumulate);  // small * big
                            accumulate = 1;
                            mma_tf32_tmem_a(tmem, tab, bsd, idesc, 1);  // big * small
                            mma_tf32_tmem_a(tmem, tab, bd, idesc, 1);   // big * big
                        } else {
                            const uint64_t ad = a_desc0 + (off + kk * a_kstep);
                            mma_tf32(tmem, ad, bd, idesc, accumulate);
                            accumulate = 1;
                        }
                    }
                }
                mma_commit(empty0 + 8 * s);  // slot reusable once these MMAs have read it
                if (SPLIT3) mma_commit(small_empty0 + 8 * j);  // and so is the remainder slot
                if (SK && --seg_left == 0) {  // the segment's sums are complete
                    mma_commit(accum_bar);
                    if (++seg < sk_nsegs) seg_left = seg_len[SK ? seg : 0];
                }
                if (++s == S) {
                    s = 0;
                    phase ^= 1;
                }
                if (SS > 0 && ++j == SS) j = 0;
            }
            // the accumulator is complete (also after an abort); stream-K: every MMA has finished
            mma_commit(SK ? done_bar : accum_bar);
        }
        __syncwarp();
    } else if (warp >= 6) {
        // ---------------- 3xTF32 transform (warps 6..9) ----------------
        if constexpr (SPLIT3) {
            const int grp = (warp - 6) >> 2;
            const int t = threadIdx.x - 192 - 128 * grp;  // thread within the group
            const int q = warp & 3;  // TMEM lane quarter: A rows 32q .. 32q + 31
            for (int it = grp; it < nst; it += Cfg::XF_GROUPS) {
                const int s = it % S;
                const int j = it % SS;
                // The MMAs of slot fill it - SS have released remainder slot j and its
                // TMEM stage, then fill it has landed.  A parity wait is exact only
                // while the awaited phase is the barrier's current or next one.  This
                // group's previous fill, it - XF_GROUPS >= it - SS, already saw the
                // release of fill it - XF_GROUPS - SS >= it - 2 SS, so small_empty[j]
                // is at most one phase behind.  MMAs complete in order, so once the
                // MMAs of it - SS are done those of it - S <= it - SS are too, whose
                // slot had landed before: full[s] is then at most one phase behind.
                const bool landed = __all_sync(
                    0xffffffffu,
                    mbar_wait_bounded(small_empty0 + 8 * j, ((it / SS) & 1) ^ 1, p.timeout_ns, abort_flag) &&
                        mbar_wait_bounded(full0 + 8 * s, (it / S) & 1, p.timeout_ns, abort_flag));
                if (!landed) {
                    if (lane == 0) raise_abort(abort_flag, p.status);
                    break;
                }
                const int nsub = SK ? 1 : min(KPS, nkb - it * KPS);  // stream-K: one k-block per slot
                for (int u = 0; u < nsub; ++u) {
                    uint8_t* slot = smem + s * Cfg::STAGE_BYTES + u * Cfg::SUB_BYTES;
                    // A row 32q + lane: its BK values.  K-major: 128-byte row in the
                    // 128-byte swizzle (16-byte chunk c at c ^ (row % 8)), read as float4s
                    // (the 8 rows of a quarter-warp hit 8 distinct chunk positions).
                    // M-major: row group q, BK lines of 32 rows, no swizzle.
                    const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + Cfg::A_TMEM_COL +
                                        Cfg::A_STAGE_COLS * j + 64 * u;
#pragma unroll
                    for (int h = 0; h < Cfg::BK / 16; ++h) {  // 16 values of the row at a time
                        float a[16];
                        if (p.a_kmajor) {
                            const uint32_t row = smem_u32(slot) + (32 * q + lane) * (Cfg::BK * 4);
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const float4 v = lds128(row + (((4 * h + c) ^ (lane & 7)) << 4));
                                a[4 * c] = v.x;
                                a[4 * c + 1] = v.y;
                                a[4 * c + 2] = v.z;
                                a[4 * c + 3] = v.w;
                            }
                        } else {
                            const float* col = reinterpret_cast<const float*>(slot + q * Cfg::A_BOX_BYTES) + lane;
#pragma unroll
                            for (int k = 0; k < 16; ++k) a[k] = col[32 * (16 * h + k)];
                        }
                        uint32_t big[16], sml[16];
                        split_tf32_batch<16>(a, big, sml);
                        tmem_st_32x32b_x16(ta + 16 * h, big);
                        tmem_st_32x32b_x16(ta + 32 + 16 * h, sml);
                    }
                    if (!b_presplit)
                        split_tile_in_place<Cfg::B_BYTES, 128>(
                            slot + Cfg::B_OFF,
                            Cfg::FUSED ? slot + Cfg::A_BYTES : small_ring + j * Cfg::SMALL_BYTES + u * Cfg::B_BYTES,
                            t);
                }
                tmem_wait_st();
                fence_proxy_async_smem();  // the tensor core reads the B writes
                tc_fence_before_sync();    // ... and the TMEM stores
                __syncwarp();
                if (lane == 0) mbar_arrive(ready0 + 8 * s);
            }
        }
    } else if (SK) {
        // ---------------- stream-K epilogue (warps 2..5) ----------------
        // Per segment: the accumulator (the two halves of the fused form added)
        // goes to the segment's partial block as [column][row] -- lane = row, so
        // every store of a warp covers 128 contiguous bytes -- and is handed back.
        const int q = warp & 3;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
        constexpr int EC = 16;
        for (int seg = 0; seg < sk_nsegs; ++seg) {
            const bool ready =
                __all_sync(0xffffffffu, mbar_wait_bounded(accum_bar, seg & 1, p.timeout_ns, abort_flag));
            if (!ready) {
                if (lane == 0) raise_abort(abort_flag, p.status);
                break;
            }
            tc_fence_after_sync();
            float* part = p.sk_P + static_cast<int64_t>(seg_slot[SK ? seg : 0]) * (Cfg::BM * BN) + 32 * q + lane;
#pragma unroll 1
            for (int c = 0; c < BN / EC; ++c) {
                uint32_t v[EC], w[EC];
                tmem_ld_32x32b_x16(lane_base + EC * c, v);
                tmem_ld_32x32b_x16(lane_base + BN + EC * c, w);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < EC; ++t)
                    part[(EC * c + t) * Cfg::BM] = __uint_as_float(v[t]) + __uint_as_float(w[t]);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty_bar);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;
        const bool ready =
            __all_sync(0xffffffffu, mbar_wait_bounded(accum_bar, 0, p.timeout_ns, abort_flag));
        if (!ready) {
            if (lane == 0) raise_abort(abort_flag, p.status);
        } else if (!*abort_flag) {
            tc_fence_after_sync();
            const int64_t i = m0 + 32 * q + lane;
            const bool row_ok = i < p.m;
            const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
            const float alpha = p.alpha, beta = p.beta;
            // Chunks of EC columns: 32, or 16 in 3xTF32, whose extra warps leave 128
            // registers a thread (two 32-value arrays would spill).
            constexpr int EC = SPLIT3 ? 16 : 32;
#pragma unroll 1
            for (int c = 0; c < BN / EC; ++c) {
                const int64_t jb = n0 + EC * c;
                if (jb >= p.n) break;  // uniform across the warp
                const int jn = (p.n - jb < EC) ? static_cast<int>(p.n - jb) : EC;
                // All EC loads of C are issued before the tensor-memory read and
                // before any store: interleaved with the stores, each load would wait
                // for the previous store (the compiler cannot rule out that they
                // alias) and the epilogue would run at DRAM latency.
                float* dst = p.C + jb * p.ldc + i;
                const bool read_c = row_ok && p.split == 1 && beta != 0.0f;
                float cv[EC];
#pragma unroll
                for (int t = 0; t < EC; ++t) cv[t] = (read_c && t < jn) ? dst[t * p.ldc] : 0.0f;
                uint32_t v[EC];
                if constexpr (EC == 32)
                    tmem_ld_32x32b_x32(lane_base + EC * c, v);
                else
                    tmem_ld_32x32b_x16(lane_base + EC * c, v);
                if constexpr (Cfg::FUSED) {
                    // the two partial accumulators: big * small, and big * big + small * big
                    uint32_t w[EC];
                    tmem_ld_32x32b_x16(lane_base + BN + EC * c, w);
                    tmem_wait_ld();
#pragma unroll
                    for (int t = 0; t < EC; ++t) v[t] = __float_as_uint(__uint_as_float(v[t]) + __uint_as_float(w[t]));
                }
                tmem_wait_ld();
                if (!row_ok) continue;
                if (p.split > 1) {
                    float* part = p.P + slice * p.p_stride + jb * p.ldp + i;
#pragma unroll
                    for (int t = 0; t < EC; ++t)
                        if (t < jn) part[t * p.ldp] = __uint_as_float(v[t]);
                } else {
#pragma unroll
                    for (int t = 0; t < EC; ++t) {
                        if (t < jn) {
                            float o = alpha * __uint_as_float(v[t]);
                            if (beta != 0.0f) o = fmaf(beta, cv[t], o);
                            dst[t * p.ldc] = o;
                        }
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        if (*abort_flag) {
            // MMAs issued before an abort must finish before TMEM is released.
            if (lane == 0) mbar_wait_bounded(SK ? done_bar : accum_bar, 0, p.timeout_ns, nullptr);
            __syncwarp();
        }
        tc_fence_after_sync();
        tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

template <int BN, bool SPLIT3, bool SK = false>
cudaError_t launch_impl(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmBs, const GemmParams& p,
                        dim3 grid, cudaStream_t stream) {
    using Cfg = TcCfg<BN, SPLIT3>;
    auto kern = tc_gemm_kernel<BN, SPLIT3, SK>;
    static std::atomic<uint64_t> smem_set{0};
    cudaError_t e = set_smem_limit_once(smem_set, reinterpret_cast<const void*>(kern), static_cast<int>(Cfg::SMEM));
    if (e != cudaSuccess) return e;
    return launch_kernel(p.after_prep != 0, kern, grid, dim3(Cfg::THREADS), Cfg::SMEM, stream, tmA, tmB, tmBs, p);
}

template <bool SPLIT3>
cudaError_t launch_bn(int bn, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& bs, const GemmParams& p,
                      dim3 grid, cudaStream_t st) {
    switch (bn) {
        case 64: return launch_impl<64, SPLIT3>(a, b, bs, p, grid, st);
        case 128: return launch_impl<128, SPLIT3>(a, b, bs, p, grid, st);
        case 256: return launch_impl<256, SPLIT3>(a, b, bs, p, grid, st);
        default: return cudaErrorInvalidValue;
    }
}

template <bool SPLIT3>
constexpr int stages_of(int bn) {
    return bn == 64 ? TcCfg<64, SPLIT3>::STAGES
                    : bn == 128 ? TcCfg<128, SPLIT3>::STAGES : TcCfg<256, SPLIT3>::STAGES;
}

template <bool SPLIT3>
constexpr size_t smem_of(int bn) {
    return bn == 64 ? TcCfg<64, SPLIT3>::SMEM : bn == 128 ? TcCfg<128, SPLIT3>::SMEM : TcCfg<256, SPLIT3>::SMEM;
}

}  // namespace

int tc_bk(bool split3) { return split3 ? TcCfg<256, true>::BK : TcCfg<256, false>::BK; }
int tc_stages(int bn, bool split3) { return split3 ? stages_of<true>(bn) : stages_of<false>(bn); }
int tc_threads(int bn, bool split3) {
    if (!split3) return TcCfg<256, false>::THREADS;
    return bn == 64 ? TcCfg<64, true>::THREADS : (bn == 128 ? TcCfg<128, true>::THREADS : TcCfg<256, true>::THREADS);
}
size_t tc_smem_bytes(int bn, bool split3) { return split3 ? smem_of<true>(bn) : smem_of<false>(bn); }

cudaError_t launch_tc_sk(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmBs, const GemmParams& p,
                         int bn, int ctas, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(ctas), 1);
    if (bn != 128) return cudaErrorInvalidValue;  // the planner takes stream-K for the 128-wide tile only
    return launch_impl<128, true, true>(tmA, tmB, tmBs, p, grid, stream);
}

cudaError_t launch_tc(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmBs, const GemmParams& p,
                      int bn, bool split3, dim3 grid, cudaStream_t stream) {
    if (p.b_presplit && !(split3 && bn <= 128)) return cudaErrorInvalidValue;  // pre-split B: fused 3xTF32 only
    return split3 ? launch_bn<true>(bn, tmA, tmB, tmBs, p, grid, stream)
                  : launch_bn<false>(bn, tmA, tmB, tmBs, p, grid, stream);
}

}  // namespace pg
