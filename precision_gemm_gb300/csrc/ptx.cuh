// Thin inline-PTX wrappers for the sm_103a features the kernels use:
// mbarriers, TMA tile loads, tcgen05 (tensor memory + MMA), and the timer
// that bounds every wait.  Each wrapper is one PTX instruction (or a short
// fixed sequence) as documented in the PTX ISA for sm_100-family targets.
#pragma once

#include <cuda.h>
#include <cstdint>

#include "internal.h"

namespace pg {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The dynamic shared-memory base rounded up to 1 KiB (the 128-byte swizzle
// atom).  The offset is added to the __shared__ array itself so the compiler
// keeps the shared address space: loads through the result are ld.shared with
// 32-bit addresses, not generic loads.
__device__ __forceinline__ uint8_t* align_smem_1024(uint8_t* base) {
    return base + ((1024u - (smem_u32(base) & 1023u)) & 1023u);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ----------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

// CLUSTER: acquire at cluster scope, for phases completed by arrivals from other
// CTAs of the cluster whose shared-memory writes the waiter must then see.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    if (CLUSTER)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with parity `parity` to complete, for at most
// `timeout_ns`.  Returns false when the limit passes, or (when abort_flag is
// non-null) as soon as another thread of the CTA has raised the abort flag.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                                  const volatile int* abort_flag) {
    if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
#pragma unroll 1
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait<CLUSTER>(bar, parity)) return true;
        if (abort_flag != nullptr && *abort_flag) return false;
        if (global_timer_ns() - t0 > timeout_ns) return false;
    }
}

// A warp's wait for a phase of `bar`: lane 0 alone polls (bounded); once it has
// seen the phase complete, every lane runs its own wait, which then succeeds at
// its first test and gives that lane the acquire ordering on the data the phase
// guards (a lane's reads of TMA-written shared memory are ordered only by its
// own acquire).  One polling lane instead of 32 keeps the barrier's shared-memory
// traffic off the banks the operand reads use.  Returns the warp-uniform outcome.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                               const volatile int* abort_flag) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait_bounded(bar, parity, timeout_ns, abort_flag);
    if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) return false;
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, timeout_ns, abort_flag));
}

// Record a failed wait: raise the CTA's abort flag and the device status word.
__device__ __forceinline__ void raise_abort(volatile int* abort_flag, int* status) {
    *abort_flag = 1;
    __threadfence_block();
    atomicCAS(status, 0, kStatusTimeout);
}

// ---- 3xTF32 split ------------------------------------------------------------------

// x = big + small with big holding x's leading 11 significant bits (the TF32
// format: 8-bit exponent, 10 stored mantissa bits), rounded to nearest with
// ties away from zero by adding half a TF32 unit to the magnitude bits before
// clearing the low 13 bits.  small = x - big is exact in FP32 (|small| is at
// most half a TF32 unit of x); a finite value whose rounding would overflow is
// truncated.  An infinity becomes big = +-1, small = +-infinity: its products
// then carry the infinity through the remainder only, so infinity times a
// finite nonzero value is an infinity of the right sign and times zero is NaN,
// as in FP32 (with big = infinity, the big * small term would add an infinity
// of the other remainder's sign, or NaN for a zero remainder).  NaN: both NaN.
__device__ __forceinline__ void split_tf32(float x, float& big, float& small) {
    const uint32_t u = __float_as_uint(x);
    if (!isfinite(x)) {
        big = isnan(x) ? x : __uint_as_float((u & 0x80000000u) | 0x3F800000u);
        small = x;
        return;
    }
    float b = __uint_as_float((u + 0x1000u) & 0xFFFFE000u);
    if (!isfinite(b)) b = __uint_as_float(u & 0xFFFFE000u);
    big = b;
    small = x - b;
}

// split_tf32 over N values at once, for the on-chip splits: the rounding (add
// half a TF32 unit, clear the 13 low bits) and the exact remainder for every
// value, then one test for the rare inputs that need split_tf32's care -- an
// infinite or NaN input, or a finite one whose rounding reaches the all-ones
// exponent -- which redoes the batch value by value.  Same results as
// split_tf32 on every input, in fewer instructions per value.
template <int N>
__device__ __forceinline__ void split_tf32_batch(const float (&x)[N], uint32_t (&big)[N], uint32_t (&small)[N]) {
    // The rare inputs are NaN and magnitudes from 0x7F7FF000 up (infinities, and
    // finite values that round to the all-ones exponent): one NaN-propagating
    // maximum of the magnitudes per value finds them (one instruction where
    // tracking the exponents of x and big took two; 8192 x 64 x 8192 3xTF32
    // 0.0774 -> 0.0748 ms).
    float vmax = 0.0f;
#pragma unroll
    for (int k = 0; k < N; ++k) {
        const uint32_t u = __float_as_uint(x[k]);
        const uint32_t b = (u + 0x1000u) & 0xFFFFE000u;
        big[k] = b;
        small[k] = __float_as_uint(x[k] - __uint_as_float(b));
        asm("max.NaN.xorsign.abs.f32 %0, %0, %1;" : "+f"(vmax) : "f"(x[k]));
    }
    if (!(fabsf(vmax) < __uint_as_float(0x7F7FF000u))) {
#pragma unroll
        for (int k = 0; k < N; ++k) {
            float bf, sf;
            split_tf32(x[k], bf, sf);
            big[k] = __float_as_uint(bf);
            small[k] = __float_as_uint(sf);
        }
    }
}

// Split the BYTES of FP32 values at `tile` (shared memory, TMA-written) in
// place: each value becomes its TF32 big part and its remainder goes to the same
// offset in `small`.  A swizzled layout is a function of the byte address inside
// 1 KiB-aligned atoms, so with both regions 1 KiB aligned the remainder tile has
// the layout of the big one.  Thread t of NTHREADS takes the 16-byte chunks t,
// t + NTHREADS, ... (a warp covers 512 contiguous bytes) and loads all of its
// chunks before it stores any: a load that might alias an earlier store of the
// same thread would otherwise wait for it.
template <int BYTES, int NTHREADS>
__device__ __forceinline__ void split_tile_in_place(uint8_t* tile, uint8_t* small, int t) {
    static_assert(BYTES % (16 * NTHREADS) == 0, "whole chunks per thread");
    constexpr int CH = BYTES / (16 * NTHREADS);
    float4 v[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) v[c] = *reinterpret_cast<const float4*>(tile + 16 * (t + c * NTHREADS));
    constexpr int G = CH < 4 ? CH : 4;  // chunks split per batch
    static_assert(CH % G == 0, "whole batches");
#pragma unroll
    for (int c0 = 0; c0 < CH; c0 += G) {
        float x[4 * G];
#pragma unroll
        for (int c = 0; c < G; ++c) {
            x[4 * c] = v[c0 + c].x;
            x[4 * c + 1] = v[c0 + c].y;
            x[4 * c + 2] = v[c0 + c].z;
            x[4 * c + 3] = v[c0 + c].w;
        }
        uint32_t big[4 * G], sml[4 * G];
        split_tf32_batch<4 * G>(x, big, sml);
#pragma unroll
        for (int c = 0; c < G; ++c) {
            const int off = 16 * (t + (c0 + c) * NTHREADS);
            *reinterpret_cast<uint4*>(tile + off) = make_uint4(big[4 * c], big[4 * c + 1], big[4 * c + 2], big[4 * c + 3]);
            *reinterpret_cast<uint4*>(small + off) = make_uint4(sml[4 * c], sml[4 * c + 1], sml[4 * c + 2], sml[4 * c + 3]);
        }
    }
}

// ---- programmatic dependent launch ---------------------------------------------

// In a kernel launched with launch_after_previous: block until the previous
// kernel in the stream has completed and its memory operations are visible.
// Returns at once in a kernel launched the ordinary way.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Let a dependent kernel (launched with launch_after_previous) be scheduled
// once every CTA of this grid has issued this or exited.  The dependent still
// waits for this grid's completion before it reads anything.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Where the GEMM kernels let their dependent kernel be scheduled: at their
// start (1), or once their main loop has issued its last copy (0).
#ifndef PG_PDL_EARLY
#define PG_PDL_EARLY 0
#endif

// ---- TMA -----------------------------------------------------------------------

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of the box at (x, y) (x is the contiguous coordinate, always a
// multiple of 4 elements here) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 3-D tiled load of the box at (x, y, z) (x contiguous, a multiple of 4 elements).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// 2-D tiled store of the shared-memory box at `src` to (x, y) of the tensor (x
// contiguous, a multiple of 4 elements, never negative); elements of the box
// outside the tensor are not written.  Completes through the bulk-group
// mechanism: bulk_commit() then bulk_wait_read() before `src` may be reused or
// the CTA may exit.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// ---- tcgen05 -----------------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t holder_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(holder_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::tf32, one CTA.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc], kind::tf32, one CTA: A is read from
// tensor memory, row i of the M = 128 rows in lane i, one TF32 value per 32-bit
// column (K = 8 columns from a_tmem on).
__device__ __forceinline__ void mma_tf32_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every previously issued tcgen05 operation of this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 consecutive 32-bit columns of the warp's 32 TMEM lanes: thread t gets
// lane (base lane + t), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Thread t writes r[0..31] to lane (base lane + t), columns [col, col + 32).
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Thread t writes r[0..15] to lane (base lane + t), columns [col, col + 16).
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// 16 consecutive 32-bit columns of the warp's 32 TMEM lanes: thread t gets
// lane (base lane + t), columns [col, col + 16).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (all in 16-byte units), fixed version bits 46-47 = 1,
// base offset 0, and the swizzle layout in bits 61-63.
// kSwizzle128B32 is the 128-byte swizzle with 32-byte atoms (32-byte chunks of
// each 128-byte row XOR-ed with row % 4, atoms of 4 rows = 512 B): the layout an
// M/N-major TF32 operand needs, written by TMA's SWIZZLE_128B_ATOM_32B mode.
enum SmemLayout : uint32_t {
    kSwizzleNone = 0,
    kSwizzle128B32 = 1,
    kSwizzle128B = 2,
    kSwizzle64B = 4,
    kSwizzle32B = 6
};

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t layout) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(layout & 7u) << 61;
    return d;
}

// Descriptor of the 8-deep k-step kk of an operand tile at shared address `tile`
// (BK k-values per ring slot), in one of the two canonical TF32 layouts:
//   K-major  : one row of BK floats per M/N index, the 128-byte swizzle (BK 32,
//              8-row atoms of 1 KiB) or 64-byte swizzle (BK 16, 512-B atoms);
//              the k-step starts 32 bytes further into each row.
//   M/N-major: groups of 32 M/N indices, each BK rows of 128 bytes (one per k) in
//              the 128-byte swizzle with 32-byte atoms; leading byte offset (between
//              groups) 128*BK, stride byte offset (between 4-row atoms) 512; the
//              k-step starts 8 rows (1 KiB) further.
template <int BK>
__device__ __forceinline__ uint64_t operand_desc(uint32_t tile, int kk, bool k_major) {
    if (k_major)
        return smem_desc(tile + 32 * kk, 16, BK == 32 ? 1024 : 512, BK == 32 ? kSwizzle128B : kSwizzle64B);
    return smem_desc(tile + 1024 * kk, 128 * BK, 512, kSwizzle128B32);
}

// Instruction descriptor for kind::tf32 with FP32 accumulation: D format F32
// (bits 4-5 = 1), A and B format TF32 (bits 7-9 and 10-12 = 2), A major-ness
// (bit 15: 1 = M-major), B major-ness (bit 16: 0 = K-major), N/8 in bits 17-22,
// M/16 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// ---- shared-memory vector access -----------------------------------------------------

__device__ __forceinline__ float4 lds128(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}

// Stream-K: the CTA whose range [c T / G, (c + 1) T / G) of the T (tile,
// k-block) iterations holds iteration `it` -- the largest c with c T / G <= it.
__device__ __forceinline__ int sk_cta_of(int64_t it, int G, int64_t T) {
    return static_cast<int>(((it + 1) * G - 1) / T);
}

// Output tile position for CTA `tile` under grouped rasterisation: consecutive
// CTAs walk `group_m` tile rows of one tile column before moving right, so a
// wave of CTAs shares A row-panels and B column-panels in L2.
__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int group_m, int& tm,
                                            int& tn) {
    const int per_group = group_m * tiles_n;
    const int g = tile / per_group;
    const int first = g * group_m;
    const int rows = min(tiles_m - first, group_m);
    const int r = tile - g * per_group;
    tm = first + r % rows;
    tn = r / rows;
}

}  // namespace pg
