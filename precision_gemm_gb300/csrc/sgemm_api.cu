// C ABI of the library (declared in include/precision_gemm.h): argument checks,
// planning (kernel, tile, split-K, operand preparation), the per-(device,
// stream) workspace, TMA tensor-map encoding and the launch sequence.
//
// The host-side flow follows the lecture's matmatgpu1 ("HPC - Lecture 13 -
// MatMat GPU"): operands with leading dimensions are brought into the layout the
// kernel wants, the kernel runs, and C is written back -- except that here the
// operands already live on the device, the "packing" is a device pre-pass that
// runs only when TMA cannot read an operand in place, and nothing is copied
// through the host (sgemm_host is the variant that starts from host arrays).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/precision_gemm.h"
#include "host_sgemm.h"
#include "internal.h"

#define PG_EXPORT extern "C" __attribute__((visibility("default")))

namespace pg {

// Per-device status word written by kernels whose bounded wait expired.
__device__ int g_device_status;

namespace {

// FFMA: whole-tile results with beta = 0 leave through TMA stores (1) or
// through thread stores of whole columns (0).
#ifndef PG_FFMA_TMA_STORE
#define PG_FFMA_TMA_STORE 1
#endif
// Tile rows per rasterisation group (a compile-time tunable; 4, 8 and 16 measured
// within noise of each other at 8192^3; 8 and 32 slower than 16 for the SM-pair
// kernels: TF32 1.087 -> 1.096 / 1.098 ms).
#ifndef PG_GROUP_M
#define PG_GROUP_M 16
#endif
// The FFMA kernel's own group: at 8192^3 (128 x 64 tiles) groups of 8 tile rows
// cut its DRAM reads from 5.00 to 4.08 GB a launch (2: 9.55, 4: 5.69) at the same
// time (17.13 ms), and 4096^3, 6144^3 and 2048^3 run the same with any of them.
#ifndef PG_FFMA_GROUP_M
#define PG_FFMA_GROUP_M 8
#endif

// FFMA stream-K (a compile-time switch): products whose tiles fill less than
// PG_FFMA_SK_FILL percent of one wave of CTA slots, even after a K split, with
// at least 4 k-blocks per CTA, run on the stream-K kernel.
#ifndef PG_FFMA_SK
#define PG_FFMA_SK 1
#endif
#ifndef PG_FFMA_SK_FILL
#define PG_FFMA_SK_FILL 90
#endif
// K slices of a last-wave tile at most: FFMA (measured, 128 x 64 tiles at 2048^2 x
// 4096: 0.587 -> 0.574 ms with 8 against 4) and SM pairs
#ifndef PG_TAIL_MAX_SPLIT
#define PG_TAIL_MAX_SPLIT 8
#endif
#ifndef PG_TAIL_MAX_SPLIT_PAIRS
#define PG_TAIL_MAX_SPLIT_PAIRS 4
#endif
#ifndef PG_FFMA_SK_MIN_KB
#define PG_FFMA_SK_MIN_KB 4  // k-blocks per CTA at least
#endif
constexpr int kSkMaxSegsPerCta = 8;  // the kernels' segment tables
// 3xTF32 stream-K on the single-SM tensor-core kernel (a compile-time switch),
// at least PG_TC_SK_MIN_KB k-blocks per CTA.
#ifndef PG_TC_SK
#define PG_TC_SK 1
#endif
#ifndef PG_TC_SK_MIN_KB
#define PG_TC_SK_MIN_KB 32
#endif


constexpr int kMaxDevices = 64;
constexpr const char* kVersion = "precision_gemm_gb300 0.1.0 (sm_103a; FFMA, TF32, 3xTF32)";

thread_local char t_err[512] = "no error";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof t_err, fmt, ap);
    va_end(ap);
    return code;
}

int fail_cuda(cudaError_t e, const char* what) {
    return fail(SGEMM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

std::atomic<uint64_t> g_timeout_ns{4000000000ull};
std::atomic<int> g_force_bn{0};
std::atomic<int> g_force_split{0};
std::atomic<int> g_debug{0};
std::atomic<uint64_t> g_launches{0};

bool is_notrans(char t) { return t == 'N' || t == 'n'; }
bool valid_trans(char t) { return t == 'N' || t == 'n' || t == 'T' || t == 't' || t == 'C' || t == 'c'; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int64_t round_up(int64_t x, int64_t q) { return (x + q - 1) / q * q; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1024;  // TMA coordinates (tile + box) are 32-bit
constexpr int64_t kMaxLd = (int64_t(1) << 37);        // TMA strides are < 2^40 bytes

// Checks in the order of the signature; returns 0 or -i.
int validate(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha, const void* A,
             int64_t lda, const void* B, int64_t ldb, float beta, const void* C, int64_t ldc, int mode) {
    if (!valid_trans(transa)) return fail(-1, "argument 1 (transa): '%c' is not N, T or C", transa);
    if (!valid_trans(transb)) return fail(-2, "argument 2 (transb): '%c' is not N, T or C", transb);
    if (m < 0 || m > kMaxDim) return fail(-3, "argument 3 (m): %lld out of [0, 2^31-1024]", (long long)m);
    if (n < 0 || n > kMaxDim) return fail(-4, "argument 4 (n): %lld out of [0, 2^31-1024]", (long long)n);
    if (k < 0 || k > kMaxDim) return fail(-5, "argument 5 (k): %lld out of [0, 2^31-1024]", (long long)k);
    const bool reads_ab = m > 0 && n > 0 && k > 0 && alpha != 0.0f;
    if (reads_ab && A == nullptr) return fail(-7, "argument 7 (A): null pointer");
    const int64_t rows_a = is_notrans(transa) ? m : k;
    if (lda < std::max<int64_t>(1, rows_a) || lda > kMaxLd)
        return fail(-8, "argument 8 (lda): %lld < max(1, %lld) or too large", (long long)lda, (long long)rows_a);
    if (reads_ab && B == nullptr) return fail(-9, "argument 9 (B): null pointer");
    const int64_t rows_b = is_notrans(transb) ? k : n;
    if (ldb < std::max<int64_t>(1, rows_b) || ldb > kMaxLd)
        return fail(-10, "argument 10 (ldb): %lld < max(1, %lld) or too large", (long long)ldb, (long long)rows_b);
    const bool touches_c = m > 0 && n > 0 && (reads_ab || beta != 1.0f);
    if (touches_c && C == nullptr) return fail(-12, "argument 12 (C): null pointer");
    if (ldc < std::max<int64_t>(1, m) || ldc > kMaxLd)
        return fail(-13, "argument 13 (ldc): %lld < max(1, %lld) or too large", (long long)ldc, (long long)m);
    if (mode != SGEMM_FFMA && mode != SGEMM_TF32 && mode != SGEMM_3XTF32)
        return fail(-14, "argument 14 (mode): %d is not SGEMM_FFMA, SGEMM_TF32 or SGEMM_3XTF32", mode);
    (void)beta;
    return 0;
}

size_t region(int64_t elems) { return static_cast<size_t>(round_up(elems * 4, 256)); }

// Stream-K: the CTA whose range [c T / G, (c + 1) T / G) holds iteration it, and
// the most segments (CTAs) any tile is cut into -- the partial-block slots per tile.
int64_t sk_cta_of(int64_t it, int64_t G, int64_t T) { return ((it + 1) * G - 1) / T; }
// The most tiles (segments) any CTA's range touches.
int sk_segs_per_cta(int64_t tiles, int64_t kb, int64_t G) {
    const int64_t T = tiles * kb;
    int64_t most = 0;
    for (int64_t c = 0; c < G; ++c) {
        const int64_t it0 = c * T / G, it1 = (c + 1) * T / G;
        if (it1 > it0) most = std::max(most, (it1 - 1) / kb - it0 / kb + 1);
    }
    return static_cast<int>(most);
}
int sk_maxseg(int64_t tiles, int64_t kb, int64_t G) {
    const int64_t T = tiles * kb;
    int64_t most = 1;
    for (int64_t t = 0; t < tiles; ++t)
        most = std::max(most, sk_cta_of(t * kb + kb - 1, G, T) - sk_cta_of(t * kb, G, T) + 1);
    return static_cast<int>(most);
}

// Workspace of the last-wave split: the partial blocks, and one arrival counter
// per (tail tile, epilogue warp region).
size_t tail_bytes(const sgemm_plan_t& pl) {
    return region(static_cast<int64_t>(pl.tail_tiles) * pl.tail_split * pl.bm * pl.bn);
}
size_t tail_counter_bytes(const sgemm_plan_t& pl) {
    const int per_tile = pl.kernel == SGEMM_KERNEL_TC2 ? 2 * tc2_epilogue_warps() : pl.threads / 32;
    return region(static_cast<int64_t>(pl.tail_tiles) * per_tile);
}

// The planner.  Pure host arithmetic: no device is touched.  allow_tail = false
// (the allocation-free entry) never plans a last-wave split.
void make_plan(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha, const void* A,
               int64_t lda, const void* B, int64_t ldb, float beta, int mode, int num_sms, sgemm_plan_t* pl,
               bool allow_tail = true, int ffma_bn = 0) {
    std::memset(pl, 0, sizeof *pl);
    pl->mode = mode;
    pl->split_k = 1;
    pl->tail_split = 1;
    pl->bm = kBM;
    if (m == 0 || n == 0) {
        pl->kernel = SGEMM_KERNEL_NONE;
        return;
    }
    if (k == 0 || alpha == 0.0f) {
        pl->kernel = (beta == 1.0f) ? SGEMM_KERNEL_NONE : SGEMM_KERNEL_SCALE;
        pl->launches = (pl->kernel == SGEMM_KERNEL_SCALE) ? 1 : 0;
        return;
    }
    const bool tc = mode != SGEMM_FFMA;
    const bool split3 = mode == SGEMM_3XTF32;

    // Tile width: 64 for n <= 64; otherwise 128 for the FFMA kernel (two CTAs per
    // SM measured fastest) and the narrowest of 128/256 covering n for tcgen05 --
    // except that a tensor-core product whose 128 x 64 tiles fit in one wave of
    // SMs runs on those (single-SM kernel) when it is 3xTF32 (which there splits
    // on chip instead of running two pre-passes over A and B) or a TF32 product
    // under 4 GFLOP (lowest latency up to ~1024^3; with long K the SM pairs and a
    // K split stream A faster).
    // Tiny FFMA products (under 2 GFLOP, their 128 x 64 tiles filling at most half
    // the SMs) take the 64-wide tile too, with thinner K slices below: more CTAs
    // share the few k-blocks; so do FFMA products with K <= 64 (below).
    int bn = n <= 64 ? 64 : ((n <= 128 || !tc) ? 128 : 256);
    const int64_t tiles64 = cdiv(m, kBM) * cdiv(n, 64);
    const bool one_wave64 = tc && tiles64 <= std::max(num_sms, 1);
    if (one_wave64 && (split3 || 2.0 * m * n * k <= 4e9)) bn = 64;
    // 128-wide tiles on single SMs (128 x 128 x 8 MMAs run at the full rate,
    // 128 x 64 x 8 ones at two thirds, and each issue carries twice the work):
    //  - one row of tiles (m <= 128) whose 128-wide tiles fit in one wave, for
    //    3xTF32 and for TF32 above 4 GFLOP: 3xTF32 128 x 4096 x 8192 0.099 ->
    //    0.071 ms, 128 x 128 x 262144 0.087 -> 0.065; TF32 128 x 4096 x 8192
    //    0.044 -> 0.040 (256-wide tiles before);
    //  - 3xTF32 whose 64-wide tiles fit in one wave and whose K is long (>= 2048):
    //    4096 x 128 x 8192 0.098 -> 0.070 ms, 512 x 256 x 32768 0.087 -> 0.062;
    //    with short K the halved tile count costs more (1024^3 0.031 -> 0.034).
    const bool single128 =
        tc && n > 64 &&
        ((m <= kBM && cdiv(n, 128) <= std::max(num_sms, 1) && (split3 || 2.0 * m * n * k > 4e9)) ||
         (split3 && one_wave64 && k >= 2048));
    if (single128) bn = 128;
    const bool tiny_ffma = !tc && 2 * tiles64 <= std::max(num_sms, 1) && 2.0 * m * n * k <= 2e9;
    if (tiny_ffma) bn = 64;
    // FFMA with at most two k-blocks (K <= 64): a CTA's prologue and epilogue weigh
    // as much as its arithmetic, and three 128 x 64 CTAs per SM overlap them better
    // than two 128 x 128 ones: 16384^2 x 64 0.654 -> 0.611 ms, 16384^2 x 32 0.422 ->
    // 0.345, 8192^2 x 64 0.169 -> 0.158 (K = 128 1 % slower, K = 256 even).
    if (!tc && k <= 2 * kFfmaBK) bn = 64;
    // FFMA over several waves: 128 x 128 tiles (two CTAs per SM) and 128 x 64 tiles
    // (three) reach the same throughput within a wave, so the tile whose grid fills
    // its waves better wins (the 128 x 64 one on a tie); the estimate counts a last
    // wave at most half full as 1/s of a wave when it is split s ways along K.  Only with K >= 2048, where
    // the split slices stay long, or with K >= 512 and two or more waves of 128 x 64
    // tiles (the ragged 3000 x 1500 x 777 problem, 1.26 waves, ran 16 % slower on
    // 128 x 64 tiles).  Measured (L2 flushed): 4096^3 0.962 -> 0.998 of the waves
    // filled, 2.250 -> 2.174 ms; 6144^3 7.61 -> 7.25; 4096^2 x 2048 1.140 -> 1.099;
    // 4096^2 x 1024 0.585 -> 0.563; 4096 x 8192 x 1536 1.682 -> 1.627; 8192^2 x 512
    // 1.112 -> 1.092; ties: 8192^2 x 1024 2.179 -> 2.162, 16384^2 x 1024 even,
    // 1024 x 15409 x 1903 1.045 -> 1.051.
    const bool ffma_waves64 = k >= 2048 || (k >= 512 && tiles64 >= 2 * std::max(num_sms, 1) * ffma_ctas_per_sm(64));
    if (!tc && bn == 128 && ffma_bn == 0 && ffma_waves64) {
        const int64_t kb = cdiv(k, kFfmaBK);
        auto filled = [&](int64_t tiles, int64_t cap) {
            const int64_t full = tiles / cap, rem = tiles % cap;
            double waves = static_cast<double>(full) + (rem > 0 ? 1.0 : 0.0);
            if (rem > 0 && full >= 1 && 2 * rem <= cap && allow_tail) {
                const int64_t sp = std::min<int64_t>({cap / rem, PG_TAIL_MAX_SPLIT, kb / 8});
                if (sp >= 2) waves = static_cast<double>(full) + 1.0 / static_cast<double>(sp);
            }
            return static_cast<double>(tiles) / (static_cast<double>(cap) * waves);
        };
        const int64_t sms = std::max(num_sms, 1);
        const int64_t t128 = cdiv(m, kBM) * cdiv(n, 128);
// On a tie (within 0.01) the 128 x 64 tile: it also runs spill-free (158
// registers at three CTAs per SM against 48 B of spills at the 128-register cap
// of the 128 x 128 tile) and measured a little faster: 8192^3 17.168 -> 17.132
// ms, 16384^3 137.02 -> 136.64, 8192^2 x 2048 4.345 -> 4.318 (beta = 1).
#ifndef PG_FFMA_PREFER64
#define PG_FFMA_PREFER64 1
#endif
        const double f64 = filled(tiles64, sms * ffma_ctas_per_sm(64));
        const double f128 = filled(t128, sms * ffma_ctas_per_sm(128));
        if (t128 >= sms * ffma_ctas_per_sm(128) && (PG_FFMA_PREFER64 ? f64 >= f128 - 0.01 : f64 > f128 + 0.01))
            bn = 64;
    }
    if (ffma_bn) bn = ffma_bn;  // the re-plan below
    // TF32 on SM pairs: 256 x 512 tiles (two N = 256 MMAs per k-step) need 48 B/clk
    // per SM of operand feed at the full MMA rate against 64 for 256 x 256 tiles
    // (bulk copies sustain ~65 per SM), at the price of a single TMEM accumulator
    // (the epilogue of a tile no longer overlaps the next tile's MMAs).  With K >=
    // 2048 a wave of 256 x 512 tiles takes about 1.8 times as long as a wave of
    // 256 x 256 ones (half the tiles), so the wider tile wins when 1.8 x its waves
    // (a partial last wave counted whole: it is not split, the split's 512-column
    // partial blocks measured slower than a whole extra wave) is under the 256-wide
    // grid's waves (a last wave at most half full split s ways counted as 1/s + 0.4,
    // the 0.4 for the slices' partial blocks and their sum).  Measured (L2 flushed,
    // ms, 256 -> 512): 4096^3 0.178 -> 0.160, 4096^2 x 2048 0.106 -> 0.089, 8192^2 x
    // 2048 0.321 -> 0.302, 16384 x 4096 x 4096 0.611 -> 0.562, 3000 x 5000 x 4096
    // 0.202 -> 0.163, 8192^3 1.17 -> 1.09; kept at 256: 3072 x 4096 x 4096 0.134
    // (0.170 on 512), 4096 x 2560 x 4096 0.142 (0.179).
    if (tc && !split3 && m > kBM && bn == 256 && k >= 2048) {
        const int64_t pairs = std::max(num_sms / 2, 1);
        const int64_t t512 = cdiv(m, 2 * kBM) * cdiv(n, 512), t256 = cdiv(m, 2 * kBM) * cdiv(n, 256);
        if (t512 >= pairs) {
            const int64_t full = t256 / pairs, rem = t256 % pairs;
            double w256 = static_cast<double>(full) + (rem > 0 ? 1.0 : 0.0);
            if (rem > 0 && full >= 1 && 2 * rem <= pairs && allow_tail) {
                const int64_t sp = std::min<int64_t>({pairs / rem, PG_TAIL_MAX_SPLIT_PAIRS, cdiv(k, tc2_bk(false)) / 8});
                if (sp >= 2) w256 = static_cast<double>(full) + 1.0 / static_cast<double>(sp) + 0.4;
            }
            if (1.8 * static_cast<double>(cdiv(t512, pairs)) < w256) bn = 512;
        }
    }
    const int fbn = g_force_bn.load();
    if (fbn) bn = (fbn == 512 && (!tc || split3 || m <= kBM)) ? 256 : fbn;  // 512: TF32 on SM pairs only
    pl->bn = bn;
    // Tensor-core modes run on SM pairs (256-row tiles, cta_group::2) when m > 128;
    // a single-SM 128-row tile serves m <= 128, the 64-wide tile and the 128-wide
    // tiles chosen above.
    const bool pair = tc && m > kBM && bn >= 128 && !(single128 && fbn == 0);

    // Operand preparation: TMA needs a 16-byte aligned base and a leading
    // dimension that is a multiple of 16 bytes.  The tensor-core kernels read
    // either orientation of A and B (K-major or M/N-major descriptors), so their
    // copies and 3xTF32 splits keep the stored orientation; the FFMA kernel reads
    // A M-major and B K-major only, so a transposed operand is copied transposed.
    // 3xTF32 on SM pairs reads operands split by a pre-pass (the large shapes, where
    // the pre-pass is cheap next to the product); the single-SM kernel splits them
    // itself on chip (the narrow shapes, where a pre-pass would dominate).
    // The single-SM kernel's on-chip split of B is repeated by every row of tiles
    // that shares B; from four rows of tiles and K >= 4096 on, a pre-pass splits B
    // once and TMA brings both parts (64- and 128-wide tiles, whose sub-slots keep
    // room for B's remainders): 3xTF32 8192 x 64 x 8192 0.0925 -> 0.0870 ms,
    // 8192 x 128 x 8192 0.121 -> 0.103; with short K the pre-pass launch costs more
    // than it saves (1024^3 0.027 -> 0.033).
    const bool a_ok = aligned16(A) && (lda % 4 == 0);
    const bool b_ok = aligned16(B) && (ldb % 4 == 0);
    const bool presplit_b = split3 && !pair && bn <= 128 && cdiv(m, kBM) >= 4 && k >= 4096;
    if (split3 && pair) {
        pl->prep_a = SGEMM_PREP_SPLIT;
        pl->prep_b = SGEMM_PREP_SPLIT;
    } else if (tc) {
        pl->prep_a = a_ok ? SGEMM_PREP_NONE : SGEMM_PREP_COPY;
        pl->prep_b = presplit_b ? SGEMM_PREP_SPLIT : (b_ok ? SGEMM_PREP_NONE : SGEMM_PREP_COPY);
    } else {
        pl->prep_a = (a_ok && is_notrans(transa)) ? SGEMM_PREP_NONE
                                                  : (is_notrans(transa) ? SGEMM_PREP_COPY : SGEMM_PREP_TRANSPOSE);
        pl->prep_b = (b_ok && is_notrans(transb)) ? SGEMM_PREP_NONE
                                                  : (is_notrans(transb) ? SGEMM_PREP_COPY : SGEMM_PREP_TRANSPOSE);
    }
    // Stored rows of each operand as the kernel reads it.
    const int64_t rows_a = (tc && !is_notrans(transa)) ? k : m;
    const int64_t rows_b = (tc && !is_notrans(transb)) ? n : k;
    pl->ld_a = pl->prep_a == SGEMM_PREP_NONE ? lda : round_up(rows_a, 4);
    pl->ld_b = pl->prep_b == SGEMM_PREP_NONE ? ldb : round_up(rows_b, 4);

    pl->kernel = !tc ? SGEMM_KERNEL_FFMA : (pair ? SGEMM_KERNEL_TC2 : SGEMM_KERNEL_TC);
    pl->bm = pair ? 2 * kBM : kBM;
    pl->bk = !tc ? kFfmaBK : (pair ? tc2_bk(split3) : tc_bk(split3));
    pl->stages = !tc ? ffma_stages(bn) : (pair ? tc2_stages(bn, split3) : tc_stages(bn, split3));
    pl->threads = !tc ? ffma_threads(bn) : (pair ? tc2_threads() : tc_threads(bn, split3));
    pl->ctas_per_sm = tc ? 1 : ffma_ctas_per_sm(bn);
    pl->smem_bytes = !tc ? ffma_smem_bytes(bn) : (pair ? tc2_smem_bytes(bn, split3) : tc_smem_bytes(bn, split3));
    pl->tiles_m = static_cast<int>(cdiv(m, pl->bm));
    pl->tiles_n = static_cast<int>(cdiv(n, bn));
    pl->k_blocks = static_cast<int>(cdiv(k, pl->bk));

    // Split-K when the output tiles cannot fill one wave of the machine: give
    // each tile up to floor(capacity / tiles) K slices (capacity counts SM pairs
    // for the pair kernel).  A slice must carry enough work to repay the partial
    // sums' round trip and the reduction launch, which the tensor cores reach
    // only with longer K: FFMA splits into slices of at least 128 of K; TF32 only
    // when K >= 2048, into slices of at least 512; 3xTF32 only when K >= 512,
    // into slices of at least 128; tiny FFMA products into slices of 64
    // (measured on 256^3 .. 2048^3, K up to 262144).
    const int64_t tiles = static_cast<int64_t>(pl->tiles_m) * pl->tiles_n;
    const int64_t capacity =
        pair ? std::max(num_sms / 2, 1) : static_cast<int64_t>(std::max(num_sms, 1)) * pl->ctas_per_sm;
    int64_t split = 1;
    const int fs = g_force_split.load();
    if (fs > 0) {
        split = fs;
    } else {
        const int64_t min_k_slice = (tc && !split3) ? 512 : (tiny_ffma ? 64 : 128);
        const int64_t min_k_total = !tc ? 0 : (split3 ? 512 : 2048);
        if (tiles < capacity && k >= min_k_total)
            split = std::min<int64_t>(capacity / tiles, pl->k_blocks / cdiv(min_k_slice, pl->bk));
    }
    split = std::max<int64_t>(1, std::min<int64_t>({split, static_cast<int64_t>(pl->k_blocks), 65535}));
    int64_t per = cdiv(pl->k_blocks, split);
    split = cdiv(pl->k_blocks, per);  // no empty slice

    // FFMA stream-K: when the tiles (times their K slices) leave more than a
    // tenth of the wave's CTA slots idle, every slot takes an equal share of all
    // (tile, k-block) iterations instead -- at least 4 k-blocks each (measured:
    // 2048^3 0.341 -> 0.324 ms and 8192 x 64 x 8192 0.191 -> 0.169 at 54 per CTA).
    // The minimum was 32 while the fix-up was an ordinary launch and the tiles
    // 128 wide (1024^3 at 7 and 1000 x 1300 x 1500 at 14 per CTA were slower than
    // the K split then); with the fix-up dependent-launched and 128 x 64 tiles at
    // three CTAs per SM, 4 measured best: row-major 1024^3 0.0549 -> 0.0532 ms,
    // 1024^2 x 2048 0.0948 -> 0.0908, 1000 x 1300 x 1500 0.0948 -> 0.0903.
    if (PG_FFMA_SK && !tc && (bn == 64 || bn == 128) && fs == 0 && allow_tail && tiles < capacity &&
        100 * tiles * split < PG_FFMA_SK_FILL * capacity && tiles * pl->k_blocks >= PG_FFMA_SK_MIN_KB * capacity &&
        sk_segs_per_cta(tiles, pl->k_blocks, capacity) <= kSkMaxSegsPerCta) {
        split = 1;
        per = pl->k_blocks;
        pl->sk_ctas = static_cast<int>(capacity);
    }
    // 3xTF32 stream-K on the single-SM kernel's 128-wide tiles whose products
    // fill less than 90 % of the SMs even with a K split: every SM is given an
    // equal share.  Measured (L2 flushed): 8192 x 128 x 8192 0.102 -> 0.097 ms,
    // 4096 x 128 x 8192 0.064 -> 0.062, 128 x 4096 x 8192 0.067 -> 0.063; on the
    // 64-wide tile slower (8192 x 64 x 8192 0.083 -> 0.089, 5000 x 60 x 12000
    // 0.082 -> 0.084), so it keeps the K split there.
    if (PG_TC_SK && split3 && !pair && bn == 128 && fs == 0 && allow_tail && tiles < capacity &&
        100 * tiles * split < PG_FFMA_SK_FILL * capacity && tiles * pl->k_blocks >= PG_TC_SK_MIN_KB * capacity &&
        sk_segs_per_cta(tiles, pl->k_blocks, capacity) <= kSkMaxSegsPerCta) {
        split = 1;
        per = pl->k_blocks;
        pl->sk_ctas = static_cast<int>(capacity);
    }
    pl->split_k = static_cast<int>(split);
    pl->k_blocks_per_split = static_cast<int>(per);

    // Last-wave split (SM pairs, and FFMA): when the tiles fill whole waves and a
    // last wave at most half full, cut each last-wave tile's K into s slices (at
    // least 8 K blocks each; s <= 4 on SM pairs, <= 8 for FFMA) so the last wave
    // keeps every pair (every FFMA CTA slot) busy.
    if ((pair || !tc) && split == 1 && pl->sk_ctas == 0 && g_force_split.load() == 0 && allow_tail &&
        (pl->bn != 512 || fbn == 512)) {  // 256 x 512 tiles: only when forced (slower than a whole wave)
        const int64_t waves = tiles / capacity, rem = tiles % capacity;
        if (waves >= 1 && rem > 0 && 2 * rem <= capacity) {
            const int64_t s = std::min<int64_t>(
                {capacity / rem, pair ? PG_TAIL_MAX_SPLIT_PAIRS : PG_TAIL_MAX_SPLIT, pl->k_blocks / 8});
            if (s >= 2) {
                pl->tail_tiles = static_cast<int>(rem);
                pl->tail_split = static_cast<int>(s);
            }
        }
    }

    size_t ws = 0;
    const int parts_a = pl->prep_a == SGEMM_PREP_SPLIT ? 2 : 1, parts_b = pl->prep_b == SGEMM_PREP_SPLIT ? 2 : 1;
    if (pl->prep_a != SGEMM_PREP_NONE) ws += parts_a * region(pl->ld_a * (rows_a == m ? k : m));
    if (pl->prep_b != SGEMM_PREP_NONE) ws += parts_b * region(pl->ld_b * (rows_b == k ? n : k));
    if (split > 1) ws += region(split * round_up(m, 4) * n);
    if (pl->tail_split > 1) ws += tail_bytes(*pl) + tail_counter_bytes(*pl);
    if (pl->sk_ctas > 0) ws += region(tiles * sk_maxseg(tiles, pl->k_blocks, pl->sk_ctas) * pl->bm * pl->bn);
    pl->workspace_bytes = ws;
    pl->launches = (pl->prep_a != SGEMM_PREP_NONE) + (pl->prep_b != SGEMM_PREP_NONE) + 1 + (split > 1) +
                   (pl->sk_ctas > 0);

    // FFMA products whose 128-wide tiles would run stream-K (under a wave of 304
    // CTA slots) run 128 x 64 tiles at three CTAs per SM instead (456 slots; stream-K
    // again, or a wave plus a last-wave split), which overlap the CTAs' prologues,
    // segment switches and epilogues better.  Measured (L2 flushed): 2048^3 0.3185 ->
    // 0.3065 ms, 1000 x 1300 x 4000 0.2208 -> 0.2075, 1100 x 700 x 6000 0.2024 ->
    // 0.1881, 1500 x 1300 x 6000 0.458 -> 0.445, 2048^2 x 4096 0.606 -> 0.587,
    // 1700^2 x 2048 0.2505 -> 0.2423; 1024^2 x 8192 even; 1250 x 1650 x 5000 0.3954
    // -> 0.4031.
    if (!tc && ffma_bn == 0 && pl->bn == 128 && pl->sk_ctas > 0 && g_force_bn.load() == 0)
        make_plan(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, mode, num_sms, pl, allow_tail, 64);
}

// ---- devices ------------------------------------------------------------------------

struct DeviceState {
    bool init = false;
    int sms = 0;
    int major = 0, minor = 0;
    int* status = nullptr;
};
std::mutex g_dev_mu;
DeviceState g_dev[kMaxDevices];

int current_device(int* dev_out, DeviceState** ds_out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return fail(SGEMM_ERR_NO_DEVICE, "no usable CUDA device: %s", cudaGetErrorString(e));
    }
    if (dev >= kMaxDevices) return fail(SGEMM_ERR_NO_DEVICE, "device ordinal %d unsupported", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceState& d = g_dev[dev];
    if (!d.init) {
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return fail_cuda(e, "cudaDeviceGetAttribute");
        if (d.major == 10 && d.minor == 3) {
            if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_device_status)) != cudaSuccess)
                return fail_cuda(e, "cudaGetSymbolAddress(status word)");
        }
        d.init = true;
    }
    if (!(d.major == 10 && d.minor == 3))
        return fail(SGEMM_ERR_ARCH, "device %d is compute capability %d.%d; this library is built for 10.3 (sm_103a)",
                    dev, d.major, d.minor);
    *dev_out = dev;
    *ds_out = &d;
    return 0;
}

// ---- workspace: one growing buffer per (device, stream, purpose) ---------------------

struct Buf {
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mu;
std::map<std::pair<std::pair<int, uintptr_t>, int>, Buf> g_bufs;
// Workspaces supplied by the caller (sgemm_set_workspace), per (device, stream):
// used in place of the library's own workspace buffer, never grown or freed here.
std::map<std::pair<int, uintptr_t>, Buf> g_user_ws;

constexpr int kPurposeWorkspace = 0;
constexpr int kPurposeStaging = 1;

int get_buffer(int dev, cudaStream_t st, int purpose, size_t need, void** out) {
    *out = nullptr;
    if (need == 0) return 0;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    if (purpose == kPurposeWorkspace) {
        auto u = g_user_ws.find({dev, reinterpret_cast<uintptr_t>(st)});
        if (u != g_user_ws.end()) {
            if (u->second.bytes < need)
                return fail(SGEMM_ERR_WORKSPACE,
                            "the call needs %zu bytes of workspace; the workspace given by sgemm_set_workspace for "
                            "this stream holds %zu",
                            need, u->second.bytes);
            *out = u->second.ptr;
            return 0;
        }
    }
    Buf& b = g_bufs[{{dev, reinterpret_cast<uintptr_t>(st)}, purpose}];
    if (b.bytes >= need) {
        *out = b.ptr;
        return 0;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone)
        return fail(SGEMM_ERR_CAPTURE,
                    "workspace must grow to %zu bytes during stream capture; make one call of this size "
                    "before capturing", need);
    if (g_debug.load() & SGEMM_DEBUG_FAIL_ALLOC)
        return fail(SGEMM_ERR_ALLOC, "injected allocation failure (SGEMM_DEBUG_FAIL_ALLOC) for %zu bytes", need);
    if (b.ptr) {
        if ((e = cudaFreeAsync(b.ptr, st)) != cudaSuccess) return fail_cuda(e, "cudaFreeAsync(workspace)");
        b.ptr = nullptr;
        b.bytes = 0;
    }
    const size_t bytes = static_cast<size_t>(round_up(static_cast<int64_t>(need), int64_t(2) << 20));
    if ((e = cudaMallocAsync(&b.ptr, bytes, st)) != cudaSuccess) {
        cudaGetLastError();
        b.ptr = nullptr;
        return fail(SGEMM_ERR_ALLOC, "cudaMallocAsync(%zu bytes) for the workspace: %s", bytes, cudaGetErrorString(e));
    }
    b.bytes = bytes;
    *out = b.ptr;
    return 0;
}

// [base, base + size) of the device allocation holding `p` (driver call
// cuMemGetAddressRange, reached through the runtime's entry-point query), or
// false when the driver cannot say.
bool allocation_range(const void* p, uintptr_t* base, size_t* size) {
    using RangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);
    static std::once_flag once;
    static RangeFn fn = nullptr;
    std::call_once(once, [] {
        void* q = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &q, 12000, cudaEnableDefault, &r) ==
                cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<RangeFn>(q);
    });
    if (!fn) return false;
    CUdeviceptr b = 0;
    size_t s = 0;
    if (fn(&b, &s, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS) return false;
    *base = static_cast<uintptr_t>(b);
    *size = s;
    return true;
}

// ---- TMA tensor maps ------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// A tensor map depends only on the arguments it is encoded from, so the maps of
// repeated calls on the same buffers are kept instead of re-encoded (a driver
// call each, two to four per product): a direct-mapped table of 256 entries,
// each with the arguments it was made from.
struct MapKey {
    const void* base;
    uint32_t rank;
    int32_t swizzle;
    cuuint64_t dims[3];
    cuuint64_t strides[2];
    cuuint32_t box[3];
};
struct MapEntry {
    MapKey key;
    CUtensorMap map;
    bool valid;
};
std::mutex g_map_mu;
MapEntry g_maps[256];

CUresult encode_cached(EncodeTiledFn fn, CUtensorMap* map, uint32_t rank, const float* base, const cuuint64_t* dims,
                       const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swizzle) {
    MapKey key;
    std::memset(&key, 0, sizeof key);  // padding included: keys compare as bytes
    key.base = base;
    key.rank = rank;
    key.swizzle = static_cast<int32_t>(swizzle);
    for (uint32_t i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
        if (i + 1 < rank) key.strides[i] = strides[i];
    }
    uint64_t h = 1469598103934665603ull;  // FNV-1a over the key's bytes
    const unsigned char* kb = reinterpret_cast<const unsigned char*>(&key);
    for (size_t i = 0; i < sizeof key; ++i) h = (h ^ kb[i]) * 1099511628211ull;
    MapEntry& slot = g_maps[h & 255];
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        if (slot.valid && std::memcmp(&slot.key, &key, sizeof key) == 0) {
            *map = slot.map;
            return CUDA_SUCCESS;
        }
    }
    const cuuint32_t elem[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<float*>(base), dims, strides, box,
                          elem, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) {
        std::lock_guard<std::mutex> lk(g_map_mu);
        slot.key = key;
        slot.map = *map;
        slot.valid = true;
    }
    return r;
}

// An M/N-major operand (rows x cols, leading dimension ld, rows % 32 == 0) as the
// 3-D tensor {32 rows, cols, rows / 32} with box {32, box_cols, groups}: one copy
// fetches 32 * groups rows as `groups` [box_cols][32] row groups, the layout that
// `groups` 2-D boxes of 32 rows give.  Row groups past rows/32 are out of range of
// the third dimension and read as zero, so no element beyond the matrix is read.
int encode_mn3d(CUtensorMap* map, const float* base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_cols,
                uint32_t groups, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(SGEMM_ERR_TENSOR_MAP, "cuTensorMapEncodeTiled is unavailable from the driver");
    if (g_debug.load() & SGEMM_DEBUG_FAIL_TENSOR_MAP)
        return fail(SGEMM_ERR_TENSOR_MAP, "injected tensor-map failure (SGEMM_DEBUG_FAIL_TENSOR_MAP)");
    const cuuint64_t dims[3] = {32, static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows / 32)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 4, 32 * 4};
    const cuuint32_t box[3] = {32, box_cols, groups};
    const CUresult r = encode_cached(fn, map, 3, base, dims, strides, box, swizzle);
    if (r != CUDA_SUCCESS)
        return fail(SGEMM_ERR_TENSOR_MAP, "cuTensorMapEncodeTiled (3-D) failed (%d) for a %lld x %lld matrix, ld %lld",
                    static_cast<int>(r), (long long)rows, (long long)cols, (long long)ld);
    return 0;
}

// 2-D fp32 column-major matrix rows x cols with leading dimension ld (elements),
// box {box_rows, box_cols}; out-of-range elements of a box read as zero.
int encode_2d(CUtensorMap* map, const float* base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows,
              uint32_t box_cols, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(SGEMM_ERR_TENSOR_MAP, "cuTensorMapEncodeTiled is unavailable from the driver");
    if (g_debug.load() & SGEMM_DEBUG_FAIL_TENSOR_MAP)
        return fail(SGEMM_ERR_TENSOR_MAP, "injected tensor-map failure (SGEMM_DEBUG_FAIL_TENSOR_MAP)");
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    const cuuint32_t box[2] = {box_rows, box_cols};
    const CUresult r = encode_cached(fn, map, 2, base, dims, strides, box, swizzle);
    if (r != CUDA_SUCCESS)
        return fail(SGEMM_ERR_TENSOR_MAP, "cuTensorMapEncodeTiled failed (%d) for a %lld x %lld matrix, ld %lld",
                    static_cast<int>(r), (long long)rows, (long long)cols, (long long)ld);
    return 0;
}

// Encode the tensor maps the planned kernel reads, launch it, then the split-K
// reduction when the plan splits K.  Operands are in the kernels' layout here
// (A M-major with ld pl.ld_a, B K-major with ld pl.ld_b).
int launch_gemm(const sgemm_plan_t& pl, bool split3, bool a_kmajor, bool b_mnmajor, const float* a_big,
                const float* a_small, const float* b_big, const float* b_small, int64_t m, int64_t n, int64_t k,
                GemmParams& gp, int num_sms, cudaStream_t st) {
    int rc;
    cudaError_t e;
    CUtensorMap tmA, tmB;
    if (pl.kernel == SGEMM_KERNEL_FFMA) {
        // one block per tile and K slice; the last wave's tiles take tail_split blocks each
        const dim3 grid(static_cast<unsigned>(pl.tiles_m * pl.tiles_n + pl.tail_tiles * (pl.tail_split - 1)),
                        static_cast<unsigned>(pl.split_k));
        if ((rc = encode_2d(&tmA, a_big, m, k, pl.ld_a, kBM, kFfmaBK, CU_TENSOR_MAP_SWIZZLE_NONE))) return rc;
        if ((rc = encode_2d(&tmB, b_big, k, n, pl.ld_b, kFfmaBK, pl.bn, CU_TENSOR_MAP_SWIZZLE_128B))) return rc;
        // C by TMA stores (boxes of 32 rows x bn columns, 128-byte swizzle) when
        // the tile's result is final and needs no read of C.
        CUtensorMap tmC{};
        gp.c_tma = 0;
        if (PG_FFMA_TMA_STORE && pl.sk_ctas == 0 && gp.split == 1 && gp.beta == 0.0f && gp.c_vec) {
            if ((rc = encode_2d(&tmC, gp.C, m, n, gp.ldc, 32, pl.bn, CU_TENSOR_MAP_SWIZZLE_128B))) return rc;
            gp.c_tma = 1;
        }
        if (pl.sk_ctas > 0) {
            if ((e = launch_ffma_sk(tmA, tmB, gp, pl.bn, pl.sk_ctas, num_sms, st)) != cudaSuccess)
                return fail_cuda(e, "FFMA stream-K kernels");
        } else if ((e = launch_ffma(tmA, tmB, tmC, gp, pl.bn, grid, st)) != cudaSuccess) {
            return fail_cuda(e, "FFMA GEMM kernel");
        }
    } else {
        // tcgen05: A in 32-row boxes (M-major, 32-byte-atom swizzle), B in boxes of
        // pl.bk x (bn, or bn/2 per CTA on SM pairs).
        const bool pair = pl.kernel == SGEMM_KERNEL_TC2;
        // (the 512-wide pair tile stages each CTA's B columns as two halves of 128)
        const uint32_t b_cols = pair ? (pl.bn == 512 ? 128 : pl.bn / 2) : pl.bn;
        // K-major operands: rows of BK floats, 128- or 64-byte swizzle.  M/N-major
        // operands: groups of 32 rows in the 32-byte-atom 128-byte swizzle, as one
        // 3-D box when the extent is a multiple of 32, else as 2-D boxes.
        const CUtensorMapSwizzle ksw = pl.bk == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
        const CUtensorMapSwizzle msw = CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B;
        gp.a_kmajor = a_kmajor ? 1 : 0;
        gp.b_mnmajor = b_mnmajor ? 1 : 0;
        gp.a3d = (!a_kmajor && m % 32 == 0) ? 1 : 0;
        gp.b3d = (b_mnmajor && n % 32 == 0) ? 1 : 0;
        // The single-SM 3xTF32 kernel splits A into tensor memory: its M-major A
        // tile is read only by threads, so it lands without a swizzle.
        const CUtensorMapSwizzle msw_a = (!pair && split3) ? CU_TENSOR_MAP_SWIZZLE_NONE : msw;
        auto encode_a = [&](CUtensorMap* map, const float* base) {
            if (a_kmajor) return encode_2d(map, base, k, m, pl.ld_a, pl.bk, kBM, ksw);
            return gp.a3d ? encode_mn3d(map, base, m, k, pl.ld_a, pl.bk, 4, msw_a)
                          : encode_2d(map, base, m, k, pl.ld_a, 32, pl.bk, msw_a);
        };
        auto encode_b = [&](CUtensorMap* map, const float* base) {
            if (!b_mnmajor) return encode_2d(map, base, k, n, pl.ld_b, pl.bk, b_cols, ksw);
            return gp.b3d ? encode_mn3d(map, base, n, k, pl.ld_b, pl.bk, b_cols / 32, msw)
                          : encode_2d(map, base, n, k, pl.ld_b, 32, pl.bk, msw);
        };
        if ((rc = encode_a(&tmA, a_big))) return rc;
        if ((rc = encode_b(&tmB, b_big))) return rc;
        if (pair) {
            // 3xTF32 on SM pairs reads the pre-split parts: big through tmA/tmB, small through tmAs/tmBs
            CUtensorMap tmAs = tmA, tmBs = tmB;
            if (split3) {
                if ((rc = encode_a(&tmAs, a_small))) return rc;
                if ((rc = encode_b(&tmBs, b_small))) return rc;
            }
            int pairs = 0;
            const int units = pl.tail_split > 1
                                  ? pl.tiles_m * pl.tiles_n + pl.tail_tiles * (pl.tail_split - 1)
                                  : pl.tiles_m * pl.tiles_n * pl.split_k;
            if ((e = launch_tc2(tmA, tmAs, tmB, tmBs, gp, pl.bn, split3, units, num_sms, st, &pairs)) != cudaSuccess)
                return fail_cuda(e, "tcgen05 SM-pair GEMM kernel");
        } else {
            // 3xTF32 with B split by the pre-pass: remainders through tmBs
            CUtensorMap tmBs = tmB;
            gp.b_presplit = (split3 && b_small != nullptr) ? 1 : 0;
            if (gp.b_presplit && (rc = encode_b(&tmBs, b_small))) return rc;
            if (pl.sk_ctas > 0) {
                if ((e = launch_tc_sk(tmA, tmB, tmBs, gp, pl.bn, pl.sk_ctas, st)) != cudaSuccess)
                    return fail_cuda(e, "tcgen05 stream-K GEMM kernel");
                if ((e = launch_streamk_fixup(gp, pl.bn, pl.sk_ctas, num_sms, st)) != cudaSuccess)
                    return fail_cuda(e, "stream-K fix-up");
            } else {
                const dim3 grid(static_cast<unsigned>(pl.tiles_m * pl.tiles_n), static_cast<unsigned>(pl.split_k));
                if ((e = launch_tc(tmA, tmB, tmBs, gp, pl.bn, split3, grid, st)) != cudaSuccess)
                    return fail_cuda(e, "tcgen05 GEMM kernel");
            }
        }
    }
    if (pl.split_k > 1) {
        if ((e = launch_splitk_reduce(gp, num_sms, st)) != cudaSuccess) return fail_cuda(e, "split-K reduction");
    }
    g_launches += pl.launches;
    return 0;
}

// ---- the call ---------------------------------------------------------------------------

// Operand A already in the layout a plan's kernel reads (copied, transposed or
// TF32-split once by a caller that runs several products on the same A, as
// sgemm_host does for its column slabs).
struct PreparedA {
    const float* big = nullptr;
    const float* small = nullptr;  // 3xTF32 remainder part (split pre-pass)
};

// Device bytes of A's preparation under plan pl (0 when A is read in place).
size_t prep_a_bytes(const sgemm_plan_t& pl, char transa, int64_t m, int64_t k) {
    if (pl.prep_a == SGEMM_PREP_NONE) return 0;
    const int parts = pl.prep_a == SGEMM_PREP_SPLIT ? 2 : 1;
    const int64_t cols_a = (pl.kernel != SGEMM_KERNEL_FFMA && !is_notrans(transa)) ? m : k;
    return parts * region(pl.ld_a * cols_a);
}

// Prepare A as plan pl asks into dst (prep_a_bytes(pl, ...) bytes); one launch.
int prepare_a(const sgemm_plan_t& pl, char transa, int64_t m, int64_t k, const float* A, int64_t lda, char* dst,
              int num_sms, cudaStream_t st, PreparedA* out) {
    float* d = reinterpret_cast<float*>(dst);
    float* ds2 = pl.prep_a == SGEMM_PREP_SPLIT
                     ? reinterpret_cast<float*>(dst + prep_a_bytes(pl, transa, m, k) / 2)
                     : nullptr;
    const bool tr = pl.prep_a == SGEMM_PREP_TRANSPOSE;  // FFMA only: transposed into M-major
    const bool kmaj = !tr && !is_notrans(transa);      // tensor cores: stored k x m, kept as is
    cudaError_t e = launch_prep(A, lda, tr, kmaj ? k : m, kmaj ? m : k, d, ds2, pl.ld_a, num_sms, st, false);
    if (e != cudaSuccess) return fail_cuda(e, "operand preparation (A)");
    out->big = d;
    out->small = ds2;
    return 0;
}

// pre != null: A is already prepared as this call's plan asks (same mode, transa,
// m and k); the call then neither prepares A nor reserves workspace for it.
int run(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha, const float* A, int64_t lda,
        const float* B, int64_t ldb, float beta, float* C, int64_t ldc, int mode, cudaStream_t st,
        const PreparedA* pre = nullptr) {
    int dev;
    DeviceState* ds;
    int rc = current_device(&dev, &ds);
    if (rc) return rc;
    sgemm_plan_t pl;
    make_plan(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, mode, ds->sms, &pl);
    cudaError_t e;
    if (pl.kernel == SGEMM_KERNEL_NONE) return 0;
    if (pl.kernel == SGEMM_KERNEL_SCALE) {
        if ((e = launch_scale(C, ldc, m, n, beta, ds->sms, st)) != cudaSuccess) return fail_cuda(e, "scale kernel");
        g_launches += 1;
        return 0;
    }
    const size_t a_prep = prep_a_bytes(pl, transa, m, k);
    const bool a_given = pre != nullptr && a_prep > 0;
    if (a_given) {
        pl.workspace_bytes -= a_prep;
        pl.launches -= 1;
    }
    void* ws = nullptr;
    if ((rc = get_buffer(dev, st, kPurposeWorkspace, pl.workspace_bytes, &ws))) return rc;
    const bool split3 = mode == SGEMM_3XTF32;
    char* cursor = static_cast<char*>(ws);

    const float* a_big = A;
    const float* a_small = nullptr;
    bool a_prepped = false;  // this call launched A's pass
    if (a_given) {
        a_big = pre->big;
        a_small = pre->small;
    } else if (a_prep > 0) {
        PreparedA pa;
        if ((rc = prepare_a(pl, transa, m, k, A, lda, cursor, ds->sms, st, &pa))) return rc;
        a_prepped = true;
        cursor += a_prep;
        a_big = pa.big;
        a_small = pa.small;
    }
    const float* b_big = B;
    const float* b_small = nullptr;
    if (pl.prep_b != SGEMM_PREP_NONE) {
        float* d = reinterpret_cast<float*>(cursor);
        const int64_t cols_b = (pl.kernel != SGEMM_KERNEL_FFMA && !is_notrans(transb)) ? k : n;
        cursor += region(pl.ld_b * cols_b);
        float* ds2 = nullptr;
        if (pl.prep_b == SGEMM_PREP_SPLIT) {
            ds2 = reinterpret_cast<float*>(cursor);
            cursor += region(pl.ld_b * cols_b);
        }
        const bool tr = pl.prep_b == SGEMM_PREP_TRANSPOSE;  // FFMA only: transposed into K-major
        const bool nmaj = !tr && !is_notrans(transb);      // tensor cores: stored n x k, kept as is
        if ((e = launch_prep(B, ldb, tr, nmaj ? n : k, nmaj ? k : n, d, ds2, pl.ld_b, ds->sms, st, a_prepped)) !=
            cudaSuccess)
            return fail_cuda(e, "operand preparation (B)");
        b_big = d;
        b_small = ds2;
    }

    GemmParams gp{};
    gp.m = m;
    gp.n = n;
    gp.k = k;
    gp.alpha = alpha;
    gp.beta = beta;
    gp.C = C;
    gp.ldc = ldc;
    gp.split = pl.split_k;
    if (pl.split_k > 1) {
        gp.P = reinterpret_cast<float*>(cursor);
        gp.ldp = round_up(m, 4);
        gp.p_stride = gp.ldp * n;
        cursor += region(pl.split_k * gp.ldp * n);
    }
    gp.tiles_m = pl.tiles_m;
    gp.tiles_n = pl.tiles_n;
    gp.kb_total = pl.k_blocks;
    gp.kb_per_split = pl.k_blocks_per_split;
    gp.tail_split = pl.tail_split;
    gp.tail_first = pl.tiles_m * pl.tiles_n - pl.tail_tiles;
    if (pl.tail_split > 1) {
        gp.tail_kb = static_cast<int32_t>(cdiv(pl.k_blocks, pl.tail_split));
        gp.tail_P = reinterpret_cast<float*>(cursor);
        cursor += tail_bytes(pl);
        gp.tail_cnt = reinterpret_cast<int*>(cursor);
        if ((e = cudaMemsetAsync(gp.tail_cnt, 0, tail_counter_bytes(pl), st)) != cudaSuccess)
            return fail_cuda(e, "cudaMemsetAsync (last-wave counters)");
    }
    if (pl.sk_ctas > 0) {
        const int64_t tiles = static_cast<int64_t>(pl.tiles_m) * pl.tiles_n;
        gp.sk_iters = tiles * pl.k_blocks;
        gp.sk_maxseg = sk_maxseg(tiles, pl.k_blocks, pl.sk_ctas);
        gp.sk_P = reinterpret_cast<float*>(cursor);
        cursor += region(tiles * gp.sk_maxseg * pl.bm * pl.bn);
    }
    gp.group_m = (pl.kernel == SGEMM_KERNEL_FFMA) ? PG_FFMA_GROUP_M : PG_GROUP_M;
    gp.c_vec = aligned16(C) && (ldc % 4 == 0);
    gp.debug_flags = g_debug.load();
    gp.timeout_ns = g_timeout_ns.load();
    gp.status = ds->status;
    // the GEMM right after this call's operand pass (no memset between them)
    gp.after_prep = (PG_PDL_PREP && (a_prepped || pl.prep_b != SGEMM_PREP_NONE) && pl.tail_split <= 1) ? 1 : 0;

    const bool tcm = pl.kernel != SGEMM_KERNEL_FFMA;
    return launch_gemm(pl, split3, tcm && !is_notrans(transa), tcm && !is_notrans(transb), a_big, a_small, b_big,
                       b_small, m, n, k, gp, ds->sms, st);
}

// ---- the allocation-free variant (sgemm_noalloc) ---------------------------------------
//
// Callers that cannot call cudaMalloc -- a process whose device memory is all
// reserved up front by another allocator, or a latency-critical loop in which
// cudaMalloc/cudaFree (which may synchronise the device) are not allowed -- get
// one entry point whose only scratch, the split-K partial sums, lives in this
// fixed array.  Every GPU that loads the library holds the array until the
// process exits.  Host code cannot use the array's name as a device address (it
// names a host-side stand-in), so each device's address is taken once with
// cudaGetSymbolAddress while that device is current.

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

float* g_noalloc_ptr[kMaxDevices];  // device address of the array, per device (guarded by g_dev_mu)

int noalloc_scratch(int dev, float** out) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        float* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_scratch);
        if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(no-allocation scratch)");
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return 0;
}

int run_noalloc(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha, const float* A,
                int64_t lda, const float* B, int64_t ldb, float beta, float* C, int64_t ldc, int mode,
                cudaStream_t st) {
    // The limits below concern how the kernels read A and B in place; a call that
    // only scales C (k == 0 or alpha == 0) reads neither and is not limited.
    // Checked in signature order.
    const bool reads_ab = k > 0 && alpha != 0.0f;
    if (reads_ab) {
        if (!is_notrans(transa)) return fail(-1, "argument 1 (transa): sgemm_noalloc reads A untransposed ('N')");
        if (!is_notrans(transb)) return fail(-2, "argument 2 (transb): sgemm_noalloc reads B untransposed ('N')");
        if (!aligned16(A)) return fail(-7, "argument 7 (A): sgemm_noalloc needs a 16-byte aligned A");
        if (lda % 4 != 0) return fail(-8, "argument 8 (lda): sgemm_noalloc needs lda to be a multiple of 4");
        if (!aligned16(B)) return fail(-9, "argument 9 (B): sgemm_noalloc needs a 16-byte aligned B");
        if (ldb % 4 != 0) return fail(-10, "argument 10 (ldb): sgemm_noalloc needs ldb to be a multiple of 4");
        if (mode != SGEMM_FFMA && mode != SGEMM_TF32)
            return fail(-14, "argument 14 (mode): sgemm_noalloc supports SGEMM_FFMA and SGEMM_TF32 only (3xTF32 "
                             "needs split operands in a workspace)");
    }
    int dev;
    DeviceState* ds;
    int rc = current_device(&dev, &ds);
    if (rc) return rc;
    sgemm_plan_t pl;
    make_plan(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, mode, ds->sms, &pl, false);
    cudaError_t e;
    if (pl.kernel == SGEMM_KERNEL_NONE) return 0;
    if (pl.kernel == SGEMM_KERNEL_SCALE) {
        if ((e = launch_scale(C, ldc, m, n, beta, ds->sms, st)) != cudaSuccess) return fail_cuda(e, "scale kernel");
        g_launches += 1;
        return 0;
    }
    const int64_t ldp = round_up(m, 4);
    // split_k * ldp * n floats must fit; compared by division so that no product
    // can wrap (ldp * n < 2^62 by the size limits, split_k <= 65535).
    if (pl.split_k > 1 &&
        ldp * n > static_cast<int64_t>(kNoAllocScratchBytes / sizeof(float)) / pl.split_k)
        return fail(SGEMM_ERR_SCRATCH,
                    "sgemm_noalloc: %d K slices of a %lld x %lld result (%.0f bytes of partial sums) do not fit the "
                    "fixed device array of %zu bytes",
                    pl.split_k, (long long)m, (long long)n, 4.0 * pl.split_k * static_cast<double>(ldp * n),
                    kNoAllocScratchBytes);
    float* scratch = nullptr;
    if ((rc = noalloc_scratch(dev, &scratch))) return rc;

    GemmParams gp{};
    gp.m = m;
    gp.n = n;
    gp.k = k;
    gp.alpha = alpha;
    gp.beta = beta;
    gp.C = C;
    gp.ldc = ldc;
    gp.split = pl.split_k;
    if (pl.split_k > 1) {
        gp.P = scratch;  // every partial read by the reduction is written first: nothing to clear
        gp.ldp = ldp;
        gp.p_stride = ldp * n;
    }
    gp.tiles_m = pl.tiles_m;
    gp.tiles_n = pl.tiles_n;
    gp.kb_total = pl.k_blocks;
    gp.kb_per_split = pl.k_blocks_per_split;
    gp.group_m = (pl.kernel == SGEMM_KERNEL_FFMA) ? PG_FFMA_GROUP_M : PG_GROUP_M;
    gp.c_vec = aligned16(C) && (ldc % 4 == 0);
    gp.debug_flags = g_debug.load();
    gp.timeout_ns = g_timeout_ns.load();
    gp.status = ds->status;

    return launch_gemm(pl, false, false, false, A, nullptr, B, nullptr, m, n, k, gp, ds->sms, st);
}

// ---- the host-array entry: internal copy streams ------------------------------------------

// Two non-blocking streams per (device, caller stream) for the host-array calls'
// copies in and out, with a pool of events that order them against the caller's
// stream.  Calls on different caller streams get different pipes, so their
// copies share the host link instead of queueing behind each other; the mutex
// serialises the queueing of calls on the same caller stream.
struct HostPipe {
    std::mutex mu;
    cudaStream_t in = nullptr, out = nullptr;
    std::vector<cudaEvent_t> events;
    cudaEvent_t ev(size_t i) {
        while (events.size() <= i) {
            cudaEvent_t e = nullptr;
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
            events.push_back(e);
        }
        return events[i];
    }
};
std::map<std::pair<int, cudaStream_t>, std::unique_ptr<HostPipe>> g_pipes;  // never shrinks
std::mutex g_pipe_init_mu;

int host_pipe(int dev, cudaStream_t caller, HostPipe** out) {
    std::lock_guard<std::mutex> lk(g_pipe_init_mu);
    std::unique_ptr<HostPipe>& slot = g_pipes[std::make_pair(dev, caller)];
    if (!slot) slot.reset(new HostPipe());
    HostPipe& hp = *slot;
    cudaError_t e;
    if (!hp.in && (e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking)) != cudaSuccess)
        return fail_cuda(e, "cudaStreamCreateWithFlags");
    if (!hp.out && (e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking)) != cudaSuccess)
        return fail_cuda(e, "cudaStreamCreateWithFlags");
    {
        std::lock_guard<std::mutex> lk2(hp.mu);
        for (size_t i = 0; i < 19; ++i)
            if (!hp.ev(i)) return fail(SGEMM_ERR_CUDA, "cudaEventCreateWithFlags failed");
    }
    *out = &hp;
    return 0;
}

}  // namespace
}  // namespace pg

using namespace pg;

PG_EXPORT int sgemm(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha, const float* A,
                    int64_t lda, const float* B, int64_t ldb, float beta, float* C, int64_t ldc, int mode,
                    void* stream) {
    int rc = validate(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode);
    if (rc) return rc;
    if (m == 0 || n == 0 || ((k == 0 || alpha == 0.0f) && beta == 1.0f)) return 0;  // C unchanged
    return run(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode,
               static_cast<cudaStream_t>(stream));
}

namespace pg {
namespace {

// The host-array call: queue the copies in, the product and the copies out on
// `stream` (and the device's internal copy streams), then, when `wait`, wait for
// all of it.  Without `wait`, `stream` is left ordered after the last copy out,
// so synchronising it -- or the next call on it, whose copies reuse the staging
// buffers -- waits for every copy of this call.
int host_call_gpu(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha, const float* A,
                  int64_t lda, const float* B, int64_t ldb, float beta, float* C, int64_t ldc, int mode,
                  void* stream, bool wait) {
    int rc = 0;
    if (m == 0 || n == 0) return 0;
    int dev;
    DeviceState* ds;
    if ((rc = current_device(&dev, &ds))) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool reads_ab = k > 0 && alpha != 0.0f;
    const int64_t ra = is_notrans(transa) ? m : k, ca = is_notrans(transa) ? k : m;
    const int64_t rb = is_notrans(transb) ? k : n, cb = is_notrans(transb) ? n : k;
    const int64_t lda_d = round_up(ra, 4), ldb_d = round_up(rb, 4), ldc_d = round_up(m, 4);
    const size_t a_bytes = reads_ab ? region(lda_d * ca) : 0;
    const size_t b_bytes = reads_ab ? region(ldb_d * cb) : 0;
    const size_t c_bytes = region(ldc_d * n);

    // Column slabs of C: A is copied in (and, if its kernel wants it transposed or
    // split, prepared) once; each slab's columns of B (and of C when beta != 0)
    // are copied in on one internal stream, the slab is computed on `stream`, and
    // its result is copied out on a second internal stream, so the copies of one
    // slab overlap the arithmetic of its neighbours.  Slabs stay at least 2048
    // columns wide so each product still fills the GPU.  (Fewer, wider slabs sized
    // to whole waves of the kernel measured slower end to end: the host link, not
    // the arithmetic, bounds the tensor-core modes, and it is best kept busy by
    // fine slabs.)
#ifndef PG_HOST_SLAB_COLS
#define PG_HOST_SLAB_COLS 2048  // compile-time tunable: narrowest slab
#endif
    const int64_t slab_min = PG_HOST_SLAB_COLS;
    const int slabs = (reads_ab && is_notrans(transb) && n >= 2 * slab_min)
                          ? static_cast<int>(std::min<int64_t>(8, n / slab_min))
                          : 1;
    sgemm_plan_t full{};
    size_t pre_bytes = 0;
    if (slabs > 1) {
        // staging buffers are 256-byte aligned with ld multiples of 4: plan with them
        const void* aligned = reinterpret_cast<const void*>(uintptr_t(256));
        make_plan(transa, transb, m, n, k, alpha, aligned, lda_d, aligned, ldb_d, beta, mode, ds->sms, &full);
        pre_bytes = prep_a_bytes(full, transa, m, k);
    }
    void* stage = nullptr;
    if ((rc = get_buffer(dev, st, kPurposeStaging, a_bytes + b_bytes + c_bytes + pre_bytes, &stage))) return rc;
    float* dA = reinterpret_cast<float*>(static_cast<char*>(stage));
    float* dB = reinterpret_cast<float*>(static_cast<char*>(stage) + a_bytes);
    float* dC = reinterpret_cast<float*>(static_cast<char*>(stage) + a_bytes + b_bytes);
    char* dPre = static_cast<char*>(stage) + a_bytes + b_bytes + c_bytes;
    HostPipe* hp = nullptr;
    if (slabs > 1 && (rc = host_pipe(dev, st, &hp))) return rc;
    std::unique_lock<std::mutex> lk;
    if (hp) lk = std::unique_lock<std::mutex>(hp->mu);
    cudaStream_t s_in = hp ? hp->in : st;
    cudaStream_t s_out = hp ? hp->out : st;
    cudaError_t e = cudaSuccess;
    auto note = [&](cudaError_t err, const char* what) {
        if (err != cudaSuccess && rc == 0) rc = fail_cuda(err, what);
        return rc == 0;
    };
    if (hp) {  // the internal streams start after the work already queued on `stream`
        note(cudaEventRecord(hp->ev(0), st), "cudaEventRecord");
        note(cudaStreamWaitEvent(s_in, hp->ev(0), 0), "cudaStreamWaitEvent");
        note(cudaStreamWaitEvent(s_out, hp->ev(0), 0), "cudaStreamWaitEvent");
    }
    if (rc == 0 && reads_ab) {
        note(cudaMemcpy2DAsync(dA, lda_d * 4, A, lda * 4, ra * 4, ca, cudaMemcpyHostToDevice, s_in),
             "copy of A to the device");
        if (hp) {
            note(cudaEventRecord(hp->ev(1), s_in), "cudaEventRecord");
            note(cudaStreamWaitEvent(st, hp->ev(1), 0), "cudaStreamWaitEvent");
        }
    }
    PreparedA pre;
    if (rc == 0 && pre_bytes > 0) {
        rc = prepare_a(full, transa, m, k, dA, lda_d, dPre, ds->sms, st, &pre);
        if (rc == 0) g_launches += 1;
    }
    for (int sl = 0; sl < slabs && rc == 0; ++sl) {
        const int64_t j0 = n * sl / slabs, j1 = n * (sl + 1) / slabs, w = j1 - j0;
        if (reads_ab) {
            // slabs > 1 only with B untransposed: columns j0..j1 of B are contiguous storage columns
            const int64_t b_cols = (slabs > 1) ? w : cb;
            note(cudaMemcpy2DAsync(dB + j0 * ldb_d, ldb_d * 4, B + j0 * ldb, ldb * 4, rb * 4, b_cols,
                                   cudaMemcpyHostToDevice, s_in),
                 "copy of B to the device");
        }
        if (rc == 0 && beta != 0.0f)
            note(cudaMemcpy2DAsync(dC + j0 * ldc_d, ldc_d * 4, C + j0 * ldc, ldc * 4, m * 4, w, cudaMemcpyHostToDevice,
                                   s_in),
                 "copy of C to the device");
        if (rc == 0 && hp) {
            note(cudaEventRecord(hp->ev(2 + 2 * sl), s_in), "cudaEventRecord");
            note(cudaStreamWaitEvent(st, hp->ev(2 + 2 * sl), 0), "cudaStreamWaitEvent");
        }
        if (rc == 0)
            rc = run(transa, transb, m, w, k, alpha, reads_ab ? dA : nullptr, reads_ab ? lda_d : 1,
                     reads_ab ? dB + j0 * ldb_d : nullptr, reads_ab ? ldb_d : 1, beta, dC + j0 * ldc_d, ldc_d, mode, st,
                     pre_bytes > 0 ? &pre : nullptr);
        if (rc == 0 && hp) {
            note(cudaEventRecord(hp->ev(3 + 2 * sl), st), "cudaEventRecord");
            note(cudaStreamWaitEvent(s_out, hp->ev(3 + 2 * sl), 0), "cudaStreamWaitEvent");
        }
        if (rc == 0)
            note(cudaMemcpy2DAsync(C + j0 * ldc, ldc * 4, dC + j0 * ldc_d, ldc_d * 4, m * 4, w, cudaMemcpyDeviceToHost,
                                   s_out),
                 "copy of C to the host");
    }
    if (hp) {
        // `stream` waits for everything queued on the internal streams (also after a
        // failure: those copies touch the caller's arrays and the staging buffers).
        for (cudaStream_t s : {s_in, s_out}) {
            cudaEvent_t done = hp->ev(18);
            if ((e = cudaEventRecord(done, s)) != cudaSuccess || (e = cudaStreamWaitEvent(st, done, 0)) != cudaSuccess)
                if (rc == 0) rc = fail_cuda(e, "ordering the caller's stream after the copies");
        }
    }
    if (!wait && rc == 0) return 0;
    // Every queued copy touches the caller's host arrays: wait for all of them
    // (also after a failure) before returning.
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess && rc == 0) rc = fail_cuda(e, "cudaStreamSynchronize");
    if (hp) {
        if ((e = cudaStreamSynchronize(s_in)) != cudaSuccess && rc == 0) rc = fail_cuda(e, "cudaStreamSynchronize");
        if ((e = cudaStreamSynchronize(s_out)) != cudaSuccess && rc == 0) rc = fail_cuda(e, "cudaStreamSynchronize");
    }
    return rc;
}

// ---- the hybrid CPU + GPU column split ("HPC - Lecture 13 - MatMat GPU", sections
// "Load distribution" and "the hybrid function matmatgpu3") ----------------------
//
// With a ratio Q set (sgemm_set_host_split), a host call gives the first
// n - floor(n / (Q + 1)) columns of C to the GPU path above and the last
// floor(n / (Q + 1)) to the host co-worker (host_sgemm), which runs in the
// calling thread while the GPU's copies and kernels proceed: the lecture's
// asynchronous kernel launch followed by matmatthreadomp, then the wait.  The
// host columns of B and C never cross the host link.  Q < 0 selects the
// automatic ratio: every synchronous call measures its two parts (the GPU part
// by events around its queued work, the host part by the host clock) and sets
// the next Q of its mode to the ratio of their speeds, GFLOP/s of the GPU part
// over GFLOP/s of the host part -- the lecture's rule of splitting in
// proportion to the measured performance ratio, re-measured call by call.  It
// starts from the lecture's Q = 15.

std::atomic<double> g_split_q{0.0};                 // 0: off, > 0: fixed Q, < 0: automatic
std::atomic<double> g_split_auto[3] = {{15.0}, {15.0}, {15.0}};  // automatic Q per mode

double split_ratio(int mode) {
    const double q = g_split_q.load();
    if (q == 0.0) return 0.0;
    return q > 0.0 ? q : g_split_auto[mode].load();
}

int host_call(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha, const float* A, int64_t lda,
              const float* B, int64_t ldb, float beta, float* C, int64_t ldc, int mode, void* stream, bool wait) {
    int rc = validate(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode);
    if (rc) return rc;
    const double q = split_ratio(mode);
    const bool product = m > 0 && n > 1 && k > 0 && alpha != 0.0f;
    const int64_t n_cpu = (q > 0.0 && product) ? static_cast<int64_t>(std::floor(n / (q + 1.0))) : 0;
    if (n_cpu <= 0 || n_cpu >= n)
        return host_call_gpu(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode, stream, wait);
    const int64_t n_gpu = n - n_cpu;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool measure = wait && g_split_q.load() < 0.0;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    cudaError_t e;
    if (measure) {
        if ((e = cudaEventCreate(&e0)) != cudaSuccess || (e = cudaEventCreate(&e1)) != cudaSuccess ||
            (e = cudaEventRecord(e0, st)) != cudaSuccess) {
            if (e0) cudaEventDestroy(e0);
            if (e1) cudaEventDestroy(e1);
            return fail_cuda(e, "events of the host split");
        }
    }
    // the GPU's columns: queued, not waited for
    rc = host_call_gpu(transa, transb, m, n_gpu, k, alpha, A, lda, B, ldb, beta, C, ldc, mode, stream, false);
    if (rc == 0 && measure && (e = cudaEventRecord(e1, st)) != cudaSuccess) rc = fail_cuda(e, "cudaEventRecord");
    // the host's columns, meanwhile (B's columns n_gpu.. are B + n_gpu*ldb when B is
    // stored k x n, its rows n_gpu.. when stored n x k)
    double cpu_s = 0.0;
    if (rc == 0) {
        const float* Bc = is_notrans(transb) ? B + n_gpu * ldb : B + n_gpu;
        const auto t0 = std::chrono::steady_clock::now();
        host_sgemm(transa, transb, m, n_cpu, k, alpha, A, lda, Bc, ldb, beta, C + n_gpu * ldc, ldc, 0);
        cpu_s = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
    }
    // the GPU's copies touch the caller's arrays: also after a failure, wait for
    // what was queued before returning an error
    if ((wait || rc != 0) && (e = cudaStreamSynchronize(st)) != cudaSuccess && rc == 0)
        rc = fail_cuda(e, "cudaStreamSynchronize");
    if (rc == 0 && measure) {
        float gpu_ms = 0.0f;
        if (cudaEventElapsedTime(&gpu_ms, e0, e1) == cudaSuccess && gpu_ms > 0.0f && cpu_s > 0.0) {
            const double r_gpu = static_cast<double>(n_gpu) / (1e-3 * gpu_ms);  // columns per second
            const double r_cpu = static_cast<double>(n_cpu) / cpu_s;
            g_split_auto[mode] = std::min(1e6, std::max(1.0, r_gpu / r_cpu));
        }
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    return rc;
}

}  // namespace
}  // namespace pg

PG_EXPORT int sgemm_set_host_split(double q) {
    if (std::isnan(q) || std::isinf(q)) return fail(-1, "argument 1 (q): %g is not a finite ratio", q);
    g_split_q = q;
    return 0;
}

PG_EXPORT double sgemm_host_split_ratio(int mode) {
    if (mode != SGEMM_FFMA && mode != SGEMM_TF32 && mode != SGEMM_3XTF32) return -1.0;
    return split_ratio(mode);
}

PG_EXPORT int sgemm_host(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha, const float* A,
                         int64_t lda, const float* B, int64_t ldb, float beta, float* C, int64_t ldc, int mode,
                         void* stream) {
    return host_call(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode, stream, true);
}

PG_EXPORT int sgemm_host_async(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha,
                               const float* A, int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                               int64_t ldc, int mode, void* stream) {
    return host_call(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode, stream, false);
}

PG_EXPORT int sgemm_noalloc(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha,
                            const float* A, int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                            int64_t ldc, int mode, void* stream) {
    int rc = validate(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode);
    if (rc) return rc;
    if (m == 0 || n == 0 || ((k == 0 || alpha == 0.0f) && beta == 1.0f)) return 0;  // C unchanged
    return run_noalloc(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode,
                       static_cast<cudaStream_t>(stream));
}

PG_EXPORT int sgemm_set_workspace(void* workspace, size_t bytes, void* stream) {
    if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(-1, "argument 1 (workspace): %p is not 256-byte aligned", workspace);
    if (workspace == nullptr && bytes != 0)
        return fail(-2, "argument 2 (bytes): must be 0 when the workspace is null (null restores the library's own)");
    int dev;
    DeviceState* ds;
    int rc = current_device(&dev, &ds);
    if (rc) return rc;
    cudaError_t e;
    if (workspace != nullptr) {
        cudaPointerAttributes at{};
        if ((e = cudaPointerGetAttributes(&at, workspace)) != cudaSuccess) {
            cudaGetLastError();
            return fail(-1, "argument 1 (workspace): %p is not memory the CUDA runtime knows (%s)", workspace,
                        cudaGetErrorString(e));
        }
        if (!((at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == dev))
            return fail(-1, "argument 1 (workspace): %p is not device memory of the current device %d", workspace,
                        dev);
        uintptr_t base = 0;
        size_t size = 0;
        if (allocation_range(workspace, &base, &size) &&
            (bytes > size || reinterpret_cast<uintptr_t>(workspace) - base > size - bytes))
            return fail(-2, "argument 2 (bytes): %zu bytes from %p run past the end of its allocation", bytes,
                        workspace);
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const std::pair<int, uintptr_t> key{dev, reinterpret_cast<uintptr_t>(st)};
    std::lock_guard<std::mutex> lk(g_ws_mu);
    if (workspace == nullptr) {
        g_user_ws.erase(key);
        return 0;
    }
    // The library's own workspace for this stream is no longer used: free it in
    // stream order (after the work already queued that may still use it).
    auto it = g_bufs.find({key, kPurposeWorkspace});
    if (it != g_bufs.end() && it->second.ptr != nullptr) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if ((e = cudaStreamIsCapturing(st, &cs)) != cudaSuccess) return fail_cuda(e, "cudaStreamIsCapturing");
        if (cs != cudaStreamCaptureStatusNone)
            return fail(SGEMM_ERR_CAPTURE, "sgemm_set_workspace would free the stream's workspace during capture");
        if ((e = cudaFreeAsync(it->second.ptr, st)) != cudaSuccess) return fail_cuda(e, "cudaFreeAsync(workspace)");
        g_bufs.erase(it);
    }
    g_user_ws[key] = Buf{workspace, bytes};
    return 0;
}

PG_EXPORT int sgemm_plan(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha, const void* A,
                         int64_t lda, const void* B, int64_t ldb, float beta, const void* C, int64_t ldc, int mode,
                         int num_sms, sgemm_plan_t* plan) {
    int rc = validate(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, C, ldc, mode);
    if (rc) return rc;
    if (num_sms <= 0) return fail(-15, "argument 15 (num_sms): %d must be positive", num_sms);
    if (plan == nullptr) return fail(-16, "argument 16 (plan): null pointer");
    make_plan(transa, transb, m, n, k, alpha, A, lda, B, ldb, beta, mode, num_sms, plan);
    return 0;
}

PG_EXPORT int sgemm_device_status(void* stream, int clear) {
    int dev;
    DeviceState* ds;
    int rc = current_device(&dev, &ds);
    if (rc) return rc;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
    int v = 0;
    if ((e = cudaMemcpy(&v, ds->status, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return fail_cuda(e, "reading the status word");
    if (clear && (e = cudaMemset(ds->status, 0, sizeof v)) != cudaSuccess) return fail_cuda(e, "clearing the status word");
    if (v != 0) return fail(v, "a kernel on device %d recorded status %d (bounded wait expired)", dev, v);
    return 0;
}

PG_EXPORT uint64_t sgemm_set_wait_timeout(uint64_t ns) { return g_timeout_ns.exchange(ns); }

PG_EXPORT int sgemm_force_plan(int bn, int split_k) {
    if (!(bn == 0 || bn == 64 || bn == 128 || bn == 256 || bn == 512))
        return fail(-1, "bn %d is not 0, 64, 128, 256 or 512", bn);
    if (split_k < 0) return fail(-2, "split_k %d is negative", split_k);
    g_force_bn = bn;
    g_force_split = split_k;
    return 0;
}

PG_EXPORT int sgemm_debug_flags(int flags) { return g_debug.exchange(flags); }

PG_EXPORT uint64_t sgemm_launch_count(void) { return g_launches.load(); }

PG_EXPORT int sgemm_workspace_release(void) {
    std::lock_guard<std::mutex> lk(g_ws_mu);
    int prev = -1;
    cudaGetDevice(&prev);
    int rc = 0;
    for (auto& kv : g_bufs) {
        if (!kv.second.ptr) continue;
        cudaSetDevice(kv.first.first.first);
        cudaError_t e = cudaDeviceSynchronize();
        if (e == cudaSuccess) e = cudaFree(kv.second.ptr);
        if (e != cudaSuccess && !rc) rc = fail_cuda(e, "releasing the workspace");
        kv.second = Buf{};
    }
    g_bufs.clear();
    if (prev >= 0) cudaSetDevice(prev);
    return rc;
}

PG_EXPORT const char* sgemm_last_error_string(void) { return t_err; }

PG_EXPORT const char* sgemm_version(void) { return kVersion; }
