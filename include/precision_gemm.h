/*
 * precision_gemm.h -- C ABI of the GB300 (sm_103a) single-precision GEMM library.
 *
 * The operation is dense single-precision matrix multiply,
 *
 *     C = alpha * op(A) * op(B) + beta * C,
 *
 * on column-major storage with leading dimensions.  Sources for this contract:
 *   - "Optimizing SGEMM on NVIDIA Turing GPUs" (README): SGEMM with column-major
 *     A and B, not transposed, is the primary case.
 *   - "HPC - Lecture 13 - MatMat GPU", sections "Kernel 1: Global Memory Access"
 *     and "function matmatgpu1": the product accumulates into C (C += A*B), and
 *     the host routine takes strided arrays with leading dimensions lda, ldb,
 *     ldc, moves them to the device, launches, and copies C back.
 *   - "V3. Vectorized and double buffer" (Explore-GPU-performance wiki),
 *     section 2: a row-major kernel that overwrites C; row-major storage is
 *     the column-major storage of the transpose, so it needs no entry of its
 *     own (C^T = B^T * A^T, with the operands and m/n swapped).
 *
 * Conventions shared by every call below:
 *   - Element (i, j) of a stored matrix X with leading dimension ldx is
 *     X[i + j*ldx].  op(A) is m x k, op(B) is k x n, C is m x n.
 *   - trans is one of 'N','n' (op(X) = X) or 'T','t','C','c' (op(X) = X^T).
 *   - The library reads A, B and C only inside their logical extents and writes
 *     only C[i + j*ldc] for i < m, j < n; the leading-dimension gaps are never
 *     touched.  When beta == 0 C is not read (NaN there does not propagate);
 *     when alpha == 0 or k == 0, A and B are not read.
 *   - Return value: 0 on success; -i when the i-th argument (1-based, in the
 *     order of the signature) is invalid, checked in signature order and before
 *     any device work; a positive SGEMM_ERR_* code for device-side failures.
 *     sgemm_last_error_string() describes the last failure on the calling
 *     thread.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream) unless stated otherwise.
 *   - Threads: calls on different streams may come from any host threads at
 *     once.  Calls on ONE stream must not overlap in time on the host (make
 *     them from one thread, or hold a lock around each call): a call that needs
 *     a larger workspace than the stream's frees the old one in stream order,
 *     so a concurrent call that took the old workspace's address could enqueue
 *     its kernels after that free.
 *   - A failure detected inside a running kernel (a bounded wait that
 *     expired) cannot be returned by the launching call; it is recorded in a
 *     per-device status word that sgemm_device_status() reads.
 */
#ifndef PRECISION_GEMM_H
#define PRECISION_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Arithmetic modes (argument `mode`). */
#define SGEMM_FFMA 0   /* exact FP32 fused multiply-add on the CUDA cores          */
#define SGEMM_TF32 1   /* tensor cores (tcgen05), TF32 inputs, FP32 accumulation  */
#define SGEMM_3XTF32 2 /* tensor cores, each operand split x = big + small (both
                          TF32); small*big + big*small + big*big accumulated in
                          FP32, which recovers FP32-level accuracy               */
/* Subnormal operands: SGEMM_FFMA keeps them (no flush to zero).  The two
 * tensor-core modes read every operand (3xTF32: each of its two parts) in TF32,
 * whose 10 mantissa-field bits hold a subnormal only down to 2^-136: operand
 * values below 2^-137 in magnitude act as zero there (so infinity times such a
 * value gives NaN), and 3xTF32 keeps FP32-level accuracy for operands of
 * magnitude 2^-118 and above.  The tensor core itself does not flush subnormal
 * TF32 operands or FP32 sums. */

/* Status codes. */
#define SGEMM_SUCCESS 0
#define SGEMM_ERR_CUDA 1       /* a CUDA runtime call or launch failed          */
#define SGEMM_ERR_NO_DEVICE 2  /* no CUDA device is usable                      */
#define SGEMM_ERR_ARCH 3       /* the current device is not compute capability 10.3 */
#define SGEMM_ERR_TIMEOUT 4    /* a bounded in-kernel wait expired              */
#define SGEMM_ERR_ALLOC 5      /* device or host allocation failed              */
#define SGEMM_ERR_TENSOR_MAP 6 /* a TMA tensor map could not be encoded         */
#define SGEMM_ERR_CAPTURE 7    /* workspace must grow while the stream is being
                                  captured into a CUDA graph                    */
#define SGEMM_ERR_SCRATCH 8    /* sgemm_noalloc: the call needs more scratch than
                                  its fixed device array holds                  */
#define SGEMM_ERR_WORKSPACE 9  /* the workspace given by sgemm_set_workspace is
                                  smaller than the call needs                   */

/* Kernel families reported by sgemm_plan(). */
#define SGEMM_KERNEL_NONE 0    /* nothing to do (m == 0, n == 0, or C unchanged) */
#define SGEMM_KERNEL_SCALE 1   /* C = beta * C only (k == 0 or alpha == 0)       */
#define SGEMM_KERNEL_FFMA 2    /* CUDA-core FP32 kernel                         */
#define SGEMM_KERNEL_TC 3      /* tcgen05 tensor-core kernel, one SM per tile   */
#define SGEMM_KERNEL_TC2 4     /* tcgen05 on SM pairs (cta_group::2), 256-row
                                  tiles, persistent                              */

/* How an operand reaches the GEMM kernel (sgemm_plan_t.prep_a / prep_b). */
#define SGEMM_PREP_NONE 0      /* read in place through TMA                     */
#define SGEMM_PREP_COPY 1      /* copied into the workspace with an aligned ld  */
#define SGEMM_PREP_TRANSPOSE 2 /* copied transposed (trans = 'T')               */
#define SGEMM_PREP_SPLIT 3     /* split into big/small TF32 parts (3xTF32 on SM pairs) */

/*
 * sgemm -- C = alpha*op(A)*op(B) + beta*C on device memory.
 *
 *   transa, transb  'N'/'n' or 'T'/'t'/'C'/'c' (arguments 1, 2)
 *   m, n, k         sizes, >= 0 (arguments 3, 4, 5)
 *   alpha           scalar (6)
 *   A, lda          device pointer; m x k matrix (k x m if transa is 'T'),
 *                   lda >= max(1, rows of the stored matrix) (7, 8)
 *   B, ldb          device pointer; k x n matrix (n x k if transb is 'T'),
 *                   ldb >= max(1, rows of the stored matrix) (9, 10)
 *   beta            scalar (11)
 *   C, ldc          device pointer; m x n, ldc >= max(1, m) (12, 13)
 *   mode            SGEMM_FFMA, SGEMM_TF32 or SGEMM_3XTF32 (14)
 *   stream          cudaStream_t as void*, or NULL (15)
 *
 * Ownership: the caller owns A, B and C and keeps them alive until the work
 * on `stream` completes.  The library owns a workspace per (device, stream)
 * for operand copies, 3xTF32 split operands and split-K partial sums; it grows
 * on demand with stream-ordered allocation and is released by
 * sgemm_workspace_release() -- unless the caller has given the stream a
 * workspace of its own with sgemm_set_workspace().  Calls on the same stream are ordered; calls on
 * different streams use different workspaces.  The workspaces are keyed by
 * the stream handle and outlive the stream: synchronise a stream before
 * destroying it (a stream created later may get the same handle, and with it
 * the cached workspace), and call sgemm_workspace_release() to free them.  A
 * null pointer is an invalid argument only when the call would read or write
 * through it.
 *
 * Results are deterministic: the same inputs, mode and device give bitwise
 * identical C on every run (split-K partial sums are added in a fixed order).
 */
int sgemm(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha,
          const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
          float *C, int64_t ldc, int mode, void *stream);

/*
 * sgemm_host -- the same operation on HOST arrays (the shape of the lecture's
 * matmatgpu1: copy the operands in, run the product, copy C back).
 *
 * Arguments as sgemm, but A, B and C are host pointers (pinned memory gives
 * the fastest copies; pageable memory works).  The call copies the logical
 * extents of A, B and (when beta != 0) C into library-owned device buffers on
 * `stream`, runs sgemm, copies the m x n result back into C (its ld gaps are
 * not written), and synchronises `stream` before returning, so C is ready
 * when it returns 0.
 */
int sgemm_host(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha,
               const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
               float *C, int64_t ldc, int mode, void *stream);

/*
 * sgemm_host_async -- sgemm_host without the final synchronisation: the
 * copies in, the product and the copy of C out are queued in `stream` order
 * (after the work already queued on `stream`) and the call returns; C holds
 * the result once `stream` has been synchronised (or an event recorded on it
 * after the call has completed).  Until then the caller must not write A, B
 * or C, nor read C.  Calls on different streams overlap one call's copies
 * with another's arithmetic (the host link and the SMs are separate
 * resources).  With page-locked (pinned) host arrays the call does not wait;
 * with pageable arrays the CUDA runtime may block in the copies.  Returns as
 * sgemm_host; an error detected after queueing is reported by the stream.
 */
int sgemm_host_async(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha,
                     const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                     float *C, int64_t ldc, int mode, void *stream);

/*
 * sgemm_set_host_split -- the hybrid CPU + GPU column split of the host-array
 * calls ("HPC - Lecture 13 - MatMat GPU", sections "Load distribution" and "the
 * hybrid function matmatgpu3": the columns of C are divided between the two
 * devices in proportion to their measured speeds, the GPU kernel runs
 * asynchronously while the host cores compute their share, then both are
 * waited for).
 *
 *   q  > 0  fixed ratio Q: sgemm_host and sgemm_host_async give the last
 *           floor(n / (Q + 1)) columns of C to the library's host co-worker (a
 *           blocked FP32 product on the host cores, OpenMP; every output one
 *           fused multiply-add chain in increasing p, so deterministic) and the
 *           rest to the GPU path;
 *      < 0  automatic: Q per mode starts at the lecture's 15 and every
 *           synchronous sgemm_host call re-measures it as the ratio of the two
 *           parts' speeds (columns per second);
 *      = 0  off (the default): everything on the GPU.
 *   (1)
 *
 * The split applies to calls with a product (k > 0, alpha != 0) and n >= 2;
 * the host part runs in the calling thread during the call (sgemm_host_async
 * therefore returns with the host columns of C already written and the GPU
 * columns queued).  The host columns of B and C never cross the host link.
 * The host part computes in FP32 in every mode, within every mode's accuracy.
 * sgemm (device pointers) is not affected.  Applies to calls made afterwards
 * from any thread.  Returns 0, or -1 when q is not finite.
 */
int sgemm_set_host_split(double q);

/*
 * sgemm_host_split_ratio -- the Q the next host call in `mode` would use: the
 * fixed ratio, the automatic one as last measured, or 0 when the split is off;
 * -1 for an invalid mode.
 */
double sgemm_host_split_ratio(int mode);

/*
 * sgemm_noalloc -- sgemm without any device allocation.  (The pages have no
 * counterpart: this entry exists for callers of this library, not for the
 * method.)
 *
 * Who needs it: callers that cannot call cudaMalloc -- a process in which
 * another allocator has reserved the device memory up front, or a
 * latency-critical loop in which cudaMalloc/cudaFree, which may synchronise
 * the device, are not allowed.  sgemm itself may allocate its workspace on
 * first use of a size; this call never does.  Its only scratch, the split-K
 * partial sums, lives in a fixed 16 MiB array in device memory that every
 * GPU loading the library holds until the process exits.
 *
 * Arguments are those of sgemm.  When the call reads A and B (k > 0 and
 * alpha != 0) these limits apply, checked in signature order: transa and
 * transb are 'N' (else -1, -2); A and B are 16-byte aligned with lda and ldb
 * multiples of 4 (else -7/-8, -9/-10), so the kernels read them in place; mode
 * is SGEMM_FFMA or SGEMM_TF32 (else -14).  A call that only scales C
 * (k == 0 or alpha == 0) takes any arguments sgemm takes.  The call's split-K
 * partial sums, split_k * round_up(m, 4) * n * 4 bytes as sgemm_plan reports
 * split_k, must fit in the 16 MiB array (else SGEMM_ERR_SCRATCH, and nothing
 * is launched).  sgemm_noalloc never splits the last partial wave of tiles
 * along K as sgemm may (sgemm_plan's tail_split > 1), so its results equal
 * sgemm's within the mode's tolerance, and bit for bit when sgemm_plan
 * reports tail_split == 1.
 *
 * The first call on a device takes the array's device address (a
 * cudaGetSymbolAddress call with that device current, done once per device);
 * make that first call before any stream capture.  Every call shares the one
 * array and leaves its contents behind; each call writes every partial sum
 * before reading it, so nothing needs clearing, but calls whose work overlaps
 * on the GPU (different streams, or different host threads) race on the array
 * and must be serialised by the caller.
 */
int sgemm_noalloc(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha,
                  const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                  float *C, int64_t ldc, int mode, void *stream);

/*
 * sgemm_set_workspace -- give the library device memory to use as the
 * workspace of calls on `stream` (a cudaStream_t as void*, NULL for the legacy
 * default stream) on the current device, instead of memory it allocates
 * itself: for callers whose device memory comes from their own allocator (a
 * framework's caching allocator, a memory pool reserved at start-up).  The
 * pages have no counterpart; the lecture's host routine allocates its device
 * arrays itself.
 *
 *   workspace  device memory of the current device, 256-byte aligned (1), or
 *              NULL to return the stream to the library's own workspace
 *   bytes      its size; 0 when workspace is NULL (2).  The buffer must lie
 *              inside one allocation (checked when the driver can tell)
 *   stream     the stream whose calls use it (3)
 *
 * sgemm, and the product step of sgemm_host / sgemm_host_async, on that
 * stream then take their workspace (operand copies, 3xTF32 split operands,
 * split-K and last-wave partial sums: sgemm_plan's workspace_bytes) from this
 * buffer and never allocate one; a call needing more than `bytes` returns
 * SGEMM_ERR_WORKSPACE before launching anything.  The host entries' staging
 * buffers (the device copies of host A, B and C) are still the library's.
 * Setting a buffer frees the library's own workspace for that stream in stream
 * order (SGEMM_ERR_CAPTURE if the stream is being captured).
 *
 * Ownership: the caller owns the buffer and keeps it alive, unwritten by
 * anything else, until the work queued on `stream` by the calls that used it
 * has completed, and until another sgemm_set_workspace call replaces it for
 * that stream.  Calls on one stream are ordered and may share the buffer;
 * giving one buffer to two streams makes their calls race.
 * sgemm_workspace_release does not touch it.  Returns 0, -i for an invalid
 * argument, or SGEMM_ERR_NO_DEVICE / SGEMM_ERR_ARCH.
 */
int sgemm_set_workspace(void *workspace, size_t bytes, void *stream);

/* The choices sgemm would make for a call (see sgemm_plan). */
typedef struct sgemm_plan {
    int kernel;              /* SGEMM_KERNEL_*                                  */
    int mode;                /* the mode argument                               */
    int bm, bn, bk, stages;  /* output tile (bm = 256 on SM pairs), ring depth  */
    int split_k;             /* number of K slices (1: no split)                */
    int k_blocks;            /* BK-sized blocks of K in total                   */
    int k_blocks_per_split;  /* BK-sized blocks each slice reduces              */
    int tiles_m, tiles_n;    /* output tiles                                    */
    int prep_a, prep_b;      /* SGEMM_PREP_* per operand                        */
    int threads;             /* threads per CTA of the GEMM kernel              */
    int ctas_per_sm;         /* CTAs the kernel is built to co-schedule per SM  */
    int64_t ld_a, ld_b;      /* leading dimension the kernel reads A and B with */
    size_t smem_bytes;       /* dynamic shared memory of the GEMM kernel        */
    size_t workspace_bytes;  /* device workspace the call needs                 */
    int launches;            /* kernels the call launches                       */
    int tail_tiles;          /* SM pairs and FFMA: last-wave tiles whose K is split ... */
    int tail_split;          /* ... into this many slices (1: none)             */
    int sk_ctas;             /* FFMA stream-K: CTAs sharing all (tile, k-block)
                                iterations in equal ranges (0: not used)        */
} sgemm_plan_t;

/*
 * sgemm_plan -- fill *plan with what sgemm would do for these arguments on a
 * device with `num_sms` multiprocessors, without touching any device.
 * The pointers are only inspected for alignment, never dereferenced, so this
 * works on a machine without a GPU.  Returns 0, or -i for an invalid argument
 * exactly as sgemm would (mode is argument 14, num_sms 15, plan 16).
 */
int sgemm_plan(char transa, char transb, int64_t m, int64_t n, int64_t k, float alpha,
               const void *A, int64_t lda, const void *B, int64_t ldb, float beta,
               const void *C, int64_t ldc, int mode, int num_sms, sgemm_plan_t *plan);

/*
 * sgemm_device_status -- synchronise `stream`, then return SGEMM_SUCCESS, or
 * SGEMM_ERR_TIMEOUT if any kernel of this library on the current device found
 * a bounded wait expired since the status was last cleared, or SGEMM_ERR_CUDA
 * if the synchronisation itself failed.  clear != 0 resets the status word.
 */
int sgemm_device_status(void *stream, int clear);

/*
 * sgemm_set_wait_timeout -- limit, in nanoseconds, of every in-kernel wait of
 * kernels launched afterwards from any thread (default 4e9 = 4 s).  A kernel
 * whose wait expires records SGEMM_ERR_TIMEOUT, waits (bounded) for its own
 * copies in flight, frees its tensor memory and exits; its C is unspecified.
 * Returns the previous limit.
 */
uint64_t sgemm_set_wait_timeout(uint64_t ns);

/*
 * sgemm_force_plan -- tuning override for later calls from any thread:
 * bn in {0, 64, 128, 256, 512} fixes the CTA tile width (512 exists for TF32 on
 * SM pairs only and means 256 elsewhere), split_k > 0 fixes the number of K
 * slices (clamped to the number of K blocks).  0 restores the automatic choice.
 * Returns -1 for an unsupported bn, -2 for a negative split_k.
 */
int sgemm_force_plan(int bn, int split_k);

/*
 * sgemm_debug_flags -- test hooks for failure detection, injected on the
 * host or as a wait that cannot complete, never as a GPU fault.
 *   SGEMM_DEBUG_STALL_PRODUCER     the operand loader of later GEMM kernels
 *                                  issues nothing, so the rest of the CTA's
 *                                  bounded waits expire (SGEMM_ERR_TIMEOUT in
 *                                  sgemm_device_status);
 *   SGEMM_DEBUG_FAIL_ALLOC         a workspace or staging allocation the call
 *                                  needs fails: the call returns SGEMM_ERR_ALLOC
 *                                  before any GEMM kernel is launched;
 *   SGEMM_DEBUG_FAIL_TENSOR_MAP    the TMA tensor-map encoding fails: the call
 *                                  returns SGEMM_ERR_TENSOR_MAP before the GEMM
 *                                  kernel is launched (operand preparation may
 *                                  have run; C is not written).
 * 0 clears.  Returns the previous flags.
 */
#define SGEMM_DEBUG_STALL_PRODUCER 1
#define SGEMM_DEBUG_FAIL_ALLOC 2
#define SGEMM_DEBUG_FAIL_TENSOR_MAP 4
int sgemm_debug_flags(int flags);

/* Kernels this library has launched in this process (all devices). */
uint64_t sgemm_launch_count(void);

/* Free every cached workspace and staging buffer the library allocated
 * (synchronises the device); buffers given by sgemm_set_workspace stay in use. */
int sgemm_workspace_release(void);

/* Human-readable description of the last failure on the calling thread. */
const char *sgemm_last_error_string(void);

/* Library version string. */
const char *sgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PRECISION_GEMM_H */
