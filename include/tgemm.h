/*
 * tgemm.h -- C ABI of libtgemm, the tiled dense matrix multiply for NVIDIA
 * GB300 (sm_103a).
 *
 * The operation (hecess.blogspot.com "[Multi-Core & GPU Programming] CUDA -
 * Matrix Multiplication", section "[Matrix Multiplication]", the loop that
 * keeps the running sum in a register and writes P(i,j) once; generalised from
 * the page's square Width x Width case to rectangular row-major matrices):
 *
 *     C[i*ldc + j] = sum_{kk=0}^{k-1} A[i*lda + kk] * B[kk*ldb + j]
 *     for 0 <= i < m, 0 <= j < n.
 *
 * A is m x k, B is k x n and C is m x n, all row-major with leading dimensions
 * (element strides between consecutive rows) lda, ldb and ldc -- the page's
 * flattened indices M[row*width+k] and N[k*width+col] (section
 * "[Coalescing]") with one "width" per matrix.  C is overwritten, never
 * accumulated into.  k == 0 gives C = 0 (the empty sum).
 *
 * Memory and ownership.  A, B and C are DEVICE pointers (cudaMalloc'd or
 * managed memory on the current device) owned by the caller; the library
 * never frees them and keeps no reference after the call returns.  The
 * library may take temporary stream-ordered workspace on `stream` (for
 * operands whose base address or leading dimension is not a multiple of 16
 * bytes, for B transposed on the TF32 path, and for the partial sums of
 * tiles that a call splits along k between several blocks) and returns it on
 * the same stream.
 *
 * Execution.  Every call is asynchronous on `stream` (NULL is the legacy
 * default stream) and returns once the work is queued.  Argument errors are
 * found on the host before anything is queued.  A launch failure returns
 * TGEMM_ERR_CUDA.  Faults during execution surface at the caller's next
 * synchronisation; a kernel whose internal pipeline wait exceeds its time
 * limit stops, records TGEMM_ERR_TIMEOUT in a per-device status word and
 * exits, and tgemm_get_device_status() reports it.  Some kernels are
 * launched as programmatic dependents of the kernel queued before them: they
 * may start early, but wait on the device for that kernel to complete before
 * they touch global memory, and a call's last kernel completes only after
 * all of the call's work, so stream order holds for every buffer.
 *
 * Results.  tgemm_f32 multiplies in fp32 with fused multiply-add (one
 * rounding per term); tgemm_tf32 feeds fp32 inputs to the tensor cores as
 * TF32 and accumulates in fp32; tgemm_bf16 takes bf16 inputs and accumulates
 * and writes fp32.  Each element of C is written exactly once.  The order in
 * which the k terms are added is fixed per shape, so repeated calls give
 * bit-identical results.
 *
 * Thread safety.  All entry points may be called from several host threads
 * at once.  Calls on different streams may overlap on the GPU; C of one call
 * must not overlap A, B or C of a call that can run at the same time.
 */
#ifndef TGEMM_H
#define TGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;   /* cudaStream_t is `struct CUstream_st *` */

typedef enum tgemm_status {
    TGEMM_OK = 0,
    /* A size, leading dimension or pointer breaks the rules below, or C
     * overlaps A or B. */
    TGEMM_ERR_INVALID_VALUE = 1,
    /* Reserved: misaligned operands are repacked, never rejected. */
    TGEMM_ERR_MISALIGNED = 2,
    /* The current device is not an sm_103 GPU (the kernels are built for
     * sm_103a only; there is no fallback of any kind). */
    TGEMM_ERR_UNSUPPORTED_DEVICE = 3,
    /* A CUDA runtime or driver call failed; tgemm_last_error() has its text. */
    TGEMM_ERR_CUDA = 4,
    /* A kernel gave up on a pipeline wait after its time limit. */
    TGEMM_ERR_TIMEOUT = 5,
    /* Temporary workspace could not be allocated. */
    TGEMM_ERR_WORKSPACE = 6,
    /* A device-side consistency check failed: an index outside its buffer or
     * a pipeline wait that found the wrong phase.  Only the debug build
     * (libtgemm_debug.so, compiled with TGEMM_DEBUG) carries these checks;
     * tgemm_get_device_status() reports the file and line. */
    TGEMM_ERR_INTERNAL = 7
} tgemm_status;

/*
 * Argument rules shared by the three products:
 *   m, n, k >= 0 and each < 2^31;
 *   lda >= max(1, k), ldb >= max(1, n), ldc >= max(1, n);
 *   A may be NULL only when m == 0 or k == 0; B only when k == 0 or n == 0;
 *   C only when m == 0 or n == 0;
 *   non-NULL pointers are device or managed memory of the current device;
 *   C[0 .. (m-1)*ldc + n) overlaps neither A's nor B's span.
 * m == 0 or n == 0 is a no-op returning TGEMM_OK.
 */

/* fp32 x fp32 -> fp32 on the FMA pipes: register-blocked, TMA-staged tiles in
 * bank-conflict-free shared memory fed through an mbarrier pipeline. */
tgemm_status tgemm_f32(int64_t m, int64_t n, int64_t k,
                       const float *A, int64_t lda,
                       const float *B, int64_t ldb,
                       float *C, int64_t ldc,
                       struct CUstream_st *stream);

/* fp32 inputs multiplied as TF32 on the tcgen05 tensor cores, fp32
 * accumulation in tensor memory, fp32 output. */
tgemm_status tgemm_tf32(int64_t m, int64_t n, int64_t k,
                        const float *A, int64_t lda,
                        const float *B, int64_t ldb,
                        float *C, int64_t ldc,
                        struct CUstream_st *stream);

/* bf16 inputs (A and B point at IEEE bfloat16 values, 2 bytes each) on the
 * tcgen05 tensor cores, fp32 accumulation, fp32 output.  For m <= 64 the
 * product is formed as C^T = B^T A^T with the k range split across CTAs and
 * the partial sums added in a fixed order. */
tgemm_status tgemm_bf16(int64_t m, int64_t n, int64_t k,
                        const void *A, int64_t lda,
                        const void *B, int64_t ldb,
                        float *C, int64_t ldc,
                        struct CUstream_st *stream);

/* dst = transpose of src: dst[j*ld_dst + i] = src[i*ld_src + j] for
 * 0 <= i < rows, 0 <= j < cols; 4-byte elements (fp32), device pointers.
 * note.jhbae.stream "Lec 29 · GPU Architecture (2)", matrix transpose case
 * study: tiles read with coalesced row accesses into shared memory padded by
 * one word per row, columns written back coalesced; with 16-byte aligned
 * matrices and pitches (ld % 4 == 0) every access is 128 bits wide.  This is
 * the kernel that gives tgemm_tf32 its k-contiguous copy of B.  Rules: rows,
 * cols >= 0 and < 2^31, ld_src >= cols, ld_dst >= rows, dst must not overlap
 * src; rows == 0 or cols == 0 is a no-op. */
tgemm_status tgemm_transpose_f32(int64_t rows, int64_t cols,
                                 const float *src, int64_t ld_src,
                                 float *dst, int64_t ld_dst,
                                 struct CUstream_st *stream);

/* Size of the static device array used by tgemm_tf32_noalloc (32 MiB). */
#define TGEMM_NOALLOC_SCRATCH_BYTES (32ull << 20)

/*
 * tgemm_tf32 without allocating.  Same operation, argument rules and status
 * codes as tgemm_tf32 (the pages have no counterpart: this concerns only where
 * the library keeps its temporary data).  It never splits an output tile along
 * k between CTAs, so on shapes where tgemm_tf32 does (a partly filled last
 * wave of tiles, or fewer tiles than SMs) the k terms are added in another
 * order: the results agree
 * with tgemm_tf32 within the TF32 error bound, exactly on integer-valued
 * inputs, and may take longer there.
 *
 * Who needs it: callers that cannot let a library allocate device memory --
 * programs whose device memory is wholly managed by their own allocator or a
 * fixed arena, and hot paths that must not pay for, or synchronise on, an
 * allocation.  tgemm_tf32 takes a transposed copy of B (and, for a misaligned
 * A, a re-pitched copy of A) from the stream-ordered allocator on each call;
 * this entry point keeps them in a static device array of
 * TGEMM_NOALLOC_SCRATCH_BYTES instead, and calls no allocation routine.
 *
 * Limit: the shape must need at most TGEMM_NOALLOC_SCRATCH_BYTES of scratch,
 * namely 4 * n * k4 bytes plus 4 * m * k4 more when A's base address or lda*4
 * is not a multiple of 16 (k4 = k rounded up to a multiple of 4, each part
 * rounded up to 256 bytes); a larger shape returns TGEMM_ERR_INVALID_VALUE
 * before any work is queued, with the sizes in tgemm_last_error().
 *
 * The array: one copy per GPU that loads the library, held until the process
 * exits.  The first call on a device looks up its device address (with that
 * device current), which also makes CUDA load it; make that first call before
 * any stream capture.  All calls on a device share the one array and it keeps
 * whatever the last call left in it (nothing in it needs to start at zero), so
 * two calls whose GPU work can overlap -- on different streams, or on one
 * stream from different threads without ordering -- race on it.  Serialise
 * them, for example by issuing them on one stream.
 */
tgemm_status tgemm_tf32_noalloc(int64_t m, int64_t n, int64_t k,
                                const float *A, int64_t lda,
                                const float *B, int64_t ldb,
                                float *C, int64_t ldc,
                                struct CUstream_st *stream);

/* Static English text of a status code (never NULL). */
const char *tgemm_status_string(tgemm_status status);

/* Text of the last failure seen by the calling host thread ("" if none). */
const char *tgemm_last_error(void);

/* Waits for `stream`, then reads and clears the current device's status word.
 * Returns TGEMM_OK, TGEMM_ERR_TIMEOUT if a kernel gave up on a wait since the
 * last read, TGEMM_ERR_INTERNAL if a device-side check of the debug build
 * failed, or TGEMM_ERR_CUDA if the synchronisation itself failed. */
tgemm_status tgemm_get_device_status(struct CUstream_st *stream);

/* Test of the failure path (the pages have no counterpart).  Queues on
 * `stream` a one-thread kernel that waits, with the same bounded wait the
 * product kernels use but a limit of `limit_ns` nanoseconds (1e3 .. 1e9), on a
 * barrier that nothing ever arrives at.  The kernel gives up after the limit,
 * records TGEMM_ERR_TIMEOUT in the device status word and returns, so a
 * following tgemm_get_device_status() must report TGEMM_ERR_TIMEOUT and the
 * CUDA context stays usable.  Returns TGEMM_OK once the kernel is queued,
 * TGEMM_ERR_INVALID_VALUE for a limit outside the range. */
tgemm_status tgemm_selftest_wait_timeout(int64_t limit_ns, struct CUstream_st *stream);

/* Test of the debug checks' reporting path (the pages have no counterpart).
 * Queues on `stream` a one-thread kernel that records a failed consistency
 * check in the device status word, exactly as a failing check of the debug
 * build does, and returns; it touches no other memory.  A following
 * tgemm_get_device_status() must report TGEMM_ERR_INTERNAL with the check's
 * file and line.  Available in every build. */
tgemm_status tgemm_selftest_debug_check(struct CUstream_st *stream);

/* 1 if this library was built with the device-side consistency checks
 * (libtgemm_debug.so), else 0. */
int tgemm_debug_build(void);

/* Kernels launched by this library in this process so far (all devices). */
uint64_t tgemm_kernel_launches(void);

/* The tensor-core tiles tgemm_tf32 (tf32 != 0) or tgemm_bf16 would use for an
 * m x n x k product on a GPU with sm_count SMs: with the workspace those calls
 * take (workspace != 0), or without it, as tgemm_tf32_noalloc.  Host arithmetic
 * only: no CUDA call, no device needed.  Writes out[0] = tile rows (128 or
 * 256), out[1] = tile columns (256 or 224), out[2] = 1 where the last tiles
 * are split along k between two CTAs (stream-K), out[3] = split-K pieces per
 * tile (0: none), out[4] = 1 for multicast CTA pairs; all five are 0 for bf16
 * with m <= 64, which takes the cluster split-K kernel instead.  Returns
 * TGEMM_OK, or TGEMM_ERR_INVALID_VALUE (out untouched) for a NULL out, sizes
 * outside 1 .. 2^31 - 1 or sm_count outside 1 .. 4096. */
tgemm_status tgemm_plan(int tf32, int64_t m, int64_t n, int64_t k, int sm_count, int workspace, int *out);

/* The same for tgemm_f32 (128 x 128 tiles on the FMA pipes): writes out[0] =
 * tiles run whole, out[1] = tiles of a partly filled last round that are cut
 * along k instead, out[2] = pieces per such tile (0: none; their partial sums
 * are then added in piece order).  Host arithmetic only.  Returns TGEMM_OK, or
 * TGEMM_ERR_INVALID_VALUE (out untouched) for a NULL out, sizes outside
 * 1 .. 2^31 - 1 or sm_count outside 1 .. 4096. */
tgemm_status tgemm_plan_f32(int64_t m, int64_t n, int64_t k, int sm_count, int64_t *out);

/* Library version: major * 10000 + minor * 100 + patch. */
int tgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TGEMM_H */
