/*
 * tgemm_probes.h -- C ABI of libtgemm_probes, calibration kernels: read streams
 * and the paired-FMA rate.  The read-stream probes serve the roofline of the
 * bandwidth-bound skinny product (the pages have no
 * counterpart: they only state that DRAM bandwidth, not arithmetic, bounds
 * such kernels -- note.jhbae.stream "Lec 29 · GPU Architecture (2)", tiling
 * strategy: reducing DRAM accesses is what tiling is for).
 *
 * Each probe reads `bytes` bytes of device memory at `buf` exactly once and
 * adds every 32-bit word of it, as an unsigned integer, into the 64-bit
 * counter at `sum` (device memory, modulo 2^64; the caller zeroes it first).
 * The sum proves that every byte was read and keeps the reads from being
 * optimised away; timing a probe with events on `stream` gives the rate at
 * which this GPU streams memory into its SMs by that route:
 *
 *  - tgemm_probe_read_tma: persistent CTAs (two per SM), each streaming a
 *    contiguous share of the buffer through a 3-stage shared-memory ring of
 *    32 KiB bulk copies (cp.async.bulk, the TMA unit), as the skinny product
 *    streams B;
 *  - tgemm_probe_read_ldg: 1024 threads per SM, each with four 128-bit loads
 *    in flight, grid-strided over the buffer.
 *
 * Rules: buf and sum are device pointers of the current device; buf is
 * 16-byte aligned; bytes >= 0 is a multiple of 16 and < 2^40; sum is 8-byte
 * aligned.  bytes == 0 is a no-op.  Returns 0 when the kernel is queued,
 * 1 for an argument outside these rules, 4 for a CUDA failure (the codes of
 * tgemm_status in tgemm.h).
 */
#ifndef TGEMM_PROBES_H
#define TGEMM_PROBES_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;

int tgemm_probe_read_tma(const void *buf, int64_t bytes, uint64_t *sum, struct CUstream_st *stream);
int tgemm_probe_read_ldg(const void *buf, int64_t bytes, uint64_t *sum, struct CUstream_st *stream);

/*
 * tgemm_probe_ffma2: the FFMA product kernel's inner update with register
 * operands only -- the arithmetic ceiling of its consumer loop (the pages tie
 * a kernel's speed to how many operations it does per loaded element;
 * hecess.blogspot.com "[Multi-Core & GPU Programming] CUDA - Matrix
 * Multiplication", "Memory 분석"; this probe removes the loads altogether).
 *
 * One CTA of 32 * warps_per_sm threads per SM.  Every thread reads a[0..7] =
 * ab[0..7] and b[0..7] = ab[8..15], keeps acc[i][j] = 0 (i, j = 0..7) in
 * registers and `iters` times does acc[i][j] = fma(a[i], b[j], acc[i][j])
 * for all 64 (i, j), as 32 paired FMAs (fma.rn.f32x2), i.e. 128 flops per
 * thread per step; it then adds its 64 accumulators, in double, into *out
 * (device memory; the caller zeroes it).  With every a[i] * b[j] a power of
 * two and iters < 2^24 every accumulator is exact (iters * a[i] b[j]), and
 * so is *out = threads * iters * (sum a)(sum b) as long as the largest and
 * smallest |a[i] b[j]| are at most 2^10 apart.  Timing a call with
 * events on `stream` gives the paired-FMA rate: 128 * threads * iters flops.
 *
 * Rules: 1 <= warps_per_sm <= 16; 0 <= iters < 2^40; ab (16 floats, 4-byte
 * aligned) and out (8-byte aligned) are device pointers of the current
 * device.  Returns 0 when the kernel is queued, 1 for an argument outside
 * these rules, 4 for a CUDA failure.
 */
int tgemm_probe_ffma2(int warps_per_sm, int64_t iters, const float *ab, double *out, struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* TGEMM_PROBES_H */
