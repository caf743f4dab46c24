/*
 * tgemm_probes.h -- C ABI of libtgemm_probes, read-stream calibration kernels
 * for the roofline of the bandwidth-bound skinny product (the pages have no
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

#ifdef __cplusplus
}
#endif

#endif /* TGEMM_PROBES_H */
