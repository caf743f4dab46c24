/*
 * tgemm_pages.h -- C ABI of libtgemm_pages, the two matrix-multiply kernels the
 * pages describe, kept as comparators for the tiled library (they are not used
 * by libtgemm's entry points).
 *
 * Both compute exactly what tgemm_f32 computes (see tgemm.h): row-major
 * C[i*ldc + j] = sum_kk A[i*lda + kk] * B[kk*ldb + j], fp32 inputs and output,
 * one fused multiply-add per term in ascending kk into a register, C written
 * once.  They differ only in how the data reaches the multiply:
 *
 *  - tgemm_pages_naive_f32: hecess.blogspot.com "[Multi-Core & GPU
 *    Programming] CUDA - Matrix Multiplication", sections "가장 단순한 CUDA 행렬
 *    곱셈 Kernel" and "Work Flow": one thread per element of C,
 *    col = blockIdx.x*blockDim.x + threadIdx.x, row = blockIdx.y*blockDim.y +
 *    threadIdx.y, every M and N element read from global memory; 16 x 16
 *    threads per block.
 *  - tgemm_pages_tiled_f32: same page, sections "[Shared Memory]" and "Tiled
 *    Matrix Multiplication Kernel" (and note.jhbae.stream "Lec 29 · GPU
 *    Architecture (2)"): TILE_WIDTH x TILE_WIDTH threads per block, one element
 *    of C each; per phase every thread copies one element of M and one of N
 *    into the block's two shared tiles, __syncthreads(), adds TILE_WIDTH
 *    products, __syncthreads(); tile_width is 16 or 32.  Sizes that are not
 *    multiples of the tile read zeros outside M and N and store nothing
 *    outside C.
 *
 * tgemm_pages_transpose_f32 is the matrix-transpose case study of note.jhbae.stream
 * "Lec 29 · GPU Architecture (2)": dst[j*ld_dst + i] = src[i*ld_src + j] with
 * 32 x 32 tiles and 32 x 8 threads, 4 elements per thread.  variant 0 reads
 * rows and writes columns straight from global memory (uncoalesced writes);
 * variant 1 goes through a shared tile[32][32] and writes coalesced (a column
 * read of the tile is a 32-way bank conflict); variant 2 pads the tile to
 * [32][33], which removes the conflicts.
 *
 * Arguments, ownership and status codes are those of tgemm.h (device
 * pointers owned by the caller, asynchronous on `stream`).  The status values
 * are the tgemm_status codes.
 */
#ifndef TGEMM_PAGES_H
#define TGEMM_PAGES_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;

int tgemm_pages_naive_f32(int64_t m, int64_t n, int64_t k,
                          const float *A, int64_t lda,
                          const float *B, int64_t ldb,
                          float *C, int64_t ldc,
                          struct CUstream_st *stream);

int tgemm_pages_tiled_f32(int64_t m, int64_t n, int64_t k,
                          const float *A, int64_t lda,
                          const float *B, int64_t ldb,
                          float *C, int64_t ldc,
                          int tile_width,
                          struct CUstream_st *stream);

int tgemm_pages_transpose_f32(int64_t rows, int64_t cols,
                              const float *src, int64_t ld_src,
                              float *dst, int64_t ld_dst,
                              int variant,
                              struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* TGEMM_PAGES_H */
