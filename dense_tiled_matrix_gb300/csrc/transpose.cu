// transpose.cu -- dst (cols x rows, pitch ld_dst) = transpose of src (rows x
// cols, pitch ld_src), 4-byte elements.
//
// The TF32 tensor-core path needs B with K contiguous, the opposite of the
// caller's row-major B (N contiguous); this kernel makes that copy.  It is the
// shared-memory transpose of note.jhbae.stream "Lec 29 · GPU Architecture
// (2)" (matrix transpose case study): a 32 x 32 tile read with coalesced row
// accesses, a barrier, and a coalesced write of the tile's columns; the tile
// is declared [32][33] so that reading a column touches 32 different banks
// instead of replaying 32 times on one bank; blocks of 32 x 8 threads each move
// 4 elements per tile to amortise index arithmetic.
#include "device.cuh"
#include "host.h"

namespace tgemm {
namespace {

constexpr int kTile = 32;
constexpr int kRowsPerPass = 8;

__global__ void __launch_bounds__(kTile * kRowsPerPass)
transpose_kernel(const uint32_t* __restrict__ src, int64_t ld_src, uint32_t* __restrict__ dst,
                 int64_t ld_dst, int rows, int cols) {
    __shared__ uint32_t tile[kTile][kTile + 1];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int tiles_c = (cols + kTile - 1) / kTile;
    const int tiles_r = (rows + kTile - 1) / kTile;
    for (int64_t t = blockIdx.x; t < static_cast<int64_t>(tiles_c) * tiles_r; t += gridDim.x) {
        const int r0 = static_cast<int>(t / tiles_c) * kTile;
        const int c0 = static_cast<int>(t % tiles_c) * kTile;
#pragma unroll
        for (int j = 0; j < kTile; j += kRowsPerPass) {
            const int r = r0 + ty + j, c = c0 + tx;
            if (r < rows && c < cols) tile[ty + j][tx] = src[static_cast<int64_t>(r) * ld_src + c];
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kTile; j += kRowsPerPass) {
            const int c = c0 + ty + j, r = r0 + tx;   // dst row c, column r
            if (c < cols && r < rows) dst[static_cast<int64_t>(c) * ld_dst + r] = tile[tx][ty + j];
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_transpose(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows,
                             int64_t cols, cudaStream_t stream, const Device& dev) {
    const int64_t tiles = ((rows + kTile - 1) / kTile) * ((cols + kTile - 1) / kTile);
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 64;
    const unsigned grid = static_cast<unsigned>(tiles < cap ? tiles : cap);
    transpose_kernel<<<grid, dim3(kTile, kRowsPerPass), 0, stream>>>(
        static_cast<const uint32_t*>(src), ld_src, static_cast<uint32_t*>(dst), ld_dst, static_cast<int>(rows),
        static_cast<int>(cols));
    count_launch();
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) set_error("transpose_kernel launch: %s", cudaGetErrorString(err));
    return err;
}

}  // namespace tgemm
