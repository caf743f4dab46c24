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
//
// When both matrices are 16-byte aligned with 16-byte pitches, a wider form
// moves the data with 128-bit accesses: a 64 x 32 tile per 256 threads, each
// thread loading two float4 from input rows and storing two float4 to output
// rows; the tile is [64][33], so both the row-wise writes into it and the
// column-wise reads out of it hit 32 distinct banks per warp instruction.
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

constexpr int kVRows = 64;   // input rows per tile of the 128-bit form
constexpr int kVCols = 32;   // input columns per tile

__global__ void __launch_bounds__(256)
transpose_v4_kernel(const float* __restrict__ src, int64_t ld_src, float* __restrict__ dst, int64_t ld_dst,
                    int rows, int cols) {
    __shared__ float tile[kVRows][kVCols + 1];
    const int t = threadIdx.x;
    const int lr = t >> 3;         // input row (and output row) within a 32-row half / the tile
    const int lq = (t & 7) * 4;    // first of 4 consecutive elements
    const int64_t tiles_c = (cols + kVCols - 1) / kVCols;
    const int64_t tiles = tiles_c * ((rows + kVRows - 1) / kVRows);
    for (int64_t idx = blockIdx.x; idx < tiles; idx += gridDim.x) {
        const int r0 = static_cast<int>(idx / tiles_c) * kVRows;
        const int c0 = static_cast<int>(idx % tiles_c) * kVCols;
        const bool whole = r0 + kVRows <= rows && c0 + kVCols <= cols;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = r0 + lr + 32 * i;
            if (whole) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(src + static_cast<int64_t>(r) * ld_src + c0 + lq));
                tile[lr + 32 * i][lq + 0] = v.x;
                tile[lr + 32 * i][lq + 1] = v.y;
                tile[lr + 32 * i][lq + 2] = v.z;
                tile[lr + 32 * i][lq + 3] = v.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = c0 + lq + j;
                    tile[lr + 32 * i][lq + j] = (r < rows && c < cols) ? src[static_cast<int64_t>(r) * ld_src + c] : 0.0f;
                }
            }
        }
        __syncthreads();
        const int c = c0 + lr;   // output row
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int rr = lq + 32 * i;   // first of 4 output columns (input rows) within the tile
            if (whole) {
                const float4 w = make_float4(tile[rr][lr], tile[rr + 1][lr], tile[rr + 2][lr], tile[rr + 3][lr]);
                *reinterpret_cast<float4*>(dst + static_cast<int64_t>(c) * ld_dst + r0 + rr) = w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int r = r0 + rr + j;
                    if (c < cols && r < rows) dst[static_cast<int64_t>(c) * ld_dst + r] = tile[rr + j][lr];
                }
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_transpose(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows,
                             int64_t cols, cudaStream_t stream, const Device& dev) {
    const bool v4 = reinterpret_cast<uintptr_t>(src) % 16 == 0 && reinterpret_cast<uintptr_t>(dst) % 16 == 0 &&
                    ld_src % 4 == 0 && ld_dst % 4 == 0;
    if (v4) {
        const int64_t tiles = ((rows + kVRows - 1) / kVRows) * ((cols + kVCols - 1) / kVCols);
        const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
        const unsigned grid = static_cast<unsigned>(tiles < cap ? tiles : cap);
        transpose_v4_kernel<<<grid, 256, 0, stream>>>(static_cast<const float*>(src), ld_src,
                                                       static_cast<float*>(dst), ld_dst, static_cast<int>(rows),
                                                       static_cast<int>(cols));
    } else {
        const int64_t tiles = ((rows + kTile - 1) / kTile) * ((cols + kTile - 1) / kTile);
        const int64_t cap = static_cast<int64_t>(dev.sm_count) * 64;
        const unsigned grid = static_cast<unsigned>(tiles < cap ? tiles : cap);
        transpose_kernel<<<grid, dim3(kTile, kRowsPerPass), 0, stream>>>(
            static_cast<const uint32_t*>(src), ld_src, static_cast<uint32_t*>(dst), ld_dst,
            static_cast<int>(rows), static_cast<int>(cols));
    }
    count_launch();
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) set_error("transpose kernel launch: %s", cudaGetErrorString(err));
    return err;
}

}  // namespace tgemm
