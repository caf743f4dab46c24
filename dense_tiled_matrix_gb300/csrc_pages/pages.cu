// pages.cu -- the pages' naive and shared-memory tiled matrix multiply, as
// comparators (libtgemm_pages; see include/tgemm_pages.h for what each
// computes and where the pages describe it).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "tgemm.h"
#include "tgemm_pages.h"

namespace {

// One thread per element of C, operands straight from global memory.
__global__ void naive_kernel(const float* __restrict__ M, int64_t ldm, const float* __restrict__ N,
                             int64_t ldn, float* __restrict__ P, int64_t ldp, int rows, int cols, int width) {
    const int col = blockIdx.x * blockDim.x + threadIdx.x;
    const int row = blockIdx.y * blockDim.y + threadIdx.y;
    if (row >= rows || col >= cols) return;
    float value = 0.0f;
    for (int k = 0; k < width; ++k)
        value = fmaf(M[static_cast<int64_t>(row) * ldm + k], N[static_cast<int64_t>(k) * ldn + col], value);
    P[static_cast<int64_t>(row) * ldp + col] = value;
}

// TILE x TILE threads; per phase one element of each operand per thread into
// shared memory, a barrier, TILE products, a barrier.
template <int TILE>
__global__ void tiled_kernel(const float* __restrict__ M, int64_t ldm, const float* __restrict__ N,
                             int64_t ldn, float* __restrict__ P, int64_t ldp, int rows, int cols, int width) {
    __shared__ float subTileM[TILE][TILE];
    __shared__ float subTileN[TILE][TILE];
    const int tx = threadIdx.x, ty = threadIdx.y;
    const int row = blockIdx.y * TILE + ty;
    const int col = blockIdx.x * TILE + tx;
    float pvalue = 0.0f;
    const int phases = (width + TILE - 1) / TILE;
    for (int ph = 0; ph < phases; ++ph) {
        const int mk = ph * TILE + tx;   // M element of this thread: (row, mk)
        const int nk = ph * TILE + ty;   // N element of this thread: (nk, col)
        subTileM[ty][tx] = (row < rows && mk < width) ? M[static_cast<int64_t>(row) * ldm + mk] : 0.0f;
        subTileN[ty][tx] = (nk < width && col < cols) ? N[static_cast<int64_t>(nk) * ldn + col] : 0.0f;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < TILE; ++k) pvalue = fmaf(subTileM[ty][k], subTileN[k][tx], pvalue);
        __syncthreads();
    }
    if (row < rows && col < cols) P[static_cast<int64_t>(row) * ldp + col] = pvalue;
}

// Transposes of the lecture's case study: TILE x TILE tiles, TILE x 8 threads,
// each thread moving 4 elements (rows ty, ty+8, ty+16, ty+24 of the tile).
constexpr int kTT = 32;
constexpr int kTR = 8;

// Naive: read row-wise (coalesced), write column-wise (strided, uncoalesced).
__global__ void transpose_naive_kernel(const float* __restrict__ in, int64_t ld_in, float* __restrict__ out,
                                       int64_t ld_out, int rows, int cols) {
    const int x = blockIdx.x * kTT + threadIdx.x;   // input column
    const int y0 = blockIdx.y * kTT + threadIdx.y;  // input row
    for (int j = 0; j < kTT; j += kTR) {
        const int y = y0 + j;
        if (x < cols && y < rows) out[static_cast<int64_t>(x) * ld_out + y] = in[static_cast<int64_t>(y) * ld_in + x];
    }
}

// Shared-memory tile: coalesced read into the tile, barrier, block offsets
// swapped, a column of the tile written out coalesced.  PAD = 0 is tile[32][32]
// (a warp reading a column hits one bank 32 times), PAD = 1 is tile[32][33].
template <int PAD>
__global__ void transpose_tiled_kernel(const float* __restrict__ in, int64_t ld_in, float* __restrict__ out,
                                       int64_t ld_out, int rows, int cols) {
    __shared__ float tile[kTT][kTT + PAD];
    int x = blockIdx.x * kTT + threadIdx.x;
    int y = blockIdx.y * kTT + threadIdx.y;
    for (int j = 0; j < kTT; j += kTR)
        if (x < cols && y + j < rows) tile[threadIdx.y + j][threadIdx.x] = in[static_cast<int64_t>(y + j) * ld_in + x];
    __syncthreads();
    x = blockIdx.y * kTT + threadIdx.x;   // output column = input row
    y = blockIdx.x * kTT + threadIdx.y;   // output row = input column
    for (int j = 0; j < kTT; j += kTR)
        if (x < rows && y + j < cols) out[static_cast<int64_t>(y + j) * ld_out + x] = tile[threadIdx.x][threadIdx.y + j];
}

using AddressRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);

AddressRangeFn address_range() {
    static AddressRangeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<AddressRangeFn>(p);
    });
    return fn;
}

// Device memory of the current device holding `bytes` from p.
bool span_ok(const void* p, uint64_t bytes) {
    if (bytes == 0) return true;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    int dev = -1;
    cudaGetDevice(&dev);
    if (!((a.type == cudaMemoryTypeDevice && a.device == dev) || a.type == cudaMemoryTypeManaged)) return false;
    if (AddressRangeFn f = address_range()) {
        CUdeviceptr base = 0;
        size_t size = 0;
        if (f(&base, &size, reinterpret_cast<CUdeviceptr>(p)) == CUDA_SUCCESS &&
            reinterpret_cast<uint64_t>(p) - base + bytes > size)
            return false;
    }
    return true;
}

uint64_t span(int64_t r, int64_t c, int64_t ld) {
    return (r == 0 || c == 0) ? 0 : (static_cast<uint64_t>(r - 1) * ld + c) * 4;
}

int check(int64_t m, int64_t n, int64_t k, const float* A, int64_t lda, const float* B, int64_t ldb, float* C,
          int64_t ldc) {
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (m < 0 || n < 0 || k < 0 || m > lim || n > lim || k > lim) return TGEMM_ERR_INVALID_VALUE;
    if (m == 0 || n == 0) return TGEMM_OK;
    if (lda < (k > 1 ? k : 1) || ldb < n || ldc < n) return TGEMM_ERR_INVALID_VALUE;
    if (!C || (k > 0 && (!A || !B))) return TGEMM_ERR_INVALID_VALUE;
    if (!span_ok(C, span(m, n, ldc)) || (k > 0 && (!span_ok(A, span(m, k, lda)) || !span_ok(B, span(k, n, ldb)))))
        return TGEMM_ERR_INVALID_VALUE;
    int dev = -1, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return TGEMM_ERR_CUDA;
    if (major != 10 || minor != 3) return TGEMM_ERR_UNSUPPORTED_DEVICE;
    return -1;   // proceed
}

}  // namespace

extern "C" int tgemm_pages_naive_f32(int64_t m, int64_t n, int64_t k, const float* A, int64_t lda, const float* B,
                                     int64_t ldb, float* C, int64_t ldc, struct CUstream_st* stream) {
    const int st = check(m, n, k, A, lda, B, ldb, C, ldc);
    if (st >= 0) return st;
    const dim3 block(16, 16);
    const dim3 grid(static_cast<unsigned>((n + 15) / 16), static_cast<unsigned>((m + 15) / 16));
    if (grid.y > 65535) return TGEMM_ERR_INVALID_VALUE;
    naive_kernel<<<grid, block, 0, stream>>>(A, lda, B, ldb, C, ldc, static_cast<int>(m), static_cast<int>(n),
                                             static_cast<int>(k));
    return cudaGetLastError() == cudaSuccess ? TGEMM_OK : TGEMM_ERR_CUDA;
}

extern "C" int tgemm_pages_tiled_f32(int64_t m, int64_t n, int64_t k, const float* A, int64_t lda, const float* B,
                                     int64_t ldb, float* C, int64_t ldc, int tile_width,
                                     struct CUstream_st* stream) {
    if (tile_width != 16 && tile_width != 32) return TGEMM_ERR_INVALID_VALUE;
    const int st = check(m, n, k, A, lda, B, ldb, C, ldc);
    if (st >= 0) return st;
    const int T = tile_width;
    const dim3 block(T, T);
    const dim3 grid(static_cast<unsigned>((n + T - 1) / T), static_cast<unsigned>((m + T - 1) / T));
    if (grid.y > 65535) return TGEMM_ERR_INVALID_VALUE;
    if (T == 16)
        tiled_kernel<16><<<grid, block, 0, stream>>>(A, lda, B, ldb, C, ldc, static_cast<int>(m),
                                                      static_cast<int>(n), static_cast<int>(k));
    else
        tiled_kernel<32><<<grid, block, 0, stream>>>(A, lda, B, ldb, C, ldc, static_cast<int>(m),
                                                      static_cast<int>(n), static_cast<int>(k));
    return cudaGetLastError() == cudaSuccess ? TGEMM_OK : TGEMM_ERR_CUDA;
}

extern "C" int tgemm_pages_transpose_f32(int64_t rows, int64_t cols, const float* src, int64_t ld_src, float* dst,
                                         int64_t ld_dst, int variant, struct CUstream_st* stream) {
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (variant < 0 || variant > 2 || rows < 0 || cols < 0 || rows > lim || cols > lim) return TGEMM_ERR_INVALID_VALUE;
    if (rows == 0 || cols == 0) return TGEMM_OK;
    if (ld_src < cols || ld_dst < rows || !src || !dst) return TGEMM_ERR_INVALID_VALUE;
    const uint64_t sb = span(rows, cols, ld_src), db = span(cols, rows, ld_dst);
    const uintptr_t a = reinterpret_cast<uintptr_t>(src), b = reinterpret_cast<uintptr_t>(dst);
    if (a < b + db && b < a + sb) return TGEMM_ERR_INVALID_VALUE;
    if (!span_ok(src, sb) || !span_ok(dst, db)) return TGEMM_ERR_INVALID_VALUE;
    int dev = -1, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return TGEMM_ERR_CUDA;
    if (major != 10 || minor != 3) return TGEMM_ERR_UNSUPPORTED_DEVICE;
    const dim3 block(kTT, kTR);
    const dim3 grid(static_cast<unsigned>((cols + kTT - 1) / kTT), static_cast<unsigned>((rows + kTT - 1) / kTT));
    if (grid.y > 65535) return TGEMM_ERR_INVALID_VALUE;
    const int r = static_cast<int>(rows), c = static_cast<int>(cols);
    if (variant == 0)
        transpose_naive_kernel<<<grid, block, 0, stream>>>(src, ld_src, dst, ld_dst, r, c);
    else if (variant == 1)
        transpose_tiled_kernel<0><<<grid, block, 0, stream>>>(src, ld_src, dst, ld_dst, r, c);
    else
        transpose_tiled_kernel<1><<<grid, block, 0, stream>>>(src, ld_src, dst, ld_dst, r, c);
    return cudaGetLastError() == cudaSuccess ? TGEMM_OK : TGEMM_ERR_CUDA;
}
