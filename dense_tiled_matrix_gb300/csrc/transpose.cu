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
// When both matrices are 16-byte aligned with 16-byte pitches, a TMA form
// (below) moves whole 128-byte lines in and out instead.
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
    griddep_launch_dependents();   // the product that reads dst may be launched now; it waits for us
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

// TMA form: a persistent grid whose CTAs take 128 x 32 input tiles (128 rows
// of one 128-byte line each) in turn.  One thread keeps kXStages tile loads in
// flight (TMA with the 128-byte swizzle: 16-byte chunk c of tile row r sits at
// chunk c ^ (r % 8), so the 8 lanes of a quarter-warp reading chunk j of 8
// consecutive rows hit 8 different bank groups); the CTA turns each tile into
// a 32 x 128 output tile in a plain shared buffer (a warp writes 32
// consecutive words per instruction) and one thread stores it with a TMA bulk
// store, which skips rows and columns outside dst.  Two output buffers
// alternate, so a tile's store overlaps the next tile's shuffle.
constexpr int kXR = 128;                               // input rows per tile = output columns
constexpr int kXC = 32;                                // input columns per tile = output rows
constexpr int kXStages = 4;
constexpr int kXThreads = 256;
constexpr uint32_t kXTileBytes = kXR * kXC * 4;        // 16 KiB
constexpr size_t kXSmem = 1024 + (kXStages + 2) * kXTileBytes + kXStages * sizeof(uint64_t);

__global__ void __launch_bounds__(kXThreads, 2)
transpose_tma_kernel(const __grid_constant__ CUtensorMap tm_src, const __grid_constant__ CUtensorMap tm_dst,
                     int rows, int cols, uint32_t* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = smem_align_1024(smem_raw);
    uint8_t* in = base;                                           // kXStages swizzled input tiles
    float* out = reinterpret_cast<float*>(base + kXStages * kXTileBytes);   // 2 x [kXC][kXR]
    uint64_t* full = reinterpret_cast<uint64_t*>(base + (kXStages + 2) * kXTileBytes);

    griddep_launch_dependents();   // the product that reads dst may be launched now; it waits for us
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tiles_c = (cols + kXC - 1) / kXC;
    const int64_t tiles = static_cast<int64_t>((rows + kXR - 1) / kXR) * tiles_c;
    const int n = tiles > blockIdx.x ? static_cast<int>((tiles - 1 - blockIdx.x) / gridDim.x) + 1 : 0;
    auto load = [&](int i) {
        const int64_t t = blockIdx.x + static_cast<int64_t>(i) * gridDim.x;
        const int s = i % kXStages;
        mbar_arrive_expect_tx(&full[s], kXTileBytes);
        tma_load_2d(in + s * kXTileBytes, &tm_src, &full[s], static_cast<int>(t % tiles_c) * kXC,
                    static_cast<int>(t / tiles_c) * kXR);
    };
    int issued = 0;   // loads issued (thread 0)
    if (tid == 0) {
        tma_prefetch_map(&tm_src);
        tma_prefetch_map(&tm_dst);
        for (int s = 0; s < kXStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
        for (int i = 0; i < n && i < kXStages; ++i) load(i);
        issued = n < kXStages ? n : kXStages;
    }
    __syncthreads();

    bool ok = true;
    for (int i = 0; i < n; ++i) {
        const int s = i % kXStages;
        float* o = out + (i & 1) * (kXC * kXR);
        if (ok && !mbar_wait(&full[s], static_cast<uint32_t>(i / kXStages) & 1u, status)) ok = false;
        if (tid == 0) bulk_wait_group_read<1>();   // the store that last used `o` has read it
        __syncthreads();
        // Warp w moves 4 strips of 32 rows x 4 columns: lane l reads row
        // 32 rb + l, chunk j (columns 4j .. 4j+3) and writes them to output
        // rows 4j .. 4j+3, column 32 rb + l.
        const uint8_t* tile = in + s * kXTileBytes;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int u = warp * 4 + q, rb = u >> 3, j = u & 7;
            const int r = rb * 32 + lane;
            const float4 v = *reinterpret_cast<const float4*>(tile + r * 128 + ((j ^ (r & 7)) << 4));
            o[(4 * j + 0) * kXR + r] = v.x;
            o[(4 * j + 1) * kXR + r] = v.y;
            o[(4 * j + 2) * kXR + r] = v.z;
            o[(4 * j + 3) * kXR + r] = v.w;
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            const int64_t t = blockIdx.x + static_cast<int64_t>(i) * gridDim.x;
            tma_store_2d(&tm_dst, o, static_cast<int>(t / tiles_c) * kXR, static_cast<int>(t % tiles_c) * kXC);
            bulk_commit_group();
            // Every thread has read stage s (barrier above): refill it.
            if (ok && i + kXStages < n) {
                fence_proxy_async_smem();
                load(i + kXStages);
                ++issued;
            }
        }
    }
    if (tid == 0) {
        drain_ring(full, kXStages, issued, status);   // loads left unwaited after a timeout
        bulk_wait_group<0>();
    }
}

}  // namespace

cudaError_t launch_transpose(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows,
                             int64_t cols, cudaStream_t stream, const Device& dev) {
    const bool aligned = reinterpret_cast<uintptr_t>(src) % 16 == 0 && reinterpret_cast<uintptr_t>(dst) % 16 == 0 &&
                         ld_src % 4 == 0 && ld_dst % 4 == 0;
    cudaError_t err = cudaSuccess;
    if (aligned) {
        CUtensorMap ts, td;
        if (!make_tensor_map(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, src, rows, cols, ld_src, kXR, kXC,
                             CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_tensor_map(&td, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dst, cols, rows, ld_dst, kXC, kXR,
                             CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        err = cudaFuncSetAttribute(transpose_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(kXSmem));
        if (err != cudaSuccess) {
            set_error("cudaFuncSetAttribute(transpose_tma_kernel): %s", cudaGetErrorString(err));
            return err;
        }
        const int64_t tiles = ((rows + kXR - 1) / kXR) * ((cols + kXC - 1) / kXC);
        const int64_t cap = static_cast<int64_t>(dev.sm_count) * 2;
        const unsigned grid = static_cast<unsigned>(tiles < cap ? tiles : cap);
        transpose_tma_kernel<<<grid, kXThreads, kXSmem, stream>>>(ts, td, static_cast<int>(rows),
                                                                  static_cast<int>(cols), dev.status);
    } else {
        const int64_t tiles = ((rows + kTile - 1) / kTile) * ((cols + kTile - 1) / kTile);
        const int64_t cap = static_cast<int64_t>(dev.sm_count) * 64;
        const unsigned grid = static_cast<unsigned>(tiles < cap ? tiles : cap);
        transpose_kernel<<<grid, dim3(kTile, kRowsPerPass), 0, stream>>>(
            static_cast<const uint32_t*>(src), ld_src, static_cast<uint32_t*>(dst), ld_dst,
            static_cast<int>(rows), static_cast<int>(cols));
    }
    count_launch();
    err = cudaGetLastError();
    if (err != cudaSuccess) set_error("transpose kernel launch: %s", cudaGetErrorString(err));
    return err;
}

}  // namespace tgemm
