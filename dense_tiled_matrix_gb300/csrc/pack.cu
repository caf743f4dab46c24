// pack.cu -- copies an operand into a pitched workspace that TMA can describe.
//
// A TMA descriptor needs a 16-byte aligned base and a row pitch that is a
// multiple of 16 bytes.  When the caller's A or B breaks either rule (for
// instance a 4097 x 1023 fp32 A with lda = 1023), the entry point copies it
// into workspace rows of ld_dst elements (ld_dst rounded up to 16 bytes) and
// zero-fills the padding columns, then runs the tiled kernel on the copy.
// The copy is plain coalesced memory traffic: consecutive threads move
// consecutive elements of a row.
#include "device.cuh"
#include "host.h"

namespace tgemm {
namespace {

template <typename T>
__global__ void __launch_bounds__(256)
pack_kernel(const T* __restrict__ src, int64_t ld_src, T* __restrict__ dst, int64_t ld_dst,
            int64_t rows, int64_t cols) {
    const int64_t col = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (col >= ld_dst) return;
    for (int64_t r = blockIdx.y; r < rows; r += gridDim.y) {
        dst[r * ld_dst + col] = col < cols ? src[r * ld_src + col] : T(0);
    }
}

}  // namespace

cudaError_t launch_pack(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows,
                        int64_t cols, int elem_bytes, cudaStream_t stream, const Device& dev) {
    const dim3 block(256);
    const int64_t gx = (ld_dst + 255) / 256;
    int64_t gy = rows < 65535 ? rows : 65535;
    if (gy < 1) gy = 1;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
    if (elem_bytes == 4)
        pack_kernel<uint32_t><<<grid, block, 0, stream>>>(static_cast<const uint32_t*>(src), ld_src,
                                                          static_cast<uint32_t*>(dst), ld_dst, rows, cols);
    else
        pack_kernel<uint16_t><<<grid, block, 0, stream>>>(static_cast<const uint16_t*>(src), ld_src,
                                                          static_cast<uint16_t*>(dst), ld_dst, rows, cols);
    count_launch();
    (void)dev;
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) set_error("pack_kernel launch: %s", cudaGetErrorString(err));
    return err;
}

}  // namespace tgemm
