// pack.cu -- copies operands into pitched workspace that TMA can describe.
//
// A TMA descriptor needs a 16-byte aligned base and a row pitch that is a
// multiple of 16 bytes.  When the caller's A or B breaks either rule (for
// instance a 4097 x 1023 fp32 A with lda = 1023), the entry point copies it
// into workspace rows of ld_dst elements (ld_dst rounded up to 16 bytes) and
// zero-fills the padding columns, then runs the tiled kernel on the copy.
//
// The copy is plain coalesced memory traffic (note.jhbae.stream "Lec 29 · GPU
// Architecture (2)", coalescing: consecutive threads touch consecutive
// addresses): each thread writes one aligned 16-byte vector of each of four
// destination rows, gathering its 4 (fp32) or 8 (bf16) elements from each
// source row with element-sized loads (all of them in flight together), so a
// warp reads and writes 512 contiguous bytes per row.  Up to
// two matrices go out in one launch, and the kernel lets the dependent product
// kernel start its set-up at once (that kernel waits for this one to finish
// before it reads memory).
#include "device.cuh"
#include "host.h"

namespace tgemm {
namespace {

constexpr int kPackThreads = 256;
constexpr int kPackRows = 4;   // rows per thread: their loads are all in flight together

struct PackJob {
    const void* src;
    int64_t ld_src;
    void* dst;
    int64_t ld_dst;   // a multiple of 16 / element size
    int64_t rows, cols;
};

template <typename T>
__global__ void __launch_bounds__(kPackThreads)
pack_kernel(PackJob j0, PackJob j1) {
    griddep_launch_dependents();
    constexpr int kVec = 16 / sizeof(T);
    const PackJob& j = blockIdx.z == 0 ? j0 : j1;
    const int64_t vec = static_cast<int64_t>(blockIdx.x) * kPackThreads + threadIdx.x;
    if (vec * kVec >= j.ld_dst) return;
    const T* __restrict__ src = static_cast<const T*>(j.src);
    T* __restrict__ dst = static_cast<T*>(j.dst);
    const int64_t c0 = vec * kVec;
    const bool full = c0 + kVec <= j.cols;
    for (int64_t r0 = static_cast<int64_t>(blockIdx.y) * kPackRows; r0 < j.rows;
         r0 += static_cast<int64_t>(gridDim.y) * kPackRows) {
        union V {
            uint4 v;
            T e[kVec];
        } u[kPackRows];
#pragma unroll
        for (int q = 0; q < kPackRows; ++q) {
            const int64_t r = r0 + q < j.rows ? r0 + q : j.rows - 1;   // rows past the end repeat the last
            const T* srow = src + r * j.ld_src + c0;
#pragma unroll
            for (int e = 0; e < kVec; ++e) u[q].e[e] = (full || c0 + e < j.cols) ? srow[e] : T(0);
        }
#pragma unroll
        for (int q = 0; q < kPackRows; ++q)
            if (r0 + q < j.rows) *reinterpret_cast<uint4*>(dst + (r0 + q) * j.ld_dst + c0) = u[q].v;
    }
}

}  // namespace

cudaError_t launch_pack2(const PackSpec* specs, int count, int elem_bytes, cudaStream_t stream, const Device& dev) {
    if (count < 1 || count > 2) return cudaErrorInvalidValue;
    PackJob job[2] = {};
    int64_t vecs = 0, rows = 0;
    const int64_t vec_elems = 16 / elem_bytes;
    for (int i = 0; i < count; ++i) {
        job[i] = PackJob{specs[i].src, specs[i].ld_src, specs[i].dst, specs[i].ld_dst, specs[i].rows, specs[i].cols};
        const int64_t v = specs[i].ld_dst / vec_elems;
        vecs = v > vecs ? v : vecs;
        rows = specs[i].rows > rows ? specs[i].rows : rows;
    }
    if (count == 1) job[1] = job[0];
    const int64_t gx = (vecs + kPackThreads - 1) / kPackThreads;
    // kPackRows destination rows per block row (grid-stride beyond the grid's y limit)
    int64_t gy = (rows + kPackRows - 1) / kPackRows;
    gy = gy < 65535 ? gy : 65535;
    if (gy < 1) gy = 1;
    const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(count));
    if (elem_bytes == 4)
        pack_kernel<uint32_t><<<grid, kPackThreads, 0, stream>>>(job[0], job[1]);
    else
        pack_kernel<uint16_t><<<grid, kPackThreads, 0, stream>>>(job[0], job[1]);
    count_launch();
    (void)dev;
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) set_error("pack_kernel launch: %s", cudaGetErrorString(err));
    return err;
}

cudaError_t launch_pack(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows, int64_t cols,
                        int elem_bytes, cudaStream_t stream, const Device& dev) {
    const PackSpec s{src, ld_src, dst, ld_dst, rows, cols};
    return launch_pack2(&s, 1, elem_bytes, stream, dev);
}

}  // namespace tgemm
