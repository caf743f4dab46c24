// host.h -- declarations shared by the host parts of libtgemm: the per-device
// context, the problem description handed to each kernel's launcher, and the
// launchers themselves (one per kernel family, defined next to its kernel).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "tgemm.h"

namespace tgemm {

struct Device {
    int ordinal = -1;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int smem_optin = 0;           // max dynamic shared memory per block (bytes)
    uint32_t* status = nullptr;   // device address of this device's status word
};

// One product C = A * B, row-major, as validated by the C entry points.
// `A`/`B` point at fp32 or bf16 elements depending on the entry point.
struct Problem {
    int m = 0, n = 0, k = 0;
    const void* A = nullptr;
    int64_t lda = 0;
    const void* B = nullptr;
    int64_t ldb = 0;
    float* C = nullptr;
    int64_t ldc = 0;
    cudaStream_t stream = nullptr;
};

// Counts a kernel launch made by the library.
void count_launch();

// Encodes a 2-D tiled TMA descriptor over a row-major matrix of `rows` x
// `cols` elements (cols contiguous) with a row pitch of `ld` elements and a
// box of `box_rows` x `box_cols`.  Returns false with a message on failure.
bool make_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem_bytes,
                     const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                     uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle swizzle);

// Records a failure text for tgemm_last_error(); clear_error() empties it.
void set_error(const char* fmt, ...);
void clear_error();

// Host-side checks shared by the entry points (tgemm_api.cu).
// The current device, set up on first use (sm_103 check, SM count, status word).
tgemm_status current_device(Device** out);
// `p` is device or managed memory of device `ord` and [p, p + bytes) lies in one allocation.
tgemm_status check_span(const char* name, const void* p, uint64_t bytes, int ord);
// Records "what: <CUDA error text>" and returns TGEMM_ERR_CUDA.
tgemm_status cuda_fail(const char* what, cudaError_t err);
// TMA can describe the matrix: 16-byte aligned base and 16-byte row pitch.
bool tma_ok(const void* p, int64_t ld, int es);
// Bytes spanned by a rows x cols row-major matrix with pitch ld.
uint64_t span_bytes(int64_t rows, int64_t cols, int64_t ld, int es);
// The byte ranges [a, a+na) and [b, b+nb) intersect.
bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb);

// ------------------------------------------------------------ launchers --
// Each returns cudaSuccess or the launch error (with set_error called).

// The persistent kernels' plan (stream_k.cuh) has a stream-K region -- T = qG
// + r tiles on G CTAs with q >= 1, r > 0 and r * KT >= G -- so its last G + r
// tiles are split along k into G equal runs.
inline bool sk_has_region(int64_t tiles, int64_t KT, int64_t G) {
    const int64_t r = tiles % G;
    return tiles >= G && r > 0 && r * KT >= G;
}

// fp32 FFMA kernel; A and B must be 16-byte aligned with 16-byte row pitches.
// Shapes that take its split-tile form need ffma_f32_workspace_bytes() of
// stream-ordered device memory (256-byte aligned, no initial contents), valid
// until the kernel has run; others need none and take nullptr.
uint64_t ffma_f32_workspace_bytes(const Problem& p, const Device& dev);
cudaError_t launch_ffma_f32(const Problem& p, const Device& dev, void* workspace);
// The tiles launch_ffma_f32 would run (host arithmetic only, only dev.sm_count
// read): out[0] whole tiles, out[1] remainder tiles cut along k, out[2] pieces
// per remainder tile (0: none).
void ffma_f32_plan(const Problem& p, const Device& dev, int64_t out[3]);

// tcgen05 kernels; same alignment rule.  `tf32` selects kind::tf32 on fp32
// inputs, and then p.B must hold B TRANSPOSED (n x k, pitch p.ldb, k
// contiguous); otherwise bf16 inputs under kind::f16 with B as k x n.  With
// umma_workspace_bytes() of stream-ordered workspace (no initial contents)
// the last partial wave of tiles is split along k (stream-K), or, with fewer
// tiles than SMs, every tile (split-K pieces); with nullptr whole tiles only.
uint64_t umma_workspace_bytes(const Problem& p, const Device& dev, bool tf32);
cudaError_t launch_umma(const Problem& p, const Device& dev, bool tf32, void* workspace);
// The tiles launch_umma would use (host arithmetic only, only dev.sm_count read):
// out[0] tile rows, out[1] tile columns, out[2] stream-K, out[3] split-K pieces
// per tile, out[4] multicast CTA pairs.
void umma_plan(const Problem& p, const Device& dev, bool tf32, bool workspace, int out[5]);

// bf16 tcgen05 kernel for m <= 64: C^T = B^T A^T with k split across the CTAs
// of a cluster and the partials added through distributed shared memory.
cudaError_t launch_umma_skinny(const Problem& p, const Device& dev);

// dst (cols x rows, pitch ld_dst) = transpose of src (rows x cols, pitch
// ld_src), 4-byte elements.
cudaError_t launch_transpose(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows,
                             int64_t cols, cudaStream_t stream, const Device& dev);

// Copies a rows x cols matrix of `elem_bytes`-byte elements with pitch `ld_src`
// into `dst` with pitch `ld_dst` (elements; dst 16-byte aligned and ld_dst a
// multiple of 16 bytes), zero-filling columns cols .. ld_dst-1.
cudaError_t launch_pack(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows,
                        int64_t cols, int elem_bytes, cudaStream_t stream, const Device& dev);

// One or two such copies (same element size) in one launch.
struct PackSpec {
    const void* src;
    int64_t ld_src;
    void* dst;
    int64_t ld_dst;
    int64_t rows, cols;
};
cudaError_t launch_pack2(const PackSpec* specs, int count, int elem_bytes, cudaStream_t stream, const Device& dev);

}  // namespace tgemm
