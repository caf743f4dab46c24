// noalloc.cu -- tgemm_tf32_noalloc: the TF32 product without any device
// memory allocation on the call path.
//
// tgemm_tf32 needs temporary device memory: a transposed (K-contiguous) copy
// of B for the tensor cores, and a re-pitched copy of A when A's base or row
// pitch is not a multiple of 16 bytes.  It takes that memory from the stream-
// ordered allocator on every call.  Some callers cannot let a library
// allocate: code whose device memory is entirely owned by its own allocator
// or arena (so an outside allocation can fail or break its accounting), and
// code that must not risk the synchronisation or latency of an allocation on
// its hot path.  For them this entry point uses a fixed array in the
// library's static device memory instead, sized TGEMM_NOALLOC_SCRATCH_BYTES.
//
// The array exists once per GPU that loads this part of the library and stays
// allocated until the process exits.  Host code cannot use the array's name as
// a device address; the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current) and every later call on that
// device reuses it.
#include <mutex>

#include "host.h"
#include "tgemm.h"

namespace tgemm {
namespace {

constexpr uint64_t kScratchBytes = TGEMM_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte sub-buffers aligned");

static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices];

// Device address of this device's copy of the scratch array; the device must
// be current.  Looked up once per device.
tgemm_status scratch_address(int ord, void** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[ord]) {
        void* p = nullptr;
        const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return cuda_fail("cudaGetSymbolAddress(noalloc scratch)", err);
        g_scratch_addr[ord] = p;
    }
    *out = g_scratch_addr[ord];
    return TGEMM_OK;
}

uint64_t round256(uint64_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace tgemm

extern "C" tgemm_status tgemm_tf32_noalloc(int64_t m, int64_t n, int64_t k, const float* A, int64_t lda,
                                           const float* B, int64_t ldb, float* C, int64_t ldc,
                                           struct CUstream_st* stream) {
    using namespace tgemm;
    clear_error();
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (m < 0 || n < 0 || k < 0 || m > lim || n > lim || k > lim) {
        set_error("sizes must satisfy 0 <= m, n, k < 2^31");
        return TGEMM_ERR_INVALID_VALUE;
    }
    if (m == 0 || n == 0) return TGEMM_OK;
    if (lda < (k > 1 ? k : 1) || ldb < n || ldc < n || lda > (int64_t(1) << 40) || ldb > (int64_t(1) << 40) ||
        ldc > (int64_t(1) << 40)) {
        set_error("leading dimensions must satisfy lda >= max(1,k), ldb >= max(1,n), ldc >= max(1,n)");
        return TGEMM_ERR_INVALID_VALUE;
    }
    if (!C || (k > 0 && (!A || !B))) {
        set_error("NULL pointer for a matrix with nonzero extent");
        return TGEMM_ERR_INVALID_VALUE;
    }
    const uint64_t a_bytes = k > 0 ? span_bytes(m, k, lda, 4) : 0;
    const uint64_t b_bytes = k > 0 ? span_bytes(k, n, ldb, 4) : 0;
    const uint64_t c_bytes = span_bytes(m, n, ldc, 4);
    if (overlaps(C, c_bytes, A, a_bytes) || overlaps(C, c_bytes, B, b_bytes)) {
        set_error("C overlaps A or B");
        return TGEMM_ERR_INVALID_VALUE;
    }
    if (reinterpret_cast<uintptr_t>(C) % 4 || reinterpret_cast<uintptr_t>(A) % 4 ||
        reinterpret_cast<uintptr_t>(B) % 4) {
        set_error("pointers must be aligned to 4 bytes");
        return TGEMM_ERR_INVALID_VALUE;
    }
    // Scratch needed: B^T (n x k4) always, A re-pitched (m x k4) when TMA
    // cannot describe A as given; k4 = k rounded up to a multiple of 4.
    const int64_t k4 = (k + 3) / 4 * 4;
    const bool pack_a = k > 0 && !tma_ok(A, lda, 4);
    const uint64_t a_ws = pack_a ? round256(static_cast<uint64_t>(m) * k4 * 4) : 0;
    const uint64_t b_ws = k > 0 ? round256(static_cast<uint64_t>(n) * k4 * 4) : 0;
    if (a_ws + b_ws > kScratchBytes) {
        set_error("tgemm_tf32_noalloc needs %llu bytes of scratch for this shape; its static array holds %llu "
                  "(TGEMM_NOALLOC_SCRATCH_BYTES)",
                  (unsigned long long)(a_ws + b_ws), (unsigned long long)kScratchBytes);
        return TGEMM_ERR_INVALID_VALUE;
    }

    Device* dev = nullptr;
    tgemm_status st = current_device(&dev);
    if (st != TGEMM_OK) return st;
    if ((st = check_span("C", C, c_bytes, dev->ordinal)) != TGEMM_OK) return st;
    if (k == 0) {
        const cudaError_t err = cudaMemset2DAsync(C, static_cast<size_t>(ldc) * 4, 0,
                                                  static_cast<size_t>(n) * 4, static_cast<size_t>(m), stream);
        return err == cudaSuccess ? TGEMM_OK : cuda_fail("cudaMemset2DAsync(C)", err);
    }
    if ((st = check_span("A", A, a_bytes, dev->ordinal)) != TGEMM_OK) return st;
    if ((st = check_span("B", B, b_bytes, dev->ordinal)) != TGEMM_OK) return st;
    void* scratch = nullptr;
    if ((st = scratch_address(dev->ordinal, &scratch)) != TGEMM_OK) return st;
    uint8_t* w = static_cast<uint8_t*>(scratch);

    Problem p;
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.A = A;
    p.lda = lda;
    p.C = C;
    p.ldc = ldc;
    p.stream = stream;
    cudaError_t err = cudaSuccess;
    if (pack_a) {
        err = launch_pack(A, lda, w, k4, m, k, 4, stream, *dev);
        p.A = w;
        p.lda = k4;
    }
    if (err == cudaSuccess) {
        // Every element of B^T that the product reads is written here; the
        // padding columns k .. k4-1 lie outside the descriptor and are never read.
        err = launch_transpose(B, ldb, w + a_ws, k4, k, n, stream, *dev);
        p.B = w + a_ws;
        p.ldb = k4;
    }
    if (err == cudaSuccess) err = launch_umma(p, *dev, true, nullptr);   // whole tiles: no partial-sum workspace
    if (err != cudaSuccess) {
        if (tgemm_last_error()[0] == '\0') set_error("CUDA: %s", cudaGetErrorString(err));
        return TGEMM_ERR_CUDA;
    }
    return TGEMM_OK;
}
