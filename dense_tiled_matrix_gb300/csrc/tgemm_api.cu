// tgemm_api.cu -- the C entry points of libtgemm: argument checks, device
// checks, TMA descriptor encoding, workspace for misaligned operands, and the
// choice of kernel.  The operation and the argument rules are those stated in
// include/tgemm.h.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "device.cuh"
#include "host.h"
#include "tgemm.h"

// Per-device status word: a kernel that gives up on a pipeline wait writes a
// nonzero code here (every device that loads the library has its own copy).
__device__ uint32_t g_tgemm_status;

namespace tgemm {

namespace {

thread_local char t_last_error[512];
std::atomic<uint64_t> g_launches{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
using AddressRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);

struct DriverFns {
    EncodeTiledFn encode = nullptr;
    AddressRangeFn address_range = nullptr;
    bool loaded = false;
};

DriverFns& driver() {
    static DriverFns fns;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.encode = reinterpret_cast<EncodeTiledFn>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.address_range = reinterpret_cast<AddressRangeFn>(fn);
        fns.loaded = true;
    });
    return fns;
}

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
Device g_devices[kMaxDevices];
tgemm_status g_dev_state[kMaxDevices];   // TGEMM_OK once set up; error otherwise
bool g_dev_ready[kMaxDevices];

}  // namespace

tgemm_status cuda_fail(const char* what, cudaError_t err) {
    set_error("%s: %s", what, cudaGetErrorString(err));
    return TGEMM_ERR_CUDA;
}

// Current device, set up on first use: compute capability check, SM count,
// shared-memory limit and the address of its status word.
tgemm_status current_device(Device** out) {
    int ord = -1;
    cudaError_t err = cudaGetDevice(&ord);
    if (err != cudaSuccess) return cuda_fail("cudaGetDevice", err);
    if (ord < 0 || ord >= kMaxDevices) {
        set_error("device ordinal %d out of range", ord);
        return TGEMM_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!g_dev_ready[ord]) {
        Device d;
        d.ordinal = ord;
        tgemm_status st = TGEMM_OK;
        if ((err = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, ord)) != cudaSuccess ||
            (err = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, ord)) != cudaSuccess ||
            (err = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, ord)) != cudaSuccess ||
            (err = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, ord)) !=
                cudaSuccess) {
            return cuda_fail("cudaDeviceGetAttribute", err);
        }
        if (d.cc_major != 10 || d.cc_minor != 3) {
            set_error("device %d is sm_%d%d; libtgemm is built for sm_103a only", ord, d.cc_major, d.cc_minor);
            st = TGEMM_ERR_UNSUPPORTED_DEVICE;
        } else {
            void* p = nullptr;
            if ((err = cudaGetSymbolAddress(&p, g_tgemm_status)) != cudaSuccess)
                return cuda_fail("cudaGetSymbolAddress(status)", err);
            d.status = static_cast<uint32_t*>(p);
            if (!driver().encode) {
                set_error("cuTensorMapEncodeTiled is not available from the driver");
                st = TGEMM_ERR_CUDA;
            }
        }
        g_devices[ord] = d;
        g_dev_state[ord] = st;
        g_dev_ready[ord] = true;
    }
    if (g_dev_state[ord] != TGEMM_OK) {
        set_error("device %d is not usable by libtgemm (sm_%d%d)", ord, g_devices[ord].cc_major,
                  g_devices[ord].cc_minor);
        return g_dev_state[ord];
    }
    *out = &g_devices[ord];
    return TGEMM_OK;
}

// The pointer must be device (or managed) memory reachable from device `ord`,
// and [p, p + bytes) must lie inside one allocation.
tgemm_status check_span(const char* name, const void* p, uint64_t bytes, int ord) {
    cudaPointerAttributes attr;
    cudaError_t err = cudaPointerGetAttributes(&attr, p);
    if (err != cudaSuccess) {
        cudaGetLastError();
        set_error("%s: not a CUDA pointer (%s)", name, cudaGetErrorString(err));
        return TGEMM_ERR_INVALID_VALUE;
    }
    if (attr.type == cudaMemoryTypeDevice) {
        if (attr.device != ord) {
            set_error("%s lives on device %d, the current device is %d", name, attr.device, ord);
            return TGEMM_ERR_INVALID_VALUE;
        }
    } else if (attr.type != cudaMemoryTypeManaged) {
        set_error("%s is host memory; libtgemm takes device pointers", name);
        return TGEMM_ERR_INVALID_VALUE;
    }
    AddressRangeFn range = driver().address_range;
    if (range) {
        CUdeviceptr base = 0;
        size_t size = 0;
        if (range(&base, &size, reinterpret_cast<CUdeviceptr>(p)) == CUDA_SUCCESS) {
            const uint64_t off = reinterpret_cast<uint64_t>(p) - static_cast<uint64_t>(base);
            if (off + bytes > size) {
                set_error("%s: %llu bytes from the pointer run past the end of its allocation", name,
                          static_cast<unsigned long long>(bytes));
                return TGEMM_ERR_INVALID_VALUE;
            }
        }
    }
    return TGEMM_OK;
}

bool tma_ok(const void* p, int64_t ld, int es) {
    return (reinterpret_cast<uintptr_t>(p) % 16 == 0) && ((ld * es) % 16 == 0);
}

enum class Kind { F32, TF32, BF16 };

// Bytes spanned by a rows x cols row-major matrix with pitch ld.
uint64_t span_bytes(int64_t rows, int64_t cols, int64_t ld, int es) {
    if (rows == 0 || cols == 0) return 0;
    return (static_cast<uint64_t>(rows - 1) * static_cast<uint64_t>(ld) + static_cast<uint64_t>(cols)) *
           static_cast<uint64_t>(es);
}

bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
    if (na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

namespace {

tgemm_status run(Kind kind, int64_t m, int64_t n, int64_t k, const void* A, int64_t lda, const void* B,
                 int64_t ldb, float* C, int64_t ldc, cudaStream_t stream) {
    t_last_error[0] = '\0';
    const int es = kind == Kind::BF16 ? 2 : 4;
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (m < 0 || n < 0 || k < 0 || m > lim || n > lim || k > lim) {
        set_error("sizes must satisfy 0 <= m, n, k < 2^31 (got %lld, %lld, %lld)", (long long)m,
                  (long long)n, (long long)k);
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
    const uint64_t a_bytes = k > 0 ? span_bytes(m, k, lda, es) : 0;
    const uint64_t b_bytes = k > 0 ? span_bytes(k, n, ldb, es) : 0;
    const uint64_t c_bytes = span_bytes(m, n, ldc, 4);
    if (overlaps(C, c_bytes, A, a_bytes) || overlaps(C, c_bytes, B, b_bytes)) {
        set_error("C overlaps A or B");
        return TGEMM_ERR_INVALID_VALUE;
    }
    if (reinterpret_cast<uintptr_t>(C) % 4 != 0 || (A && reinterpret_cast<uintptr_t>(A) % es != 0) ||
        (B && reinterpret_cast<uintptr_t>(B) % es != 0)) {
        set_error("pointers must be aligned to their element size");
        return TGEMM_ERR_INVALID_VALUE;
    }

    Device* dev = nullptr;
    tgemm_status st = current_device(&dev);
    if (st != TGEMM_OK) return st;
    if ((st = check_span("C", C, c_bytes, dev->ordinal)) != TGEMM_OK) return st;
    if (k == 0) {
        cudaError_t err = cudaMemset2DAsync(C, static_cast<size_t>(ldc) * 4, 0, static_cast<size_t>(n) * 4,
                                            static_cast<size_t>(m), stream);
        return err == cudaSuccess ? TGEMM_OK : cuda_fail("cudaMemset2DAsync(C)", err);
    }
    if ((st = check_span("A", A, a_bytes, dev->ordinal)) != TGEMM_OK) return st;
    if ((st = check_span("B", B, b_bytes, dev->ordinal)) != TGEMM_OK) return st;

    Problem p;
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    p.A = A;
    p.lda = lda;
    p.B = B;
    p.ldb = ldb;
    p.C = C;
    p.ldc = ldc;
    p.stream = stream;

    // Operands TMA cannot describe are copied into 16-byte pitched workspace;
    // the TF32 path also needs B transposed (k contiguous), made here too.
    const int64_t align_elems = 16 / es;
    const bool pack_a = !tma_ok(A, lda, es);
    const bool transpose_b = kind == Kind::TF32;
    const bool pack_b = !transpose_b && !tma_ok(B, ldb, es);
    int64_t a_ld2 = 0, b_ld2 = 0;
    uint64_t a_ws = 0, b_ws = 0;
    if (pack_a) {
        a_ld2 = (k + align_elems - 1) / align_elems * align_elems;
        a_ws = static_cast<uint64_t>(m) * a_ld2 * es;
    }
    if (transpose_b) {
        b_ld2 = (k + align_elems - 1) / align_elems * align_elems;   // B^T is n x k
        b_ws = static_cast<uint64_t>(n) * b_ld2 * es;
    } else if (pack_b) {
        b_ld2 = (n + align_elems - 1) / align_elems * align_elems;
        b_ws = static_cast<uint64_t>(k) * b_ld2 * es;
    }
    // Split tiles of the persistent kernels need room for partial sums (size
    // known from the shape).
    const bool skinny = kind == Kind::BF16 && m <= 64;
    const uint64_t c_ws = kind == Kind::F32 ? ffma_f32_workspace_bytes(p, *dev)
                          : skinny          ? 0
                                            : umma_workspace_bytes(p, *dev, kind == Kind::TF32);
    void* work = nullptr;
    cudaError_t err = cudaSuccess;
    const uint64_t b_off = (a_ws + 255) / 256 * 256;
    const uint64_t c_off = (b_off + b_ws + 255) / 256 * 256;
    if (a_ws + b_ws + c_ws > 0) {
        err = cudaMallocAsync(&work, c_off + c_ws, stream);
        if (err != cudaSuccess) {
            cudaGetLastError();
            set_error("workspace of %llu bytes: %s", (unsigned long long)(c_off + c_ws), cudaGetErrorString(err));
            return TGEMM_ERR_WORKSPACE;
        }
        uint8_t* w = static_cast<uint8_t*>(work);
        PackSpec specs[2];
        int packs = 0;
        if (pack_a) {
            specs[packs++] = PackSpec{A, lda, w, a_ld2, m, k};
            p.A = w;
            p.lda = a_ld2;
        }
        if (pack_b) {
            specs[packs++] = PackSpec{B, ldb, w + b_off, b_ld2, k, n};
            p.B = w + b_off;
            p.ldb = b_ld2;
        }
        if (packs > 0) err = launch_pack2(specs, packs, es, stream, *dev);   // both operands in one launch
        if (err == cudaSuccess && transpose_b) {
            err = launch_transpose(B, ldb, w + b_off, b_ld2, k, n, stream, *dev);
            p.B = w + b_off;
            p.ldb = b_ld2;
        }
    }
    if (err == cudaSuccess) {
        const int64_t tiles_m = (m + 127) / 128, tiles_n = (n + 127) / 128;
        if (tiles_m * tiles_n > lim) {
            set_error("problem too large: %lld output tiles", (long long)(tiles_m * tiles_n));
            st = TGEMM_ERR_INVALID_VALUE;
        } else if (kind == Kind::F32) {
            err = launch_ffma_f32(p, *dev, c_ws ? static_cast<uint8_t*>(work) + c_off : nullptr);
        } else if (skinny) {
            err = launch_umma_skinny(p, *dev);
        } else {
            err = launch_umma(p, *dev, kind == Kind::TF32, c_ws ? static_cast<uint8_t*>(work) + c_off : nullptr);
        }
    }
    if (work) {
        cudaError_t ferr = cudaFreeAsync(work, stream);
        if (err == cudaSuccess && ferr != cudaSuccess) err = ferr;
    }
    if (st != TGEMM_OK) return st;
    if (err != cudaSuccess) {
        if (t_last_error[0] == '\0') set_error("CUDA: %s", cudaGetErrorString(err));
        return TGEMM_ERR_CUDA;
    }
    return TGEMM_OK;
}

}  // namespace

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
    va_end(ap);
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void clear_error() { t_last_error[0] = '\0'; }

bool make_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem_bytes, const void* base,
                     uint64_t rows, uint64_t cols, uint64_t ld, uint32_t box_rows, uint32_t box_cols,
                     CUtensorMapSwizzle swizzle) {
    EncodeTiledFn encode = driver().encode;
    if (!encode) {
        set_error("cuTensorMapEncodeTiled unavailable");
        return false;
    }
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {ld * elem_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed (CUresult %d) for %llu x %llu, ld %llu, box %u x %u", (int)r,
                  (unsigned long long)rows, (unsigned long long)cols, (unsigned long long)ld, box_rows, box_cols);
        return false;
    }
    return true;
}

}  // namespace tgemm

extern "C" {

tgemm_status tgemm_f32(int64_t m, int64_t n, int64_t k, const float* A, int64_t lda, const float* B,
                       int64_t ldb, float* C, int64_t ldc, struct CUstream_st* stream) {
    return tgemm::run(tgemm::Kind::F32, m, n, k, A, lda, B, ldb, C, ldc, stream);
}

tgemm_status tgemm_tf32(int64_t m, int64_t n, int64_t k, const float* A, int64_t lda, const float* B,
                        int64_t ldb, float* C, int64_t ldc, struct CUstream_st* stream) {
    return tgemm::run(tgemm::Kind::TF32, m, n, k, A, lda, B, ldb, C, ldc, stream);
}

tgemm_status tgemm_bf16(int64_t m, int64_t n, int64_t k, const void* A, int64_t lda, const void* B,
                        int64_t ldb, float* C, int64_t ldc, struct CUstream_st* stream) {
    return tgemm::run(tgemm::Kind::BF16, m, n, k, A, lda, B, ldb, C, ldc, stream);
}

tgemm_status tgemm_transpose_f32(int64_t rows, int64_t cols, const float* src, int64_t ld_src, float* dst,
                                 int64_t ld_dst, struct CUstream_st* stream) {
    using namespace tgemm;
    clear_error();
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (rows < 0 || cols < 0 || rows > lim || cols > lim) {
        set_error("sizes must satisfy 0 <= rows, cols < 2^31");
        return TGEMM_ERR_INVALID_VALUE;
    }
    if (rows == 0 || cols == 0) return TGEMM_OK;
    if (ld_src < cols || ld_dst < rows || ld_src > (int64_t(1) << 40) || ld_dst > (int64_t(1) << 40)) {
        set_error("leading dimensions must satisfy ld_src >= cols and ld_dst >= rows");
        return TGEMM_ERR_INVALID_VALUE;
    }
    if (!src || !dst) {
        set_error("NULL pointer for a matrix with nonzero extent");
        return TGEMM_ERR_INVALID_VALUE;
    }
    if (reinterpret_cast<uintptr_t>(src) % 4 || reinterpret_cast<uintptr_t>(dst) % 4) {
        set_error("pointers must be aligned to 4 bytes");
        return TGEMM_ERR_INVALID_VALUE;
    }
    const uint64_t s_bytes = span_bytes(rows, cols, ld_src, 4);
    const uint64_t d_bytes = span_bytes(cols, rows, ld_dst, 4);
    if (overlaps(src, s_bytes, dst, d_bytes)) {
        set_error("dst overlaps src");
        return TGEMM_ERR_INVALID_VALUE;
    }
    Device* dev = nullptr;
    tgemm_status st = current_device(&dev);
    if (st != TGEMM_OK) return st;
    if ((st = check_span("src", src, s_bytes, dev->ordinal)) != TGEMM_OK) return st;
    if ((st = check_span("dst", dst, d_bytes, dev->ordinal)) != TGEMM_OK) return st;
    return launch_transpose(src, ld_src, dst, ld_dst, rows, cols, stream, *dev) == cudaSuccess ? TGEMM_OK
                                                                                               : TGEMM_ERR_CUDA;
}

const char* tgemm_status_string(tgemm_status status) {
    switch (status) {
        case TGEMM_OK: return "success";
        case TGEMM_ERR_INVALID_VALUE: return "invalid argument";
        case TGEMM_ERR_MISALIGNED: return "misaligned operand";
        case TGEMM_ERR_UNSUPPORTED_DEVICE: return "unsupported device (sm_103 required)";
        case TGEMM_ERR_CUDA: return "CUDA error";
        case TGEMM_ERR_TIMEOUT: return "kernel pipeline wait timed out";
        case TGEMM_ERR_WORKSPACE: return "workspace allocation failed";
        case TGEMM_ERR_INTERNAL: return "device-side consistency check failed";
    }
    return "unknown status";
}

const char* tgemm_last_error(void) { return tgemm::t_last_error; }

tgemm_status tgemm_get_device_status(struct CUstream_st* stream) {
    tgemm::t_last_error[0] = '\0';
    tgemm::Device* dev = nullptr;
    tgemm_status st = tgemm::current_device(&dev);
    if (st != TGEMM_OK) return st;
    cudaError_t err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return tgemm::cuda_fail("cudaStreamSynchronize", err);
    uint32_t value = 0;
    err = cudaMemcpyFromSymbol(&value, g_tgemm_status, sizeof value);
    if (err != cudaSuccess) return tgemm::cuda_fail("reading the status word", err);
    if (value != 0) {
        const uint32_t zero = 0;
        err = cudaMemcpyToSymbol(g_tgemm_status, &zero, sizeof zero);
        if (err != cudaSuccess) return tgemm::cuda_fail("clearing the status word", err);
        if ((value & 0xFFu) == tgemm::kStatusDebugCheck) {
            static const char* const files[] = {"?", "ffma_f32.cu", "umma.cu", "umma_skinny.cu", "transpose.cu",
                                                "selftest.cu"};
            const uint32_t file = (value >> 8) & 0xFu;
            tgemm::set_error("device check failed in %s at line %u", file < 6 ? files[file] : "?", value >> 12);
            return TGEMM_ERR_INTERNAL;
        }
        tgemm::set_error("a kernel reported status %u (pipeline wait timed out)", value);
        return TGEMM_ERR_TIMEOUT;
    }
    return TGEMM_OK;
}

uint64_t tgemm_kernel_launches(void) { return tgemm::g_launches.load(std::memory_order_relaxed); }

tgemm_status tgemm_plan(int tf32, int64_t m, int64_t n, int64_t k, int sm_count, int workspace, int* out) {
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (!out || m < 1 || n < 1 || k < 1 || m > lim || n > lim || k > lim || sm_count < 1 || sm_count > 4096)
        return TGEMM_ERR_INVALID_VALUE;
    int plan[5] = {0, 0, 0, 0, 0};
    if (tf32 || m > 64) {   // bf16 with m <= 64 takes the skinny kernel: all zero
        tgemm::Problem p;
        p.m = static_cast<int>(m);
        p.n = static_cast<int>(n);
        p.k = static_cast<int>(k);
        tgemm::Device d;
        d.sm_count = sm_count;
        tgemm::umma_plan(p, d, tf32 != 0, workspace != 0, plan);
    }
    for (int i = 0; i < 5; ++i) out[i] = plan[i];
    return TGEMM_OK;
}

tgemm_status tgemm_plan_f32(int64_t m, int64_t n, int64_t k, int sm_count, int64_t* out) {
    const int64_t lim = (int64_t(1) << 31) - 1;
    if (!out || m < 1 || n < 1 || k < 1 || m > lim || n > lim || k > lim || sm_count < 1 || sm_count > 4096)
        return TGEMM_ERR_INVALID_VALUE;
    tgemm::Problem p;
    p.m = static_cast<int>(m);
    p.n = static_cast<int>(n);
    p.k = static_cast<int>(k);
    tgemm::Device d;
    d.sm_count = sm_count;
    int64_t plan[3];
    tgemm::ffma_f32_plan(p, d, plan);
    for (int i = 0; i < 3; ++i) out[i] = plan[i];
    return TGEMM_OK;
}

int tgemm_version(void) { return 200; }

int tgemm_debug_build(void) { return tgemm::kDebugBuild ? 1 : 0; }

}  // extern "C"
