// probes.cu -- calibration kernels (include/tgemm_probes.h).
//
// Two ways to stream a buffer from HBM into the SMs, each reading every byte
// once and adding every 32-bit word into a 64-bit checksum (integer addition,
// so the result does not depend on the order): bulk copies by the TMA unit
// into a shared-memory ring, as the skinny product streams B, and 128-bit
// loads from many threads.  Timed by the caller, they give the two read-stream
// ceilings the skinny product's bandwidth is compared with.  A third kernel
// runs the FFMA product's register-tile update with no memory operands: the
// paired-FMA rate its consumer loop is compared with.
#include <cuda_runtime.h>

#include <cstdint>

#include "device.cuh"
#include "tgemm_probes.h"

namespace {

constexpr int kChunk = 32768;        // bytes per bulk copy / ring stage
constexpr int kStages = 3;           // 96 KiB of ring: two CTAs per SM
constexpr int kThreads = 256;
constexpr size_t kTmaSmem = kStages * kChunk + kStages * 8 + 16;

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(tgemm::smem_addr(dst)), "l"(src), "r"(bytes), "r"(tgemm::smem_addr(bar)) : "memory");
}

// Bounded wait for phase `parity` of `bar` (2 s); false if it ran out.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const uint32_t a = tgemm::smem_addr(bar);
    const uint64_t start = tgemm::global_timer_ns();
    while (!tgemm::mbar_try_wait(a, parity))
        if (tgemm::global_timer_ns() - start > limit_ns) return false;
    return true;
}

__device__ __forceinline__ uint64_t add_words(uint4 v) {
    return static_cast<uint64_t>(v.x) + v.y + v.z + v.w;
}

// The block's total of `acc` added to *sum.
__device__ __forceinline__ void block_sum(uint64_t acc, unsigned long long* sum) {
    __shared__ uint64_t warp_sums[kThreads / 32];
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_down_sync(0xFFFFFFFFu, acc, o);
    if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint64_t t = 0;
        for (int w = 0; w < kThreads / 32; ++w) t += warp_sums[w];
        atomicAdd(sum, static_cast<unsigned long long>(t));
    }
}

// CTA b streams chunks [C b / G, C (b+1) / G) of the buffer through the ring.
__global__ void __launch_bounds__(kThreads, 2)
probe_tma_kernel(const uint8_t* __restrict__ buf, int64_t bytes, unsigned long long* sum) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kChunk);
    __shared__ int s_ok;
    const int64_t chunks = (bytes + kChunk - 1) / kChunk;
    const int64_t c0 = chunks * blockIdx.x / gridDim.x, c1 = chunks * (blockIdx.x + 1) / gridDim.x;
    const int n = static_cast<int>(c1 - c0);
    auto chunk_bytes = [&](int i) {
        const int64_t left = bytes - (c0 + i) * kChunk;
        return static_cast<uint32_t>(left < kChunk ? left : kChunk);
    };
    auto issue = [&](int i) {
        const int s = i % kStages;
        tgemm::mbar_arrive_expect_tx(&full[s], chunk_bytes(i));
        bulk_load(ring + s * kChunk, buf + (c0 + i) * kChunk, chunk_bytes(i), &full[s]);
    };
    int issued = 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) tgemm::mbar_init(&full[s], 1);
        tgemm::fence_barrier_init();
        for (; issued < n && issued < kStages; ++issued) issue(issued);
    }
    __syncthreads();
    uint64_t acc = 0;
    int i = 0;
    for (; i < n; ++i) {
        const int s = i % kStages;
        if (threadIdx.x == 0) s_ok = wait_phase(&full[s], static_cast<uint32_t>(i / kStages) & 1u, 2000000000ull);
        __syncthreads();
        if (!s_ok) break;   // the checksum comes out wrong; the caller sees it
        const uint32_t size = chunk_bytes(i);
        const uint8_t* stage = ring + s * kChunk;
        for (uint32_t off = threadIdx.x * 16; off < size; off += kThreads * 16)
            acc += add_words(*reinterpret_cast<const uint4*>(stage + off));
        __syncthreads();   // the stage is consumed: refill it
        if (threadIdx.x == 0 && issued < n) issue(issued++);
    }
    if (threadIdx.x == 0) {
        // no copy outlives the CTA: wait (bounded) for the ones still landing
        for (int j = i; j < issued; ++j)
            wait_phase(&full[j % kStages], static_cast<uint32_t>(j / kStages) & 1u, 200000000ull);
    }
    block_sum(acc, sum);
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Grid-strided 128-bit loads, four in flight per thread.
__global__ void __launch_bounds__(kThreads)
probe_ldg_kernel(const uint4* __restrict__ buf, int64_t nvec, unsigned long long* sum) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    uint64_t acc = 0;
    for (; i + 3 * stride < nvec; i += 4 * stride) {
        const uint4 a = ld_stream(buf + i), b = ld_stream(buf + i + stride);
        const uint4 c = ld_stream(buf + i + 2 * stride), d = ld_stream(buf + i + 3 * stride);
        acc += add_words(a) + add_words(b) + add_words(c) + add_words(d);
    }
    for (; i < nvec; i += stride) acc += add_words(ld_stream(buf + i));
    block_sum(acc, sum);
}

// Paired-FMA throughput: each thread keeps the FFMA product kernel's 8 x 8
// register tile (32 accumulator pairs) and updates it from registers only, 32
// fma.rn.f32x2 per step, `iters` steps; then adds its 64 accumulators, in
// double, into *out.  The operands are read from memory, so the compiler can
// neither fold nor merge the chains.
constexpr int kFfmaMaxWarps = 16;
__global__ void __launch_bounds__(kFfmaMaxWarps * 32, 1)
probe_ffma2_kernel(const float* __restrict__ ab, int64_t iters, double* out) {
    float a[8];
    float2 b[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = ab[i];
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = make_float2(ab[8 + 2 * j], ab[9 + 2 * j]);
    float2 acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.0f, 0.0f);
#pragma unroll 4
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i][j] = __ffma2_rn(make_float2(a[i], a[i]), b[j], acc[i][j]);
    }
    double s = 0.0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) s += static_cast<double>(acc[i][j].x) + static_cast<double>(acc[i][j].y);
    for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xFFFFFFFFu, s, o);
    if ((threadIdx.x & 31) == 0) atomicAdd(out, s);
}

int check(const void* buf, int64_t bytes, const uint64_t* sum, int* sms) {
    if (bytes < 0 || bytes % 16 != 0 || bytes >= (int64_t(1) << 40)) return 1;
    if (bytes > 0 && (!buf || reinterpret_cast<uintptr_t>(buf) % 16 != 0)) return 1;
    if (!sum || reinterpret_cast<uintptr_t>(sum) % 8 != 0) return 1;
    if (bytes == 0) return 0;   // nothing to read: no CUDA call at all
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 4;
    if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 4;
    return 0;
}

}  // namespace

extern "C" int tgemm_probe_read_tma(const void* buf, int64_t bytes, uint64_t* sum, struct CUstream_st* stream) {
    int sms = 0;
    const int rc = check(buf, bytes, sum, &sms);
    if (rc != 0 || bytes == 0) return rc;
    if (cudaFuncSetAttribute(probe_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kTmaSmem)) != cudaSuccess)
        return 4;
    const int64_t chunks = (bytes + kChunk - 1) / kChunk;
    const int64_t grid = chunks < 2 * sms ? chunks : 2 * sms;
    probe_tma_kernel<<<static_cast<unsigned>(grid), kThreads, kTmaSmem, stream>>>(
        static_cast<const uint8_t*>(buf), bytes, reinterpret_cast<unsigned long long*>(sum));
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

extern "C" int tgemm_probe_read_ldg(const void* buf, int64_t bytes, uint64_t* sum, struct CUstream_st* stream) {
    int sms = 0;
    const int rc = check(buf, bytes, sum, &sms);
    if (rc != 0 || bytes == 0) return rc;
    const int64_t nvec = bytes / 16;
    const int64_t want = (nvec + kThreads - 1) / kThreads;
    const int64_t grid = want < 4 * sms ? want : 4 * sms;
    probe_ldg_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(
        static_cast<const uint4*>(buf), nvec, reinterpret_cast<unsigned long long*>(sum));
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

extern "C" int tgemm_probe_ffma2(int warps_per_sm, int64_t iters, const float* ab, double* out,
                                 struct CUstream_st* stream) {
    if (warps_per_sm < 1 || warps_per_sm > kFfmaMaxWarps || iters < 0 || iters >= (int64_t(1) << 40)) return 1;
    if (!ab || reinterpret_cast<uintptr_t>(ab) % 4 != 0 || !out || reinterpret_cast<uintptr_t>(out) % 8 != 0)
        return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 4;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 4;
    probe_ffma2_kernel<<<static_cast<unsigned>(sms), static_cast<unsigned>(warps_per_sm * 32), 0, stream>>>(
        ab, iters, out);
    return cudaGetLastError() == cudaSuccess ? 0 : 4;
}
