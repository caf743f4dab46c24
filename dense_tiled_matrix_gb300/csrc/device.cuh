// device.cuh -- inline-PTX building blocks shared by the libtgemm kernels
// (sm_103a): shared-memory addresses, mbarriers with bounded waits, TMA tile
// loads, and the tcgen05 tensor-core / tensor-memory instructions.
//
// Every wait on an mbarrier is bounded by a wall-clock limit read from
// %globaltimer.  When the limit passes, the waiting thread records a status
// code in the kernel's status word and returns false; the kernel then leaves
// its main loop, so a lost arrival ends the launch with an error instead of
// hanging the GPU.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace tgemm {

// Wall-clock limit of one pipeline wait.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

// Status word values written by kernels (host side maps them to tgemm_status).
// The low byte is the code; a failed debug check also records where it sits
// (file id in bits 8-11, source line from bit 12).
constexpr uint32_t kStatusTimeout = 5u;
constexpr uint32_t kStatusDebugCheck = 7u;

// File ids of the debug checks.
constexpr uint32_t kFileFfma = 1, kFileUmma = 2, kFileSkinny = 3, kFileTranspose = 4, kFileSelftest = 5;

// Records a failed consistency check in the status word (the first failure
// is kept).  Used by the checks of debug builds and by the self-test.
__device__ __forceinline__ void debug_fail(uint32_t* status, uint32_t file, uint32_t line) {
    atomicCAS(status, 0u, kStatusDebugCheck | (file << 8) | (line << 12));
}

// Device-side consistency checks of the debug build (-DTGEMM_DEBUG): the
// condition is evaluated, a failure is recorded with its file and line, and
// the caller skips the access the check guards.  In normal builds the checks
// compile to nothing and always pass.
#ifdef TGEMM_DEBUG
#define TGEMM_DCHECK(cond, status, file) \
    ((cond) ? true : (::tgemm::debug_fail((status), (file), static_cast<uint32_t>(__LINE__)), false))
constexpr bool kDebugBuild = true;
#else
#define TGEMM_DCHECK(cond, status, file) true
constexpr bool kDebugBuild = false;
#endif

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    return done != 0;
}

// Waits until the phase with the given parity of `bar` has completed.
// Returns false (after recording kStatusTimeout) if that takes longer than
// `limit_ns` (kWaitLimitNs unless given).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t start = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(a, parity)) return true;
        if (global_timer_ns() - start > limit_ns) {
            atomicCAS(status, 0u, kStatusTimeout);
            return false;
        }
    }
}

// A CTA must not exit while a bulk copy it issued may still write its shared
// memory or signal its barriers.  On the normal path every copy has been
// waited for by the time a producer gets here; after a timeout some may not
// have been.  `issued` copies (or groups of copies) went out in ring order --
// number i into stage i mod `stages`, completing phase i / stages of full[s]
// -- and this waits, each wait bounded by `limit_ns`, for the last phase
// armed on every stage.
constexpr uint64_t kDrainLimitNs = 200000000ull;   // 200 ms per stage
__device__ __forceinline__ void drain_ring(uint64_t* full, int stages, int issued, uint32_t* status) {
#pragma unroll 1
    for (int s = 0; s < stages && s < issued; ++s) {
        const int fills = issued / stages + (s < issued % stages ? 1 : 0);
        mbar_wait(&full[s], static_cast<uint32_t>(fills - 1) & 1u, status, kDrainLimitNs);
    }
}

// Rounds a dynamic shared-memory pointer up to a 1024-byte boundary (the
// alignment of 128-byte-swizzled TMA tiles) by pointer arithmetic on the
// pointer itself.  Rounding through an integer cast hides from the compiler
// that the result still points into shared memory, and every access through
// it becomes a generic load or store (measured on GB300: the FFMA kernel's
// shared-memory operand reads, 59.1 -> 63.5 TFLOP/s at 4096^3 once they were
// shared loads again).
__device__ __forceinline__ uint8_t* smem_align_1024(uint8_t* raw) {
    return raw + ((1024u - static_cast<uint32_t>(reinterpret_cast<uintptr_t>(raw) & 1023u)) & 1023u);
}

// --------------------------------------------------------------------- TMA --

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled bulk copy global -> shared; completion is signalled on `bar` as
// transaction bytes.  c0 is the innermost (contiguous) coordinate.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)),
           "r"(c0), "r"(c1)
        : "memory");
}

// The same copy delivered to every CTA of the cluster whose bit is set in
// `mask`: the box lands at the same shared-memory offset in each of them and
// completes transaction bytes on the barrier at `bar`'s offset in each.
__device__ __forceinline__ void tma_load_2d_multicast(void* dst, const CUtensorMap* map, uint64_t* bar,
                                                      int32_t c0, int32_t c1, uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%3, %4}], [%2], %5;"
        :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)),
           "r"(c0), "r"(c1), "h"(mask)
        : "memory");
}

// 2-D tiled bulk copy shared -> global of the box at (c0, c1), added to the
// thread's current bulk group.  Rows and columns outside the tensor are not
// written.  c0 and c1 must not be negative.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t c0, int32_t c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(src)), "r"(c0), "r"(c1)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until at most N of the thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory");
}

// Waits until at most N of the thread's bulk groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" :: "n"(N) : "memory");
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialisation may start while the kernel before it in the stream is still
// running; griddep_wait() returns once that kernel has completed and its
// memory operations are visible, so everything before it must not touch
// global memory the previous kernel writes.  griddep_launch_dependents()
// lets the next such kernel be launched before this one finishes.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Orders this thread's ordinary shared-memory accesses before later accesses
// by the async proxy (TMA) and vice versa.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- tcgen05 --

// Allocates `ncols` tensor-memory columns (power of two, 32..512); the base
// address is written to shared memory at `dst`.  Whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_addr(dst)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], one instruction of the shape and kinds
// encoded in `idesc`.  kind::f16 covers bf16 inputs.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void umma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_addr(bar)) : "memory");
}

// As umma_commit, arriving on the barrier at `bar`'s offset in every CTA of
// the cluster whose bit is set in `mask`.
__device__ __forceinline__ void umma_commit_multicast(uint64_t* bar, uint16_t mask) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                 :: "r"(smem_addr(bar)), "h"(mask) : "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_load_32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_load_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of tcgen05 (sm_100 family): start address,
// leading- and stride-dimension byte offsets (all >> 4), the fixed version
// field 0b001 at bits 46-48, base offset 0, and the swizzle mode at bits 61-63
// (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle_mode) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= static_cast<uint64_t>(swizzle_mode & 7u) << 61;
    return d;
}

// Instruction descriptor for kind::f16 / kind::tf32 with fp32 accumulation:
// D format F32 (bits 4-5 = 1), A and B formats (bits 7-9, 10-12), major-ness
// of A and B (bits 15, 16: 0 = K-major, 1 = MN-major), N >> 3 (bits 17-22),
// M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t instr_desc(uint32_t ab_format, uint32_t a_mn_major,
                                                  uint32_t b_mn_major, uint32_t mma_m, uint32_t mma_n) {
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | (a_mn_major << 15) |
           (b_mn_major << 16) | ((mma_n >> 3) << 17) | ((mma_m >> 4) << 24);
}

constexpr uint32_t kFormatBF16 = 1u;   // under kind::f16
constexpr uint32_t kFormatTF32 = 2u;   // under kind::tf32
constexpr uint32_t kSwizzle128B = 2u;

}  // namespace tgemm

namespace tgemm {

// ---------------------------------------------------- thread-block clusters --

__device__ __forceinline__ uint32_t cluster_cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Shared-memory address of the same variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t local_saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t cluster_saddr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_saddr) : "memory");
    return v;
}

// Every thread of every CTA of the cluster must call this (it is the
// cluster-wide counterpart of __syncthreads, with release/acquire ordering of
// shared-memory writes).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_load_16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

}  // namespace tgemm
