// ffma_f32.cu -- fp32 C = A * B on the FMA pipes (tgemm_f32).
//
// The tiled matrix multiply of hecess.blogspot.com "[Multi-Core & GPU
// Programming] CUDA - Matrix Multiplication" (sections "[Shared Memory]" and
// "Tiled Matrix Multiplication Kernel"), rebuilt for sm_103a:
//
//  * Output tiles.  Each CTA owns a 128 x 128 tile of C (the page's block owns
//    a TILE_WIDTH x TILE_WIDTH tile); tiles are numbered in groups of 8 tile
//    rows so that CTAs running together share A and B tiles in L2.
//  * Phases.  K is walked in phases of BK = 16.  Instead of every thread
//    copying one element and a __syncthreads, one thread issues two TMA bulk
//    tensor copies per phase into an 8-stage ring of shared-memory tiles; an
//    mbarrier per stage ("full") replaces the first __syncthreads (data has
//    landed) and a second per stage ("empty", one arrival per warp) replaces
//    the second one (nobody still reads the tile that the next copy
//    overwrites).  Out-of-range rows and columns are zero-filled by TMA.
//  * More outputs per thread (the page's remedy for unused shared memory, end
//    of "Tile Size 결정"): 256 threads each keep an 8 x 8 block of C in
//    registers (the page's Pvalue, 64 of them), so every shared-memory value
//    read feeds 8 FMAs.  Pairs of neighbouring columns are updated with
//    Blackwell's paired FMA (fma.rn.f32x2), halving the FMA instruction count.
//  * Bank conflicts (note.jhbae.stream "Lec 29 · GPU Architecture (2)": 32
//    banks of 4 bytes, N-way conflicts replay, one word read by many threads is
//    a broadcast).  A tiles (128 rows x 64 bytes) are stored with TMA's 64-byte
//    swizzle; a warp's 128-bit reads of A touch 4 rows whose 16-byte chunks
//    land in 4 distinct bank groups, and lanes reading the same row broadcast.
//    B tiles (16 rows x 512 bytes) are stored plain; 8 consecutive lanes read
//    128 consecutive bytes.  Neither pattern has a bank conflict (one pass
//    in the pages' bank model, checked on the host in the tests); measured
//    on GB300 an A read takes 2 shared-memory wavefronts and a B read 4, the
//    least a 128-bit load of that many distinct bytes takes.
//  * The tiles are addressed through a pointer derived from the shared-memory
//    array itself, so every operand read is a shared load (an address rounded
//    through an integer made them generic loads: 7 % slower).
//  * Coalescing / corner turning (section "[Coalescing]"): TMA moves whole
//    tile rows; the epilogue writes 4 rows x 128 contiguous bytes per warp
//    instruction with 128-bit stores.
//
//  * Roles.  The kernel is warp-specialised: one warp group only streams
//    tiles with TMA, two multiply, and the register file is re-split between
//    them (setmaxnreg).
//  * The last wave.  With T = q G + r tiles on G SMs (r < 0.9 G), the one-tile
//    grid runs the q G tiles of the full rounds and the r tiles left are cut
//    along k into `parts` pieces that fill whole rounds best; each piece's
//    partial sums go to a workspace slot and a reduce kernel adds a tile's
//    pieces in part order.
//
// Each C element is the sum over k, in ascending k, of fused multiply-adds
// into one fp32 register that starts at 0 (for a split tile: per piece, then
// the pieces added in order), then stored once.
#include <cstdio>

#include "device.cuh"
#include "host.h"

namespace tgemm {
namespace {

constexpr int kBN = 128;
constexpr int kBK = 16;                  // 16 (64-byte A rows, 64-byte swizzle) or 32 (128-byte, 128-byte swizzle)
constexpr int kStages = 8;               // 4 -> 8: 57.8 -> 59.0 TFLOP/s at 4096^3
constexpr int kTR = 8;                   // rows of C per consumer thread (8 or 16)
constexpr int kRowGroup = 8;             // rows of a thread processed together (4 or 8)
constexpr int kChunkUnroll = 4;          // unrolling of the 4-wide k chunks of a stage (1..4)
constexpr int kWarpsM = 4;               // consumer warps along M (two along N); 6 (192-row tiles,
                                         // 160 registers a consumer) measured 4 % slower at 4096^3
constexpr int kGroupM = 8;
constexpr uint32_t kStageB = kBK * kBN * 4;   // 8 KiB

// kWarpsM x 2 consumer warps, each warp 4 kTR rows x 64 columns: kWarpsM = 4
// and kTR = 8 give eight warps and 128 x 128 tiles.  (A 64-row form, two CTAs per
// SM, served k < 2048 until the warp-specialised 128-row kernel beat it
// there too: 4096 x 4096 x 1024 50.9 -> 55.6 TFLOP/s.)
struct FCfg {
    static constexpr int BM = 4 * kTR * kWarpsM;
    static constexpr int THREADS = 64 * kWarpsM;
    static constexpr int WARPS = THREADS / 32;
    static constexpr uint32_t STAGE_A = BM * kBK * 4;   // 8 KiB at 128 rows
    static constexpr size_t SMEM = 1024 + kStages * (STAGE_A + kStageB) + 2 * kStages * sizeof(uint64_t);
};

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int& tm, int& tn) {
    const int per_group = kGroupM * tiles_n;
    const int group = tile / per_group;
    const int first = group * kGroupM;
    const int rows = min(tiles_m - first, kGroupM);
    const int in_group = tile - group * per_group;
    tm = first + in_group % rows;
    tn = in_group / rows;
}

// Per-thread register tile: acc[i][p] holds row a_row0 + 4i and columns
// b_col0 + 2p, +1 (p < 2) or b_col0 + 32 + 2(p-2), +1 (p >= 2) of the CTA
// tile.  Pairs of columns are updated by one paired FMA (fma.rn.f32x2): each
// lane is an ordinary fused multiply-add with one rounding, exactly as fmaf.
using Acc = float2[kTR][4];

__device__ __forceinline__ void zero(Acc& acc) {
#pragma unroll
    for (int i = 0; i < kTR; ++i)
#pragma unroll
        for (int p = 0; p < 4; ++p) acc[i][p] = make_float2(0.0f, 0.0f);
}

// One k-phase (kBK terms) from a staged A tile (rows of kBK floats, swizzled)
// and B tile (kBK rows of kBN floats).  Per 4 k-values: the thread's rows in
// groups of kRowGroup, one 128-bit A read per row (4 consecutive k), two
// 128-bit B reads per k and group.
__device__ __forceinline__ void fma_phase(Acc& acc, const float* As, const float* Bs, int a_row0, int b_col0,
                                          int swz_even) {
#pragma unroll kChunkUnroll
    for (int kc = 0; kc < kBK / 4; ++kc) {
#pragma unroll
        for (int g = 0; g < kTR / kRowGroup; ++g) {
            float4 av[kRowGroup];
#pragma unroll
            for (int ii = 0; ii < kRowGroup; ++ii) {
                const int i = kRowGroup * g + ii;
                const int r = a_row0 + 4 * i;
                const int chunk = kc ^ (swz_even ^ ((i & 1) << (kBK == 16 ? 1 : 2)));
                av[ii] = *reinterpret_cast<const float4*>(As + r * kBK + chunk * 4);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float* brow = Bs + (kc * 4 + kk) * kBN + b_col0;
                const float4 b0 = *reinterpret_cast<const float4*>(brow);
                const float4 b1 = *reinterpret_cast<const float4*>(brow + 32);
                const float2 bp[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                                      make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
                for (int p = 0; p < 4; ++p) {
#pragma unroll
                    for (int ii = 0; ii < kRowGroup; ++ii) {
                        const float a = kk == 0 ? av[ii].x : kk == 1 ? av[ii].y : kk == 2 ? av[ii].z : av[ii].w;
                        acc[kRowGroup * g + ii][p] = __ffma2_rn(make_float2(a, a), bp[p], acc[kRowGroup * g + ii][p]);
                    }
                }
            }
        }
    }
}

// Writes the thread's part of the tile at (m0, n0); every element of C is
// written exactly once, rows and columns outside C are skipped.
__device__ __forceinline__ void store_tile(const Acc& acc, float* C, int64_t ldc, int M, int N, int m0, int n0,
                                           int a_row0, int b_col0, int vec_store) {
#pragma unroll
    for (int i = 0; i < kTR; ++i) {
        const int gm = m0 + a_row0 + 4 * i;
        if (gm >= M) continue;
        float* crow = C + static_cast<int64_t>(gm) * ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int gn = n0 + b_col0 + 32 * h;
            const float v[4] = {acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x, acc[i][2 * h + 1].y};
            if (vec_store && gn + 3 < N) {
                *reinterpret_cast<float4*>(crow + gn) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (gn + j < N) crow[gn + j] = v[j];
            }
        }
    }
}

// Shared-memory layout: kStages A stages, kStages B stages,
// then the full and empty mbarriers, from a 1024-byte aligned base.
struct Smem {
    float* sA;
    float* sB;
    uint64_t* full;
    uint64_t* empty;
    __device__ __forceinline__ explicit Smem(uint8_t* raw) {
        uint8_t* base = smem_align_1024(raw);
        sA = reinterpret_cast<float*>(base);
        sB = reinterpret_cast<float*>(base + kStages * FCfg::STAGE_A);
        full = reinterpret_cast<uint64_t*>(base + kStages * (FCfg::STAGE_A + kStageB));
        empty = full + kStages;
    }
};

// 128-row tiles, warp-specialised.  Warp group 0 streams the operand tiles:
// one thread issues the TMA copies of each k-phase as soon as its stage is
// free; warp groups 1-2 (8 warps, the thread layout below) multiply.  The
// register file is re-split once at the start -- the producer group keeps
// 24 registers a thread, the consumer groups take 240 -- so the consumers
// keep the 8 x 8 register tile while their loop carries no producer branch
// (measured on GB300: 4096^3 54.0 -> 57.0 TFLOP/s; with the producer in lane
// 0 of every warp in turn it fell to 51.2).  Block u computes, with
// parts == 1, tile tile0 + u and stores it in C; with parts > 1, piece
// u % parts (k-phases [KT p / parts, KT (p + 1) / parts)) of tile
// tile0 + u / parts, whose partial sums go to slot u of `ws` (float4 j of
// consumer thread t at j * 256 + t) for ffma_f32_reduce_kernel.
constexpr int kWsThreads = 128 + FCfg::THREADS;
constexpr int kProducerRegs = 24;
constexpr int kConsumerRegs = (65536 - 128 * kProducerRegs) / FCfg::THREADS / 8 * 8 > 240
                                  ? 240
                                  : (65536 - 128 * kProducerRegs) / FCfg::THREADS / 8 * 8;
static_assert(128 * kProducerRegs + FCfg::THREADS * kConsumerRegs <= 65536, "register split exceeds the file");

__global__ void __launch_bounds__(kWsThreads, 1)
ffma_f32_ws_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   float* __restrict__ C, int64_t ldc, int M, int N, int K, int vec_store, uint32_t* status,
                   int tile0, int parts, float* __restrict__ ws) {
    using F = FCfg;
    constexpr int kBM = F::BM;
    extern __shared__ uint8_t smem_raw[];
    const Smem sm(smem_raw);
#ifdef TGEMM_DEBUG
    // Debug build: how often each stage was filled (producer) and released
    // (one count per consumer warp), to check every wait's phase.
    __shared__ uint32_t dbg_fills[kStages], dbg_releases[kStages];
#endif
    const int warp_all = threadIdx.x >> 5;
    // A whole-tile grid is launched as a programmatic dependent of the kernel
    // before it (e.g. the re-pitch of a misaligned operand): every thread
    // waits here until that kernel has completed, before any global access.
    // Only then may the next launch of a split product (the pieces after the
    // whole tiles, the reduce after the pieces) start on SMs this grid frees;
    // it reads nothing this grid writes (the reduce waits for the pieces on
    // the device, the pieces for this grid at their end).
    if (parts == 1) griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    // Tile origin and k-range of this block (recomputed where needed rather
    // than held in registers through the consumers' loop).
    auto origin = [&](int& m0, int& n0) {
        int tile_m, tile_n;
        tile_coords(tile0 + (parts > 1 ? static_cast<int>(blockIdx.x) / parts : static_cast<int>(blockIdx.x)),
                    (M + kBM - 1) / kBM, (N + kBN - 1) / kBN, tile_m, tile_n);
        m0 = tile_m * kBM;
        n0 = tile_n * kBN;
    };
    auto k_range = [&](int& k0, int& NI) {
        const int KT = (K + kBK - 1) / kBK;
        const int part = parts > 1 ? static_cast<int>(blockIdx.x) % parts : 0;
        k0 = static_cast<int>(static_cast<int64_t>(KT) * part / parts);
        NI = static_cast<int>(static_cast<int64_t>(KT) * (part + 1) / parts) - k0;
    };
    if (threadIdx.x == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], F::WARPS);
#ifdef TGEMM_DEBUG
            dbg_fills[s] = 0;
            dbg_releases[s] = 0;
#endif
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp_all < 4) {
        // ---------------------------------------------------- producer --
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kProducerRegs));
        if (threadIdx.x == 0) {
            int m0, n0, k0, NI;
            origin(m0, n0);
            k_range(k0, NI);
            int issued = 0;
            for (int i = 0; i < NI; ++i) {
                const int s = i % kStages;
                if (i >= kStages && !mbar_wait(&sm.empty[s], static_cast<uint32_t>(i / kStages - 1) & 1u, status))
                    break;   // the consumers time out on the stages never filled
#ifdef TGEMM_DEBUG
                // every consumer warp has released every earlier fill of this stage
                TGEMM_DCHECK(dbg_releases[s] == static_cast<uint32_t>(i / kStages) * F::WARPS, status, kFileFfma);
                dbg_fills[s] = static_cast<uint32_t>(i / kStages) + 1;
#endif
                mbar_arrive_expect_tx(&sm.full[s], F::STAGE_A + kStageB);
                tma_load_2d(sm.sA + s * (kBM * kBK), &tmA, &sm.full[s], (k0 + i) * kBK, m0);
                tma_load_2d(sm.sB + s * (kBK * kBN), &tmB, &sm.full[s], n0, (k0 + i) * kBK);
                issued = i + 1;
            }
            // This thread keeps the CTA alive until its copies have landed
            // (consumers that timed out may have left some unwaited).
            drain_ring(sm.full, kStages, issued, status);
        }
        return;
    }

    // --------------------------------------------------------- consumers --
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(kConsumerRegs));
    const int ctid = threadIdx.x - 128;
    const int warp = ctid >> 5;
    // Thread layout: warp (wm, wn) covers rows 4 kTR wm .. + 4 kTR - 1 and
    // columns 64*wn .. +63; lane (tm, tn) takes rows tm + 4i (i < kTR) and columns
    // 4*tn .. +3 and 32 + 4*tn .. +3 of that warp tile.
    const int wm = warp >> 1, wn = warp & 1;
    const int tm = lane >> 3, tn = lane & 7;
    const int a_row0 = 4 * kTR * wm + tm;
    const int b_col0 = 64 * wn + 4 * tn;
    // 64-byte swizzle: 16-byte chunk c of tile row r sits at chunk c ^ ((r >> 1) & 3).
    // For r = a_row0 + 4i this is (tm >> 1) ^ (2 * (i & 1)).
    const int swz_even = kBK == 16 ? (tm >> 1) : tm;
    // The thread's shared-memory reads stay inside a stage: A rows a_row0 + 4i
    // (i < kTR), swizzled 16-byte chunks < kBK / 4; B columns b_col0 .. +3 and
    // b_col0 + 32 .. +35.
    if (!TGEMM_DCHECK(a_row0 + 4 * (kTR - 1) < kBM && (swz_even ^ (kBK == 16 ? 3 : 7)) < kBK / 4 &&
                          b_col0 + 32 + 3 < kBN,
                      status, kFileFfma))
        return;
    int k0, NI;
    k_range(k0, NI);
    Acc acc;
    zero(acc);
    int s = 0;
    uint32_t phase = 0;
    for (int i = 0; i < NI; ++i) {
        if (!mbar_wait(&sm.full[s], phase, status)) return;   // status records the timeout
#ifdef TGEMM_DEBUG
        // the stage holds fill i / kStages: neither an older one nor a refill
        TGEMM_DCHECK(dbg_fills[s] == static_cast<uint32_t>(i / kStages) + 1, status, kFileFfma);
#endif
        fma_phase(acc, sm.sA + s * (kBM * kBK), sm.sB + s * (kBK * kBN), a_row0, b_col0, swz_even);
        __syncwarp();
        if (lane == 0) {
#ifdef TGEMM_DEBUG
            atomicAdd(&dbg_releases[s], 1u);
#endif
            mbar_arrive(&sm.empty[s]);
        }
        if (++s == kStages) { s = 0; phase ^= 1u; }
    }
    if (parts == 1) {
        int m0, n0;
        origin(m0, n0);
        store_tile(acc, C, ldc, M, N, m0, n0, a_row0, b_col0, vec_store);
        return;
    }
    float4* dst = reinterpret_cast<float4*>(ws + static_cast<int64_t>(blockIdx.x) * kBM * kBN) + ctid;
#pragma unroll
    for (int i = 0; i < kTR; ++i)
#pragma unroll
        for (int p = 0; p < 4; p += 2)
            dst[(i * 2 + p / 2) * F::THREADS] = make_float4(acc[i][p].x, acc[i][p].y, acc[i][p + 1].x, acc[i][p + 1].y);
    // Launched as a dependent of the whole-tile grid, the pieces may finish
    // first; waiting for that grid here makes this grid's completion (which
    // the reduce waits for) imply that every tile of C has been written.
    griddep_wait();
}

// C of the remainder tiles: tile tile0 + b is the sum of the pieces in
// slots b * parts .. b * parts + parts - 1, added in part order.  Four blocks
// share a tile, one per 32-row quarter (the rows of the piece kernel's
// consumer warps wm = q): reduce thread t takes consumer thread
// 64 q + (t % 64)'s float4 slots j = 4 (t / 64) .. +3 (rows a_row0 + 4 (j / 2),
// columns b_col0 + 32 (j % 2) .. +3), so consecutive threads read consecutive
// float4s of the workspace and store neighbouring 16-byte pieces of C.
constexpr int kReduceSplit = 4;

__global__ void __launch_bounds__(FCfg::THREADS)
ffma_f32_reduce_kernel(const float* __restrict__ ws, float* __restrict__ C, int64_t ldc, int M, int N, int tile0,
                       int parts, int vec_store) {
    using F = FCfg;
    constexpr int kBM = F::BM;
    constexpr int kSlots = kTR * 2;                         // float4 slots per consumer thread
    constexpr int kPer = kSlots * 64 / F::THREADS;          // slots per reduce thread (4)
    const int tile = static_cast<int>(blockIdx.x) / kReduceSplit;
    const int q = static_cast<int>(blockIdx.x) % kReduceSplit;
    const int src = 64 * q + (threadIdx.x & 63);             // consumer thread whose slots this thread adds
    const int j0 = (threadIdx.x >> 6) * kPer;
    const int warp = src >> 5, lane = src & 31;
    const int wm = warp >> 1, wn = warp & 1;
    const int tm = lane >> 3, tn = lane & 7;
    const int a_row0 = 4 * kTR * wm + tm;
    const int b_col0 = 64 * wn + 4 * tn;
    int tile_m, tile_n;
    tile_coords(tile0 + tile, (M + kBM - 1) / kBM, (N + kBN - 1) / kBN, tile_m, tile_n);
    griddep_wait();   // the pieces have been written (launched as their dependent)
    float4 acc[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) acc[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    const float4* slot = reinterpret_cast<const float4*>(ws + static_cast<int64_t>(tile) * parts * kBM * kBN) + src;
    for (int p = 0; p < parts; ++p) {
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const float4 v = __ldcs(slot + (j0 + j) * F::THREADS);
            acc[j].x += v.x;
            acc[j].y += v.y;
            acc[j].z += v.z;
            acc[j].w += v.w;
        }
        slot += kBM * kBN / 4;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int gm = tile_m * kBM + a_row0 + 4 * ((j0 + j) >> 1);
        const int gn = tile_n * kBN + b_col0 + 32 * ((j0 + j) & 1);
        if (gm >= M) continue;
        float* crow = C + static_cast<int64_t>(gm) * ldc;
        if (vec_store && gn + 3 < N) {
            *reinterpret_cast<float4*>(crow + gn) = acc[j];
        } else {
            const float v[4] = {acc[j].x, acc[j].y, acc[j].z, acc[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (gn + e < N) crow[gn + e] = v[e];
        }
    }
}

// The warp-specialised 128-row kernel over `grid` blocks (see its comment).
// Launch configuration on p.stream; with `dependent`, as a programmatic
// dependent of the kernel before it (it may start while that one finishes).
cudaLaunchConfig_t launch_config(const Problem& p, unsigned grid, unsigned threads, size_t smem, bool dependent,
                                 cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = p.stream;
    if (dependent) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cfg;
}

cudaError_t launch_ws(const Problem& p, const CUtensorMap& ta, const CUtensorMap& tb, int64_t grid, int64_t tile0,
                      int parts, float* ws, int vec_store, const Device& dev, bool dependent) {
    cudaError_t err = cudaFuncSetAttribute(ffma_f32_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(FCfg::SMEM));
    if (err != cudaSuccess) {
        set_error("cudaFuncSetAttribute(ffma_f32_ws_kernel): %s", cudaGetErrorString(err));
        return err;
    }
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg =
        launch_config(p, static_cast<unsigned>(grid), kWsThreads, FCfg::SMEM, dependent, attr);
    err = cudaLaunchKernelEx(&cfg, ffma_f32_ws_kernel, ta, tb, p.C, p.ldc, p.m, p.n, p.k, vec_store, dev.status,
                             static_cast<int>(tile0), parts, ws);
    count_launch();
    return err;
}

bool make_maps(const Problem& p, CUtensorMap* ta, CUtensorMap* tb) {
    using F = FCfg;
    return make_tensor_map(ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.A, p.m, p.k, p.lda, F::BM, kBK,
                           kBK == 16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_tensor_map(tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.B, p.k, p.n, p.ldb, kBK, kBN,
                           CU_TENSOR_MAP_SWIZZLE_NONE);
}

int vec_store_ok(const Problem& p) { return (reinterpret_cast<uintptr_t>(p.C) % 16 == 0) && (p.ldc % 4 == 0); }

// Split remainder: the kernel runs the tiles of the full rounds (152 a round
// on GB300); the r tiles left (r < 0.9 G) are cut along k into `parts`
// pieces, chosen so that r * parts pieces fill whole rounds best (each round
// of pieces takes 1/parts of a tile's time); a reduce kernel adds the pieces.
// 4096^3: 1024 = 6 x 152 + 112 tiles; 112 x 4 quarters = 2.95 rounds of
// quarter tiles instead of one round of whole tiles.
struct SplitTail {
    int64_t full;   // tiles of the full rounds
    int64_t rest;   // remainder tiles
    int parts;
};

bool split_tail(const Problem& p, const Device& dev, SplitTail* st) {
    using F = FCfg;
    const int64_t G = dev.sm_count;
    const int64_t tiles = static_cast<int64_t>((p.m + F::BM - 1) / F::BM) * ((p.n + kBN - 1) / kBN);
    const int64_t KT = (p.k + kBK - 1) / kBK;
    const int64_t r = tiles % G;
    if (r == 0 || 10 * r >= 9 * G) return false;
    double best = 0.95;   // a round of whole tiles costs 1; require a 5 % gain
    int parts = 1;
    for (int s = 2; s <= 8 && KT / s >= 2 * kStages; ++s) {
        const double t = static_cast<double>((r * s + G - 1) / G) / s;
        if (t < best) {
            best = t;
            parts = s;
        }
    }
    if (parts == 1) return false;
    *st = SplitTail{tiles - r, r, parts};
    return true;
}

cudaError_t launch_tiles(const Problem& p, const Device& dev) {
    using F = FCfg;
    CUtensorMap ta, tb;
    if (!make_maps(p, &ta, &tb)) return cudaErrorInvalidValue;
    const int64_t tiles = static_cast<int64_t>((p.m + F::BM - 1) / F::BM) * ((p.n + kBN - 1) / kBN);
    cudaError_t err = launch_ws(p, ta, tb, tiles, 0, 1, nullptr, vec_store_ok(p), dev, true);
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) set_error("ffma_f32_ws_kernel launch: %s", cudaGetErrorString(err));
    return err;
}

cudaError_t launch_split_tail(const Problem& p, const Device& dev, void* workspace, const SplitTail& st) {
    using F = FCfg;
    if (!workspace) {
        set_error("ffma_f32: split remainder launched without its workspace");
        return cudaErrorInvalidValue;
    }
    CUtensorMap ta, tb;
    if (!make_maps(p, &ta, &tb)) return cudaErrorInvalidValue;
    const int vec_store = vec_store_ok(p);
    float* ws = static_cast<float*>(workspace);
    cudaError_t err = cudaSuccess;
    // Whole tiles first (a dependent launch whose CTAs wait for the kernel
    // before them), then the pieces of the remainder, which read only A and B
    // and so start as soon as the whole-tile grid frees SMs, then the reduce,
    // which waits on the device for the pieces.
    if (st.full > 0) err = launch_ws(p, ta, tb, st.full, 0, 1, nullptr, vec_store, dev, true);
    if (err == cudaSuccess)
        err = launch_ws(p, ta, tb, st.rest * st.parts, st.full, st.parts, ws, vec_store, dev, st.full > 0);
    if (err != cudaSuccess) {
        set_error("ffma_f32_ws_kernel launch: %s", cudaGetErrorString(err));
        return err;
    }
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg =
        launch_config(p, static_cast<unsigned>(st.rest * kReduceSplit), F::THREADS, 0, true, attr);
    err = cudaLaunchKernelEx(&cfg, ffma_f32_reduce_kernel, static_cast<const float*>(ws), p.C, p.ldc, p.m, p.n,
                             static_cast<int>(st.full), st.parts, vec_store);
    count_launch();
    if (err == cudaSuccess) err = cudaGetLastError();
    if (err != cudaSuccess) set_error("ffma_f32 split launches: %s", cudaGetErrorString(err));
    return err;
}

}  // namespace

uint64_t ffma_f32_workspace_bytes(const Problem& p, const Device& dev) {
    SplitTail st;
    if (!split_tail(p, dev, &st)) return 0;
    return static_cast<uint64_t>(st.rest) * st.parts * FCfg::BM * kBN * sizeof(float);
}

void ffma_f32_plan(const Problem& p, const Device& dev, int64_t out[3]) {
    SplitTail st;
    if (split_tail(p, dev, &st)) {
        out[0] = st.full;
        out[1] = st.rest;
        out[2] = st.parts;
        return;
    }
    out[0] = static_cast<int64_t>((p.m + FCfg::BM - 1) / FCfg::BM) * ((p.n + kBN - 1) / kBN);
    out[1] = out[2] = 0;
}

cudaError_t launch_ffma_f32(const Problem& p, const Device& dev, void* workspace) {
    SplitTail st;
    return split_tail(p, dev, &st) ? launch_split_tail(p, dev, workspace, st) : launch_tiles(p, dev);
}

}  // namespace tgemm
