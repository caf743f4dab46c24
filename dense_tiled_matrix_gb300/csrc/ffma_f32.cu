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
//    tensor copies per phase into a 4-stage ring of shared-memory tiles; an
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
//    128 consecutive bytes.  Both patterns take one shared-memory wavefront
//    per instruction (checked by the host-side bank model in the tests).
//  * Coalescing / corner turning (section "[Coalescing]"): TMA moves whole
//    tile rows; the epilogue writes 4 rows x 128 contiguous bytes per warp
//    instruction with 128-bit stores.
//
// Each C element is the sum over k, in ascending k, of fused multiply-adds
// into one fp32 register that starts at 0, then stored once.
#include <cstdio>

#include "device.cuh"
#include "host.h"

namespace tgemm {
namespace {

constexpr int kBN = 128;
constexpr int kBK = 16;                  // 16 (64-byte A rows, 64-byte swizzle) or 32 (128-byte, 128-byte swizzle)
constexpr int kStages = 4;
constexpr int kRowGroup = 4;             // rows of a thread processed together (4 or 8)
constexpr int kChunkUnroll = 4;          // unrolling of the 4-wide k chunks of a stage (1..4)
constexpr int kGroupM = 8;
constexpr uint32_t kStageB = kBK * kBN * 4;   // 8 KiB

// WR warps stacked along M (each warp 32 rows x 64 columns, two warps across
// N): WR = 4 gives 128 x 128 tiles and one 256-thread CTA per SM; WR = 2 gives
// 64 x 128 tiles and two 128-thread CTAs per SM, whose barrier and prologue
// waits overlap each other (better when k is short).
template <int WR>
struct FCfg {
    static constexpr int BM = 32 * WR;
    static constexpr int THREADS = 64 * WR;
    static constexpr int WARPS = THREADS / 32;
    static constexpr int MIN_BLOCKS = WR == 2 ? 2 : 1;
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

template <int WR>
__global__ void __launch_bounds__(FCfg<WR>::THREADS, FCfg<WR>::MIN_BLOCKS)
ffma_f32_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                float* __restrict__ C, int64_t ldc, int M, int N, int K, int vec_store,
                uint32_t* status) {
    using F = FCfg<WR>;
    constexpr int kBM = F::BM;
    constexpr int kWarps = F::WARPS;
    constexpr uint32_t kStageA = F::STAGE_A;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    float* sA = reinterpret_cast<float*>(smem);
    float* sB = reinterpret_cast<float*>(smem + kStages * kStageA);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * (kStageA + kStageB));
    uint64_t* empty = full + kStages;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int tiles_m = (M + kBM - 1) / kBM;
    const int tiles_n = (N + kBN - 1) / kBN;
    int tile_m, tile_n;
    tile_coords(blockIdx.x, tiles_m, tiles_n, tile_m, tile_n);
    const int m0 = tile_m * kBM;
    const int n0 = tile_n * kBN;
    const int KT = (K + kBK - 1) / kBK;

    if (tid == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (tid == 0) {
        const int first = KT < kStages ? KT : kStages;
        for (int s = 0; s < first; ++s) {
            mbar_arrive_expect_tx(&full[s], kStageA + kStageB);
            tma_load_2d(sA + s * (kBM * kBK), &tmA, &full[s], s * kBK, m0);
            tma_load_2d(sB + s * (kBK * kBN), &tmB, &full[s], n0, s * kBK);
        }
    }

    // Thread layout: warp (wm, wn) covers rows 32*wm .. +31 and columns
    // 64*wn .. +63; lane (tm, tn) takes rows tm + 4i (i < 8) and columns
    // 4*tn .. +3 and 32 + 4*tn .. +3 of that warp tile.
    const int wm = warp >> 1, wn = warp & 1;
    const int tm = lane >> 3, tn = lane & 7;
    const int a_row0 = 32 * wm + tm;
    const int b_col0 = 64 * wn + 4 * tn;
    // 64-byte swizzle: 16-byte chunk c of tile row r sits at chunk c ^ ((r >> 1) & 3).
    // For r = a_row0 + 4i this is (tm >> 1) ^ (2 * (i & 1)).
    // 128-byte swizzle (kBK = 32): chunk c of tile row r sits at c ^ (r & 7),
    // which for r = a_row0 + 4i is tm ^ (4 * (i & 1)).
    const int swz_even = kBK == 16 ? (tm >> 1) : tm;

    // acc[i][p]: row a_row0 + 4i, columns b_col0 + 2p, +1 (p < 2) and
    // b_col0 + 32 + 2(p-2), +1 (p >= 2).  Pairs of columns are updated by one
    // paired FMA (fma.rn.f32x2): each lane is an ordinary fused multiply-add
    // with one rounding, exactly as fmaf.
    float2 acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int p = 0; p < 4; ++p) acc[i][p] = make_float2(0.0f, 0.0f);

    bool ok = true;
    int s = 0;
    uint32_t phase = 0;
    for (int kt = 0; kt < KT; ++kt) {
        // Refill the stage drained in the previous phase with phase kt-1+kStages.
        if (tid == 0 && kt > 0) {
            const int next = kt - 1 + kStages;
            if (next < KT) {
                const int ps = (kt - 1) % kStages;
                const uint32_t pph = static_cast<uint32_t>((kt - 1) / kStages) & 1u;
                if (!mbar_wait(&empty[ps], pph, status)) { ok = false; break; }
                mbar_arrive_expect_tx(&full[ps], kStageA + kStageB);
                tma_load_2d(sA + ps * (kBM * kBK), &tmA, &full[ps], next * kBK, m0);
                tma_load_2d(sB + ps * (kBK * kBN), &tmB, &full[ps], n0, next * kBK);
            }
        }
        if (!mbar_wait(&full[s], phase, status)) { ok = false; break; }

        const float* As = sA + s * (kBM * kBK);
        const float* Bs = sB + s * (kBK * kBN);
        // Per 4 k-values: the thread's rows in groups of kRowGroup, one 128-bit A
        // read per row (4 consecutive k), two 128-bit B reads per k and group.
#pragma unroll kChunkUnroll
        for (int kc = 0; kc < kBK / 4; ++kc) {
#pragma unroll
            for (int g = 0; g < 8 / kRowGroup; ++g) {
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
                    for (int ii = 0; ii < kRowGroup; ++ii) {
                        const float a = kk == 0 ? av[ii].x : kk == 1 ? av[ii].y : kk == 2 ? av[ii].z : av[ii].w;
                        const float2 aa = make_float2(a, a);
#pragma unroll
                        for (int p = 0; p < 4; ++p)
                            acc[kRowGroup * g + ii][p] = __ffma2_rn(aa, bp[p], acc[kRowGroup * g + ii][p]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == kStages) { s = 0; phase ^= 1u; }
    }
    if (!ok) return;   // status already records the timeout; C is left unwritten

    // Epilogue: every element written exactly once.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
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

template <int WR>
cudaError_t launch_wr(const Problem& p, const Device& dev) {
    using F = FCfg<WR>;
    CUtensorMap ta, tb;
    if (!make_tensor_map(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.A, p.m, p.k, p.lda, F::BM, kBK,
                         kBK == 16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.B, p.k, p.n, p.ldb, kBK, kBN,
                         CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    auto kernel = ffma_f32_kernel<WR>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(F::SMEM));
    if (err != cudaSuccess) {
        set_error("cudaFuncSetAttribute(ffma_f32_kernel): %s", cudaGetErrorString(err));
        return err;
    }
    const int64_t tiles = static_cast<int64_t>((p.m + F::BM - 1) / F::BM) * ((p.n + kBN - 1) / kBN);
    const int vec_store = (reinterpret_cast<uintptr_t>(p.C) % 16 == 0) && (p.ldc % 4 == 0);
    kernel<<<static_cast<unsigned>(tiles), F::THREADS, F::SMEM, p.stream>>>(ta, tb, p.C, p.ldc, p.m, p.n, p.k,
                                                                            vec_store, dev.status);
    count_launch();
    err = cudaGetLastError();
    if (err != cudaSuccess) set_error("ffma_f32_kernel launch: %s", cudaGetErrorString(err));
    return err;
}

// Measured on GB300: 4096^3 53.2 TFLOP/s with 128-row CTAs vs 52.6 with two
// 64-row CTAs per SM; 4097 x 3001 x 1024 42.8 vs 46.3.
constexpr int kShortK = 2048;

}  // namespace

cudaError_t launch_ffma_f32(const Problem& p, const Device& dev) {
    return p.k < kShortK ? launch_wr<2>(p, dev) : launch_wr<4>(p, dev);
}

}  // namespace tgemm
