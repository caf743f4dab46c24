// umma.cu -- C = A * B on the tcgen05 tensor cores (tgemm_tf32, tgemm_bf16).
//
// The tiled matrix multiply of hecess.blogspot.com "[Multi-Core & GPU
// Programming] CUDA - Matrix Multiplication" ("[Shared Memory]", "Tiled Matrix
// Multiplication Kernel"), with the per-thread register accumulator (the
// page's Pvalue) moved into tensor memory and the per-phase inner product done
// by tcgen05.mma:
//
//  * Output tiles of 256 x 256 (k >= 3072: two 128-row MMAs share each B tile,
//    one accumulator spanning all 512 tensor-memory columns, 3 stages) or
//    128 x 256 (two accumulators, 4 stages), visited by a persistent grid of
//    one CTA per SM in groups of tile rows (neighbouring CTAs share A and B
//    tiles in L2).
//  * Phases of 128 bytes of K (64 bf16 or 32 fp32 elements).  Warp 0 streams
//    the A tile (128 x BK, K-major) and the B tile into a 4-stage shared-memory
//    ring with TMA, 128-byte swizzled so the tensor core reads them without
//    bank conflicts.  bf16 reads B as the caller stores it (BK x 256, N
//    contiguous: "MN-major" for the tensor core).  kind::tf32 does not take an
//    MN-major operand (it yields zeros), so the TF32 path is handed B already
//    transposed to N x K (K contiguous, "K-major") and loads 256 x BK boxes.
//    mbarriers replace the page's two __syncthreads: "full" (TMA bytes landed)
//    and "empty" (the MMAs reading the stage have completed, signalled by
//    tcgen05.commit).
//  * One thread of warp 1 issues the MMAs: 128 x 256 x (32 bytes of K) per
//    instruction, accumulating in fp32 in tensor memory.  With 128 x 256
//    tiles, two accumulators of 256 columns let the epilogue of one tile
//    overlap the MMAs of the next.
//  * Warps 2-5 drain an accumulator with tcgen05.ld (warp w reads lanes
//    32*(w%4) .. +31, i.e. 32 rows of C), and store each row's values with
//    128-bit stores, masked at the edges of C.
//
// Every C element is written exactly once.  The tensor cores add the k terms
// in a fixed order, so repeated runs are bit-identical.
#include <cstdio>

#include "device.cuh"
#include "host.h"

namespace tgemm {
namespace {

template <bool kTF32, bool kBKMajor, bool kWide>
struct Cfg {
    // kWide: 256 x 256 C tiles, two 128-row MMAs sharing each B tile, the whole
    // tensor memory as one accumulator; otherwise 128 x 256 tiles with two
    // accumulators so the epilogue of a tile overlaps the next tile's MMAs.
    static constexpr int HALVES = kWide ? 2 : 1;
    static constexpr int BM = 128 * HALVES;
    static constexpr int BN = 256;
    static constexpr int ES = kTF32 ? 4 : 2;        // bytes per input element
    static constexpr int BK = 128 / ES;             // elements of K per stage (128 bytes)
    static constexpr int UK = 32 / ES;              // elements of K per MMA (32 bytes)
    static constexpr int STAGES = kWide ? 3 : 4;
    static constexpr int ACCS = kWide ? 1 : 2;      // accumulator buffers in tensor memory
    static constexpr int CH = 128 / ES;             // B columns per 128-byte swizzle chunk
    static constexpr int NCH = BN / CH;             // TMA boxes per B stage
    static constexpr uint32_t CH_BYTES = BK * 128;  // bytes of one B chunk
    static constexpr uint32_t A_BYTES = BM * 128;
    static constexpr uint32_t B_BYTES = NCH * CH_BYTES;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int GROUP_M = kWide ? 8 : 16;
    static constexpr uint32_t IDESC =
        instr_desc(kTF32 ? kFormatTF32 : kFormatBF16, 0, kBKMajor ? 0u : 1u, 128, BN);
    static constexpr size_t SMEM = 1024 + STAGES * (A_BYTES + B_BYTES) + (2 * STAGES + 4) * 8 + 16;
    static_assert(ACCS * HALVES * BN <= 512, "accumulators exceed tensor memory");
};

constexpr int kThreads = 192;

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int group_m, int& tm,
                                            int& tn) {
    const int per_group = group_m * tiles_n;
    const int group = tile / per_group;
    const int first = group * group_m;
    const int rows = min(tiles_m - first, group_m);
    const int in_group = tile - group * per_group;
    tm = first + in_group % rows;
    tn = in_group / rows;
}

template <bool kTF32, bool kBKMajor, bool kWide>
__global__ void __launch_bounds__(kThreads, 1)
umma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            float* __restrict__ C, int64_t ldc, int M, int N, int K, int vec_store, uint32_t* status) {
    using G = Cfg<kTF32, kBKMajor, kWide>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + G::STAGES * G::A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + G::STAGES * G::B_BYTES);
    uint64_t* empty = full + G::STAGES;
    uint64_t* acc_full = empty + G::STAGES;    // [2]
    uint64_t* acc_empty = acc_full + 2;        // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles_m = (M + G::BM - 1) / G::BM;
    const int tiles_n = (N + G::BN - 1) / G::BN;
    const int tiles = tiles_m * tiles_n;
    const int KT = (K + G::BK - 1) / G::BK;

    if (threadIdx.x == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        for (int s = 0; s < G::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 128);
        }
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, G::TMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
                int tm, tn;
                tile_coords(tile, tiles_m, tiles_n, G::GROUP_M, tm, tn);
                for (int kb = 0; kb < KT; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, status)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[s], G::A_BYTES + G::B_BYTES);
                    tma_load_2d(sA + s * G::A_BYTES, &tmA, &full[s], kb * G::BK, tm * G::BM);
                    uint8_t* b_dst = sB + s * G::B_BYTES;
                    if (kBKMajor) {
                        tma_load_2d(b_dst, &tmB, &full[s], kb * G::BK, tn * G::BN);
                    } else {
#pragma unroll
                        for (int c = 0; c < G::NCH; ++c)
                            tma_load_2d(b_dst + c * G::CH_BYTES, &tmB, &full[s], tn * G::BN + c * G::CH,
                                        kb * G::BK);
                    }
                    if (++s == G::STAGES) { s = 0; ph ^= 1u; }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            int it = 0;
            for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x, ++it) {
                const uint32_t acc = it % G::ACCS;
                const uint32_t acc_ph = (it / G::ACCS) & 1;
                if (!mbar_wait(&acc_empty[acc], acc_ph ^ 1u, status)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * (G::HALVES * G::BN);
                for (int kb = 0; kb < KT; ++kb) {
                    if (!mbar_wait(&full[s], ph, status)) { ok = false; break; }
                    tc_fence_after_sync();
                    const uint32_t a0 = smem_addr(sA + s * G::A_BYTES);
                    const uint32_t b0 = smem_addr(sB + s * G::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < G::BK / G::UK; ++kk) {
                        // B, MN-major: 128-byte chunks of N (CH_BYTES apart), 8-row K
                        //    groups 1 KiB apart; the k-th slice starts UK rows down.
                        // B, K-major: laid out like A.
                        const uint64_t bd =
                            kBKMajor ? smem_desc(b0 + kk * 32, 16, 1024, kSwizzle128B)
                                     : smem_desc(b0 + kk * G::UK * 128, G::CH_BYTES, 1024, kSwizzle128B);
#pragma unroll
                        for (int h = 0; h < G::HALVES; ++h) {
                            // A: K-major, 128-byte rows, 8-row swizzle atoms 1 KiB apart;
                            //    rows 128h.. start 16 KiB in; slice kk starts 32*kk bytes in.
                            const uint64_t ad = smem_desc(a0 + h * 128 * 128 + kk * 32, 16, 1024, kSwizzle128B);
                            if (kTF32)
                                umma_tf32(d_tmem + h * G::BN, ad, bd, G::IDESC, (kb | kk) != 0);
                            else
                                umma_f16(d_tmem + h * G::BN, ad, bd, G::IDESC, (kb | kk) != 0);
                        }
                    }
                    umma_commit(&empty[s]);   // stage free once these MMAs complete
                    if (++s == G::STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&acc_full[acc]);  // accumulator ready for the epilogue
            }
        }
    } else {
        // --------------------------------------------------- epilogue --
        const int quarter = warp & 3;   // tensor-memory lanes 32*quarter .. +31
        int it = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++it) {
            const uint32_t acc = it % G::ACCS;
            const uint32_t acc_ph = (it / G::ACCS) & 1;
            if (!mbar_wait(&acc_full[acc], acc_ph, status)) break;
            tc_fence_after_sync();
            __syncwarp();   // tcgen05.ld below is warp-collective
            int tm, tn;
            tile_coords(tile, tiles_m, tiles_n, G::GROUP_M, tm, tn);
#pragma unroll
            for (int h = 0; h < G::HALVES; ++h) {
                const int row = tm * G::BM + h * 128 + quarter * 32 + lane;
                float* crow = C + static_cast<int64_t>(row) * ldc;
                const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       (acc * G::HALVES + h) * G::BN;
#pragma unroll 1
                for (int c = 0; c < G::BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_load_32(t_row + c * 32, r);
                    tmem_load_wait();
                    const int col0 = tn * G::BN + c * 32;
                    if (row < M) {
                        if (vec_store && col0 + 32 <= N) {
#pragma unroll
                            for (int j = 0; j < 32; j += 4)
                                *reinterpret_cast<float4*>(crow + col0 + j) =
                                    make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                                __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (col0 + j < N) crow[col0 + j] = __uint_as_float(r[j]);
                        }
                    }
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&acc_empty[acc]);
        }
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, G::TMEM_COLS);
    }
}

template <bool kTF32, bool kBKMajor, bool kWide>
cudaError_t launch(const Problem& p, const Device& dev) {
    using G = Cfg<kTF32, kBKMajor, kWide>;
    const CUtensorMapDataType dt = kTF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap ta, tb;
    const bool b_ok =
        kBKMajor ? make_tensor_map(&tb, dt, G::ES, p.B, p.n, p.k, p.ldb, G::BN, G::BK, CU_TENSOR_MAP_SWIZZLE_128B)
                 : make_tensor_map(&tb, dt, G::ES, p.B, p.k, p.n, p.ldb, G::BK, G::CH, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!make_tensor_map(&ta, dt, G::ES, p.A, p.m, p.k, p.lda, G::BM, G::BK, CU_TENSOR_MAP_SWIZZLE_128B) || !b_ok)
        return cudaErrorInvalidValue;
    auto kernel = umma_kernel<kTF32, kBKMajor, kWide>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(G::SMEM));
    if (err != cudaSuccess) {
        set_error("cudaFuncSetAttribute(umma_kernel): %s", cudaGetErrorString(err));
        return err;
    }
    const int64_t tiles = static_cast<int64_t>((p.m + G::BM - 1) / G::BM) * ((p.n + G::BN - 1) / G::BN);
    const int grid = static_cast<int>(tiles < dev.sm_count ? tiles : dev.sm_count);
    const int vec_store = (reinterpret_cast<uintptr_t>(p.C) % 16 == 0) && (p.ldc % 4 == 0);
    kernel<<<grid, kThreads, G::SMEM, p.stream>>>(ta, tb, p.C, p.ldc, p.m, p.n, p.k, vec_store, dev.status);
    count_launch();
    err = cudaGetLastError();
    if (err != cudaSuccess) set_error("umma_kernel launch: %s", cudaGetErrorString(err));
    return err;
}

}  // namespace

// Wide 256 x 256 tiles need two thirds of the operand bytes per MMA cycle of
// the 128 x 256 ones, which hides the L2 latency of the TMA loads better, but
// their epilogue cannot overlap the next tile's MMAs.  Measured on GB300
// (bf16): 8192^3 1726 vs 1641 TFLOP/s, 4096^3 1308 vs 1272, but
// 8192 x 8192 x 2048 1235 vs 1346: long k favours the wide tiles.
constexpr int kWideMinK = 3072;

cudaError_t launch_umma(const Problem& p, const Device& dev, bool tf32) {
    const bool wide = p.k >= kWideMinK;
    if (tf32) return wide ? launch<true, true, true>(p, dev) : launch<true, true, false>(p, dev);
    return wide ? launch<false, false, true>(p, dev) : launch<false, false, false>(p, dev);
}

}  // namespace tgemm
