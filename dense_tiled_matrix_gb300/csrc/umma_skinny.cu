// umma_skinny.cu -- bf16 C = A * B for m <= 64 (tgemm_bf16 on short, wide A).
//
// With only m <= 64 rows of C there are too few 128 x 256 output tiles to
// occupy the GPU, and the product is bound by streaming B (k x n) from HBM
// once.  This kernel therefore
//
//  * forms the transposed product C^T = B^T A^T, so that n (large) is the
//    tensor core's M dimension (128 columns of C per CTA) and m is its N
//    dimension (16, 32 or 64).  B^T is read as stored: n contiguous, i.e. an
//    MN-major operand; A is read as stored: k contiguous, K-major;
//  * splits k across the S CTAs of a thread-block cluster (grid n/128 x S,
//    cluster 1 x S), each streaming its k-slice of B through a 4-stage TMA
//    ring (two 64 x 64 boxes of B and one NM x 64 box of A per stage) into
//    tcgen05.mma, with the partial 128 x NM sums in tensor memory.  S is
//    chosen so that about 5/3 CTAs per SM stream B;
//  * adds the S partial sums through distributed shared memory (coffeejoa.com
//    "CUDA.3 Writing CUDA SIMT Kernels", "Distributed Shared Memory": the
//    cluster's shared memories form one address space, cluster.sync aligns the
//    CTAs): every CTA parks its partial in its own shared memory, the cluster
//    synchronises, and CTA r adds row m of all S partials, in rank order
//    0..S-1, for the rows m = r, r+S, ... and writes them to C with coalesced
//    stores.  No workspace, no atomics: the result is deterministic.
//
// All mbarrier waits are bounded (a timeout records TGEMM_ERR_TIMEOUT and
// skips the remaining work), and every CTA always reaches both cluster
// barriers, so no CTA can be left waiting for another.
#include "device.cuh"
#include "host.h"

namespace tgemm {
namespace {

constexpr int kThreads = 128;
constexpr int kBK = 64;                     // k per stage (128 bytes of bf16)
constexpr int kUK = 16;                     // k per MMA
constexpr int kTileN = 128;                 // columns of C per CTA (tensor-core M)
constexpr uint32_t kChunkBytes = kBK * 128; // one 64-column box of B: 64 k-rows x 128 bytes
// 128-column sub-tiles of C per CTA: each k-phase runs one MMA per sub-tile,
// all sharing the A^T operand; wider CTAs read longer contiguous row segments
// of B and need fewer clusters.
constexpr int kSubTiles = 1;
constexpr int kMaxSplit = 8;
// k is split until about 5/3 CTAs per SM stream B (measured best on GB300
// for 32..128 column tiles: 8 splits of 32 tiles, 4 of 64, 2 of 128).
constexpr int kTargetCtasPer3Sms = 5;

template <int NM, int NT>
struct SkinnyCfg {
    static constexpr uint32_t STAGE_B = NT * 2 * kChunkBytes;           // NT x 128 columns x 64 k
    static constexpr uint32_t STAGE_A = NM * 128;                       // NM rows x 64 bf16
    static constexpr int COLS = NM < 32 ? 32 : NM;                      // TMEM columns per sub-tile
    // 4 stages keep the CTA at ~75 KiB of shared memory; measured on GB300,
    // deeper rings (8-12 stages, one CTA per SM) stream B more slowly overall.
    static constexpr int STAGES = 4;
    static constexpr uint32_t TMEM_COLS = NT * COLS <= 32 ? 32 : NT * COLS <= 64 ? 64 : NT * COLS <= 128 ? 128 : 256;
    static constexpr uint32_t IDESC = instr_desc(kFormatBF16, 1, 0, kTileN, NM);
    static constexpr size_t SMEM = 1024 + STAGES * (STAGE_B + STAGE_A) + (2 * STAGES + 1) * 8 + 16;
    static_assert(NT * NM * kTileN * 4 <= STAGES * STAGE_B, "partial sums must fit in the B stages");
};

// The end of a skinny CTA: its 128 x NM partial sums (tensor memory, read by
// warps 0-3, warp w holding columns n0 + 128t + 32w + lane) go to its own
// shared memory, the cluster synchronises, CTA r adds rows r, r + S, ... of
// all S partials in rank order 0..S-1 through distributed shared memory
// (threads 0-127, one column each) and stores them, and a second cluster
// barrier keeps the partials alive until every CTA has read them.  Every
// thread of the CTA calls this.
template <int NM, int NT>
__device__ __forceinline__ void cluster_sum_and_store(uint32_t tmem, float* red, bool have, uint64_t* done,
                                                      int n0, int M, int N, float* __restrict__ C, int64_t ldc,
                                                      uint32_t* status) {
    using G = SkinnyCfg<NM, NT>;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_cta_rank();
    const uint32_t splits = gridDim.y;
    __syncwarp();
    if (warp < 4) {
        if (have && !mbar_wait(done, 0, status)) have = false;
        tc_fence_after_sync();
        __syncwarp();   // tcgen05.ld is warp-collective
        const int jrow = warp * 32 + lane;   // tensor-memory lane = column n0 + 128t + jrow of C
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16) + t * G::COLS;
            float* red_t = red + t * NM * kTileN;
            if (NM == 16) {
                uint32_t r[16];
                tmem_load_16(taddr, r);
                tmem_load_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) red_t[j * kTileN + jrow] = have ? __uint_as_float(r[j]) : 0.0f;
            } else {
#pragma unroll
                for (int c = 0; c < NM / 32; ++c) {
                    uint32_t r[32];
                    tmem_load_32(taddr + c * 32, r);
                    tmem_load_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        red_t[(c * 32 + j) * kTileN + jrow] = have ? __uint_as_float(r[j]) : 0.0f;
                }
            }
        }
        tc_fence_before_sync();
    }
    __syncwarp();
    cluster_sync_all();

    // --------------------------- add the S partials in rank order, store --
    const int rows = M < NM ? M : NM;
    const uint32_t my_red = smem_addr(red);
    // every rank of the cluster exists and fits the rank-order sum
    (void)TGEMM_DCHECK(splits <= kMaxSplit && rank < splits, status, kFileSkinny);
    if (threadIdx.x < kTileN) {
        for (int item = static_cast<int>(rank); item < NT * rows; item += static_cast<int>(splits)) {
            const int t = item / rows, mr = item - t * rows;
            const int n = n0 + t * kTileN + static_cast<int>(threadIdx.x);
            const uint32_t off =
                static_cast<uint32_t>(((t * NM + mr) * kTileN + static_cast<int>(threadIdx.x)) * 4);
            // the partial sum read lies inside the B stages that hold the partials
            if (!TGEMM_DCHECK(off + 4 <= G::STAGES * G::STAGE_B, status, kFileSkinny)) continue;
            // all remote loads first (they overlap), then the sum in rank order
            float part[kMaxSplit];
#pragma unroll
            for (int q = 0; q < kMaxSplit; ++q)
                part[q] = q < static_cast<int>(splits) ? ld_cluster_f32(cluster_map(my_red + off, q)) : 0.0f;
            float sum = 0.0f;
#pragma unroll
            for (int q = 0; q < kMaxSplit; ++q)
                if (q < static_cast<int>(splits)) sum += part[q];
            if (n < N) C[static_cast<int64_t>(mr) * ldc + n] = sum;
        }
    }
    __syncwarp();
    cluster_sync_all();   // partials stay readable until every CTA is done with them
}

template <int NM, int NT>
__global__ void __launch_bounds__(kThreads, 1)
umma_skinny_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   float* __restrict__ C, int64_t ldc, int M, int N, int K, int kb_per_split,
                   uint32_t* status) {
    using G = SkinnyCfg<NM, NT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align_1024(smem_raw);
    uint8_t* sB = smem;                                   // STAGES x 16 KiB
    uint8_t* sA = smem + G::STAGES * G::STAGE_B;            // STAGES x NM*128 B
    uint64_t* full = reinterpret_cast<uint64_t*>(sA + G::STAGES * G::STAGE_A);
    uint64_t* empty = full + G::STAGES;
    uint64_t* done = empty + G::STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
#ifdef TGEMM_DEBUG
    // Debug build: the fill number each stage holds, to check every wait's phase.
    __shared__ uint32_t dbg_fills[G::STAGES];
#endif
    // After the k loop the B stages hold this CTA's partial sums:
    // red[t][m][j], sub-tile t, row m of C, column n0 + 128t + j.
    float* red = reinterpret_cast<float*>(sB);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_cta_rank();
    const int n0 = blockIdx.x * kTileN * NT;
    const int KT = (K + kBK - 1) / kBK;
    const int kb0 = static_cast<int>(rank) * kb_per_split;
    const int kb1 = min(KT, kb0 + kb_per_split);
    const int nkb = kb1 > kb0 ? kb1 - kb0 : 0;

    // The first ring's worth of loads goes out as soon as the barriers exist,
    // so their HBM latency overlaps the tensor-memory allocation (warp 1) and
    // the block barrier.
    const int prefill = nkb < G::STAGES ? nkb : G::STAGES;
    auto issue = [&](int slot, int kb) {
#ifdef TGEMM_DEBUG
        dbg_fills[slot] = static_cast<uint32_t>((kb - kb0) / G::STAGES) + 1;
#endif
        mbar_arrive_expect_tx(&full[slot], G::STAGE_B + G::STAGE_A);
        uint8_t* b_dst = sB + slot * G::STAGE_B;
#pragma unroll
        for (int c = 0; c < 2 * NT; ++c)
            tma_load_2d(b_dst + c * kChunkBytes, &tmB, &full[slot], n0 + 64 * c, kb * kBK);
        tma_load_2d(sA + slot * G::STAGE_A, &tmA, &full[slot], kb * kBK, 0);
    };
    if (threadIdx.x == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        for (int s = 0; s < G::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
#ifdef TGEMM_DEBUG
        for (int s = 0; s < G::STAGES; ++s) dbg_fills[s] = 0;
#endif
        fence_barrier_init();
        for (int i = 0; i < prefill; ++i) issue(i, kb0 + i);   // empty slots: no wait needed
    }
    if (warp == 1) tmem_alloc(tmem_slot, G::TMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    bool ok = true;
    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- TMA producer --
        int s = prefill % G::STAGES;
        uint32_t ph = prefill == G::STAGES ? 1u : 0u;
        int issued = prefill;
        for (int kb = kb0 + prefill; kb < kb1; ++kb) {
            if (!mbar_wait(&empty[s], ph ^ 1u, status)) { ok = false; break; }
            issue(s, kb);
            ++issued;
            if (++s == G::STAGES) { s = 0; ph ^= 1u; }
        }
        drain_ring(full, G::STAGES, issued, status);   // no copy outlives the CTA
    } else if (warp == 1 && lane == 0) {
        // ----------------------------------------------------- MMA issuer --
        int s = 0;
        uint32_t ph = 0;
        int last_s = -1;   // stage of the last commit to an empty barrier
        uint32_t last_ph = 0;
        for (int i = 0; i < nkb; ++i) {
            if (!mbar_wait(&full[s], ph, status)) { ok = false; break; }
            tc_fence_after_sync();
#ifdef TGEMM_DEBUG
            // the stage holds fill i / STAGES (not an older one, not a refill); the
            // sub-tiles' accumulators lie inside the tensor-memory allocation
            TGEMM_DCHECK(dbg_fills[s] == static_cast<uint32_t>(i / G::STAGES) + 1, status, kFileSkinny);
            TGEMM_DCHECK((NT - 1) * G::COLS + NM <= static_cast<int>(G::TMEM_COLS), status, kFileSkinny);
#endif
            const uint32_t b0 = smem_addr(sB + s * G::STAGE_B);
            const uint32_t a0 = smem_addr(sA + s * G::STAGE_A);
#pragma unroll
            for (int kk = 0; kk < kBK / kUK; ++kk) {
                // tensor-core B = A^T: K-major rows of 128 bytes, 8-row groups 1 KiB apart.
                const uint64_t bd = smem_desc(a0 + kk * 32, 16, 1024, kSwizzle128B);
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    // tensor-core A = B^T of sub-tile t: MN-major, 64-column chunks
                    // kChunkBytes apart, 8-row k groups 1 KiB apart; slice kk starts kUK rows down.
                    const uint64_t ad =
                        smem_desc(b0 + t * 2 * kChunkBytes + kk * kUK * 128, kChunkBytes, 1024, kSwizzle128B);
                    umma_f16(tmem + t * G::COLS, ad, bd, G::IDESC, (i | kk) != 0);
                }
            }
            umma_commit(&empty[s]);
            last_s = s;
            last_ph = ph;
            if (++s == G::STAGES) { s = 0; ph ^= 1u; }
        }
        if (ok) umma_commit(done);
        // The last commit completes once every MMA issued before it has:
        // none may still run when the tensor memory is freed.
        if (last_s >= 0) mbar_wait(&empty[last_s], last_ph, status, kDrainLimitNs);
    }

    cluster_sum_and_store<NM, NT>(tmem, red, nkb > 0, done, n0, M, N, C, ldc, status);

    if (warp == 1) {   // the allocating warp frees the tensor memory
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, G::TMEM_COLS);
    }
    (void)ok;
}

// Split of k over the CTAs of a cluster: about 5/3 CTAs per SM, at most
// kMaxSplit, no empty slice.
void skinny_split(const Problem& p, const Device& dev, int tiles, int* splits_out, int* kb_per_split_out) {
    const int KT = (p.k + kBK - 1) / kBK;
    const int target = kTargetCtasPer3Sms * dev.sm_count / 3;
    int splits = (target + tiles / 2) / tiles;
    splits = splits < 1 ? 1 : splits;
    splits = splits > kMaxSplit ? kMaxSplit : splits;
    splits = splits > KT ? KT : splits;
    const int kb_per_split = (KT + splits - 1) / splits;
    *splits_out = (KT + kb_per_split - 1) / kb_per_split;
    *kb_per_split_out = kb_per_split;
}

template <int NM>
cudaError_t launch_nm(const Problem& p, const Device& dev) {
    constexpr int NT = kSubTiles;
    using G = SkinnyCfg<NM, NT>;
    CUtensorMap ta, tb;
    if (!make_tensor_map(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.A, p.m, p.k, p.lda, NM, kBK,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.B, p.k, p.n, p.ldb, kBK, 64,
                         CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    auto kernel = umma_skinny_kernel<NM, NT>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(G::SMEM));
    if (err != cudaSuccess) {
        set_error("cudaFuncSetAttribute(umma_skinny_kernel): %s", cudaGetErrorString(err));
        return err;
    }
    const int tiles = (p.n + kTileN * NT - 1) / (kTileN * NT);
    int splits = 1, kb_per_split = 1;
    skinny_split(p, dev, tiles, &splits, &kb_per_split);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles), static_cast<unsigned>(splits), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = G::SMEM;
    cfg.stream = p.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = static_cast<unsigned>(splits);
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, kernel, ta, tb, p.C, p.ldc, p.m, p.n, p.k, kb_per_split, dev.status);
    count_launch();
    if (err != cudaSuccess) set_error("umma_skinny_kernel launch: %s", cudaGetErrorString(err));
    return err;
}

}  // namespace

cudaError_t launch_umma_skinny(const Problem& p, const Device& dev) {
    if (p.m <= 16) return launch_nm<16>(p, dev);
    if (p.m <= 32) return launch_nm<32>(p, dev);
    return launch_nm<64>(p, dev);
}

}  // namespace tgemm
