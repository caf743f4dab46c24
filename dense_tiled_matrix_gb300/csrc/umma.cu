// umma.cu -- C = A * B on the tcgen05 tensor cores (tgemm_tf32, tgemm_bf16).
//
// The tiled matrix multiply of hecess.blogspot.com "[Multi-Core & GPU
// Programming] CUDA - Matrix Multiplication" ("[Shared Memory]", "Tiled Matrix
// Multiplication Kernel"), with the per-thread register accumulator (the
// page's Pvalue) moved into tensor memory and the per-phase inner product done
// by tcgen05.mma:
//
//  * Output tiles of 256 x BN (k >= 3072, or k >= 1024 where their rounds of
//    CTAs fill at least as well as those of 128-row tiles, without stream-K:
//    two 128-row MMAs share each B tile, one
//    accumulator spanning the tensor memory, 3 stages) or 128 x BN (two
//    accumulators, 4 stages), BN = 256, or 224 for TF32 shapes whose last wave
//    that fills better; visited by a persistent grid of one CTA per SM in
//    groups of tile rows (neighbouring CTAs share A and B tiles in L2).  Where
//    whole tiles would leave more than a quarter of the CTA slots idle, the
//    last G + r tiles are split along k between CTAs (stream-K, stream_k.cuh);
//    where there are fewer tiles than SMs, every tile is cut along k into
//    split-K pieces, one CTA each, whose partial sums a reduce kernel adds in
//    piece order.
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
//    overlap the MMAs of the next.  For large bf16 grids of such tiles, the
//    two CTAs of a (2 x 1) cluster take vertically adjacent tiles and share
//    their B tile: each loads half of its chunks with TMA multicast into both.
//  * Warps 2-5, or 2-9 for stream-K and C that TMA cannot describe, drain an
//    accumulator with tcgen05.ld (warp w reads lanes 32*(w%4) .. +31, i.e. 32
//    rows of C, one row per lane; with 8 warps the two of a lane quarter take
//    alternate 32-column blocks) and turn each 32 x 32
//    block through shared memory so that C is written as whole 128-byte row
//    segments: the block is staged in the layout of a TMA box and, where TMA
//    can describe C, one lane stores it with a TMA store; otherwise the warp
//    reads the rows back and stores scalars, masked at the edges of C.
//
// Every C element is written exactly once.  The tensor cores add the k terms
// in a fixed order, a stream-K tile is (head partial) + (tail partial) and a
// split-K tile the sum of its pieces in piece order, so repeated runs are
// bit-identical.
#include <cstdio>
#include <cstring>

#include "device.cuh"
#include "host.h"
#include "stream_k.cuh"

namespace tgemm {
namespace {

// Epilogue warps: 4 (one per tensor-memory lane quarter, two staging tiles
// each) or 8 (two per quarter taking alternate column blocks, one tile each).
constexpr int kMaxEpiWarps = 8;

template <bool kTF32, bool kBKMajor, bool kWide, int kBN = 256>
struct Cfg {
    // kWide: 256 x 256 C tiles, two 128-row MMAs sharing each B tile, the whole
    // tensor memory as one accumulator; otherwise 128 x 256 tiles with two
    // accumulators so the epilogue of a tile overlaps the next tile's MMAs.
    static constexpr int HALVES = kWide ? 2 : 1;
    static constexpr int BM = 128 * HALVES;
    static constexpr int BN = kBN;                   // 256, or 224 (K-major B only)
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
    static constexpr uint32_t TCOL = 256;           // tensor-memory columns between accumulators / halves
    static constexpr int GROUP_M = kWide ? 8 : 16;
    static constexpr uint32_t IDESC =
        instr_desc(kTF32 ? kFormatTF32 : kFormatBF16, 0, kBKMajor ? 0u : 1u, 128, BN);
    // per epilogue warp one 32 x 32 fp32 staging tile (4 KiB) in the layout of
    // a TMA box with 128-byte swizzle, from which a TMA store writes C (or which
    // the warp reads back where TMA cannot describe C)
    static constexpr uint32_t EPI_BUF = 32 * 32 * 4;
    static constexpr uint32_t EPI_BYTES = kMaxEpiWarps * EPI_BUF;   // 4 warps x 2 tiles or 8 x 1
    static constexpr size_t SMEM = 1024 + STAGES * (A_BYTES + B_BYTES) + EPI_BYTES + (2 * STAGES + 4) * 8 + 16;
    static_assert(ACCS * HALVES * 256 <= 512, "accumulators exceed tensor memory");
    static_assert(BN % 32 == 0 && BN <= 256, "tile width");
    static_assert(kBKMajor || BN % CH == 0, "an N-contiguous B tile is a whole number of 128-byte chunks");
};

constexpr int threads_for(int epi_warps) { return 32 * (2 + epi_warps); }   // producer, MMA issuer, epilogue
constexpr bool kPdl = true;   // whole-tile launches may start behind the previous kernel
constexpr bool kUsePairs = true;   // bf16 128-row whole tiles as multicast CTA pairs

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

// Named barrier of the epilogue warps (threads 64 .. 64 + 32 kEpiWarps - 1).
template <int kEpiWarps>
__device__ __forceinline__ void epilogue_sync() { asm volatile("bar.sync 1, %0;" :: "n"(32 * kEpiWarps) : "memory"); }

// The CTAs walk the persistent plan of stream_k.cuh: whole tiles b, b + G, ...
// and, when `ws` is given and the last wave would be partial, a stream-K
// region whose tiles may be split along k between two CTAs.  The tail of a
// split tile stores its fp32 accumulator in its CTA's `ws` slot and raises
// its flag; the head waits for the flag, adds that partial to its own
// accumulator (always head + tail) and stores the tile.  Split tiles need
// every CTA resident: the launch is cooperative.  With kSK and pieces > 0 the
// grid has one CTA per split-K piece instead, each storing its partial tile
// in its own `ws` slot for umma_pieces_reduce_kernel; nothing waits then.
template <bool kTF32, bool kBKMajor, bool kWide, int kBN, bool kSK, bool kPair, int kEpiWarps>
__global__ void __launch_bounds__(threads_for(kEpiWarps), 1)
umma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmC, float* __restrict__ C, int64_t ldc, int M, int N, int K,
            int vec_store, uint32_t* status,
            float* __restrict__ ws, unsigned* __restrict__ flags, int pieces) {
    using G = Cfg<kTF32, kBKMajor, kWide, kBN>;
    // kPair: the two CTAs of a (2 x 1) cluster take vertically adjacent 128 x 256
    // tiles, which use the same B tile: each loads half of its 128-byte chunks and
    // multicasts them to both, so each SM fetches the operand bytes per MMA of a
    // 256-row tile while keeping two accumulators.
    static_assert(!kPair || (!kWide && !kSK && !kBKMajor && G::NCH % 2 == 0), "pairs: bf16 128-row whole tiles");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align_1024(smem_raw);
    uint8_t* sA = smem;
    uint8_t* sB = smem + G::STAGES * G::A_BYTES;
    float* sEpi = reinterpret_cast<float*>(sB + G::STAGES * G::B_BYTES);   // 4 warps x 2 x 32 x 32 fp32
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + G::STAGES * G::B_BYTES + G::EPI_BYTES);
    uint64_t* empty = full + G::STAGES;
    uint64_t* acc_full = empty + G::STAGES;    // [2]
    uint64_t* acc_empty = acc_full + 2;        // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
    __shared__ int s_flag_ok;
#ifdef TGEMM_DEBUG
    // Debug build: the fill number each stage holds, to check every wait's phase.
    __shared__ uint32_t dbg_fills[G::STAGES];
#endif

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles_m = (M + G::BM - 1) / G::BM;
    const int tiles_n = (N + G::BN - 1) / G::BN;
    const int KT = (K + G::BK - 1) / G::BK;
    const int tiles = tiles_m * tiles_n;
    // Pairs: rank r of cluster c takes tile rows 2 pm + r of the pairs c, c + G / 2, ...
    const uint32_t rank = kPair ? cluster_cta_rank() : 0u;
    const int pairs_m = (tiles_m + 1) / 2;
    const int units = kPair ? pairs_m * tiles_n : tiles;
    const int unit0 = kPair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int unit_step = kPair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    auto coords = [&](int unit, int& tm, int& tn) {
        if (kPair) {
            int pm;
            tile_coords(unit, pairs_m, tiles_n, G::GROUP_M / 2, pm, tn);
            tm = 2 * pm + static_cast<int>(rank);   // past the last tile row: loads read zeros, nothing is stored
        } else {
            tile_coords(unit, tiles_m, tiles_n, G::GROUP_M, tm, tn);
        }
    };
    // kSK with pieces > 0: split-K pieces instead of the stream-K plan.  CTA u
    // (one per unit) computes piece u % pieces of tile u / pieces, k-phases
    // [KT p / pieces, KT (p + 1) / pieces), and stores its partial sums in
    // workspace slot u; umma_pieces_reduce_kernel adds a tile's pieces in order.
    const bool split = kSK && pieces > 0;
    SkPlan plan;
    if (kSK && !split) plan.init(tiles, KT, blockIdx.x, gridDim.x);
    // The CTA's segments (tile, k-phases [ka, kz)): with kSK the plan's
    // sequence or the CTA's one piece, otherwise whole tiles b, b + G, ...
    // Each role walks its own.
    struct Seq {
        SkCursor cur;
        int t_next;
    };
    auto seq_init = [&](Seq& q) {
        q.t_next = unit0;
        if (kSK && !split) q.cur.init(plan);
    };
    auto seq_next = [&](Seq& q, int& t, int& ka, int& kz) -> bool {
        if (split) {
            if (q.t_next < 0) return false;
            const int u = q.t_next;
            q.t_next = -1;
            t = u / pieces;
            const int piece = u - t * pieces;
            ka = static_cast<int>(static_cast<int64_t>(KT) * piece / pieces);
            kz = static_cast<int>(static_cast<int64_t>(KT) * (piece + 1) / pieces);
            return t < tiles;
        }
        if (kSK) return q.cur.next(plan, KT, t, ka, kz);
        if (q.t_next >= units) return false;
        t = q.t_next;
        q.t_next += unit_step;
        ka = 0;
        kz = KT;
        return true;
    };

    if (threadIdx.x == 0) {
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        for (int s = 0; s < G::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kPair ? 2 : 1);   // pairs: both CTAs' MMAs release a stage
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 32 * kEpiWarps);
        }
#ifdef TGEMM_DEBUG
        for (int s = 0; s < G::STAGES; ++s) dbg_fills[s] = 0;
#endif
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, G::TMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // pairs: the peer's barriers exist before any copy can land in its shared memory
    if (kPair) cluster_sync_all();
    const uint32_t tmem_base = *tmem_slot;
    // Launched right behind the previous kernel in the stream (e.g. the B
    // transpose of the TF32 path): wait for it before any global access.
    griddep_wait();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            int issued = 0;
            Seq sq;
            seq_init(sq);
            int tile, ka, kz;
            while (ok && seq_next(sq, tile, ka, kz)) {
                int tm, tn;
                coords(tile, tm, tn);
                for (int kb = ka; kb < kz; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, status)) { ok = false; break; }
#ifdef TGEMM_DEBUG
                    dbg_fills[s] = static_cast<uint32_t>(issued / G::STAGES) + 1;
#endif
                    mbar_arrive_expect_tx(&full[s], G::A_BYTES + G::B_BYTES);
                    tma_load_2d(sA + s * G::A_BYTES, &tmA, &full[s], kb * G::BK, tm * G::BM);
                    uint8_t* b_dst = sB + s * G::B_BYTES;
                    if (kBKMajor) {
                        tma_load_2d(b_dst, &tmB, &full[s], kb * G::BK, tn * G::BN);
                    } else if (kPair) {
                        // this CTA's half of the chunks, into both CTAs of the pair
#pragma unroll
                        for (int c = 0; c < G::NCH / 2; ++c) {
                            const int ch = static_cast<int>(rank) * (G::NCH / 2) + c;
                            tma_load_2d_multicast(b_dst + ch * G::CH_BYTES, &tmB, &full[s], tn * G::BN + ch * G::CH,
                                                  kb * G::BK, 0x3);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < G::NCH; ++c)
                            tma_load_2d(b_dst + c * G::CH_BYTES, &tmB, &full[s], tn * G::BN + c * G::CH,
                                        kb * G::BK);
                    }
                    ++issued;
                    if (++s == G::STAGES) { s = 0; ph ^= 1u; }
                }
            }
            drain_ring(full, G::STAGES, issued, status);   // no copy outlives the CTA
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer --
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            int it = 0;
            int last_s = -1;   // stage of the last commit to an empty barrier
            uint32_t last_ph = 0;
            int consumed = 0;   // stages consumed so far (debug checks)
            Seq sq;
            seq_init(sq);
            int tile, ka, kz;
            for (; ok && seq_next(sq, tile, ka, kz); ++it) {
                const uint32_t acc = it % G::ACCS;
                const uint32_t acc_ph = (it / G::ACCS) & 1;
                if (!mbar_wait(&acc_empty[acc], acc_ph ^ 1u, status)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * (G::HALVES * G::TCOL);
                // the accumulator's columns lie inside the allocation
                if (!TGEMM_DCHECK((acc * G::HALVES + G::HALVES - 1) * G::TCOL + G::BN <= G::TMEM_COLS, status,
                                  kFileUmma))
                    break;
                for (int kb = ka; kb < kz; ++kb) {
                    if (!mbar_wait(&full[s], ph, status)) { ok = false; break; }
                    tc_fence_after_sync();
                    const uint32_t a0 = smem_addr(sA + s * G::A_BYTES);
                    const uint32_t b0 = smem_addr(sB + s * G::B_BYTES);
#ifdef TGEMM_DEBUG
                    // the stage holds fill `consumed / STAGES` (not an older one, not a refill),
                    // and the last MMA's operands end inside their stage
                    TGEMM_DCHECK(dbg_fills[s] == static_cast<uint32_t>(consumed / G::STAGES) + 1, status, kFileUmma);
                    TGEMM_DCHECK(s < G::STAGES && (G::HALVES - 1) * 128 * 128 + (G::BK / G::UK - 1) * 32 + 32 <=
                                                      static_cast<int>(G::A_BYTES),
                                 status, kFileUmma);
#endif
                    ++consumed;
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
                            // The segment's first MMA overwrites the accumulator.
                            const bool accumulate = kb != ka || kk != 0;
                            if (kTF32)
                                umma_tf32(d_tmem + h * G::TCOL, ad, bd, G::IDESC, accumulate);
                            else
                                umma_f16(d_tmem + h * G::TCOL, ad, bd, G::IDESC, accumulate);
                        }
                    }
                    // stage free once these MMAs complete (pairs: in both CTAs, whose
                    // copies land in each other's stage)
                    if (kPair)
                        umma_commit_multicast(&empty[s], 0x3);
                    else
                        umma_commit(&empty[s]);
                    last_s = s;
                    last_ph = ph;
                    if (++s == G::STAGES) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&acc_full[acc]);  // accumulator ready for the epilogue
            }
            // The last commit completes once every MMA issued before it has:
            // none may still run when the tensor memory is freed.
            if (last_s >= 0) mbar_wait(&empty[last_s], last_ph, status, kDrainLimitNs);
        }
    } else {
        // --------------------------------------------------- epilogue --
        // A warp whose wait ran out keeps the others' control flow (it stops
        // waiting but still reaches every epilogue_sync), so none is left
        // waiting at a named barrier.
        const int quarter = warp & 3;   // tensor-memory lanes 32*quarter .. +31
        const int row_in_half = quarter * 32 + lane;
        static_assert(kEpiWarps == 4 || kEpiWarps == 8, "epilogue warps");
        // this warp's staging area: two tiles (4 warps) or one (8 warps)
        float* epi = sEpi + (warp - 2) * (G::EPI_BUF / 4) * (kMaxEpiWarps / kEpiWarps);
        // With 8 warps two share each lane quarter; member `col_half` drains the
        // 32-column blocks c = col_half, col_half + 2, ...
        constexpr int kColStep = kEpiWarps / 4;
        const int col_half = (warp - 2) / 4;
        uint32_t stores = 0;   // TMA stores this warp has issued
        bool ok = true;
        int it = 0;
        Seq sq;
        seq_init(sq);
        int tile, ka, kz;
        for (; seq_next(sq, tile, ka, kz); ++it) {
            const uint32_t acc = it % G::ACCS;
            const uint32_t acc_ph = (it / G::ACCS) & 1;
            if (ok && !mbar_wait(&acc_full[acc], acc_ph, status)) ok = false;
            tc_fence_after_sync();
            __syncwarp();   // tcgen05.ld below is warp-collective
            int tm, tn;
            coords(tile, tm, tn);
            // a piece stores its partial sums like a stream-K tail (no flag)
            const bool tail = kSK && (split || ka > 0);
            const bool head = kSK && !tail && kz < KT;
            // Partial tile of a CTA's slot: float4 ((h * BN/32 + c) * 8 + q) * 128 + row
            // holds columns 32c + 4q .. +3 of row `row` of half h, so a warp
            // stores or loads 512 contiguous bytes.
            float4* my_part = reinterpret_cast<float4*>(ws + static_cast<int64_t>(blockIdx.x) * G::BM * G::BN);
            const float4* next_part =
                reinterpret_cast<const float4*>(ws + static_cast<int64_t>(blockIdx.x + 1) * G::BM * G::BN);
            if (head) {
                // a head's tail is the next CTA, which exists
                if (threadIdx.x == 64)
                    s_flag_ok = ok && TGEMM_DCHECK(blockIdx.x + 1 < gridDim.x, status, kFileUmma) &&
                                        wait_flag(flags + blockIdx.x + 1, status)
                                    ? 1
                                    : 0;
                epilogue_sync<kEpiWarps>();
            }
#pragma unroll
            for (int h = 0; h < G::HALVES; ++h) {
                const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                       (acc * G::HALVES + h) * G::TCOL;
#pragma unroll 1
                for (int c = col_half; c < G::BN / 32; c += kColStep) {
                    uint32_t r[32];
                    // columns of this load inside the allocation (uniform across the warp)
                    (void)TGEMM_DCHECK((acc * G::HALVES + h) * G::TCOL + c * 32 + 32 <= G::TMEM_COLS, status,
                                       kFileUmma);
                    tmem_load_32(t_row + c * 32, r);
                    tmem_load_wait();
                    const int slot = (h * (G::BN / 32) + c) * 8;
                    if (tail) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            my_part[(slot + q) * 128 + row_in_half] =
                                make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                            __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
                        continue;
                    }
                    if (head && s_flag_ok) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 v = __ldcg(next_part + (slot + q) * 128 + row_in_half);
                            r[4 * q] = __float_as_uint(__uint_as_float(r[4 * q]) + v.x);
                            r[4 * q + 1] = __float_as_uint(__uint_as_float(r[4 * q + 1]) + v.y);
                            r[4 * q + 2] = __float_as_uint(__uint_as_float(r[4 * q + 2]) + v.z);
                            r[4 * q + 3] = __float_as_uint(__uint_as_float(r[4 * q + 3]) + v.w);
                        }
                    }
                    // Corner turn (note.jhbae.stream "Lec 29 · GPU Architecture (2)",
                    // transpose case study): lane l holds row l of this 32 x 32 block;
                    // through the warp's shared tile C is written as whole 128-byte row
                    // segments instead of 32 rows at once.
                    const int col0 = tn * G::BN + c * 32;
                    const int row0 = tm * G::BM + h * 128 + quarter * 32;
                    // A TMA store clips a row at 16-byte granularity: a block that runs
                    // past C's last column takes it only if that column ends a 16-byte
                    // granule (N a multiple of 4).  A block wholly below C issues none
                    // (the scalar path below stores nothing for it).  The conditions
                    // are uniform across the warp.
                    if (vec_store && row0 < M && (col0 + 32 <= N || (N & 3) == 0)) {
                        // The tile is a TMA box (32 rows of 128 bytes, 128-byte swizzle:
                        // 16-byte chunk q of row i at chunk q ^ (i % 8), so the eight rows a
                        // quarter warp writes fall in eight bank groups); one lane has the
                        // TMA unit store it, and rows and columns past C are not written.
                        // The warp moves on while the store drains, into its other tile (4
                        // warps) once the store issued two blocks ago has read it, or into
                        // the same tile (8 warps) once the last store has.
                        float* tile_buf = epi;
                        if (kEpiWarps == 4) {
                            tile_buf = epi + (stores & 1u) * (G::EPI_BUF / 4);
                            if (stores >= 2) {
                                if (lane == 0) bulk_wait_group_read<1>();
                                __syncwarp();
                            }
                        } else if (stores >= 1) {
                            if (lane == 0) bulk_wait_group_read<0>();
                            __syncwarp();
                        }
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            *reinterpret_cast<float4*>(tile_buf + lane * 32 + ((q ^ (lane & 7)) << 2)) =
                                make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                            __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
                        fence_proxy_async_smem();   // the generic-proxy writes, before the TMA unit reads them
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmC, tile_buf, col0, row0);
                            bulk_commit_group();
                        }
                        ++stores;
                    } else {
                        // C rows not 16-byte aligned (TMA cannot describe C), or a block at
                        // a ragged right edge: the warp writes the same swizzled tile, reads
                        // each row back (its 8 chunks are 128 contiguous bytes of one row,
                        // so the reads are conflict-free too) and stores it, one row x 128
                        // bytes per warp store.  The tile is free once this warp's TMA
                        // stores have read it.
                        if (stores > 0) {
                            if (lane == 0) bulk_wait_group_read<0>();
                            __syncwarp();
                        }
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            *reinterpret_cast<float4*>(epi + lane * 32 + ((q ^ (lane & 7)) << 2)) =
                                make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                            __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
                        __syncwarp();
                        const int col = col0 + lane;
                        const int q = lane >> 2, w = lane & 3;
#pragma unroll 8
                        for (int rr = 0; rr < 32; ++rr) {
                            const float v = epi[rr * 32 + ((q ^ (rr & 7)) << 2) + w];
                            if (row0 + rr < M && col < N) C[static_cast<int64_t>(row0 + rr) * ldc + col] = v;
                        }
                        __syncwarp();   // the tile is rewritten by the next block
                    }
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&acc_empty[acc]);
            if (tail && !split) {
                __threadfence();
                epilogue_sync<kEpiWarps>();
                if (threadIdx.x == 64) st_release_u32(flags + blockIdx.x, 1u);
            }
        }
        // every TMA store of C has completed (and read its staging tile) before the CTA ends
        if (lane == 0) bulk_wait_group<0>();
    }

    __syncthreads();
    // pairs: the peer has consumed every stage, so no copy is still landing in it
    if (kPair) cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, G::TMEM_COLS);
    }
}

// C of split-K pieces: tile t is the sum of its pieces' partial sums (slots
// t * pieces .. + pieces - 1), added in piece order, so repeated runs are
// bit-identical.  A slot has the layout the kernel's epilogue writes: float4
// ((h * BN/32 + c) * 8 + q) * 128 + r holds columns 32c + 4q .. +3 of row
// 128h + r of the tile.  Block (t, j) takes float4s 1024 j .. +1023 of tile t,
// so a warp reads 512 contiguous bytes of every slot.
template <int BM, int BN, int kGroupM>
__global__ void __launch_bounds__(256)
umma_pieces_reduce_kernel(const float4* __restrict__ ws, float* __restrict__ C, int64_t ldc, int M, int N,
                          int pieces, int vec_store) {
    constexpr int kSlot4 = BM * BN / 4;
    const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
    const int t = static_cast<int>(blockIdx.x);
    int tm, tn;
    tile_coords(t, tiles_m, tiles_n, kGroupM, tm, tn);
    const float4* src = ws + static_cast<int64_t>(t) * pieces * kSlot4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int f = static_cast<int>(blockIdx.y) * 1024 + i * 256 + static_cast<int>(threadIdx.x);
        if (f >= kSlot4) break;
        float4 v = src[f];
        for (int pc = 1; pc < pieces; ++pc) {
            const float4 w = src[static_cast<int64_t>(pc) * kSlot4 + f];
            v.x += w.x;
            v.y += w.y;
            v.z += w.z;
            v.w += w.w;
        }
        const int g = f >> 7, q = g & 7, hc = g >> 3;
        const int row = tm * BM + (hc / (BN / 32)) * 128 + (f & 127);
        const int col = tn * BN + (hc % (BN / 32)) * 32 + q * 4;
        if (row >= M) continue;
        float* dst = C + static_cast<int64_t>(row) * ldc + col;
        if (vec_store && col + 3 < N) {
            *reinterpret_cast<float4*>(dst) = v;
        } else {
            const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (col + j < N) dst[j] = e[j];
        }
    }
}

template <bool kTF32, bool kBKMajor, bool kWide, int kBN>
int64_t tile_count(const Problem& p) {
    using G = Cfg<kTF32, kBKMajor, kWide, kBN>;
    return static_cast<int64_t>((p.m + G::BM - 1) / G::BM) * ((p.n + G::BN - 1) / G::BN);
}

// Stream-K when the plan has a region and the whole-tile grid would fill
// less than 3/4 of its CTA slots.  Measured on GB300 (TFLOP/s, whole tiles ->
// stream-K): 3300 x 3000 x 3100 TF32 354 -> 479, bf16 477 -> 559 (51 %
// filled); 2000 x 2600 x 1000 TF32 219 -> 228 (58 %); but 4096^3 TF32 685 ->
// 649 (84 %) and 8192^3 bf16 1802 -> 1603 (96 %): the runs start at scattered
// k, so the region's A and B are live in L2 all at once (ncu: DRAM reads
// 0.87 -> 1.92 GB, L2 hit rate 77 -> 62 %), whereas whole tiles step through
// k together.
template <bool kTF32, bool kBKMajor, bool kWide, int kBN>
bool has_sk(const Problem& p, const Device& dev) {
    using G = Cfg<kTF32, kBKMajor, kWide, kBN>;
    const int64_t tiles = tile_count<kTF32, kBKMajor, kWide, kBN>(p);
    const int64_t waves = (tiles + dev.sm_count - 1) / dev.sm_count;
    return sk_has_region(tiles, (p.k + G::BK - 1) / G::BK, dev.sm_count) && 4 * tiles < 3 * waves * dev.sm_count;
}

// Split-K pieces where the whole tiles fill less than one round of CTAs (no
// stream-K plan then): each tile is cut along k into P pieces, P = the most
// that fit in one round with at least kMinPiecePhases k-phases each; the
// pieces' partial sums are added by umma_pieces_reduce_kernel.
constexpr int64_t kMinPiecePhases = 8;

template <bool kTF32, bool kBKMajor, bool kWide, int kBN>
int pieces_for(const Problem& p, const Device& dev) {
    using G = Cfg<kTF32, kBKMajor, kWide, kBN>;
    const int64_t tiles = tile_count<kTF32, kBKMajor, kWide, kBN>(p);
    if (tiles <= 0 || tiles >= dev.sm_count) return 0;
    const int64_t KT = (p.k + G::BK - 1) / G::BK;
    int64_t pieces = dev.sm_count / tiles;
    if (pieces > KT / kMinPiecePhases) pieces = KT / kMinPiecePhases;
    return pieces >= 2 ? static_cast<int>(pieces) : 0;
}

template <bool kTF32, bool kBKMajor, bool kWide, int kBN>
uint64_t workspace_bytes(const Problem& p, const Device& dev) {
    using G = Cfg<kTF32, kBKMajor, kWide, kBN>;
    const uint64_t slot = static_cast<uint64_t>(G::BM) * G::BN * sizeof(float);
    if (has_sk<kTF32, kBKMajor, kWide, kBN>(p, dev))
        return static_cast<uint64_t>(dev.sm_count) * (slot + sizeof(unsigned));   // a slot and a flag per CTA
    const int pieces = pieces_for<kTF32, kBKMajor, kWide, kBN>(p, dev);
    if (pieces > 0) return static_cast<uint64_t>(tile_count<kTF32, kBKMajor, kWide, kBN>(p)) * pieces * slot;
    return 0;
}

// Stream-K (kSK, with its workspace), split-K pieces (kSK with pieces > 0,
// then the reduce kernel) or whole tiles.
template <bool kTF32, bool kBKMajor, bool kWide, int kBN, bool kSK, bool kPair = false>
cudaError_t launch(const Problem& p, const Device& dev, void* workspace, int pieces = 0) {
    using G = Cfg<kTF32, kBKMajor, kWide, kBN>;
    const CUtensorMapDataType dt = kTF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap ta, tb;
    const bool b_ok =
        kBKMajor ? make_tensor_map(&tb, dt, G::ES, p.B, p.n, p.k, p.ldb, G::BN, G::BK, CU_TENSOR_MAP_SWIZZLE_128B)
                 : make_tensor_map(&tb, dt, G::ES, p.B, p.k, p.n, p.ldb, G::BK, G::CH, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!make_tensor_map(&ta, dt, G::ES, p.A, p.m, p.k, p.lda, G::BM, G::BK, CU_TENSOR_MAP_SWIZZLE_128B) || !b_ok)
        return cudaErrorInvalidValue;
    const int64_t tiles = tile_count<kTF32, kBKMajor, kWide, kBN>(p);
    // C through TMA stores (32 x 32 boxes, 128-byte swizzle) where TMA can describe
    // it: 16-byte aligned base and row pitch; otherwise scalar stores.
    CUtensorMap tc;
    std::memset(&tc, 0, sizeof tc);
    int vec_store = (reinterpret_cast<uintptr_t>(p.C) % 16 == 0) && (p.ldc % 4 == 0);
    if (vec_store && !make_tensor_map(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.C, p.m, p.n, p.ldc, 32, 32,
                                      CU_TENSOR_MAP_SWIZZLE_128B)) {
        clear_error();
        vec_store = 0;
    }
    // Eight epilogue warps where the epilogue weighs most (stream-K hand-overs,
    // scalar stores), four otherwise.  Measured on GB300 (us per launch, 4 -> 8
    // warps): bf16 3300 x 3000 x 3100 (stream-K) 80.7 -> 73.0, 2000 x 2600 x 1000
    // (stream-K) 33.6 -> 29.5, 4097 x 3001 x 1023 (C unaligned) 50.5 -> 40.9,
    // TF32 3300 x 3000 x 3100 126.5 -> 119.7; but aligned C in whole tiles
    // 8192 x 8192 x 2048 198.9 -> 201.2, 4096 x 4096 x 1024 39.0 -> 40.8,
    // 2048^3 20.6 -> 21.2 and 8192^3 unchanged.
    const bool epi8 = kSK || !vec_store;
    auto kernel = epi8 ? umma_kernel<kTF32, kBKMajor, kWide, kBN, kSK, kPair, 8>
                       : umma_kernel<kTF32, kBKMajor, kWide, kBN, kSK, kPair, 4>;
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(G::SMEM));
    if (err != cudaSuccess) {
        set_error("cudaFuncSetAttribute(umma_kernel): %s", cudaGetErrorString(err));
        return err;
    }
    float* ws = nullptr;
    unsigned* flags = nullptr;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    cfg.blockDim = dim3(static_cast<unsigned>(threads_for(epi8 ? 8 : 4)), 1, 1);
    cfg.dynamicSmemBytes = G::SMEM;
    cfg.stream = p.stream;
    cfg.gridDim = dim3(static_cast<unsigned>(tiles < dev.sm_count ? tiles : dev.sm_count), 1, 1);
    cfg.attrs = attr;
    if (!kSK && kPdl) {
        // The prologue (barriers, tensor memory) overlaps the previous kernel's
        // tail; the kernel waits for it before touching global memory.
        attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
        ++cfg.numAttrs;
    }
    if (kPair) {
        // one (2 x 1) cluster per pair of tile rows, persistent over the pairs
        const int64_t pairs = static_cast<int64_t>((p.m + 2 * G::BM - 1) / (2 * G::BM)) * ((p.n + G::BN - 1) / G::BN);
        const int64_t clusters = pairs < dev.sm_count / 2 ? pairs : dev.sm_count / 2;
        cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
        attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attr[cfg.numAttrs].val.clusterDim.x = 2;
        attr[cfg.numAttrs].val.clusterDim.y = 1;
        attr[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
    if (kSK && !workspace) {
        set_error("umma_kernel: split form launched without its workspace");
        return cudaErrorInvalidValue;
    }
    if (kSK && pieces > 0) {
        // one CTA and one partial tile per piece; nothing waits on another CTA
        ws = static_cast<float*>(workspace);
        cfg.gridDim = dim3(static_cast<unsigned>(tiles * pieces), 1, 1);
        cfg.numAttrs = 0;
    } else if (kSK) {
        // one partial tile and one flag per CTA; the flags start cleared
        ws = static_cast<float*>(workspace);
        flags = reinterpret_cast<unsigned*>(ws + static_cast<size_t>(dev.sm_count) * G::BM * G::BN);
        err = cudaMemsetAsync(flags, 0, dev.sm_count * sizeof(unsigned), p.stream);
        if (err != cudaSuccess) {
            set_error("stream-K flags: %s", cudaGetErrorString(err));
            return err;
        }
        attr[0].id = cudaLaunchAttributeCooperative;   // all CTAs resident: a head may wait for its tail
        attr[0].val.cooperative = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(dev.sm_count), 1, 1);
        cfg.numAttrs = 1;
    }
    err = cudaLaunchKernelEx(&cfg, kernel, ta, tb, tc, p.C, p.ldc, p.m, p.n, p.k, vec_store, dev.status, ws, flags,
                             kSK ? pieces : 0);
    count_launch();
    if (err != cudaSuccess) {
        set_error("umma_kernel launch: %s", cudaGetErrorString(err));
        return err;
    }
    if constexpr (kSK) {
        if (pieces <= 0) return err;
        const int vec_c = (reinterpret_cast<uintptr_t>(p.C) % 16 == 0) && (p.ldc % 4 == 0);
        const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>((G::BM * G::BN / 4 + 1023) / 1024), 1);
        umma_pieces_reduce_kernel<G::BM, G::BN, G::GROUP_M><<<grid, 256, 0, p.stream>>>(
            reinterpret_cast<const float4*>(ws), p.C, p.ldc, p.m, p.n, pieces, vec_c);
        err = cudaGetLastError();
        count_launch();
        if (err != cudaSuccess) set_error("umma_pieces_reduce_kernel launch: %s", cudaGetErrorString(err));
    }
    return err;
}

// Pairs where the tile rows pair up evenly and fill at least two rounds (bf16
// 128 x 256 whole tiles).  Measured on GB300 (us per launch, single CTAs ->
// pairs): 8192 x 8192 x 2048 201.4 -> 194.6, 8192 x 8192 x 1024 120.6 -> 116.3,
// 6144 x 6144 x 2048 113.8 -> 110.8, 3000 x 6000 x 1024 39.8 -> 39.3; but 4097 x
// 3001 x 1023 (33 tile rows: one pair half empty) 50.3 -> 57.2 and 1000 x 1001 x
// 999 (32 tiles) 27.3 -> 28.6.
bool use_pairs(const Problem& p, const Device& dev) {
    const int64_t tiles_m = (p.m + 127) / 128;
    return kUsePairs && tiles_m % 2 == 0 && tile_count<false, false, false, 256>(p) >= 2 * dev.sm_count;
}

template <bool kTF32, bool kBKMajor, bool kWide, int kBN>
cudaError_t launch_any(const Problem& p, const Device& dev, void* workspace) {
    if (workspace && has_sk<kTF32, kBKMajor, kWide, kBN>(p, dev))
        return launch<kTF32, kBKMajor, kWide, kBN, true>(p, dev, workspace);
    if (workspace) {
        const int pieces = pieces_for<kTF32, kBKMajor, kWide, kBN>(p, dev);
        if (pieces > 0) return launch<kTF32, kBKMajor, kWide, kBN, true>(p, dev, workspace, pieces);
    }
    if constexpr (!kTF32 && !kBKMajor && !kWide && kBN == 256) {
        if (use_pairs(p, dev)) return launch<kTF32, kBKMajor, kWide, kBN, false, true>(p, dev, nullptr);
    }
    return launch<kTF32, kBKMajor, kWide, kBN, false>(p, dev, nullptr);
}

}  // namespace

// Wide 256 x 256 tiles need two thirds of the operand bytes per MMA cycle of
// the 128 x 256 ones, which hides the L2 latency of the TMA loads better, but
// their epilogue cannot overlap the next tile's MMAs.  Measured on GB300
// (bf16): 8192^3 1726 vs 1641 TFLOP/s, 4096^3 1308 vs 1272.  With the TMA-store
// epilogue they also win at shorter k where their rounds of CTAs are at least
// as full as those of the 128-row tiles and need no stream-K (us per launch,
// 128-row -> wide tiles; bf16 2900 x 5000 x 1030 56.8 -> 51.0, 3000 x 6000 x
// 1024 42.4 -> 39.1, 2048 x 4864 x 2048 32.7 -> 30.7, 4096 x 4096 x 2048 57.3
// -> 55.2; TF32 4096 x 4096 x 1024 59.1 -> 56.8, 2900 x 5000 x 1030 79.7 ->
// 73.6; equal fill and no gain at 4096 x 4096 x 1024 and 6144 x 3072 x 1024
// bf16).  They lose where their rounds are emptier (1536 x 9728 x 1024: 228
// wide tiles fill 3/4 of two rounds, 456 narrow ones three rounds exactly;
// bf16 30.6 -> 36.7), where they are too few (2048^3: 64 wide tiles) and
// where they would be split along k.
constexpr int kWideMinK = 3072;   // wide tiles from here on
constexpr int kWideMidK = 1024;   // from here, wide where the rounds fill at least as well

bool use_wide(const Problem& p, const Device& dev, bool tf32) {
    if (p.k >= kWideMinK) return true;
    if (p.k < kWideMidK) return false;
    const bool sk_wide = tf32 ? has_sk<true, true, true, 256>(p, dev) : has_sk<false, false, true, 256>(p, dev);
    if (sk_wide) return false;
    const int64_t G = dev.sm_count;
    // filled fraction of the occupied CTA slots (stream-K fills them all)
    auto fill = [&](int64_t tiles, int64_t bm) {
        return static_cast<double>(p.m) * p.n / (static_cast<double>((tiles + G - 1) / G * G) * bm * 256);
    };
    const double wide = fill(tf32 ? tile_count<true, true, true, 256>(p) : tile_count<false, false, true, 256>(p), 256);
    const bool sk_narrow = tf32 ? has_sk<true, true, false, 256>(p, dev) : has_sk<false, false, false, 256>(p, dev);
    const double narrow =
        sk_narrow ? 1.0 : fill(tf32 ? tile_count<true, true, false, 256>(p) : tile_count<false, false, false, 256>(p), 128);
    return wide >= narrow;
}

// Tile width of the TF32 kernels: 224 instead of 256 when 256-wide tiles
// would not take stream-K and 224-wide ones fill the occupied CTA slots
// better by more than 2 % (both are legal tcgen05 N for M = 128; the K-major
// B tile has no 128-byte-chunk constraint along N).  The filled fraction of
// the slots is also the time ratio: time ~ slots x tile area.  Measured on
// GB300 (TFLOP/s, 256 -> 224): 4096^3 679 -> 714 (304 tiles = 2 full waves,
// 96 % filled, against 84 %); 2048 x 2048 x 8192 377 -> 392.  With
// stream-K the wider tile is better (3300 x 3000 x 3100: 479 against 411).
bool tf32_narrow_n(const Problem& p, const Device& dev) {
    const bool wide = use_wide(p, dev, true);
    if (wide ? has_sk<true, true, true, 256>(p, dev) : has_sk<true, true, false, 256>(p, dev)) return false;
    if (wide ? pieces_for<true, true, true, 256>(p, dev) : pieces_for<true, true, false, 256>(p, dev)) return false;
    const int64_t bm = wide ? 256 : 128, G = dev.sm_count;
    auto fill = [&](int64_t bn) {
        const int64_t tiles = ((p.m + bm - 1) / bm) * ((p.n + bn - 1) / bn);
        const int64_t slots = (tiles + G - 1) / G * G;
        return static_cast<double>(p.m) * p.n / (static_cast<double>(slots) * bm * bn);
    };
    return fill(224) > 1.02 * fill(256);
}

uint64_t umma_workspace_bytes(const Problem& p, const Device& dev, bool tf32) {
    const bool wide = use_wide(p, dev, tf32);
    if (tf32) {
        if (tf32_narrow_n(p, dev)) return 0;   // 224-wide tiles: whole tiles only
        return wide ? workspace_bytes<true, true, true, 256>(p, dev) : workspace_bytes<true, true, false, 256>(p, dev);
    }
    return wide ? workspace_bytes<false, false, true, 256>(p, dev) : workspace_bytes<false, false, false, 256>(p, dev);
}

// The choice launch_umma makes, without launching (see tgemm_plan).
void umma_plan(const Problem& p, const Device& dev, bool tf32, bool workspace, int out[5]) {
    const bool wide = use_wide(p, dev, tf32);
    out[0] = wide ? 256 : 128;
    out[1] = 256;
    out[2] = out[3] = out[4] = 0;
    if (tf32 && tf32_narrow_n(p, dev)) {
        out[1] = 224;
        return;
    }
    const bool sk = tf32 ? (wide ? has_sk<true, true, true, 256>(p, dev) : has_sk<true, true, false, 256>(p, dev))
                         : (wide ? has_sk<false, false, true, 256>(p, dev) : has_sk<false, false, false, 256>(p, dev));
    if (workspace && sk) {
        out[2] = 1;
        return;
    }
    const int pieces = tf32 ? (wide ? pieces_for<true, true, true, 256>(p, dev) : pieces_for<true, true, false, 256>(p, dev))
                            : (wide ? pieces_for<false, false, true, 256>(p, dev)
                                    : pieces_for<false, false, false, 256>(p, dev));
    if (workspace && pieces > 0) {
        out[3] = pieces;
        return;
    }
    if (!tf32 && !wide && use_pairs(p, dev)) out[4] = 1;
}

cudaError_t launch_umma(const Problem& p, const Device& dev, bool tf32, void* workspace) {
    const bool wide = use_wide(p, dev, tf32);
    if (tf32) {
        if (tf32_narrow_n(p, dev))
            return wide ? launch<true, true, true, 224, false>(p, dev, nullptr)
                        : launch<true, true, false, 224, false>(p, dev, nullptr);
        return wide ? launch_any<true, true, true, 256>(p, dev, workspace)
                    : launch_any<true, true, false, 256>(p, dev, workspace);
    }
    return wide ? launch_any<false, false, true, 256>(p, dev, workspace)
                : launch_any<false, false, false, 256>(p, dev, workspace);
}

}  // namespace tgemm
