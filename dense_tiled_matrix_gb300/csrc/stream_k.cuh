// stream_k.cuh -- the persistent schedule of the tcgen05 kernels' stream-K
// form: whole-tile rounds, then a stream-K region whose tiles may be split
// along k between two CTAs, and the flag hand-over between them.
#pragma once

#include <cstdint>

#include "device.cuh"

namespace tgemm {

// The work of one CTA of a persistent kernel, as a sequence of segments
// (tile t, k-phases [ka, kz)).  With G CTAs and T tiles, T = q G + r:
//  * r = 0, or r k-phase counts too few to share (r KT < G): q (or q + 1 for
//    CTAs b < r) whole tiles b, b + G, b + 2G, ... -- the CTAs running
//    together work on G consecutive tiles, which share A and B in L2;
//  * otherwise q - 1 such rounds, then the last G + r tiles are cut into G
//    equal runs of (tile, k-phase) iterations ("stream-K"), CTA b taking the
//    b-th run, so no SM idles in a last partial wave.  Each run is longer
//    than a tile, so a tile is shared by at most two CTAs: the first segment
//    of run b + 1 may be a tail (ka > 0) and the last segment of run b a
//    head (kz < KT) of the same tile.
struct SkPlan {
    int n_dp, t_sk0;
    int64_t v0, v1;   // stream-K run: iterations [v0, v1) of the region starting at tile t_sk0

    // allow_sk = false keeps whole tiles only (the plain round-robin).
    __device__ __forceinline__ void init(int tiles, int KT, int b, int G, bool allow_sk = true) {
        int rounds = tiles / G, r = tiles % G, tiles_sk = 0;
        if (allow_sk && r > 0 && rounds >= 1 && static_cast<int64_t>(r) * KT >= G) {
            tiles_sk = G + r;
            rounds -= 1;
            r = 0;
        }
        n_dp = rounds + (b < r ? 1 : 0);
        t_sk0 = tiles - tiles_sk;
        const int64_t U = static_cast<int64_t>(tiles_sk) * KT;
        v0 = U * b / G;
        v1 = U * (b + 1) / G;
    }
    __device__ __forceinline__ int iterations(int KT) const { return n_dp * KT + static_cast<int>(v1 - v0); }
};

// A position in a CTA's SkPlan sequence: whole tiles done, then the next
// stream-K iteration.
struct SkCursor {
    int j;
    int64_t v;
    __device__ __forceinline__ void init(const SkPlan& pl) {
        j = 0;
        v = pl.v0;
    }
    // Next segment (tile t, k-phases [ka, kz)); false when there is none.
    __device__ __forceinline__ bool next(const SkPlan& pl, int KT, int& t, int& ka, int& kz) {
        if (j < pl.n_dp) {
            t = blockIdx.x + j * gridDim.x;
            ka = 0;
            kz = KT;
            ++j;
            return true;
        }
        if (v >= pl.v1) return false;
        const int64_t q = v / KT;
        t = pl.t_sk0 + static_cast<int>(q);
        ka = static_cast<int>(v - q * KT);
        kz = static_cast<int>(min(static_cast<int64_t>(KT), ka + (pl.v1 - v)));
        v += kz - ka;
        return true;
    }
};

// The flag hand-over between the tail and the head of a split tile.
__device__ __forceinline__ uint32_t ld_acquire_u32(const unsigned* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(unsigned* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Waits (bounded, like the mbarrier waits) until *flag != 0.
__device__ __forceinline__ bool wait_flag(const unsigned* flag, uint32_t* status) {
    if (ld_acquire_u32(flag)) return true;
    const uint64_t start = global_timer_ns();
    while (!ld_acquire_u32(flag)) {
        if (global_timer_ns() - start > kWaitLimitNs) {
            atomicCAS(status, 0u, kStatusTimeout);
            return false;
        }
        __nanosleep(100);
    }
    return true;
}

}  // namespace tgemm
