// Per-warp TMA ring over a window of CSR positions (sm_90+ bulk copies,
// used here on sm_103a).
//
// A warp streams the edges at CSR positions [p0, p1) in tiles of 32.  For
// each edge e = perm[j] of a tile, one lane issues two cp.async.bulk copies
// into the tile's shared-memory stage: the radial row rad[e] (3*32 floats,
// 384 bytes) and the 16-byte-aligned span holding the coupling row coup[e]
// (60 bytes inside 64 or 80 bytes).  Completion is counted in bytes on one
// mbarrier per stage.  Tiles are issued kStages - 1 ahead of the one being
// consumed, so each warp keeps about 15 KB of HBM reads in flight with no
// registers held for them.
//
// Every wait is bounded: after kMaxSpins unsuccessful tries the wait records
// a timeout in g_zs_timeouts and returns, so a lost completion can never hang
// the GPU; zs_check_timeouts() reports it.
#pragma once

#include "zs_common.cuh"

namespace zs {

// Count of bounded waits that ran out in this translation unit's kernels.
static __device__ unsigned int g_zs_timeouts;

// Host: read and clear this translation unit's count (synchronises the device).
static inline unsigned int take_timeouts_local() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_zs_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_zs_timeouts, &zero, sizeof(zero));
    return v;
}

constexpr int kTileEdges = 32;
constexpr int kRadRowBytes = 3 * 32 * 4;    // 384
constexpr int kCoupSlotFloats = 20;         // 80 bytes: the widest aligned span of one coupling row
constexpr uint32_t kMaxSpins = 1u << 22;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < kMaxSpins; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    atomicAdd(&g_zs_timeouts, 1u);
    return false;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// Shared-memory layout of one warp's ring.
template <int S>
struct RingLayout {
    static constexpr int kRad = S * kTileEdges * kRadRowBytes;              // radial rows
    static constexpr int kCoup = S * kTileEdges * kCoupSlotFloats * 4;      // coupling spans
    static constexpr int kMeta = S * kTileEdges * 8;                        // (edge id, coupling offset)
    static constexpr int kBars = S * 8;
    static constexpr int kBytes = (kRad + kCoup + kMeta + kBars + 127) / 128 * 128;
};

// One warp's stream of tiles over [p0, p1).
template <int S>
struct TileRing {
    float* rad;        // [S][32][96]
    float* coup;       // [S][32][20]
    int2* meta;        // [S][32]: x = edge id (-1 if none), y = float offset of the row in its span
    uint32_t bar0;     // shared address of the first mbarrier
    int64_t p0, p1;
    int ntiles;        // tiles covering [p0, p1)
    int issued;        // tiles issued so far
    int consumed;      // tiles waited for so far
    int pf;            // this lane's perm entry for tile `issued` (prefetched)

    __device__ __forceinline__ void init(unsigned char* base, int64_t p0_, int64_t p1_, int lane) {
        rad = reinterpret_cast<float*>(base);
        coup = reinterpret_cast<float*>(base + RingLayout<S>::kRad);
        meta = reinterpret_cast<int2*>(base + RingLayout<S>::kRad + RingLayout<S>::kCoup);
        bar0 = smem_u32(base + RingLayout<S>::kRad + RingLayout<S>::kCoup + RingLayout<S>::kMeta);
        p0 = p0_;
        p1 = p1_;
        ntiles = p1 > p0 ? (int)((p1 - p0 + kTileEdges - 1) / kTileEdges) : 0;
        issued = 0;
        consumed = 0;
        if (lane < S) mbar_init(bar0 + 8 * lane, 1);
        mbar_fence_init();
        __syncwarp();
    }

    __device__ __forceinline__ void prefetch_perm(const int32_t* __restrict__ perm, int lane) {
        const int64_t j = p0 + (int64_t)issued * kTileEdges + lane;
        pf = (issued < ntiles && j < p1) ? ld_stream_i(perm + j) : -1;
    }

    // Issue the next tile into its stage (its previous tile must be consumed).
    __device__ __forceinline__ void issue(const int32_t* __restrict__ perm, const float* __restrict__ coup_g,
                                          const float* __restrict__ rad_g, int64_t E, int lane) {
        if (issued >= ntiles) return;
        const int k = issued;
        const int st = k % S;
        const int64_t j = p0 + (int64_t)k * kTileEdges + lane;
        int e = pf;
        if ((uint32_t)e >= (uint64_t)E) e = -1;
        // next tile's perm entries, consumed at the next issue
        ++issued;
        prefetch_perm(perm, lane);
        int off = 0;
        uint32_t cbytes = 0;
        int64_t cstart = 0;
        bool plain = false;
        if (e >= 0 && j < p1) {
            const int64_t b0 = (int64_t)e * 60;
            cstart = b0 & ~(int64_t)15;
            const int64_t cend = (b0 + 60 + 15) & ~(int64_t)15;
            off = (int)((b0 - cstart) >> 2);
            if (cend <= E * 60) {
                cbytes = (uint32_t)(cend - cstart);
            } else {
                plain = true;   // span would run past the end of coup: load the row directly
            }
        } else {
            e = -1;
        }
        const uint32_t mine = (e >= 0 ? (uint32_t)kRadRowBytes : 0u) + cbytes;
        const uint32_t total = __reduce_add_sync(0xffffffffu, mine);
        const uint32_t bar = bar0 + 8 * st;
        float* cslot = coup + ((size_t)st * kTileEdges + lane) * kCoupSlotFloats;
        if (plain) {
            off = 0;
            const float* src = coup_g + (int64_t)e * 15;
#pragma unroll
            for (int r = 0; r < 15; ++r) cslot[r] = __ldg(src + r);
        }
        meta[st * kTileEdges + lane] = make_int2(e, off);
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(bar, total);
        __syncwarp();
        if (e >= 0) {
            bulk_g2s(smem_u32(rad + ((size_t)st * kTileEdges + lane) * 96), rad_g + (int64_t)e * 96,
                     kRadRowBytes, bar);
            if (cbytes) bulk_g2s(smem_u32(cslot), reinterpret_cast<const char*>(coup_g) + cstart, cbytes, bar);
        }
    }

    // Wait for the next tile in order; returns its stage.
    __device__ __forceinline__ int acquire() {
        const int k = consumed++;
        const int st = k % S;
        mbar_wait(bar0 + 8 * st, (uint32_t)((k / S) & 1));
        __syncwarp();
        return st;
    }

    // The last acquired tile is finished: reuse its stage for the next tile.
    __device__ __forceinline__ void refill(const int32_t* __restrict__ perm, const float* __restrict__ coup_g,
                                           const float* __restrict__ rad_g, int64_t E, int lane) {
        __syncwarp();
        issue(perm, coup_g, rad_g, E, lane);
    }

    // Wait for every issued tile, so the ring's memory may be reused.
    __device__ __forceinline__ void drain() {
        while (consumed < issued) {
            const int st = consumed % S;
            mbar_wait(bar0 + 8 * st, (uint32_t)((consumed / S) & 1));
            ++consumed;
        }
        __syncwarp();
    }
};

}  // namespace zs
