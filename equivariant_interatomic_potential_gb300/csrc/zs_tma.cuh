// Per-warp ring of asynchronous copies over a window of CSR positions.
//
// A warp streams the edges at CSR positions [p0, pe) in tiles of T edges
// (T <= 32, one lane per edge).  For edge e = perm[j] its lane issues
//   - one cp.async.bulk (TMA) copy of the radial row rad[e] (RadFloats
//     floats: lmax rows of 32 channels, 384 bytes at lmax 3, 16-byte
//     aligned), completion counted in bytes on the stage's mbarrier, and
//   - the 16-byte cp.async copies of the aligned span holding the coupling
//     row coup[e] (CoupRow floats, rows cld floats apart, any 4-byte
//     alignment: four or five pieces for the 15-float row), completion
//     signalled to the same mbarrier by cp.async.mbarrier.arrive.
// Tiles are issued S - 1 ahead of the one being consumed, so a warp keeps
// (S - 1) * T edges of HBM reads in flight without holding registers for
// them.  A position whose perm entry is not a valid edge id gets zero rows,
// so consumers need no branch.
//
// Every wait is bounded (zs_wait.cuh): a lost completion can never hang the
// GPU; zs_check_timeouts() and the caller's flag word report it.
#pragma once

#include "zs_common.cuh"
#include "zs_wait.cuh"

namespace zs {

constexpr int kCoupSlotFloats = 20;         // coupling slot of the 15-row ladder (coup_slot_floats(15))
// The coupling spans travel as 16-byte cp.async pieces signalled by one
// arrival per lane (default), or as one bulk copy per edge counted in bytes
// like the radial rows (ZS_RING_COUP_BULK=1: measured slower for the forward,
// 62 against 57 us on the 4096-node graph; the small bulk copies cost more
// than the pieces).
#ifndef ZS_RING_COUP_BULK
#define ZS_RING_COUP_BULK 0
#endif
constexpr bool kCoupBulk = ZS_RING_COUP_BULK != 0;
constexpr uint32_t kRingArrivals = kCoupBulk ? 1 : 33;   // the expect-tx arrival (plus one cp.async arrival per lane)

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

// Bounded wait for the phase with the given parity; false (and one timeout
// noted) when max_spins tries all fail.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t max_spins = kMaxSpins) {
    for (uint32_t i = 0; i < max_spins; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    note_timeout();
    return false;
}

__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], 4, %2;" :: "r"(dst), "l"(src), "l"(pol) : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "l"(pol) : "memory");
}

// Arrive on bar once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar, uint64_t pol) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(pol) : "memory");
}

// Coupling slot of a ring: the widest 16-byte-aligned span of a row of
// CoupRow floats that starts at any 4-byte offset, in floats (20 for the
// 15-row ladder), and the 16-byte pieces that span can take.
__host__ __device__ constexpr int coup_slot_floats(int coup_row) { return (coup_row + 3 + 3) / 4 * 4; }
__host__ __device__ constexpr int coup_max_chunks(int coup_row) { return (12 + 4 * coup_row + 15) / 16; }
static_assert(coup_slot_floats(15) == kCoupSlotFloats, "the 15-row ladder's coupling slot");

// Shared-memory layout of one warp's ring of S stages of T edges, each edge
// a radial row of RadFloats floats and a coupling row of CoupRow floats
// (defaults: the lmax = 3 ladder at C = 32).
template <int S, int T, int RadFloats = 96, int CoupRow = 15>
struct RingLayout {
    static constexpr int kRad = S * T * RadFloats * 4;                      // radial rows
    static constexpr int kCoup = S * T * coup_slot_floats(CoupRow) * 4;     // coupling spans
    static constexpr int kMeta = S * T * 8;                                 // (edge id, coupling offset)
    static constexpr int kBars = S * 8;
    static constexpr int kBytes = (kRad + kCoup + kMeta + kBars + 127) / 128 * 128;
    // copy destinations start on 16-byte boundaries, mbarriers on 8-byte ones
    static_assert(kRad % 16 == 0 && kCoup % 16 == 0 && kMeta % 8 == 0, "aligned regions");
};

// One warp's stream of tiles over [p0, pe).  kPol is the L2 policy of the
// perm entries and radial rows the ring brings in, kCoupPol that of the
// coupling spans (kL2EvictFirst for bytes read exactly once; a coupling span
// shares its 32-byte sectors with the neighbouring edges' rows, which a
// gather in CSR order reads later).
// kRadPieces: the radial rows travel as 16-byte cp.async pieces, 32 / (row
// pieces) rows per warp instruction, instead of one bulk copy per row
// (measured faster for the 128-byte rows of lmax 1 only).
// kCoupAligned: each coupling row lands at the start of its slot (4-byte
// cp.async copies by the whole warp, row offset 0) instead of as the
// 16-byte-aligned span holding it.
template <int S, int T, int kPol = kL2Normal, int RadFloats = 96, int CoupRow = 15, int kCoupPol = kPol,
          bool kRadPieces = false, bool kCoupAligned = false>
struct TileRing {
    static_assert(T >= 1 && T <= 32 && 32 % T == 0, "a tile is at most one edge per lane and divides 32");
    static_assert(RadFloats % 4 == 0, "radial rows are whole 16-byte pieces");
    static_assert(!kRadPieces || (32 % (RadFloats / 4) == 0 && T % (32 / (RadFloats / 4)) == 0),
                  "a warp instruction copies whole rows of whole steps");
    using Layout = RingLayout<S, T, RadFloats, CoupRow>;
    static constexpr int kSlot = coup_slot_floats(CoupRow);
    static constexpr int kChunks = coup_max_chunks(CoupRow);
    static constexpr uint32_t kRadBytes = RadFloats * 4;
    float* rad;        // [S][T][RadFloats]
    float* coup;       // [S][T][kSlot]
    int2* meta;        // [S][T]: x = edge id (-1 if none), y = float offset of the row in its span
    uint32_t bar0;     // shared address of the first mbarrier
    int p0, pe;
    int ntiles;        // tiles covering [p0, pe)
    int issued;        // tiles issued so far
    int consumed;      // tiles waited for so far
    // perm entries are fetched 32 positions (kPB tiles) at a time, one block
    // ahead: blk_cur holds the block of tile `issued`, blk_next the one after
    static constexpr int kPB = 32 / T;
    int blk_cur, blk_next;
    uint64_t pol;      // L2 policy of the perm entries and radial rows
    uint64_t pol_c;    // L2 policy of the coupling spans

    __device__ __forceinline__ void init(unsigned char* base, int p0_, int pe_, int lane) {
        rad = reinterpret_cast<float*>(base);
        coup = reinterpret_cast<float*>(base + Layout::kRad);
        meta = reinterpret_cast<int2*>(base + Layout::kRad + Layout::kCoup);
        bar0 = smem_u32(base + Layout::kRad + Layout::kCoup + Layout::kMeta);
        p0 = p0_;
        pe = pe_;
        ntiles = pe > p0 ? (pe - p0 + T - 1) / T : 0;
        issued = 0;
        consumed = 0;
        pol = l2_policy(kPol);
        pol_c = l2_policy(kCoupPol);
        if (lane < S) mbar_init(bar0 + 8 * lane, (kRadPieces || kCoupAligned) ? 33u : kRingArrivals);
        mbar_fence_init();
        __syncwarp();
    }

    // Narrow the range to [p0, pe_) once its end is known (the ring may have
    // been set up for a wider range so that its first perm blocks could be
    // fetched early; entries fetched past pe_ are never issued).
    __device__ __forceinline__ void set_end(int pe_) {
        pe = pe_;
        ntiles = pe > p0 ? (pe - p0 + T - 1) / T : 0;
    }

    __device__ __forceinline__ int load_block(const int32_t* __restrict__ perm, int blk, int lane) const {
        const int j = p0 + blk * 32 + lane;
        return (blk * kPB < ntiles && j < pe) ? ld_hint_i(perm + j, pol) : -1;
    }

    __device__ __forceinline__ void prefetch_perm(const int32_t* __restrict__ perm, int lane) {
        blk_cur = load_block(perm, 0, lane);
        blk_next = load_block(perm, 1, lane);
    }

    // Issue the next tile into its stage (its previous tile must be consumed).
    // Coupling row e starts at coup_g + e * cld (cld >= 15 floats, any 4-byte
    // alignment): its span is copied from the 16-byte boundary at or before it.
    __device__ __forceinline__ void issue(const int32_t* __restrict__ perm, const float* __restrict__ coup_g, int cld,
                                          const float* __restrict__ rad_g, int E, int lane) {
        if (issued >= ntiles) return;
        const int st = issued % S;
        const int sub = issued % kPB;
        const int e = __shfl_sync(0xffffffffu, blk_cur, (sub * T + lane) & 31);
        ++issued;
        if (sub == kPB - 1) {        // last tile of this block: move on, fetch the block after next
            blk_cur = blk_next;
            blk_next = load_block(perm, issued / kPB + 1, lane);
        }
        const bool valid = lane < T && (uint32_t)e < (uint32_t)E;
        const int64_t mis = (int64_t)(reinterpret_cast<uintptr_t>(coup_g) & 15u);   // bytes past a 16-byte boundary
        int64_t cstart = 0;
        int off = 0, nch = 0;
        bool tail = false;
        if (valid && !kCoupAligned) {
            const int64_t b0 = mis + (int64_t)e * cld * 4;
            cstart = b0 & ~(int64_t)15;
            off = (int)(b0 - cstart) >> 2;          // 0..3
            nch = (off * 4 + 4 * CoupRow + 15) >> 4;   // 16-byte pieces covering the row
            tail = cstart + 16 * nch > mis + ((int64_t)(E - 1) * cld + CoupRow) * 4;
        }
        const uint32_t bar = bar0 + 8 * st;
        float* cslot = coup + (st * T + lane) * kSlot;
        float* rslot = rad + (st * T + lane) * RadFloats;
        if (lane < T) {
            if (!valid || tail) {
                // rare: no edge here, or the span would run past the last row.
                // Generic-proxy writes, ordered before the consumer by the
                // syncwarps below and after the consumer's wait.
                if (valid) {
                    const float* src = coup_g + (int64_t)e * cld;
#pragma unroll
                    for (int r = 0; r < CoupRow; ++r) cslot[r] = __ldg(src + r);
                } else {
                    for (int r = 0; r < kSlot; ++r) cslot[r] = 0.f;
                    for (int c = 0; c < RadFloats; ++c) rslot[c] = 0.f;
                }
                off = 0;
            }
            meta[st * T + lane] = make_int2(valid ? e : -1, off);
        }
        const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
        const uint32_t cbytes = kCoupBulk ? __reduce_add_sync(0xffffffffu, (valid && !tail) ? 16u * nch : 0u) : 0u;
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(bar, (kRadPieces ? 0u : nvalid * kRadBytes) + cbytes);
        __syncwarp();
        if constexpr (kRadPieces) {
            constexpr int kPieces = RadFloats / 4, kRows = 32 / kPieces;
#pragma unroll
            for (int j0 = 0; j0 < T; j0 += kRows) {
                const int j = j0 + lane / kPieces, piece = lane % kPieces;
                const int ej = __shfl_sync(0xffffffffu, e, j);
                if ((uint32_t)ej < (uint32_t)E)
                    cp_async16(smem_u32(rad + (st * T + j) * RadFloats) + 16 * piece,
                               rad_g + (int64_t)ej * RadFloats + 4 * piece, pol);
            }
        }
        if constexpr (kCoupAligned) {
            // the T rows, 4 bytes a lane, each from its own first float
#pragma unroll
            for (int j = 0; j < T; ++j) {
                const int ej = __shfl_sync(0xffffffffu, e, j);
                if ((uint32_t)ej < (uint32_t)E) {
                    const uint32_t cdst = smem_u32(coup + (st * T + j) * kSlot);
#pragma unroll
                    for (int r = lane; r < CoupRow; r += 32) cp_async4(cdst + 4 * r, coup_g + (int64_t)ej * cld + r, pol_c);
                }
            }
        }
        if (valid) {
            if constexpr (!kRadPieces) bulk_g2s(smem_u32(rslot), rad_g + (int64_t)e * RadFloats, kRadBytes, bar, pol);
            if (!kCoupAligned && !tail) {
                const char* src = reinterpret_cast<const char*>(coup_g) - mis + cstart;
                const uint32_t dst = smem_u32(cslot);
                if constexpr (kCoupBulk) {
                    bulk_g2s(dst, src, 16u * nch, bar, pol_c);
                } else {
#pragma unroll
                    for (int k = 0; k < kChunks; ++k)
                        if (k < nch) cp_async16(dst + 16 * k, src + 16 * k, pol_c);
                }
            }
        }
        if constexpr (!kCoupBulk || kRadPieces || kCoupAligned) cp_async_arrive(bar);
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
    __device__ __forceinline__ void refill(const int32_t* __restrict__ perm, const float* __restrict__ coup_g, int cld,
                                           const float* __restrict__ rad_g, int E, int lane) {
        __syncwarp();
        issue(perm, coup_g, cld, rad_g, E, lane);
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
