// Forward zonal scatter (lmax = 3 shown; the ladders lmax = 1..5 the same way
// with D = (lmax+1)^2 rows):
//   out[n,0,:] = 0,  out[n,1+r,c] = sum over n's CSR positions j (in order)
//                                   of coup[e,r] * rad[e,slot(r),c], e = perm[j]
// (deepmd-kit pull request "fused Triton zonal scatter for the GIE head",
// section "What", forward bullet: a node-parallel walk of the stable
// destination CSR, message accumulated in registers, the (E,15,C) message
// never materialised, padded (N,16,C) output with a zero scalar row).  An
// optional per-node factor (the degree normalisation the pages apply after
// the operator) is applied as each node is written.
//
// Work split.  The pages use one program per node; on a 152-SM part with a
// skewed in-degree (one node can own 1/6 of all edges) that leaves most SMs
// idle while one streams.  Here every warp owns a fixed window of CSR
// POSITIONS instead, so all warps move the same number of bytes whatever the
// degree distribution:
//   * a node that lies inside one warp's window is summed in CSR order in
//     registers and written directly;
//   * a node cut by window edges is summed piecewise: the pieces inside one
//     CTA are added in shared memory in window order, and a node that crosses
//     CTA windows leaves one partial per CTA in the workspace.  On the C == 32
//     path the CTA where such a node ends adds the earlier CTAs' partials in
//     CTA order once their flags say they are written (every CTA of that
//     single-wave grid is resident, and a CTA only waits for lower ones);
//     the per-channel path leaves that to a second small kernel.
// Every sum is therefore formed in one fixed order: run to run bitwise
// deterministic, no floating-point atomics.
#include <mutex>

#include "zs_common.cuh"
#include "zs_tma.cuh"

#include <type_traits>

namespace zs {
namespace {

constexpr int kFwdWarps = 8;
constexpr int kFwdThreads = kFwdWarps * 32;
// C == 32 path: warps per CTA (one CTA per SM), ring stages and edges per tile.
#ifndef ZS_FWD_WARPS
#define ZS_FWD_WARPS 16
#endif
#ifndef ZS_FWD_STAGES
#define ZS_FWD_STAGES 2
#endif
#ifndef ZS_FWD_TILE
#define ZS_FWD_TILE 16
#endif
constexpr int kTmaWarps = ZS_FWD_WARPS;
constexpr int kTmaStages = ZS_FWD_STAGES;
constexpr int kTile = ZS_FWD_TILE;
// L2 policies of the forward's ring: radial rows (and perm) are read once,
// evict-first, so the stream does not push the rest of L2 out; a coupling
// row shares its 32-byte sectors with its neighbours in edge order, which the
// CSR-order gather reaches later, so coupling spans keep the normal policy
// (evict-first on them measured slower).
#ifndef ZS_FWD_RAD_POL
#define ZS_FWD_RAD_POL kL2EvictFirst
#endif
#ifndef ZS_FWD_COUP_POL
#define ZS_FWD_COUP_POL kL2Normal
#endif
constexpr int kFwdRadPol = ZS_FWD_RAD_POL;
constexpr int kFwdCoupPol = ZS_FWD_COUP_POL;
constexpr int kGenWin = 256;                   // CSR positions per warp (per-channel path)
constexpr int kC32 = 32;
constexpr int kNodeFloats32 = kD * kC32;       // 512 floats per node at C = 32
constexpr int kPartFloats32 = kRows * kC32;    // 480 floats per partial at C = 32
constexpr unsigned kFull = 0xffffffffu;

// --------------------------------------------------------------------------
// C == 32 path.  Lane layout: group g = lane/8 owns zonal rows 4g..4g+3 (row
// 15 is padding), quad q = lane%8 owns channels 4q..4q+3.  Rows 4g..4g+2
// share one radial slot; row 4g+3 uses slot 1 for g == 0 (row 3 is the first
// degree-2 row) and the group's own slot otherwise.
// --------------------------------------------------------------------------

struct Lane32 {
    int lane, g, q, slo, shi;
    __device__ __forceinline__ explicit Lane32(int l) : lane(l), g(l >> 3), q(l & 7) {
        slo = g == 0 ? 0 : (g == 1 ? 1 : 2);
        shi = g == 0 ? 1 : slo;
    }
};

// Write rows 1..15 of one node from acc, and the zero scalar row.
__device__ __forceinline__ void store_node32(float* __restrict__ node, const float4 acc[4], const Lane32& L) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = 4 * L.g + i;
        if (r < kRows) *reinterpret_cast<float4*>(node + (1 + r) * kC32 + 4 * L.q) = acc[i];
    }
    if (L.g == 3) *reinterpret_cast<float4*>(node + 4 * L.q) = make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ void store_part32(float* __restrict__ part, const float4 acc[4], const Lane32& L) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = 4 * L.g + i;
        if (r < kRows) *reinterpret_cast<float4*>(part + r * kC32 + 4 * L.q) = acc[i];
    }
}

__device__ __forceinline__ void load_part32(const float* __restrict__ part, float4 acc[4], const Lane32& L) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = 4 * L.g + i;
        acc[i] = r < kRows ? *reinterpret_cast<const float4*>(part + r * kC32 + 4 * L.q)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

__device__ __forceinline__ void zero_node32(float* __restrict__ node, int lane) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
        *reinterpret_cast<float4*>(node + 4 * (lane + 32 * k)) = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Where a finished node goes.  out gets scale[n] times the node's sum (the
// sum itself when scale is null: the plain operator), raw the unscaled sum
// when it is not null.  Nodes without edges are zero in both, whatever
// their scale, and the scalar row is always zero.
struct NodeOut {
    float* out;
    float* raw;
    const float* scale;
};

__device__ __forceinline__ void put_node32(const NodeOut& o, int n, const float4 acc[4], const Lane32& L) {
    const int64_t at = (int64_t)n * kNodeFloats32;
    if (o.raw) store_node32(o.raw + at, acc, L);
    if (o.scale) {
        const float sc = __ldg(o.scale + n);
        float4 t[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) t[i] = make_float4(acc[i].x * sc, acc[i].y * sc, acc[i].z * sc, acc[i].w * sc);
        store_node32(o.out + at, t, L);
    } else {
        store_node32(o.out + at, acc, L);
    }
}

__device__ __forceinline__ void zero_put32(const NodeOut& o, int n, int lane) {
    zero_node32(o.out + (int64_t)n * kNodeFloats32, lane);
    if (o.raw) zero_node32(o.raw + (int64_t)n * kNodeFloats32, lane);
}

// Add the message of the edge at tile slot j of stage st.  Rows of
// positions without an edge are zero in the ring, so there is no branch.
struct TileView {
    const float* ra;    // radial quad of slot slo of edge 0
    const float* rb;    // radial quad of slot shi of edge 0
    const float* cp;    // coupling span of edge 0, offset to this group's rows
    const int2* mt;     // (edge id, row offset in span) per edge
};

__device__ __forceinline__ void add_edge32(const TileView& v, int j, float4 acc[4]) {
    const float4 a = *reinterpret_cast<const float4*>(v.ra + j * 96);
    const float4 b = *reinterpret_cast<const float4*>(v.rb + j * 96);
    const float* crow = v.cp + j * kCoupSlotFloats + v.mt[j].y;
    acc[0] = f4_fma(crow[0], a, acc[0]);
    acc[1] = f4_fma(crow[1], a, acc[1]);
    acc[2] = f4_fma(crow[2], a, acc[2]);
    acc[3] = f4_fma(crow[3], b, acc[3]);   // row 15 of group 3 is padding, never stored
}

__device__ __forceinline__ void load_part32_cg(const float* __restrict__ part, float4 acc[4], const Lane32& L) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = 4 * L.g + i;
        acc[i] = r < kRows ? __ldcg(reinterpret_cast<const float4*>(part + r * kC32 + 4 * L.q))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Lane layouts of the single-wave forward at C = 32.  A layout owns the
// per-lane accumulator of one node and knows how to add an edge from the
// ring, finish a node and move partial sums.
//
// QuadLayout (lmax = 3): group g = lane/8 owns zonal rows 4g..4g+3 (row 15 is
// padding), quad q = lane%8 channels 4q..4q+3: per edge 2 LDS.128 + 4 LDS.32
// + 16 FFMA per lane.
struct QuadLayout {
    static constexpr int kTileEdges = kTile;
    static constexpr int kRadFloats = 3 * kC32, kCoupRow = kRows, kPartFloats = kPartFloats32;
    static constexpr int kSlot = coup_slot_floats(kCoupRow);
    struct Acc {
        float4 v[4];
    };
    Lane32 L;
    const float *rb, *hb, *cb;
    __device__ __forceinline__ explicit QuadLayout(int lane) : L(lane) {}
    template <class Ring>
    __device__ __forceinline__ void bind(const Ring& ring) {
        rb = ring.rad + L.slo * kC32 + 4 * L.q;
        hb = ring.rad + L.shi * kC32 + 4 * L.q;
        cb = ring.coup + 4 * L.g;
    }
    template <int T>
    __device__ __forceinline__ TileView view(int st, const int2* meta) const {
        return TileView{rb + st * T * kRadFloats, hb + st * T * kRadFloats, cb + st * T * kSlot, meta + st * T};
    }
    __device__ __forceinline__ static void zero(Acc& a) {
#pragma unroll
        for (int i = 0; i < 4; ++i) a.v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __device__ __forceinline__ void add(const TileView& v, int j, Acc& a) const { add_edge32(v, j, a.v); }
    __device__ __forceinline__ void put(const NodeOut& o, int n, const Acc& a) const { put_node32(o, n, a.v, L); }
    __device__ __forceinline__ void zero_node(const NodeOut& o, int n) const { zero_put32(o, n, L.lane); }
    __device__ __forceinline__ void store(float* p, const Acc& a) const { store_part32(p, a.v, L); }
    __device__ __forceinline__ void load(const float* p, Acc& a) const { load_part32(p, a.v, L); }
    __device__ __forceinline__ void load_cg(const float* p, Acc& a) const { load_part32_cg(p, a.v, L); }
    __device__ __forceinline__ static void add_to(Acc& a, const Acc& b) {
#pragma unroll
        for (int i = 0; i < 4; ++i) a.v[i] = f4_add(a.v[i], b.v[i]);
    }
};

// ChanLayout (any ladder): lane = channel, all R rows per lane; per edge
// lmax LDS.32 of radial values, R broadcast LDS.32 of coupling values (at
// lmax 4, (R + 6) / 4 broadcast LDS.128) and R FFMA per lane.  Node rows are
// written as 128-byte lines.
template <int LM>
struct ChanLayout {
    // tiles of 16 edges for the small rows of lmax 1 and 2 (8 and 32 were
    // slower); 8 for lmax 4 and 5, whose rings then fit more warps (lmax 4:
    // 16 warps of 8-edge tiles 77 us against 11 of 16-edge tiles 84 us)
    static constexpr int kTileEdges = LM <= 3 ? 16 : 8;
    // lmax 2's 256-byte rows as 16-byte pieces, two rows per warp instruction
    // (43.7 -> 42.1 us; lmax 4's 512-byte rows gained nothing, lmax 3 and 5
    // lost with them)
    static constexpr bool kRadPieces = LM == 2;
    static constexpr int R = Ladder<LM>::R, D = Ladder<LM>::D;
    static constexpr int kRadFloats = LM * kC32, kCoupRow = R, kPartFloats = R * kC32, kNodeFloats = D * kC32;
    static constexpr int kSlot = coup_slot_floats(kCoupRow);
    struct Acc {
        float v[R];
    };
    struct View {
        const float* ra;    // radial row of edge 0 of the stage, at this lane's channel
        const float* cp;    // coupling span of edge 0 of the stage
        const int2* mt;
    };
    int lane;
    const float *rb, *cb;
    __device__ __forceinline__ explicit ChanLayout(int l) : lane(l) {}
    template <class Ring>
    __device__ __forceinline__ void bind(const Ring& ring) {
        rb = ring.rad + lane;
        cb = ring.coup;
    }
    template <int T>
    __device__ __forceinline__ View view(int st, const int2* meta) const {
        return View{rb + st * T * kRadFloats, cb + st * T * kSlot, meta + st * T};
    }
    __device__ __forceinline__ static void zero(Acc& a) {
#pragma unroll
        for (int r = 0; r < R; ++r) a.v[r] = 0.f;
    }
    // At lmax 4 and 5 the coupling span is read as kSlot / 4 broadcast
    // 16-byte loads; the row starts O floats into it (O = 0..3, the same for
    // every lane), so the FMAs are unrolled once per O and picked by a
    // warp-uniform switch.  Each accumulator still takes one FMA per edge in
    // edge order.  Measured on the n4096 graph: lmax 4 98 -> 88 us, lmax 5
    // (12 warps instead of 16) 128 -> 111 us: its shared-memory instruction
    // queue had been the limit; lmax 2 unchanged and lmax 1 slower (3 rows do
    // not pay for the switch), so those keep one broadcast LDS.32 per row.
    static constexpr bool kVecCoup = R >= 16;
    // and their ring lands each coupling row at the start of its slot (4-byte
    // copies), so the row offset is 0 and no switch is needed: lmax 4 76.6 ->
    // 73.4 us, lmax 5 110.8 -> 106.6 us
    static constexpr bool kCoupAligned = kVecCoup;
    // lmax 5 holds 35 accumulators, the node's first piece and the 40-float
    // coupling span: 163 registers, so 12 warps (at 16 the 128-register cap
    // spills)
    static constexpr int kMaxWarps = LM == 5 ? 12 : 16;
    template <int O>
    __device__ __forceinline__ static void fma_rows(const float (&cf)[kSlot], const float (&rv)[LM], Acc& a) {
#pragma unroll
        for (int r = 0; r < R; ++r) a.v[r] = fmaf(cf[O + r], rv[ladder_slot(r)], a.v[r]);
    }
    __device__ __forceinline__ void add(const View& v, int j, Acc& a) const {
        float rv[LM];
#pragma unroll
        for (int k = 0; k < LM; ++k) rv[k] = v.ra[j * kRadFloats + k * kC32];
        if constexpr (kVecCoup) {
            const float4* cq = reinterpret_cast<const float4*>(v.cp + j * kSlot);
            float cf[kSlot];
#pragma unroll
            for (int k = 0; k < kSlot / 4; ++k) {
                const float4 q = cq[k];
                cf[4 * k] = q.x;
                cf[4 * k + 1] = q.y;
                cf[4 * k + 2] = q.z;
                cf[4 * k + 3] = q.w;
            }
            if constexpr (kCoupAligned) {
                fma_rows<0>(cf, rv, a);
            } else {
                switch (v.mt[j].y) {
                    case 0: fma_rows<0>(cf, rv, a); break;
                    case 1: fma_rows<1>(cf, rv, a); break;
                    case 2: fma_rows<2>(cf, rv, a); break;
                    default: fma_rows<3>(cf, rv, a); break;
                }
            }
        } else {
            const float* cr = v.cp + j * kSlot + v.mt[j].y;
#pragma unroll
            for (int r = 0; r < R; ++r) a.v[r] = fmaf(cr[r], rv[ladder_slot(r)], a.v[r]);
        }
    }
    __device__ __forceinline__ void put(const NodeOut& o, int n, const Acc& a) const {
        const int64_t at = (int64_t)n * kNodeFloats + lane;
        const float sc = o.scale ? __ldg(o.scale + n) : 1.f;
        o.out[at] = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) o.out[at + (1 + r) * kC32] = o.scale ? a.v[r] * sc : a.v[r];
        if (o.raw) {
            o.raw[at] = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) o.raw[at + (1 + r) * kC32] = a.v[r];
        }
    }
    __device__ __forceinline__ void zero_node(const NodeOut& o, int n) const {
#pragma unroll
        for (int i = 0; i < D; ++i) o.out[(int64_t)n * kNodeFloats + i * kC32 + lane] = 0.f;
        if (o.raw)
#pragma unroll
            for (int i = 0; i < D; ++i) o.raw[(int64_t)n * kNodeFloats + i * kC32 + lane] = 0.f;
    }
    __device__ __forceinline__ void store(float* p, const Acc& a) const {
#pragma unroll
        for (int r = 0; r < R; ++r) p[r * kC32 + lane] = a.v[r];
    }
    __device__ __forceinline__ void load(const float* p, Acc& a) const {
#pragma unroll
        for (int r = 0; r < R; ++r) a.v[r] = p[r * kC32 + lane];
    }
    __device__ __forceinline__ void load_cg(const float* p, Acc& a) const {
#pragma unroll
        for (int r = 0; r < R; ++r) a.v[r] = __ldcg(p + r * kC32 + lane);
    }
    __device__ __forceinline__ static void add_to(Acc& a, const Acc& b) {
#pragma unroll
        for (int r = 0; r < R; ++r) a.v[r] += b.v[r];
    }
};

// EdgeQuadLayout (small ladders): group g = lane/8 takes edge j + g of each
// step of four edges, quad q = lane%8 channels 4q..4q+3 of all R rows.  Per
// four edges a lane issues lmax LDS.128 of its edge's radial row, R LDS.32 of
// its coupling row and 4R FFMA, against 4 x (lmax + R) loads and 4R FFMA
// with lane = channel.  Each group sums every fourth edge of a node; the four
// sums are added across the groups (XOR 8, then XOR 16: the same bits in
// every lane) when the node is written or its partial stored.  A loaded
// partial sits in group 0 with zeros in the other groups, so that it takes
// the same reduction exactly.
template <int LM>
struct EdgeQuadLayout {
    static constexpr int kStep = 4;
    static constexpr int kTileEdges = 16;
    // the 128-byte rows of lmax 1 as 16-byte pieces, four rows per warp
    // instruction (30.8 -> 24.4 us against one bulk copy per row)
    static constexpr bool kRadPieces = LM == 1;
    // lmax 2 would hold 8 float4 accumulators twice: 165 registers at 12
    // warps, and no faster than ChanLayout<2> (43.7 against 43.5 us), which
    // it keeps; this layout serves lmax 1
    static constexpr int kMaxWarps = LM >= 2 ? 12 : 16;
    static constexpr int R = Ladder<LM>::R, D = Ladder<LM>::D;
    static constexpr int kRadFloats = LM * kC32, kCoupRow = R, kPartFloats = R * kC32, kNodeFloats = D * kC32;
    static constexpr int kSlot = coup_slot_floats(kCoupRow);
    struct Acc {
        float4 v[R];
    };
    struct View {
        const float* ra;    // radial rows of the stage, at this lane's channel quad
        const float* cp;    // coupling spans of the stage
        const int2* mt;
    };
    int lane, g, q;
    const float *rb, *cb;
    __device__ __forceinline__ explicit EdgeQuadLayout(int l) : lane(l), g(l >> 3), q(l & 7) {}
    template <class Ring>
    __device__ __forceinline__ void bind(const Ring& ring) {
        rb = ring.rad + 4 * q;
        cb = ring.coup;
    }
    template <int T>
    __device__ __forceinline__ View view(int st, const int2* meta) const {
        return View{rb + st * T * kRadFloats, cb + st * T * kSlot, meta + st * T};
    }
    __device__ __forceinline__ static void zero(Acc& a) {
#pragma unroll
        for (int r = 0; r < R; ++r) a.v[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // Edges j .. j + 3 of the tile; group g adds edge j + g if it is before stop.
    __device__ __forceinline__ void add_step(const View& v, int j, int stop, Acc& a) const {
        const int e = j + g;
        if (e < stop) {
            float4 rv[LM];
#pragma unroll
            for (int l = 0; l < LM; ++l) rv[l] = *reinterpret_cast<const float4*>(v.ra + e * kRadFloats + l * kC32);
            const float* cr = v.cp + e * kSlot + v.mt[e].y;
#pragma unroll
            for (int r = 0; r < R; ++r) a.v[r] = f4_fma(cr[r], rv[ladder_slot(r)], a.v[r]);
        }
    }
    __device__ __forceinline__ static Acc reduce(const Acc& a) {
        Acc s;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float4 x = f4_add(a.v[r], f4_shfl_xor(a.v[r], 8));
            s.v[r] = f4_add(x, f4_shfl_xor(x, 16));
        }
        return s;
    }
    __device__ __forceinline__ void put(const NodeOut& o, int n, const Acc& a) const {
        const Acc s = reduce(a);
        const int64_t at = (int64_t)n * kNodeFloats + 4 * q;
        const float sc = o.scale ? __ldg(o.scale + n) : 1.f;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < R; ++r)
            if ((r & 3) == g) {
                const float4 x = s.v[r];
                *reinterpret_cast<float4*>(o.out + at + (1 + r) * kC32) =
                    o.scale ? make_float4(x.x * sc, x.y * sc, x.z * sc, x.w * sc) : x;
                if (o.raw) *reinterpret_cast<float4*>(o.raw + at + (1 + r) * kC32) = x;
            }
        if (g == 3) {   // the zero scalar row
            *reinterpret_cast<float4*>(o.out + at) = z;
            if (o.raw) *reinterpret_cast<float4*>(o.raw + at) = z;
        }
    }
    __device__ __forceinline__ void zero_node(const NodeOut& o, int n) const {
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = lane; i < D * kC32 / 4; i += 32) {
            reinterpret_cast<float4*>(o.out + (int64_t)n * kNodeFloats)[i] = z;
            if (o.raw) reinterpret_cast<float4*>(o.raw + (int64_t)n * kNodeFloats)[i] = z;
        }
    }
    __device__ __forceinline__ void store(float* p, const Acc& a) const {
        const Acc s = reduce(a);
#pragma unroll
        for (int r = 0; r < R; ++r)
            if ((r & 3) == g) *reinterpret_cast<float4*>(p + r * kC32 + 4 * q) = s.v[r];
    }
    __device__ __forceinline__ void load(const float* p, Acc& a) const {
#pragma unroll
        for (int r = 0; r < R; ++r)
            a.v[r] = g == 0 ? *reinterpret_cast<const float4*>(p + r * kC32 + 4 * q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __device__ __forceinline__ void load_cg(const float* p, Acc& a) const {
#pragma unroll
        for (int r = 0; r < R; ++r)
            a.v[r] = g == 0 ? __ldcg(reinterpret_cast<const float4*>(p + r * kC32 + 4 * q))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __device__ __forceinline__ static void add_to(Acc& a, const Acc& b) {
#pragma unroll
        for (int r = 0; r < R; ++r) a.v[r] = f4_add(a.v[r], b.v[r]);
    }
};

// Whether a layout's ring puts each coupling row at the start of its slot.
template <class P, class = void>
struct CoupAlignedOf { static constexpr bool value = false; };
template <class P>
struct CoupAlignedOf<P, std::void_t<decltype(P::kCoupAligned)>> { static constexpr bool value = P::kCoupAligned; };

// Whether a layout's ring copies the radial rows as 16-byte pieces.
template <class P, class = void>
struct RadPiecesOf { static constexpr bool value = false; };
template <class P>
struct RadPiecesOf<P, std::void_t<decltype(P::kRadPieces)>> { static constexpr bool value = P::kRadPieces; };

// Edges a layout adds per call: 4 for EdgeQuadLayout (add_step), else 1 (add).
template <class P, class = void>
struct StepOf { static constexpr int value = 1; };
template <class P>
struct StepOf<P, std::void_t<decltype(P::kStep)>> { static constexpr int value = P::kStep; };

// A node whose partials come from at least this many earlier CTAs is
// combined by all warps of the CTA where it ends.
constexpr int kSplitPartials = 8;

// Single-wave forward at C = 32, fed by TMA rings.  W warps per CTA, one CTA
// per SM; warp gw owns the window [gw*KW, gw*KW + KW) of CSR positions and
// walks it in position order, closing a node when its last position is
// reached; P is the lane layout.
template <int W, int S, int T, class P>
__global__ void __launch_bounds__(W * 32, 1)
fwd_tma(const float* __restrict__ coup, int cld, const float* __restrict__ rad,
        const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ perm,
        int E, int32_t N, int KW, int Wtot, NodeOut o, float* __restrict__ cta_part,
        uint64_t* __restrict__ flags, uint64_t salt) {
    using Ring = TileRing<S, T, kFwdRadPol, P::kRadFloats, P::kCoupRow, kFwdCoupPol, RadPiecesOf<P>::value,
                          CoupAlignedOf<P>::value>;
    using Layout = typename Ring::Layout;
    using Acc = typename P::Acc;
    static_assert(2 * P::kPartFloats * 4 <= Layout::kRad + Layout::kCoup, "two partials fit a warp's idle ring");
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int sp_node[W][2];
    __shared__ int2 sp_rows[W][2];                     // (row_ptr[m], row_ptr[m + 1]) of sp_node's nodes
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    P lay(lane);
    const int gw = blockIdx.x * W + warp;
    const bool active = gw < Wtot;
    pdl_wait();
    pdl_trigger();
    const int p0 = active ? (int)imin<int64_t>((int64_t)gw * KW, E) : E;
    const int p1 = active ? (int)imin<int64_t>((int64_t)p0 + KW, E) : E;
    const bool is_last = gw == Wtot - 1;
    // Start-up.  A dependent global load costs several hundred nanoseconds,
    // so the independent ones go out together: the end of the valid
    // positions (vend), the first perm blocks and the first round of the
    // search for the window's first node; the ring's first tiles are issued
    // as soon as perm arrives, while the search finishes.
    const int vend = __ldg(row_ptr + N);              // positions from vend on hold no node
    WarpSearch ns;
    if (active) ns.begin(row_ptr, N + 1, p0, lane);
    Ring ring;
    ring.init(smem + (size_t)warp * Layout::kBytes, p0, p1, lane);
    if (active) ring.prefetch_perm(perm, lane);
    const int pe = imax(p0, imin(p1, vend));
    ring.set_end(active ? pe : p0);
    lay.bind(ring);
    if (lane < 2) sp_node[warp][lane] = -1;
    __syncwarp();

    Acc acc0, acc;
    P::zero(acc0);
    P::zero(acc);
    bool have0 = false, have1 = false;
    if (active) {
        ns.resolve();
        ns.load(row_ptr, lane);
#pragma unroll
        for (int i = 0; i < S; ++i) ring.issue(perm, coup, cld, rad, E, lane);
        while (!ns.done()) {
            ns.resolve();
            ns.load(row_ptr, lane);
        }
        // current node n covers positions [a, b); empty nodes this window owns
        // (those starting in it, or all trailing ones for the last window) are zeroed
        // a = row_ptr[n], b = row_ptr[n+1]; c = row_ptr[n+2] is fetched one node ahead.
        // The first node is n_lb (first row_ptr entry >= p0) or the one before it;
        // row_ptr[n_lb - 1 .. n_lb + 2] arrive in one round (lane k holds entry n_lb - 1 + k).
        const int n_lb = ns.lo;
        const int ik = n_lb - 1 + lane;
        const int rk = (lane < 4 && ik >= 0 && ik <= N) ? __ldg(row_ptr + ik) : 0;
        const int r0 = __shfl_sync(0xffffffffu, rk, 0), r1 = __shfl_sync(0xffffffffu, rk, 1);
        const int r2 = __shfl_sync(0xffffffffu, rk, 2), r3 = __shfl_sync(0xffffffffu, rk, 3);
        const bool back = n_lb >= 1 && n_lb <= N && (int64_t)r1 > p0;
        int n = back ? n_lb - 1 : n_lb;
        int a = n < N ? (back ? r0 : r1) : 0;
        int b = n < N ? (back ? r1 : r2) : 0;
        int c = n + 2 <= N ? (back ? r2 : r3) : 0;
        auto step = [&]() {
            ++n;
            a = b;
            b = c;
            c = n + 2 <= N ? __ldg(row_ptr + n + 2) : 0;
        };
        auto advance = [&]() {
            while (n < N && a == b && (a < p1 || is_last)) {
                lay.zero_node(o, n);
                step();
            }
        };
        advance();
        for (int k = 0; k < ring.ntiles; ++k) {
            const int st = ring.acquire();
            const auto v = lay.template view<T>(st, ring.meta);
            const int tb = p0 + k * T;
            const int jt = imin(T, pe - tb);
            int j = 0;
            while (j < jt) {
                const int stop = imin(b - tb, jt);   // the current node covers position tb + j
                if constexpr (StepOf<P>::value == 1) {
                    if (j == 0 && stop == T) {
#pragma unroll
                        for (int jj = 0; jj < T; ++jj) lay.add(v, jj, acc);
                    } else {
#pragma unroll 4
                        for (int jj = j; jj < stop; ++jj) lay.add(v, jj, acc);
                    }
                } else {
                    constexpr int kS = StepOf<P>::value;
                    if (j == 0 && stop == T) {
#pragma unroll
                        for (int jj = 0; jj < T; jj += kS) lay.add_step(v, jj, T, acc);
                    } else {
                        for (int jj = j; jj < stop; jj += kS) lay.add_step(v, jj, stop, acc);
                    }
                }
                j = stop;
                if (tb + j == b) {                   // node n ends inside this window
                    if (a >= p0) {
                        lay.put(o, n, acc);
                    } else {
                        acc0 = acc;
                        have0 = true;
                        if (lane == 0) {
                            sp_node[warp][0] = n;
                            sp_rows[warp][0] = make_int2(a, b);
                        }
                    }
                    P::zero(acc);
                    step();
                    advance();
                }
            }
            ring.refill(perm, coup, cld, rad, E, lane);
        }
        // a node still open at the end runs past p1
        if (n < N && a < pe && b > pe) {
            if (a < p0) {
                acc0 = acc;
                have0 = true;
                if (lane == 0) {
                    sp_node[warp][0] = n;
                    sp_rows[warp][0] = make_int2(a, b);
                }
            } else {
                have1 = true;
                if (lane == 0) {
                    sp_node[warp][1] = n;
                    sp_rows[warp][1] = make_int2(a, b);
                }
            }
        }
    }
    ring.drain();
    // The ring is idle: its first bytes hold this warp's two partials.
    float* part = ring.rad;
    if (have0) lay.store(part, acc0);
    if (have1) lay.store(part + P::kPartFloats, acc);
    __syncthreads();

    // Combine the warp pieces of nodes cut by window edges inside this CTA:
    // the lowest warp holding a piece of node m adds them in window order.
    const int64_t span = (int64_t)W * KW;   // CSR positions per CTA
    const int64_t P0 = imin<int64_t>((int64_t)blockIdx.x * span, E);
    const int64_t P1 = imin<int64_t>(P0 + span, E);
    int pend_node = -1;                      // a node that started in an earlier CTA and ends here
    int pend_ma = 0;                         // its first position
    Acc pend;
    __shared__ int s_stored;                 // this CTA left a partial for a later CTA
    __shared__ int s_pend_b0, s_pend_np;     // the pend node's first CTA, and how many CTAs before this one it spans
    if (threadIdx.x == 0) {
        s_stored = 0;
        s_pend_np = 0;
    }
    __syncthreads();
    // The sums of this warp's slots; the partial a later CTA needs is stored
    // and published first, the finished nodes are written after the flag.
    Acc sums[2];
    int put_node[2] = {-1, -1};
    bool wrote_part = false;
#pragma unroll
    for (int slot = 0; slot < 2; ++slot) {
        const int m = sp_node[warp][slot];
        if (m < 0) continue;
        if (warp > 0 && (sp_node[warp - 1][0] == m || sp_node[warp - 1][1] == m)) continue;
        Acc& sum = sums[slot];
        lay.load(part + slot * P::kPartFloats, sum);
        for (int w2 = warp + 1; w2 < W && sp_node[w2][0] == m; ++w2) {
            Acc t;
            lay.load(reinterpret_cast<const float*>(smem + (size_t)w2 * Layout::kBytes), t);
            P::add_to(sum, t);
        }
        const int ma = sp_rows[warp][slot].x, mb = sp_rows[warp][slot].y;
        if (ma >= P0 && mb <= P1) {
            put_node[slot] = m;
        } else if (ma < P0 && mb <= P1) {
            pend_node = m;
            pend_ma = ma;
            pend = sum;
            if (lane == 0) {
                s_pend_b0 = (int)(ma / span);
                s_pend_np = (int)blockIdx.x - (int)(ma / span);
            }
        } else {
            // slot 1: starts here and runs past this CTA; slot 0: covers all of it
            lay.store(cta_part + ((int64_t)blockIdx.x * 2 + (ma < P0 ? 0 : 1)) * P::kPartFloats, sum);
            wrote_part = true;
            if (lane == 0) s_stored = 1;
        }
    }
    // Publish this CTA's partial (a CTA leaves at most one: for the node that
    // runs past its end): its writers fence, then one release store of the
    // launch's tag.  Exactly one CTA consumes each published flag (the CTA
    // where that node ends) and resets it to 0 after its wait, so no flag
    // keeps a tag past the launch: a CUDA graph replays this launch with the
    // same tag, and must not find the previous replay's flags set.
    if (wrote_part) __threadfence();
    __syncthreads();
    const uint64_t tag = flag_tag(launch_tag(salt));
    if (threadIdx.x == 0 && s_stored) st_release_u64(flags + blockIdx.x, tag);
#pragma unroll
    for (int slot = 0; slot < 2; ++slot)
        if (put_node[slot] >= 0) lay.put(o, put_node[slot], sums[slot]);
    const int bx = (int)blockIdx.x;
    const int np = s_pend_np;                // the same in every warp (written before the barrier above)
    if (np >= kSplitPartials) {
        // A node cut by many CTAs (a hub of a skewed graph): its earlier
        // CTAs' partials are split over this CTA's warps, warp w adding those
        // of CTAs b0 + w, b0 + w + W, ... in CTA order, and the warps' sums
        // are added in warp order.  A fixed order whoever finishes first.
        const int pb0 = s_pend_b0;
        for (int k = pb0 + warp + W * lane; k < bx; k += W * 32) {
            wait_flag(flags, k, tag);
            flags[k] = 0;
        }
        __syncwarp();
        constexpr int kB = sizeof(Acc) <= 64 ? 4 : 1;
        Acc sw;
        P::zero(sw);
        for (int k0 = pb0 + warp; k0 < bx; k0 += W * kB) {
            Acc t[kB];
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int k = k0 + u * W;
                if (k < bx) lay.load_cg(cta_part + ((int64_t)k * 2 + (k == pb0 ? 1 : 0)) * P::kPartFloats, t[u]);
            }
#pragma unroll
            for (int u = 0; u < kB; ++u)
                if (k0 + u * W < bx) P::add_to(sw, t[u]);
        }
        lay.store(reinterpret_cast<float*>(smem + (size_t)warp * Layout::kBytes), sw);
        __syncthreads();
        if (pend_node < 0) return;
        Acc total;
        lay.load(reinterpret_cast<const float*>(smem), total);
        for (int w = 1; w < imin(W, np); ++w) {
            Acc t;
            lay.load(reinterpret_cast<const float*>(smem + (size_t)w * Layout::kBytes), t);
            P::add_to(total, t);
        }
        P::add_to(total, pend);
        lay.put(o, pend_node, total);
        return;
    }
    if (pend_node < 0) return;
    // node pend_node began in CTA b0 (its slot-1 partial), covered CTAs
    // b0+1 .. blockIdx.x-1 (slot-0 partials) and ends here: add in CTA order
    // (the lanes wait for the flags in parallel, and the partials are loaded
    // a few at a time before they are added, still in CTA order: a global
    // access costs several hundred nanoseconds, and on a skewed graph a node
    // spans tens of CTAs)
    const int b0 = (int)(pend_ma / span);
    for (int k = b0 + lane; k < bx; k += 32) {
        wait_flag(flags, k, tag);
        flags[k] = 0;
    }
    __syncwarp();
    constexpr int kB = sizeof(Acc) <= 64 ? 4 : 1;   // partials in flight, within the register budget
    Acc total;
    lay.load_cg(cta_part + ((int64_t)b0 * 2 + 1) * P::kPartFloats, total);
    for (int k0 = b0 + 1; k0 < bx; k0 += kB) {
        Acc t[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u)
            if (k0 + u < bx) lay.load_cg(cta_part + (int64_t)(k0 + u) * 2 * P::kPartFloats, t[u]);
#pragma unroll
        for (int u = 0; u < kB; ++u)
            if (k0 + u < bx) P::add_to(total, t[u]);
    }
    P::add_to(total, pend);
    lay.put(o, pend_node, total);
}

// --------------------------------------------------------------------------
// Per-channel path (any C, any alignment).  One warp per window of kGenWin
// positions, lane = channel within a chunk of 32 channels; every cut node
// leaves a partial per window in the workspace.
// --------------------------------------------------------------------------

template <int L>
__device__ __forceinline__ void accumulate_gen(const float* __restrict__ coup, int cld, const float* __restrict__ rad,
                                               const int32_t* __restrict__ perm, int64_t E, int C, int c,
                                               int s, int t, float (*cs)[Ladder<L>::R + 1], int lane,
                                               float acc[Ladder<L>::R]) {
    constexpr int R = Ladder<L>::R, S = Ladder<L>::S;
    const bool cok = c < C;
    for (int base = s; base < t; base += 32) {
        const int cnt = min(32, t - base);
        int e_l = -1;
        if (lane < cnt) {
            e_l = __ldg(perm + base + lane);
            if ((uint32_t)e_l >= (uint64_t)E) e_l = -1;
        }
        // the coupling rows of the (up to) 32 edges, staged through shared memory
#pragma unroll
        for (int it = 0; it < R; ++it) {
            const int v = it * 32 + lane;
            const int j = v / R;
            const int r = v - j * R;
            const int e = __shfl_sync(kFull, e_l, j);
            float cv = 0.f;
            if (j < cnt && e >= 0) cv = __ldg(coup + (int64_t)e * cld + r);
            cs[j][r] = cv;
        }
        __syncwarp();
        for (int j = 0; j < cnt; ++j) {
            const int e = __shfl_sync(kFull, e_l, j);
            if (e < 0 || !cok) continue;
            const float* rp = rad + (int64_t)e * S * C + c;
            float rv[S];
#pragma unroll
            for (int k = 0; k < S; ++k) rv[k] = __ldg(rp + k * C);
#pragma unroll
            for (int r = 0; r < R; ++r) acc[r] = fmaf(cs[j][r], rv[ladder_slot(r)], acc[r]);
        }
        __syncwarp();
    }
}

template <int L>
__global__ void __launch_bounds__(kFwdThreads)
fwd_gen_main(const float* __restrict__ coup, int cld, const float* __restrict__ rad,
             const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ perm,
             int64_t E, int32_t N, int C, int Wtot, NodeOut o, float* __restrict__ part,
             int32_t* __restrict__ cross) {
    constexpr int R = Ladder<L>::R, D = Ladder<L>::D;
    __shared__ float cs[kFwdWarps][32][R + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kFwdWarps + warp;
    pdl_wait();
    pdl_trigger();
    if (gw >= Wtot) return;
    const int64_t V = (int64_t)R * C;
    const int64_t p0 = (int64_t)gw * kGenWin;
    const int64_t p1 = min(p0 + kGenWin, E);
    const bool is_last = gw == Wtot - 1;
    int crossing = -1;   // the node that starts in this window and continues past it
    for (int n = first_node_warp(row_ptr, N, p0, lane); n < N; ++n) {
        const int a = __ldg(row_ptr + n), b = __ldg(row_ptr + n + 1);
        if (a >= p1 && !(is_last && a == b)) break;
        float* node = o.out + (int64_t)n * D * C;
        float* rnode = o.raw ? o.raw + (int64_t)n * D * C : nullptr;
        if (a == b) {
            for (int64_t i = lane; i < (int64_t)D * C; i += 32) node[i] = 0.f;
            if (rnode)
                for (int64_t i = lane; i < (int64_t)D * C; i += 32) rnode[i] = 0.f;
            continue;
        }
        const bool full = a >= p0 && b <= p1;
        float* dstp = full ? node + C : part + ((int64_t)gw * 2 + (a < p0 ? 0 : 1)) * V;
        const float sc = (full && o.scale) ? __ldg(o.scale + n) : 1.f;
        if (full) {
            for (int c = lane; c < C; c += 32) node[c] = 0.f;
            if (rnode)
                for (int c = lane; c < C; c += 32) rnode[c] = 0.f;
        }
        for (int c0 = 0; c0 < C; c0 += 32) {
            const int c = c0 + lane;
            float acc[R];
#pragma unroll
            for (int r = 0; r < R; ++r) acc[r] = 0.f;
            accumulate_gen<L>(coup, cld, rad, perm, E, C, c, (int)max((int64_t)a, p0), (int)min((int64_t)b, p1),
                              cs[warp], lane, acc);
            if (c < C) {
                if (full && rnode) {
#pragma unroll
                    for (int r = 0; r < R; ++r) rnode[C + (int64_t)r * C + c] = acc[r];
                }
                if (full && o.scale) {
#pragma unroll
                    for (int r = 0; r < R; ++r) dstp[(int64_t)r * C + c] = acc[r] * sc;
                } else {
#pragma unroll
                    for (int r = 0; r < R; ++r) dstp[(int64_t)r * C + c] = acc[r];
                }
            }
        }
        if (!full && a >= p0) crossing = n;
        if (b > p1) break;
    }
    if (lane == 0) cross[gw] = crossing;
}

// --------------------------------------------------------------------------
// Cross-window fix-up, one CTA per window: window c's main kernel recorded in
// cross[c] the node (if any) that starts in it and runs past its end.  That
// node's partials are those of windows c, c+1, ..., floor((b-1)/win): slot 1
// of window c (the node starts inside it), slot 0 of the later ones (it runs
// in from the previous window).  Warp w adds partials k = w, w+8, ... in
// order; the eight warp sums are then added in warp order, and rows 1..15 and
// the zero scalar row are written.
// --------------------------------------------------------------------------

constexpr int kFixVals = 256;   // values per chunk: 8 per lane

__global__ void __launch_bounds__(kFwdThreads)
fwd_fixup(const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ cross, int C, int R, int win,
          const float* __restrict__ part, NodeOut o) {
    __shared__ float red[kFwdWarps][kFixVals];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t V = (int64_t)R * C;
    const int wa = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    const int n = __ldg(cross + wa);
    if (n < 0) return;
    const int b = __ldg(row_ptr + n + 1);
    const int np = (b - 1) / win - wa + 1;
    float* node = o.out + (int64_t)n * (R + 1) * C;
    float* rnode = o.raw ? o.raw + (int64_t)n * (R + 1) * C : nullptr;
    const float sc = o.scale ? __ldg(o.scale + n) : 1.f;
    for (int c = threadIdx.x; c < C; c += kFwdThreads) {
        node[c] = 0.f;
        if (rnode) rnode[c] = 0.f;
    }
    for (int64_t v0 = 0; v0 < V; v0 += kFixVals) {
        float sacc[kFixVals / 32];
#pragma unroll
        for (int i = 0; i < kFixVals / 32; ++i) sacc[i] = 0.f;
        for (int k = warp; k < np; k += kFwdWarps) {
            const float* p = part + ((int64_t)(wa + k) * 2 + (k == 0 ? 1 : 0)) * V + v0;
#pragma unroll
            for (int i = 0; i < kFixVals / 32; ++i) {
                const int64_t v = v0 + lane + 32 * i;
                if (v < V) sacc[i] += __ldg(p + lane + 32 * i);
            }
        }
#pragma unroll
        for (int i = 0; i < kFixVals / 32; ++i) red[warp][lane + 32 * i] = sacc[i];
        __syncthreads();
        {
            const int vl = threadIdx.x;   // kFwdThreads == kFixVals
            const int64_t v = v0 + vl;
            if (v < V) {
                float t = red[0][vl];
#pragma unroll
                for (int w = 1; w < kFwdWarps; ++w) t += red[w][vl];
                if (rnode) rnode[C + v] = t;
                node[C + v] = o.scale ? t * sc : t;
            }
        }
        __syncthreads();
    }
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

unsigned int take_timeouts_forward() { return take_timeouts_local(); }
cudaError_t set_timeout_flag_forward(unsigned int* flag) { return set_timeout_flag_local(flag); }

}  // namespace zs

using namespace zs;

// Scratch for `windows` windows: a pair of (15 x C) partials, one
// crossing-node entry and one 64-bit flag per window, each array 256-byte
// aligned.
struct Scratch {
    float* part;
    int32_t* cross;
    uint64_t* flags;
};

static size_t part_bytes(int64_t windows, int C, int R) {
    return align_up((size_t)windows * 2 * (size_t)R * (size_t)C * sizeof(float), 256);
}

static size_t scratch_bytes(int64_t windows, int C, int R) {
    return part_bytes(windows, C, R) + align_up((size_t)windows * sizeof(int32_t), 256) +
           align_up((size_t)windows * sizeof(uint64_t), 256);
}

static Scratch scratch_at(void* base, int64_t windows, int C, int R) {
    char* b = static_cast<char*>(base);
    Scratch sc;
    sc.part = reinterpret_cast<float*>(b);
    sc.cross = reinterpret_cast<int32_t*>(b + part_bytes(windows, C, R));
    sc.flags = reinterpret_cast<uint64_t*>(b + part_bytes(windows, C, R) + align_up((size_t)windows * sizeof(int32_t), 256));
    return sc;
}


// Warps per CTA of the single-wave forward for a lane layout: 16, or as many
// rings as one SM's shared memory holds.
template <class P, class = void>
struct MaxWarpsOf { static constexpr int value = 16; };
template <class P>
struct MaxWarpsOf<P, std::void_t<decltype(P::kMaxWarps)>> { static constexpr int value = P::kMaxWarps; };
template <class P>
constexpr int layout_max_warps() { return MaxWarpsOf<P>::value; }

template <class P>
constexpr int tma_warps() {
    constexpr int bytes = RingLayout<kTmaStages, P::kTileEdges, P::kRadFloats, P::kCoupRow>::kBytes;
    constexpr int cap = imin(kTmaWarps, layout_max_warps<P>());
    return (232448 / bytes) < cap ? (232448 / bytes) : cap;
}

// A CTA of the single-wave path covers at least kMinTmaSpan CSR positions
// (so the workspace, sized per kMinTmaSpan positions, holds every CTA's
// partials): each warp's window is at least tma_min_window positions.
constexpr int kMinTmaSpan = 128;
template <class P>
constexpr int tma_min_window(int W) {
    return (kMinTmaSpan + W - 1) / W > P::kTileEdges
               ? ((kMinTmaSpan + W - 1) / W + P::kTileEdges - 1) / P::kTileEdges * P::kTileEdges
               : P::kTileEdges;
}

// Small graphs at lmax 3: when the full warp count would leave windows of
// fewer than kShortWindow positions, kQuadWarpsSmall warps per CTA take
// longer windows with fewer cut nodes to combine (on the 1000-node graph,
// 69-edge windows of 15 warps took 22.8 us, 104-edge windows of 10 warps
// 21.2 us, 12 and 8 warps 21.8 and 23.3 us; the 4096-node graph keeps 15).
// Either way a window has at least tma_min_window positions.
constexpr int kShortWindow = 96;
constexpr int kQuadWarpsSmall = 10;

static int tma_warps_for(int lmax, int64_t E) {
    switch (lmax) {
        case 1: return tma_warps<EdgeQuadLayout<1>>();
        case 2: return tma_warps<ChanLayout<2>>();
        case 3: {
            constexpr int W = tma_warps<QuadLayout>();
            return ceil_div(E, (int64_t)num_sms() * W) < kShortWindow ? kQuadWarpsSmall : W;
        }
        case 4: return tma_warps<ChanLayout<4>>();
        default: return tma_warps<ChanLayout<5>>();
    }
}

static int tma_min_window_for(int lmax, int W) {
    switch (lmax) {
        case 1: return tma_min_window<EdgeQuadLayout<1>>(W);
        case 2: return tma_min_window<ChanLayout<2>>(W);
        case 3: return tma_min_window<QuadLayout>(W);
        case 4: return tma_min_window<ChanLayout<4>>(W);
        default: return tma_min_window<ChanLayout<5>>(W);
    }
}

// How zs_forward splits a call: the single-wave C == 32 kernel (16-byte
// aligned radial rows; at lmax 3 also 16-byte aligned outputs for the quad
// layout's vector stores) or the per-channel kernel and its fix-up.
struct FwdPlan {
    bool fast;
    int R, W;
    int64_t KW, Wtot, ctas, windows;
};

static FwdPlan fwd_plan(const float* rad, const NodeOut& o, int64_t E, int C, int lmax) {
    FwdPlan p{};
    p.R = ladder_rows(lmax);
    // the coupling rows may have any 4-byte alignment and stride: the ring
    // copies each one's 16-byte-aligned span
    p.fast = C == kC32 && aligned16(rad) &&
             (lmax != 3 || (aligned16(o.out) && (o.raw == nullptr || aligned16(o.raw))));
    if (p.fast) {
        // Balanced single wave: one CTA of W warps per SM, every warp the same
        // number of CSR positions (at least one tile).
        p.W = tma_warps_for(lmax, E);
        const int64_t warps_max = (int64_t)num_sms() * p.W;
        // CTAs cover at least kMinTmaSpan positions: ceil(E / kMinTmaSpan) of them at most
        p.KW = imax<int64_t>(ceil_div(E, warps_max), tma_min_window_for(lmax, p.W));   // < 2^31: E < 2^31
        p.Wtot = imax<int64_t>(ceil_div(E, p.KW), 1);
        p.ctas = ceil_div(p.Wtot, p.W);
        p.windows = p.ctas;
    } else {
        p.W = kFwdWarps;
        p.Wtot = ceil_div(E > 0 ? E : 1, kGenWin);
        p.ctas = ceil_div(p.Wtot, kFwdWarps);
        p.windows = p.Wtot;
    }
    return p;
}

template <int L>
static void launch_gen(const FwdPlan& p, const float* coup, int cld, const float* rad, const int32_t* row_ptr,
                       const int32_t* perm, int64_t E, int32_t N, int C, const NodeOut& o, const Scratch& sc,
                       cudaStream_t s) {
    launch(fwd_gen_main<L>, (unsigned)p.ctas, kFwdThreads, 0, s, coup, cld, rad, row_ptr, perm, E, N, C, (int)p.Wtot,
           o, sc.part, sc.cross);
    launch(fwd_fixup, (unsigned)p.Wtot, kFwdThreads, 0, s, row_ptr, (const int32_t*)sc.cross, C, Ladder<L>::R,
           kGenWin, (const float*)sc.part, o);
}

template <class P, int W>
static void launch_tma_w(const FwdPlan& p, const float* coup, int cld, const float* rad, const int32_t* row_ptr,
                         const int32_t* perm, int64_t E, int32_t N, const NodeOut& o, const Scratch& sc,
                         cudaStream_t s) {
    auto kernel = fwd_tma<W, kTmaStages, P::kTileEdges, P>;
    const int smem = W * RingLayout<kTmaStages, P::kTileEdges, P::kRadFloats, P::kCoupRow>::kBytes;
    static std::atomic<uint64_t> attr_done[kMaxDevices];
    set_smem_limit_once(kernel, smem, attr_done);
    launch(kernel, (unsigned)p.ctas, W * 32, smem, s, coup, cld, rad, row_ptr, perm, (int)E, N, (int)p.KW,
           (int)p.Wtot, o, sc.part, sc.flags, next_salt());
}

template <class P>
static void launch_tma(const FwdPlan& p, const float* coup, int cld, const float* rad, const int32_t* row_ptr,
                       const int32_t* perm, int64_t E, int32_t N, const NodeOut& o, const Scratch& sc,
                       cudaStream_t s) {
    if constexpr (std::is_same<P, QuadLayout>::value) {
        if (p.W == kQuadWarpsSmall) {
            launch_tma_w<P, kQuadWarpsSmall>(p, coup, cld, rad, row_ptr, perm, E, N, o, sc, s);
            return;
        }
    }
    launch_tma_w<P, tma_warps<P>()>(p, coup, cld, rad, row_ptr, perm, E, N, o, sc, s);
}

static void launch_forward(const FwdPlan& p, const float* coup, int cld, const float* rad, const int32_t* row_ptr,
                           const int32_t* perm, int64_t E, int32_t N, int C, int lmax, const NodeOut& o,
                           const Scratch& sc, cudaStream_t s) {
    if (p.fast) {
        switch (lmax) {
            case 1: launch_tma<EdgeQuadLayout<1>>(p, coup, cld, rad, row_ptr, perm, E, N, o, sc, s); break;
            case 2: launch_tma<ChanLayout<2>>(p, coup, cld, rad, row_ptr, perm, E, N, o, sc, s); break;
            case 3: launch_tma<QuadLayout>(p, coup, cld, rad, row_ptr, perm, E, N, o, sc, s); break;
            case 4: launch_tma<ChanLayout<4>>(p, coup, cld, rad, row_ptr, perm, E, N, o, sc, s); break;
            default: launch_tma<ChanLayout<5>>(p, coup, cld, rad, row_ptr, perm, E, N, o, sc, s); break;
        }
        return;
    }
    switch (lmax) {
        case 1: launch_gen<1>(p, coup, cld, rad, row_ptr, perm, E, N, C, o, sc, s); break;
        case 2: launch_gen<2>(p, coup, cld, rad, row_ptr, perm, E, N, C, o, sc, s); break;
        case 3: launch_gen<3>(p, coup, cld, rad, row_ptr, perm, E, N, C, o, sc, s); break;
        case 4: launch_gen<4>(p, coup, cld, rad, row_ptr, perm, E, N, C, o, sc, s); break;
        default: launch_gen<5>(p, coup, cld, rad, row_ptr, perm, E, N, C, o, sc, s); break;
    }
}

extern "C" size_t zs_forward_workspace_bytes_lmax(int64_t E, int32_t N, int32_t C, int32_t lmax) {
    if (E < 0 || N < 0 || C < 1 || lmax < 1 || lmax > kMaxLmax) return 0;
    (void)N;
    // Sized for the smaller of the two window lengths: kGenWin positions per
    // warp on the per-channel path, at least W * (tile edges) per CTA on the
    // single-wave C == 32 path (at least kMinTmaSpan for every layout).
    const int64_t win = imin<int64_t>(kGenWin, kMinTmaSpan);
    const int64_t windows = ceil_div(E > 0 ? E : 1, win) + 1;
    return scratch_bytes(windows, C, ladder_rows(lmax));
}

extern "C" size_t zs_forward_workspace_bytes(int64_t E, int32_t N, int32_t C) {
    return zs_forward_workspace_bytes_lmax(E, N, C, 3);
}

static zs_status forward_impl(const char* name, const float* coup, int64_t cld, const float* rad,
                              const int32_t* row_ptr, const int32_t* perm, int64_t E, int32_t N, int32_t C,
                              int32_t lmax, const NodeOut& o, void* workspace, size_t workspace_bytes,
                              zs_stream_t stream) {
    if (lmax < 1 || lmax > kMaxLmax)
        return fail(ZS_ERR_UNSUPPORTED, "%s: lmax=%d, supported ladders are lmax 1..%d", name, lmax, kMaxLmax);
    if (cld < ladder_rows(lmax) || cld > (int64_t)1 << 24)
        return fail(ZS_ERR_INVALID_ARG, "%s: coupling row stride %lld below %d rows or too large", name, (long long)cld,
                    ladder_rows(lmax));
    if (E < 0 || N < 0 || C < 1) return fail(ZS_ERR_INVALID_ARG, "%s: bad sizes E=%lld N=%d C=%d", name, (long long)E, N, C);
    if (E >= ((int64_t)1 << 31) - 1) return fail(ZS_ERR_INVALID_ARG, "%s: E=%lld exceeds the int32 index range", name, (long long)E);
    if (!row_ptr) return fail(ZS_ERR_INVALID_ARG, "%s: row_ptr is NULL", name);
    if (N > 0 && !o.out) return fail(ZS_ERR_INVALID_ARG, "%s: out is NULL", name);
    if (E > 0 && (!coup || !rad || !perm)) return fail(ZS_ERR_INVALID_ARG, "%s: coup, rad or perm is NULL with E > 0", name);
    const size_t need = zs_forward_workspace_bytes_lmax(E, N, C, lmax);
    if (workspace_bytes < need) return fail(ZS_ERR_INVALID_ARG, "%s: workspace of %zu bytes, %zu needed", name, workspace_bytes, need);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(ZS_ERR_INVALID_ARG, "%s: workspace NULL or not 256-byte aligned", name);
    if (N == 0) return ZS_OK;
    const FwdPlan p = fwd_plan(rad, o, E, C, lmax);
    if (scratch_bytes(p.windows, C, p.R) > workspace_bytes)   // the plan never outgrows the query's size
        return fail(ZS_ERR_INVALID_ARG, "%s: plan needs %zu bytes of workspace, %zu given", name,
                    scratch_bytes(p.windows, C, p.R), workspace_bytes);
    launch_forward(p, coup, (int)cld, rad, row_ptr, perm, E, N, C, lmax, o, scratch_at(workspace, p.windows, C, p.R),
                   reinterpret_cast<cudaStream_t>(stream));
    return check_launch(name);
}

extern "C" zs_status zs_forward(const float* coup, const float* rad,
                                const int32_t* row_ptr, const int32_t* perm,
                                int64_t E, int32_t N, int32_t C, int32_t lmax,
                                float* out, void* workspace, size_t workspace_bytes,
                                zs_stream_t stream) {
    return forward_impl("zs_forward", coup, ladder_rows(lmax), rad, row_ptr, perm, E, N, C, lmax,
                        NodeOut{out, nullptr, nullptr}, workspace, workspace_bytes, stream);
}

extern "C" zs_status zs_forward_ld(const float* coup, int64_t coup_ld, const float* rad,
                                   const int32_t* row_ptr, const int32_t* perm,
                                   int64_t E, int32_t N, int32_t C, int32_t lmax,
                                   float* out, void* workspace, size_t workspace_bytes, zs_stream_t stream) {
    return forward_impl("zs_forward_ld", coup, coup_ld, rad, row_ptr, perm, E, N, C, lmax,
                        NodeOut{out, nullptr, nullptr}, workspace, workspace_bytes, stream);
}

extern "C" zs_status zs_forward_scaled(const float* coup, const float* rad,
                                       const int32_t* row_ptr, const int32_t* perm, const float* node_scale,
                                       int64_t E, int32_t N, int32_t C, int32_t lmax,
                                       float* out, float* out_raw, void* workspace, size_t workspace_bytes,
                                       zs_stream_t stream) {
    if (N > 0 && !node_scale) return fail(ZS_ERR_INVALID_ARG, "zs_forward_scaled: node_scale is NULL");
    return forward_impl("zs_forward_scaled", coup, ladder_rows(lmax), rad, row_ptr, perm, E, N, C, lmax,
                        NodeOut{out, out_raw, node_scale}, workspace, workspace_bytes, stream);
}

// --------------------------------------------------------------------------
// zs_forward_noalloc: zs_forward for callers that cannot allocate device
// memory (for example code that runs where cudaMalloc is not allowed, such
// as inside a region that must not touch the allocator, or a host framework
// that owns all device memory and hands out only the tensors themselves).
// The partial sums and flags the forward keeps between its CTAs (and, on
// the per-channel path, between its two kernels) live in a fixed, file-scope
// device array instead of a caller workspace.
// --------------------------------------------------------------------------

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB, held by every GPU that loads the library
static __device__ __align__(256) unsigned char g_forward_scratch[kNoAllocScratchBytes];

namespace {

// Device address of g_forward_scratch in the current device's context, looked
// up once per context with that device current (and again after a
// cudaDeviceReset, whose new primary context may place the array elsewhere).
// In host code the array's name is only a stand-in for the symbol, never an
// address a kernel may use.
zs_status forward_scratch_address(float** out_ptr) {
    struct Entry {
        uint64_t ctx;
        void* ptr;
    };
    static std::mutex mu;
    static Entry cached[kMaxDevices] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return fail(ZS_ERR_CUDA, "zs_forward_noalloc: cudaGetDevice: %s", cudaGetErrorString(err));
    if (dev < 0 || dev >= kMaxDevices) return fail(ZS_ERR_UNSUPPORTED, "zs_forward_noalloc: device ordinal %d", dev);
    std::lock_guard<std::mutex> lock(mu);
    const uint64_t ctx = current_context_id();
    if (ctx == 0 || cached[dev].ctx != ctx || !cached[dev].ptr) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_forward_scratch);
        if (err != cudaSuccess || !p)
            return fail(ZS_ERR_CUDA, "zs_forward_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(err));
        cached[dev] = Entry{current_context_id(), p};
    }
    *out_ptr = static_cast<float*>(cached[dev].ptr);
    return ZS_OK;
}

}  // namespace

extern "C" zs_status zs_forward_noalloc(const float* coup, const float* rad,
                                        const int32_t* row_ptr, const int32_t* perm,
                                        int64_t E, int32_t N, int32_t C, int32_t lmax,
                                        float* out, zs_stream_t stream) {
    if (lmax < 1 || lmax > kMaxLmax)
        return fail(ZS_ERR_UNSUPPORTED, "zs_forward_noalloc: lmax=%d, supported ladders are lmax 1..%d", lmax, kMaxLmax);
    if (E < 0 || N < 0 || C < 1) return fail(ZS_ERR_INVALID_ARG, "zs_forward_noalloc: bad sizes E=%lld N=%d C=%d", (long long)E, N, C);
    if (E >= ((int64_t)1 << 31) - 1) return fail(ZS_ERR_INVALID_ARG, "zs_forward_noalloc: E=%lld exceeds the int32 index range", (long long)E);
    if (!row_ptr) return fail(ZS_ERR_INVALID_ARG, "zs_forward_noalloc: row_ptr is NULL");
    if (N > 0 && !out) return fail(ZS_ERR_INVALID_ARG, "zs_forward_noalloc: out is NULL");
    if (E > 0 && (!coup || !rad || !perm)) return fail(ZS_ERR_INVALID_ARG, "zs_forward_noalloc: coup, rad or perm is NULL with E > 0");
    if (N == 0) return ZS_OK;
    // the same split as zs_forward; the scratch holds one pair of partials per window
    const NodeOut o{out, nullptr, nullptr};
    const FwdPlan p = fwd_plan(rad, o, E, C, lmax);
    const size_t need = scratch_bytes(p.windows, C, p.R);
    if (need > kNoAllocScratchBytes)
        return fail(ZS_ERR_INVALID_ARG,
                    "zs_forward_noalloc: this call needs %zu bytes of scratch but the library's static scratch holds "
                    "%zu; use zs_forward with a caller workspace", need, kNoAllocScratchBytes);
    float* base = nullptr;
    const zs_status st = forward_scratch_address(&base);
    if (st != ZS_OK) return st;
    launch_forward(p, coup, ladder_rows(lmax), rad, row_ptr, perm, E, N, C, lmax, o, scratch_at(base, p.windows, C, p.R),
                   reinterpret_cast<cudaStream_t>(stream));
    return check_launch("zs_forward_noalloc");
}
