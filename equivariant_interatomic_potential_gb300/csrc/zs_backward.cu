// Backward of the zonal scatter, one edge-parallel pass (lmax = 3 ladder shown;
// every kernel takes the ladders of degree 1..5 the same way):
//   d_coup[e,r]  = sum_c g[dst[e],1+r,c] * rad[e,slot(r),c]
//   d_rad[e,s,c] = sum over rows r of slot s of g[dst[e],1+r,c] * coup[e,r]
// (deepmd-kit pull request "fused Triton zonal scatter for the GIE head",
// section "What", backward bullet: both operand gradients in a single
// edge-parallel kernel, no materialised message gradient).
//
// zs_backward takes the edges in their own order, so coup, rad, dst, d_coup
// and d_rad stream through HBM contiguously and the only gathered operand is
// g (N x 16 x C, a few MB, resident in L2).  zs_backward_csr visits them in
// destination order instead and reads each node's g once per run of edges.
#include "zs_common.cuh"
#include "zs_tma.cuh"

// L2 policy of the CSR-order backward's coupling spans: normal, since a span
// shares its sectors with the neighbouring edges' rows, which the CSR-order
// walk reaches later (the ring's radial rows and perm are evict-first below
// lmax 4).
#ifndef ZS_BWDC_COUP_POL
#define ZS_BWDC_COUP_POL kL2Normal
#endif
namespace zs {
namespace {

constexpr int kBwdWarps = 8;
// CSR-order C == 32 path: warps per CTA (one CTA per SM), ring stages, edges per tile.
#ifndef ZS_BWD_WARPS
#define ZS_BWD_WARPS 16
#endif
#ifndef ZS_BWD_STAGES
#define ZS_BWD_STAGES 2
#endif
#ifndef ZS_BWD_TILE
#define ZS_BWD_TILE 8
#endif
constexpr int kBwdThreads = kBwdWarps * 32;
constexpr int kC32 = 32;
constexpr unsigned kFull = 0xffffffffu;

// --------------------------------------------------------------------------
// Per-channel path (any C, any alignment): lane = channel within a chunk of
// 32; d_coup is reduced over the warp after the channel loop.
// --------------------------------------------------------------------------
// Sum over the warp of 32 values at once, each lane ending with the total
// of value `lane` (a transposed butterfly: 16 + 8 + 4 + 2 + 1 shuffles).
__device__ __forceinline__ float warp_reduce_scatter32(float v[32], int lane) {
#pragma unroll
    for (int half = 16; half >= 1; half >>= 1) {
        const bool up = (lane & half) != 0;
#pragma unroll
        for (int k = 0; k < half; ++k) {
            const float keep = up ? v[k + half] : v[k];
            const float send = up ? v[k] : v[k + half];
            v[k] = keep + __shfl_xor_sync(kFull, send, half);
        }
    }
    return v[0];
}

// Gradients of one edge e whose destination is d (d < 0: no node, zero
// gradients), lane = channel within chunks of 32; ladder of degree L.
template <int L>
__device__ __forceinline__ void bwd_gen_edge(const float* __restrict__ g, const float* __restrict__ coup,
                                             const float* __restrict__ rad, int64_t e, int d, int C, int lane,
                                             float* __restrict__ d_coup, float* __restrict__ d_rad,
                                             const float* __restrict__ scale = nullptr,
                                             int64_t cld = Ladder<L>::R, int64_t dld = Ladder<L>::R) {
    constexpr int R = Ladder<L>::R, S = Ladder<L>::S, D = Ladder<L>::D;
    constexpr int RP = (R + 31) / 32 * 32;   // rows padded to whole warps for the reduction
    const bool ok = d >= 0;
    float cv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) cv[r] = __ldg(coup + e * cld + r);
    float pc[RP];
#pragma unroll
    for (int r = 0; r < RP; ++r) pc[r] = 0.f;
    const float* rp = rad + e * S * C;
    float* drp = d_rad + e * S * C;
    const float* gn = g + (int64_t)(ok ? d : 0) * D * C;
    const float sc = (ok && scale) ? __ldg(scale + d) : 1.f;   // the destination's scale (1: plain operator)
    for (int c = lane; c < C; c += 32) {
        if (!ok) {
#pragma unroll
            for (int k = 0; k < S; ++k) drp[k * C + c] = 0.f;
            continue;
        }
        float rv[S], sv[S];
#pragma unroll
        for (int k = 0; k < S; ++k) {
            rv[k] = __ldg(rp + k * C + c);
            sv[k] = 0.f;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float gv = __ldg(gn + (1 + r) * C + c);
            pc[r] = fmaf(gv, rv[ladder_slot(r)], pc[r]);
            sv[ladder_slot(r)] = fmaf(gv, cv[r], sv[ladder_slot(r)]);
        }
#pragma unroll
        for (int k = 0; k < S; ++k) drp[k * C + c] = scale ? sv[k] * sc : sv[k];
    }
#pragma unroll
    for (int r0 = 0; r0 < RP; r0 += 32) {
        const float v = warp_reduce_scatter32(pc + r0, lane);
        if (r0 + lane < R) d_coup[e * dld + r0 + lane] = ok ? (scale ? v * sc : v) : 0.f;
    }
}

template <int L>
__global__ void __launch_bounds__(kBwdThreads)
bwd_gen(const float* __restrict__ g, const float* __restrict__ coup, const float* __restrict__ rad,
        const int32_t* __restrict__ dst, int64_t E, int32_t N, int C,
        float* __restrict__ d_coup, float* __restrict__ d_rad, const float* __restrict__ scale, int cld, int dld) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    for (int64_t e = (int64_t)blockIdx.x * kBwdWarps + warp; e < E; e += (int64_t)gridDim.x * kBwdWarps) {
        const int d = __ldg(dst + e);
        bwd_gen_edge<L>(g, coup, rad, e, (d >= 0 && d < N) ? d : -1, C, lane, d_coup, d_rad, scale, cld, dld);
    }
}

// --------------------------------------------------------------------------
// CSR-order backward.  The same gradients, with the edges visited in
// destination order: each warp owns a window of CSR positions, loads the
// cotangent rows g[n] of a node once into registers and reuses them for all
// of the node's edges in the window, so g is read about once per node
// instead of once per edge.  Radial rows and coupling rows arrive through
// the warp's TMA ring; gradients are written to the edge's own rows.
// Positions at or after row_ptr[N] hold edges without a node: zeros.
// --------------------------------------------------------------------------

// Lane layout of the CSR-order C == 32 backward: the 8 lanes of group
// grp = lane/8 own one edge of every 4 consecutive positions, lane q = lane%8
// owns channels 4q..4q+3 of ALL 15 rows.  One warp instruction therefore
// advances four edges; the radial gradient needs no cross-lane traffic and
// the coupling gradient is one transposed butterfly over the group's 8 lanes.
struct QuadLane {
    int lane, grp, q;
    bool b2, b1, b0;
    __device__ __forceinline__ explicit QuadLane(int l)
        : lane(l), grp(l >> 3), q(l & 7), b2((l & 4) != 0), b1((l & 2) != 0), b0((l & 1) != 0) {}
};

// Sum of v over the 8 lanes of the group for 8K values at once, by a
// transposed butterfly (each step halves the values a lane carries): each
// lane ends with the totals of values 4K*b2 + 2K*b1 + K*b0 + {0..K-1}.
template <int K>
__device__ __forceinline__ void group_reduce(const float (&v)[8 * K], const QuadLane& Q, float (&out)[K]) {
    float w[4 * K];
#pragma unroll
    for (int k = 0; k < 4 * K; ++k) {
        const float keep = Q.b2 ? v[k + 4 * K] : v[k];
        const float send = Q.b2 ? v[k] : v[k + 4 * K];
        w[k] = keep + __shfl_xor_sync(kFull, send, 4);
    }
    float x[2 * K];
#pragma unroll
    for (int k = 0; k < 2 * K; ++k) {
        const float keep = Q.b1 ? w[k + 2 * K] : w[k];
        const float send = Q.b1 ? w[k] : w[k + 2 * K];
        x[k] = keep + __shfl_xor_sync(kFull, send, 2);
    }
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const float keep = Q.b0 ? x[k + K] : x[k];
        const float send = Q.b0 ? x[k] : x[k + K];
        out[k] = keep + __shfl_xor_sync(kFull, send, 1);
    }
}

template <int W, int S, int T, int LM>
__global__ void __launch_bounds__(W * 32, 1)
bwd_csr_quad(const float* __restrict__ g, const float* __restrict__ coup, const float* __restrict__ rad,
             const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ perm,
             int E, int32_t N, int KW, int Wtot,
             float* __restrict__ d_coup, float* __restrict__ d_rad) {
    static_assert(T % 4 == 0, "tiles hold whole groups of four edges");
    constexpr int R = Ladder<LM>::R, D = Ladder<LM>::D, RF = LM * kC32;
    constexpr int K = (R + 7) / 8;                   // coupling-gradient values per lane
    constexpr int kSlot = coup_slot_floats(R);
    // a node's R cotangent rows: in registers up to 24 rows, else in this
    // lane's own column of shared memory ([row][lane] float4, no sharing)
    constexpr bool kSmemG = R > 24;
    // radial rows and perm: evict-first, but evict-normal from lmax 4 on
    // (measured on the n4096 graph: lmax 4 147 -> 144 us, lmax 5 233 -> 227
    // us; lmax 2 and 3 were slower with it)
    // (lmax 1's 128-byte radial rows as 16-byte pieces: 47.4 -> 44.6 us; lmax 2 unchanged)
    using Ring = TileRing<S, T, (LM >= 4 ? kL2Normal : kL2EvictFirst), RF, R, ZS_BWDC_COUP_POL, LM == 1>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const QuadLane Q(threadIdx.x & 31);
    const int gw = blockIdx.x * W + warp;
    const bool active = gw < Wtot;
    pdl_wait();
    pdl_trigger();
    const int p0 = active ? (int)imin<int64_t>((int64_t)gw * KW, E) : E;
    const int p1 = active ? (int)imin<int64_t>((int64_t)p0 + KW, E) : E;
    Ring ring;
    ring.init(smem + (size_t)warp * Ring::Layout::kBytes, p0, p1, Q.lane);
    const uint64_t pol_first = l2_evict_first(), pol_last = l2_evict_last();
    if (active) {
        ring.prefetch_perm(perm, Q.lane);
#pragma unroll
        for (int i = 0; i < S; ++i) ring.issue(perm, coup, R, rad, E, Q.lane);
        const int vend = __ldg(row_ptr + N);
        // this group's node: n covers positions [.., b); G holds its rows 1..R
        int n = p0 < vend ? first_node_warp(row_ptr, N, p0, Q.lane) : N;
        int b = n < N ? __ldg(row_ptr + n + 1) : 0;
        int c = 0;   // row_ptr[n + 2], fetched one node ahead
        float4 G[kSmemG ? 1 : R];
        float4* gsm = reinterpret_cast<float4*>(smem + (size_t)W * Ring::Layout::kBytes) + (size_t)warp * R * 32 + Q.lane;
        auto put_g = [&](int r, float4 v) {
            if constexpr (kSmemG) gsm[r * 32] = v;
            else G[r] = v;
        };
        auto get_g = [&](int r) -> float4 {
            if constexpr (kSmemG) return gsm[r * 32];
            else return G[r];
        };
        const float* gq = g + 4 * Q.q;
        auto load_g = [&]() {
            const float* gn = gq + (int64_t)n * (D * kC32);
#pragma unroll
            for (int r = 0; r < R; ++r) put_g(r, ld_ro4(gn + (1 + r) * kC32));
        };
        if (p0 < vend) {
            while (b <= p0) b = __ldg(row_ptr + (++n) + 1);
            c = n + 2 <= N ? __ldg(row_ptr + n + 2) : 0;
            load_g();
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r) put_g(r, make_float4(0.f, 0.f, 0.f, 0.f));
        }
        for (int k = 0; k < ring.ntiles; ++k) {
            const int st = ring.acquire();
            const int tb = p0 + k * T;
            const int jt = imin(T, p1 - tb);
            const float* radst = ring.rad + st * T * RF + 4 * Q.q;
            const float* coupst = ring.coup + st * T * kSlot;
            const int2* metast = ring.meta + st * T;
#pragma unroll 1
            for (int i = 0; i < T / 4; ++i) {
                const int j = 4 * i + Q.grp;
                const int pos = tb + j;
                const bool in = j < jt;
                const bool has_node = in && pos < vend;
                if (has_node && pos >= b) {        // this group's edge starts a later node
                    do {
                        ++n;
                        b = c;
                        c = n + 2 <= N ? __ldg(row_ptr + n + 2) : 0;
                    } while (b <= pos);
                    load_g();
                }
                const int2 m = metast[j];
                const float* rrow = radst + j * RF;
                float4 a[LM];
#pragma unroll
                for (int l = 0; l < LM; ++l) a[l] = *reinterpret_cast<const float4*>(rrow + l * kC32);
                const float* crow = coupst + j * kSlot + m.y;
                // radial gradient: one running sum per degree slot, rows in order;
                // coupling gradient: per-row dot products over this lane's channels,
                // then summed over the group's 8 lanes
                float4 sl[LM];
                float pr[8 * K];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float cr = crow[r];
                    const float4 Gr = get_g(r);
                    const int l = ladder_slot(r);
                    if ((l + 1) * (l + 1) - 1 == r)   // first row of its degree
                        sl[l] = make_float4(cr * Gr.x, cr * Gr.y, cr * Gr.z, cr * Gr.w);
                    else
                        sl[l] = f4_fma(cr, Gr, sl[l]);
                    pr[r] = f4_dot(Gr, a[l]);
                }
#pragma unroll
                for (int r = R; r < 8 * K; ++r) pr[r] = 0.f;
                float t[K];
                group_reduce<K>(pr, Q, t);
                const int e = m.x;
                if (in && e >= 0) {
                    const int row = 4 * K * Q.b2 + 2 * K * Q.b1 + K * Q.b0;
                    float* dc = d_coup + (int64_t)e * R + row;
                    float* dr = d_rad + (int64_t)e * RF + 4 * Q.q;
                    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                    // d_rad rows are whole lines: stream them out.  d_coup rows are 4R bytes in
                    // random order: keep their lines in L2 until neighbouring rows fill them
#pragma unroll
                    for (int l = 0; l < LM; ++l) st_hint4(dr + l * kC32, has_node ? sl[l] : z, pol_first);
#pragma unroll
                    for (int q = 0; q < K; ++q)
                        if (row + q < R) st_hint(dc + q, has_node ? t[q] : 0.f, pol_last);
                }
            }
            ring.refill(perm, coup, R, rad, E, Q.lane);
        }
    }
    ring.drain();
}

// --------------------------------------------------------------------------
// Edge-order C == 32 backward fed by bulk copies.  A warp owns a window of
// consecutive edges and streams it in tiles of T edges (tiles start at
// multiples of T so every block below is 16-byte aligned): per tile one bulk
// copy of the T radial rows, one of the T coupling rows, and per edge one
// bulk copy of its destination's cotangent rows 1..R (1920 bytes at lmax 3,
// gathered from L2).  dst is read ahead with plain loads, 32 edges at a
// time, since the gathers need it.
// --------------------------------------------------------------------------

// Hot destination.  On a skewed graph one node can be the destination of a
// large share of the edges (a sixth on the Zipf(1.1) graph), and every SM
// then gathers the same 15 cotangent lines, so the few L2 slices holding them
// serialise the gathers.  A CTA that sees one destination often among the
// first 32 edges of its warps' windows copies that node's rows once into a
// hot slot of its shared memory, and its rings skip the node's gathers.  The
// consumers read every edge of that node from the slot (the rows are the same
// bytes wherever they sit, so the results are too).
#ifndef ZS_BWD_HOT
#define ZS_BWD_HOT 1
#endif
constexpr bool kHotSlot = ZS_BWD_HOT != 0;
constexpr int kNoHot = -3;                 // matches no destination and no meta marker (-1, -2)
constexpr int kHotMinSamples = 16;         // of the CTA's 32 x W samples (uniform graphs: about 1)

// The CTA's hot destination, or kNoHot: each warp votes for the most frequent
// destination among its 32 samples (sample < 0: none) with that count; the
// candidate with the largest summed count wins if it reaches kHotMinSamples.
// Every thread of the CTA must call it (it synchronises the CTA).
template <int W>
__device__ int cta_hot_node(int sample, int lane, int warp, int (*cand)[2]) {
    int cnt = 0;
#pragma unroll
    for (int k = 0; k < 32; ++k) cnt += __shfl_sync(0xffffffffu, sample, k) == sample ? 1 : 0;
    if (sample < 0) cnt = 0;
    const int best = __reduce_max_sync(0xffffffffu, cnt);
    const unsigned who = __ballot_sync(0xffffffffu, cnt == best);
    const int val = __shfl_sync(0xffffffffu, sample, __ffs(who) - 1);
    if (lane == 0) {
        cand[warp][0] = best > 0 ? val : -1;
        cand[warp][1] = best;
    }
    __syncthreads();
    // lane w < W sums the counts of the warps voting like warp w; the first
    // lane with the largest sum names the winner (every warp finds the same)
    int v = -1, c = 0;
    if (lane < W) {
        v = cand[lane][0];
        if (v >= 0)
            for (int u = 0; u < W; ++u) c += cand[u][0] == v ? cand[u][1] : 0;
    }
    const int top = __reduce_max_sync(0xffffffffu, c);
    const unsigned lead = __ballot_sync(0xffffffffu, v >= 0 && c == top);
    const int hv = lead ? __shfl_sync(0xffffffffu, v, __ffs(lead) - 1) : -1;
    return top >= kHotMinSamples && hv >= 0 ? hv : kNoHot;
}

// Per edge: the destination's cotangent rows 1..R (R x 32 floats), the
// radial row (LM x 32) and the coupling row (R), for the ladder of degree LM.
template <int S, int T, int LM = 3>
struct EdgeRingLayout {
    static constexpr int R = Ladder<LM>::R;
    static constexpr int kG = S * T * R * kC32 * 4;   // cotangent rows 1..R per edge
    static constexpr int kRad = S * T * LM * kC32 * 4;
    static constexpr int kCoup = S * T * R * 4;
    static constexpr int kMeta = (S * T * 4 + 15) / 16 * 16;
    static constexpr int kBars = S * 8;
    static constexpr int kBytes = (kG + kRad + kCoup + kMeta + kBars + 127) / 128 * 128;
    // bulk-copy destinations start on 16-byte boundaries, mbarriers on 8-byte ones
    static_assert(kG % 16 == 0 && kRad % 16 == 0 && kCoup % 16 == 0 && kMeta % 16 == 0, "16-byte aligned regions");
    static_assert((kG + kRad + kCoup + kMeta) % 8 == 0, "mbarriers 8-byte aligned");
};
template <int S, int T, int LM = 3>
struct EdgeRing {
    static_assert(32 % T == 0 && (LM != 3 || T % 4 == 0), "tiles divide 32 (whole quads at lmax 3)");
    // An edge's cotangent rows as 16-byte cp.async pieces by the whole warp
    // when they are at most 32 pieces (lmax 1: 45.1 -> 42.4 us), else one
    // bulk copy per edge.
    // (as pieces, lmax 2's 64 were no faster and lmax 3's 120 much slower)
    static constexpr bool kGPieces = Ladder<LM>::R * kC32 / 4 <= 32;
    using Layout = EdgeRingLayout<S, T, LM>;
    static constexpr int R = Ladder<LM>::R, D = Ladder<LM>::D;
    static constexpr int RF = LM * kC32;                    // radial floats per edge
    static constexpr uint32_t kGBytes = R * kC32 * 4;       // cotangent bytes per edge
    static constexpr int kPB = 32 / T;
    float* gs;      // [S][T][R*32]
    float* rads;    // [S][T][LM*32]
    float* coups;   // [S][T*R]
    int* meta;      // [S][T]: destination, -1 for an edge without a node, -2 past the window
    uint32_t bar0;
    int p0, p1, ntiles, issued, consumed;
    int blk_cur, blk_next;   // dst of the 32 edges of the current / next block
    uint64_t pol_stream, pol_g;
    int hot;        // destination whose cotangent rows the CTA holds in its hot slot, kNoHot for none

    __device__ __forceinline__ void init(unsigned char* base, int p0_, int p1_, int lane, int stream_hint) {
        gs = reinterpret_cast<float*>(base);
        rads = reinterpret_cast<float*>(base + Layout::kG);
        coups = reinterpret_cast<float*>(base + Layout::kG + Layout::kRad);
        meta = reinterpret_cast<int*>(base + Layout::kG + Layout::kRad + Layout::kCoup);
        bar0 = smem_u32(base + Layout::kG + Layout::kRad + Layout::kCoup + Layout::kMeta);
        p0 = p0_;
        p1 = p1_;
        ntiles = p1 > p0 ? (p1 - p0 + T - 1) / T : 0;
        issued = 0;
        consumed = 0;
        pol_stream = l2_policy(stream_hint);
        pol_g = l2_evict_last();
        hot = kNoHot;
        if (lane < S) mbar_init(bar0 + 8 * lane, kGPieces ? 33u : 1u);
        mbar_fence_init();
        __syncwarp();
    }

    __device__ __forceinline__ int load_block(const int32_t* __restrict__ dst, int blk, int lane) const {
        const int j = p0 + blk * 32 + lane;
        return (blk * kPB < ntiles && j < p1) ? ld_hint_i(dst + j, pol_stream) : -1;
    }

    __device__ __forceinline__ void prefetch(const int32_t* __restrict__ dst, int lane) {
        blk_cur = load_block(dst, 0, lane);
        blk_next = load_block(dst, 1, lane);
    }

    // Coupling rows are cld floats apart; coup_bulk says they are packed
    // (cld == R) from a 16-byte boundary, so a whole tile is one bulk copy.
    __device__ __forceinline__ void issue(const int32_t* __restrict__ dst, const float* __restrict__ coup_g, int cld,
                                          bool coup_bulk, const float* __restrict__ rad_g,
                                          const float* __restrict__ g_g, int N, int lane) {
        if (issued >= ntiles) return;
        const int k = issued;
        const int st = k % S;
        const int sub = k % kPB;
        const int d = __shfl_sync(0xffffffffu, blk_cur, (sub * T + lane) & 31);
        ++issued;
        if (sub == kPB - 1) {
            blk_cur = blk_next;
            blk_next = load_block(dst, issued / kPB + 1, lane);
        }
        const int e0 = p0 + k * T;
        const int cnt = imin(T, p1 - e0);
        const bool in = lane < cnt;
        const bool valid = in && d >= 0 && d < N;
        const bool fetch = valid && d != hot;
        const bool full = cnt == T && coup_bulk && (T * R) % 4 == 0;
        const uint32_t nfetch = __popc(__ballot_sync(0xffffffffu, fetch));
        const uint32_t bytes = (uint32_t)cnt * (RF * 4u) + (full ? (uint32_t)T * R * 4u : 0u) + (kGPieces ? 0u : nfetch * kGBytes);
        const uint32_t bar = bar0 + 8 * st;
        float* cst = coups + st * T * R;
        if (lane < T) meta[st * T + lane] = valid ? d : (in ? -1 : -2);
        if (!full && in) {   // ragged last tile, or rows not packed: plain loads of each row
            const float* src = coup_g + (int64_t)(e0 + lane) * cld;
#pragma unroll
            for (int r = 0; r < R; ++r) cst[lane * R + r] = __ldg(src + r);
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(smem_u32(rads + st * T * RF), rad_g + (int64_t)e0 * RF, (uint32_t)cnt * (RF * 4u), bar,
                     pol_stream);
            if (full) bulk_g2s(smem_u32(cst), coup_g + (int64_t)e0 * R, (uint32_t)T * R * 4u, bar, pol_stream);
        }
        __syncwarp();
        if constexpr (kGPieces) {
            constexpr int kPieces = R * kC32 / 4;
#pragma unroll
            for (int j = 0; j < T; ++j) {
                const int dj = __shfl_sync(0xffffffffu, d, j);
                const bool fj = __shfl_sync(0xffffffffu, fetch, j);
#pragma unroll
                for (int q = lane; q < kPieces; q += 32)
                    if (fj)
                        cp_async16(smem_u32(gs + (st * T + j) * (R * kC32)) + 16 * q,
                                   g_g + (int64_t)dj * (D * kC32) + kC32 + 4 * q, pol_g);
            }
            cp_async_arrive(bar);
        } else if (fetch) {
            bulk_g2s(smem_u32(gs + (st * T + lane) * (R * kC32)), g_g + (int64_t)d * (D * kC32) + kC32, kGBytes,
                     bar, pol_g);
        }
    }

    __device__ __forceinline__ int acquire() {
        const int k = consumed++;
        const int st = k % S;
        mbar_wait(bar0 + 8 * st, (uint32_t)((k / S) & 1));
        __syncwarp();
        return st;
    }

    __device__ __forceinline__ void drain() {
        while (consumed < issued) {
            const int st = consumed % S;
            mbar_wait(bar0 + 8 * st, (uint32_t)((consumed / S) & 1));
            ++consumed;
        }
        __syncwarp();
    }
};

// L2 policies of the edge-order backward's streams, chosen by measurement.
// While the cotangent block is small next to L2 (kSmallCotangentBytes), the
// radial, coupling and dst reads are evict-normal and the d_rad rows
// evict-last: on the 4096-node graph that made the backward 4 % faster and
// the kernel launched after it faster too (the cause was not isolated).  A
// larger block loses its lines to evict-last stores (the 32768-node backward
// was a third slower), so there the streams and the stores are evict-first.
struct StreamPolicy {
    int reads;    // L2 hint of the radial, coupling and dst reads
    int grads;    // L2 hint of the d_rad stores
};
__host__ __device__ constexpr StreamPolicy stream_policy(bool small_cotangent) {
    return small_cotangent ? StreamPolicy{kL2Normal, kL2EvictLast} : StreamPolicy{kL2EvictFirst, kL2EvictFirst};
}

// --------------------------------------------------------------------------
// The edge-order C == 32 backward for the ladder of degree LM in the quad
// lane layout: one edge per 8-lane group, lane q owns channels 4q..4q+3 of
// all R rows, each cotangent row is read once from shared memory and feeds
// both gradients (the radial slot's running sum and the row's dot product
// with the radial row), and the R coupling-gradient dot products are summed
// over the group by one transposed butterfly of 8K values, K = ceil(R / 8).
// --------------------------------------------------------------------------

template <int W, int S, int T, int LM, bool kGeneral>
__global__ void __launch_bounds__(W * 32, 1)
bwd_edge_quad(const float* __restrict__ g, const float* __restrict__ coup, const float* __restrict__ rad,
              const int32_t* __restrict__ dst, int E, int32_t N, int KW, int Wtot,
              float* __restrict__ d_coup, float* __restrict__ d_rad, const float* __restrict__ scale_arg,
              int cld_arg, int dld_arg, int coup_bulk_arg, StreamPolicy pol) {
    static_assert(T % 4 == 0, "tiles hold whole groups of four edges");
    constexpr int R = Ladder<LM>::R, D = Ladder<LM>::D, RF = LM * kC32;
    constexpr int K = (R + 7) / 8;
    constexpr bool kEarlyRefill = T == 4 && R <= 15;   // one edge per group, its rows fit in registers
    using Ring = EdgeRing<S, T, LM>;
    using Layout = EdgeRingLayout<S, T, LM>;
    const float* __restrict__ scale = kGeneral ? scale_arg : nullptr;
    const int cld = kGeneral ? cld_arg : R, dld = kGeneral ? dld_arg : R;
    const int coup_bulk = kGeneral ? coup_bulk_arg : 1;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int hot_cand[W][2];
    const int warp = threadIdx.x >> 5;
    const QuadLane Q(threadIdx.x & 31);
    const int gw = blockIdx.x * W + warp;
    const bool active = gw < Wtot;
    pdl_wait();
    pdl_trigger();
    const int p0 = active ? (int)imin<int64_t>((int64_t)gw * KW, E) : E;
    const int p1 = active ? (int)imin<int64_t>((int64_t)p0 + KW, E) : E;
    Ring ring;
    ring.init(smem + (size_t)warp * Layout::kBytes, p0, p1, Q.lane, pol.reads);
    float* hot_g = reinterpret_cast<float*>(smem + (size_t)W * Layout::kBytes);
    const uint64_t pol_out = l2_policy(pol.grads);
    int sample = -1;
    if (active) {
        ring.prefetch(dst, Q.lane);
        // votes only for destinations that are nodes (others have no cotangent rows)
        sample = (ring.blk_cur >= 0 && ring.blk_cur < N) ? ring.blk_cur : -1;
#pragma unroll
        for (int i = 0; i < S; ++i) ring.issue(dst, coup, cld, coup_bulk != 0, rad, g, N, Q.lane);
    }
    const int hot = kHotSlot ? cta_hot_node<W>(sample, Q.lane, warp, hot_cand) : kNoHot;
    if (hot >= 0) {
        const float4* src = reinterpret_cast<const float4*>(g + (int64_t)hot * (D * kC32) + kC32);
        for (int t = threadIdx.x; t < R * kC32 / 4; t += W * 32) reinterpret_cast<float4*>(hot_g)[t] = __ldg(src + t);
        __syncthreads();
    }
    ring.hot = hot;
    if (active) {
        for (int k = 0; k < ring.ntiles; ++k) {
            const int st = ring.acquire();
            const int e0 = p0 + k * T;
            if constexpr (kEarlyRefill) {
                // One edge per group: its rows go to registers first, and the
                // stage is refilled before the arithmetic, so the next tile's
                // copies are in flight a few hundred cycles sooner (the ring
                // is only two stages deep).  Same arithmetic, same order.
                const int j = Q.grp;
                const int m = ring.meta[st * T + j];
                const float sc = (scale && m >= 0) ? __ldg(scale + m) : 1.f;
                const float* gj = (m == hot ? hot_g : ring.gs + (st * T + j) * (R * kC32)) + 4 * Q.q;
                const float* rrow = ring.rads + (st * T + j) * RF + 4 * Q.q;
                float4 a[LM];
#pragma unroll
                for (int l = 0; l < LM; ++l) a[l] = *reinterpret_cast<const float4*>(rrow + l * kC32);
                const float* crow = ring.coups + st * T * R + j * R;
                float c[R];
#pragma unroll
                for (int r = 0; r < R; ++r) c[r] = crow[r];
                float4 G[R];
#pragma unroll
                for (int r = 0; r < R; ++r) G[r] = *reinterpret_cast<const float4*>(gj + r * kC32);
                __syncwarp();
                ring.issue(dst, coup, cld, coup_bulk != 0, rad, g, N, Q.lane);
                float4 sl[LM];
                float pr[8 * K];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int l = ladder_slot(r);
                    if ((l + 1) * (l + 1) - 1 == r)   // first row of its degree
                        sl[l] = make_float4(c[r] * G[r].x, c[r] * G[r].y, c[r] * G[r].z, c[r] * G[r].w);
                    else
                        sl[l] = f4_fma(c[r], G[r], sl[l]);
                    pr[r] = f4_dot(G[r], a[l]);
                }
#pragma unroll
                for (int r = R; r < 8 * K; ++r) pr[r] = 0.f;
                float t[K];
                group_reduce<K>(pr, Q, t);
                if (m == -2) continue;
                const bool ok = m >= 0;
                const int64_t e = e0 + j;
                const int row = 4 * K * Q.b2 + 2 * K * Q.b1 + K * Q.b0;
                float* dc = d_coup + e * dld + row;
                float* dr = d_rad + e * RF + 4 * Q.q;
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                if (scale && ok) {   // gradients of the scaled output: the destination's scale times these
#pragma unroll
                    for (int l = 0; l < LM; ++l) sl[l] = make_float4(sl[l].x * sc, sl[l].y * sc, sl[l].z * sc, sl[l].w * sc);
#pragma unroll
                    for (int q = 0; q < K; ++q) t[q] *= sc;
                }
#pragma unroll
                for (int l = 0; l < LM; ++l) st_hint4(dr + l * kC32, ok ? sl[l] : z, pol_out);
#pragma unroll
                for (int q = 0; q < K; ++q)
                    if (row + q < R) st_stream(dc + q, ok ? t[q] : 0.f);
            } else {
#pragma unroll
            for (int i = 0; i < T / 4; ++i) {
                const int j = 4 * i + Q.grp;
                const int m = ring.meta[st * T + j];
                const float sc = (scale && m >= 0) ? __ldg(scale + m) : 1.f;   // issued early, used at the stores
                const float* gj = (m == hot ? hot_g : ring.gs + (st * T + j) * (R * kC32)) + 4 * Q.q;
                const float* rrow = ring.rads + (st * T + j) * RF + 4 * Q.q;
                float4 a[LM];
#pragma unroll
                for (int l = 0; l < LM; ++l) a[l] = *reinterpret_cast<const float4*>(rrow + l * kC32);
                const float* crow = ring.coups + st * T * R + j * R;
                float c[R];
#pragma unroll
                for (int r = 0; r < R; ++r) c[r] = crow[r];
                float4 sl[LM];
                float pr[8 * K];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float4 G = *reinterpret_cast<const float4*>(gj + r * kC32);
                    const int l = ladder_slot(r);
                    if ((l + 1) * (l + 1) - 1 == r)   // first row of its degree
                        sl[l] = make_float4(c[r] * G.x, c[r] * G.y, c[r] * G.z, c[r] * G.w);
                    else
                        sl[l] = f4_fma(c[r], G, sl[l]);
                    pr[r] = f4_dot(G, a[l]);
                }
#pragma unroll
                for (int r = R; r < 8 * K; ++r) pr[r] = 0.f;
                float t[K];
                group_reduce<K>(pr, Q, t);
                if (m == -2) continue;
                const bool ok = m >= 0;
                const int64_t e = e0 + j;
                const int row = 4 * K * Q.b2 + 2 * K * Q.b1 + K * Q.b0;
                float* dc = d_coup + e * dld + row;
                float* dr = d_rad + e * RF + 4 * Q.q;
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                if (scale && ok) {   // gradients of the scaled output: the destination's scale times these
#pragma unroll
                    for (int l = 0; l < LM; ++l) sl[l] = make_float4(sl[l].x * sc, sl[l].y * sc, sl[l].z * sc, sl[l].w * sc);
#pragma unroll
                    for (int q = 0; q < K; ++q) t[q] *= sc;
                }
#pragma unroll
                for (int l = 0; l < LM; ++l) st_hint4(dr + l * kC32, ok ? sl[l] : z, pol_out);
#pragma unroll
                for (int q = 0; q < K; ++q)
                    if (row + q < R) st_stream(dc + q, ok ? t[q] : 0.f);
            }
            __syncwarp();
            ring.issue(dst, coup, cld, coup_bulk != 0, rad, g, N, Q.lane);
            }
        }
    }
    ring.drain();
}

// Per-channel CSR-order backward (any C, any alignment): same walk, no TMA.
template <int L>
__global__ void __launch_bounds__(kBwdThreads)
bwd_csr_gen(const float* __restrict__ g, const float* __restrict__ coup, const float* __restrict__ rad,
            const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ perm,
            int64_t E, int32_t N, int C, int64_t KW, int Wtot,
            float* __restrict__ d_coup, float* __restrict__ d_rad) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kBwdWarps + warp;
    pdl_wait();
    pdl_trigger();
    if (gw >= Wtot) return;
    const int64_t p0 = (int64_t)gw * KW;
    const int64_t p1 = imin<int64_t>(p0 + KW, E);
    const int64_t vend = __ldg(row_ptr + N);
    int n = p0 < vend ? first_node_warp(row_ptr, N, p0, lane) : N;
    for (int64_t pos = p0; pos < p1; ++pos) {
        int d = -1;
        if (pos < vend) {
            while ((int64_t)__ldg(row_ptr + n + 1) <= pos) ++n;
            d = n;
        }
        const int e = __ldg(perm + pos);
        if ((uint32_t)e >= (uint64_t)E) continue;
        bwd_gen_edge<L>(g, coup, rad, e, d, C, lane, d_coup, d_rad);
    }
}

constexpr int64_t kSmallCotangentBytes = int64_t(16) << 20;   // 16 MiB
#ifndef ZS_EDGE_SMALL_W
#define ZS_EDGE_SMALL_W 12
#endif
#ifndef ZS_EDGE_SMALL_S
#define ZS_EDGE_SMALL_S 2
#endif
#ifndef ZS_EDGE_SMALL_T
#define ZS_EDGE_SMALL_T 4
#endif
constexpr int kEdgeWarpsSmall = ZS_EDGE_SMALL_W;   // 2-stage rings of 4 edges: 12 warps fit one SM's shared memory
constexpr int kEdgeStagesSmall = ZS_EDGE_SMALL_S;
constexpr int kEdgeTileSmall = ZS_EDGE_SMALL_T;
constexpr int kEdgeWarpsLarge = 8;    // 3-stage rings of 4 edges: 8 warps

// One warp waits on an mbarrier that nothing arrives on, with a limit of
// max_spins tries: the wait gives up, counts a timeout and the kernel ends.
__global__ void __launch_bounds__(32) selftest_wait(uint32_t max_spins) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) mbar_init(b, 1);
    mbar_fence_init();
    __syncwarp();
    if (threadIdx.x == 0) mbar_wait(b, 0, max_spins);
    __syncwarp();
}

}  // namespace

unsigned int take_timeouts_backward() { return take_timeouts_local(); }
cudaError_t set_timeout_flag_backward(unsigned int* flag) { return set_timeout_flag_local(flag); }

zs_status selftest_bounded_wait(uint32_t max_spins, cudaStream_t s) {
    selftest_wait<<<1, 32, 0, s>>>(max_spins);
    return check_launch("zs_selftest_bounded_wait");
}

// Gradient of the node scale of the scaled forward: d_scale[n] = sum over
// rows 1..D-1 and channels of g[n,r,c] * out_raw[n,r,c], one warp per node,
// lane-strided products added in a fixed order (float4 steps when both rows
// are 16-byte aligned, four steps in flight per lane).
__global__ void __launch_bounds__(kBwdThreads)
bwd_scale_grad(const float* __restrict__ g, const float* __restrict__ raw, int32_t N, int64_t node_floats, int C,
               float* __restrict__ d_scale) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * kBwdWarps + warp;
    pdl_wait();
    pdl_trigger();
    if (n >= N) return;
    const float* gp = g + n * node_floats + C;        // rows 1..D-1
    const float* rp = raw + n * node_floats + C;
    const int64_t len = node_floats - C;
    float acc = 0.f;
    if (aligned16(gp) && aligned16(rp) && (len & 3) == 0) {
        const float4* g4 = reinterpret_cast<const float4*>(gp);
        const float4* r4 = reinterpret_cast<const float4*>(rp);
        const int64_t len4 = len >> 2;
        int64_t i = lane;
        for (; i + 96 < len4; i += 128) {
            float4 a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a[u] = __ldg(g4 + i + 32 * u);
                b[u] = __ldg(r4 + i + 32 * u);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) acc += a[u].x * b[u].x + a[u].y * b[u].y + a[u].z * b[u].z + a[u].w * b[u].w;
        }
        for (; i < len4; i += 32) {
            const float4 a = __ldg(g4 + i), b = __ldg(r4 + i);
            acc += a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
        }
    } else {
        for (int64_t i = lane; i < len; i += 32) acc = fmaf(__ldg(gp + i), __ldg(rp + i), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
    if (lane == 0) d_scale[n] = acc;
}

template <int LM>
constexpr int rows_pick(const int (&v)[4]) { return v[LM <= 2 ? LM - 1 : LM - 2]; }

// Quad-layout edge backward of the other ladders: tiles of whole quads;
// stages and tile per ladder (chosen by timing), as many warps as the rings
// and the hot slot leave room for, at most 16.  lmax 3 uses the fixed
// configurations below (kEdgeWarpsSmall / kEdgeWarpsLarge).
#ifndef ZS_QUAD_T1
#define ZS_QUAD_T1 8
#endif
#ifndef ZS_QUAD_T2
#define ZS_QUAD_T2 4
#endif
#ifndef ZS_QUAD_T4
#define ZS_QUAD_T4 4
#endif
#ifndef ZS_QUAD_T5
#define ZS_QUAD_T5 4
#endif
#ifndef ZS_QUAD_S1
#define ZS_QUAD_S1 3
#endif
#ifndef ZS_QUAD_S2
#define ZS_QUAD_S2 3
#endif
#ifndef ZS_QUAD_S4
#define ZS_QUAD_S4 2
#endif
#ifndef ZS_QUAD_S5
#define ZS_QUAD_S5 2
#endif
// per ladder degree 1, 2, 4, 5
constexpr int kQuadTiles[4] = {ZS_QUAD_T1, ZS_QUAD_T2, ZS_QUAD_T4, ZS_QUAD_T5};
constexpr int kQuadStages[4] = {ZS_QUAD_S1, ZS_QUAD_S2, ZS_QUAD_S4, ZS_QUAD_S5};
template <int LM>
constexpr int quad_tile() { return rows_pick<LM>(kQuadTiles); }
template <int LM>
constexpr int quad_stages() { return rows_pick<LM>(kQuadStages); }
template <int LM>
constexpr int quad_hot_bytes() { return Ladder<LM>::R * kC32 * 4; }
template <int LM>
constexpr int quad_warps() {
    constexpr int bytes = EdgeRingLayout<quad_stages<LM>(), quad_tile<LM>(), LM>::kBytes;
    constexpr int avail = 232448 - quad_hot_bytes<LM>() - 16 * 8;   // the hot slot, the votes
    return avail / bytes < 16 ? avail / bytes : 16;
}

template <int LM, int W, int S, int T>
void launch_edge_quad(const float* g, const float* coup, int cld, const float* rad, const int32_t* dst, int64_t E,
                      int32_t N, float* d_coup, int dld, float* d_rad, const float* scale, cudaStream_t s) {
    constexpr int R = Ladder<LM>::R;
    const int64_t warps_max = (int64_t)num_sms() * W;
    const int64_t KW = imax<int64_t>((E + warps_max - 1) / warps_max + T - 1, T) / T * T;   // whole tiles
    const int64_t Wtot = imax<int64_t>((E + KW - 1) / KW, 1);
    const int64_t ctas = (Wtot + W - 1) / W;
    const int smem = W * EdgeRingLayout<S, T, LM>::kBytes + quad_hot_bytes<LM>();
    static_assert(W * EdgeRingLayout<S, T, LM>::kBytes + quad_hot_bytes<LM>() + W * 8 <= 232448,
                  "rings and hot slot fit an SM");
    const int bulk = (cld == R && aligned16(coup)) ? 1 : 0;
    const StreamPolicy pol = stream_policy((int64_t)N * Ladder<LM>::D * kC32 * 4 <= kSmallCotangentBytes);
    if (scale == nullptr && dld == R && bulk) {
        static std::atomic<uint64_t> attr_done[kMaxDevices];
        set_smem_limit_once(bwd_edge_quad<W, S, T, LM, false>, smem, attr_done);
        launch(bwd_edge_quad<W, S, T, LM, false>, (unsigned)ctas, W * 32, smem, s, g, coup, rad, dst, (int)E, N,
               (int)KW, (int)Wtot, d_coup, d_rad, scale, cld, dld, bulk, pol);
    } else {
        static std::atomic<uint64_t> attr_done[kMaxDevices];
        set_smem_limit_once(bwd_edge_quad<W, S, T, LM, true>, smem, attr_done);
        launch(bwd_edge_quad<W, S, T, LM, true>, (unsigned)ctas, W * 32, smem, s, g, coup, rad, dst, (int)E, N,
               (int)KW, (int)Wtot, d_coup, d_rad, scale, cld, dld, bulk, pol);
    }
}

template <int LM>
void launch_edge_quad_auto(const float* g, const float* coup, int cld, const float* rad, const int32_t* dst,
                           int64_t E, int32_t N, float* d_coup, int dld, float* d_rad, const float* scale,
                           cudaStream_t s) {
    launch_edge_quad<LM, quad_warps<LM>(), quad_stages<LM>(), quad_tile<LM>()>(g, coup, cld, rad, dst, E, N, d_coup,
                                                                                dld, d_rad, scale, s);
}

template <int L>
void launch_gen_edges(const float* g, const float* coup, int cld, const float* rad, const int32_t* dst, int64_t E,
                      int32_t N, int C, float* d_coup, int dld, float* d_rad, const float* scale, cudaStream_t s) {
    const int64_t want = (E + kBwdWarps - 1) / kBwdWarps;
    const int grid = (int)imin<int64_t>(want, (int64_t)num_sms() * 8);
    launch(bwd_gen<L>, grid, kBwdThreads, 0, s, g, coup, rad, dst, E, N, C, d_coup, d_rad, scale, cld, dld);
}

// CSR-order quad kernel: lmax 4 keeps 24 cotangent rows (96 registers) per
// lane, so fewer warps (more registers each) than the other ladders; lmax 5
// keeps its 35 rows in shared memory (17.5 KB a warp), so fewer, smaller tiles.
constexpr int kCsrQuadWarps4 = 8;
constexpr int kCsrQuadWarps5 = 8, kCsrQuadTile5 = 4;

template <int LM, int W, int S, int T>
void launch_csr_quad(const float* g, const float* coup, const float* rad, const int32_t* row_ptr,
                     const int32_t* perm, int64_t E, int32_t N, float* d_coup, float* d_rad, cudaStream_t s) {
    constexpr int R = Ladder<LM>::R;
    using Layout = RingLayout<S, T, LM * kC32, R>;
    const int64_t warps_max = (int64_t)num_sms() * W;
    const int64_t KW = imax<int64_t>((E + warps_max - 1) / warps_max, T);
    const int64_t Wtot = imax<int64_t>((E + KW - 1) / KW, 1);
    const int64_t ctas = (Wtot + W - 1) / W;
    constexpr int kGBytes = R > 24 ? R * 32 * 16 : 0;   // shared-memory cotangent rows per warp
    static_assert(W * (Layout::kBytes + kGBytes) <= 232448, "rings and cotangent rows fit an SM");
    const int smem = W * (Layout::kBytes + kGBytes);
    static std::atomic<uint64_t> attr_done[kMaxDevices];
    set_smem_limit_once(bwd_csr_quad<W, S, T, LM>, smem, attr_done);
    launch(bwd_csr_quad<W, S, T, LM>, (unsigned)ctas, W * 32, smem, s, g, coup, rad, row_ptr, perm, (int)E, N,
           (int)KW, (int)Wtot, d_coup, d_rad);
}

template <int L>
void launch_gen_csr(const float* g, const float* coup, const float* rad, const int32_t* row_ptr,
                    const int32_t* perm, int64_t E, int32_t N, int C, float* d_coup, float* d_rad, cudaStream_t s) {
    const int64_t KW = 64;
    const int64_t Wtot = (E + KW - 1) / KW;
    const int64_t ctas = (Wtot + kBwdWarps - 1) / kBwdWarps;
    launch(bwd_csr_gen<L>, (unsigned)ctas, kBwdThreads, 0, s, g, coup, rad, row_ptr, perm, E, N, C, KW, (int)Wtot,
           d_coup, d_rad);
}

}  // namespace zs

using namespace zs;

static zs_status backward_impl(const char* name, const float* g, const float* coup, int64_t cld, const float* rad,
                               const int32_t* dst, int64_t E, int32_t N, int32_t C, int32_t lmax,
                               float* d_coup, int64_t dld, float* d_rad, const float* scale, cudaStream_t s) {
    if (lmax < 1 || lmax > kMaxLmax)
        return fail(ZS_ERR_UNSUPPORTED, "%s: lmax=%d, supported ladders are lmax 1..%d", name, lmax, kMaxLmax);
    if (E < 0 || N < 0 || C < 1) return fail(ZS_ERR_INVALID_ARG, "%s: bad sizes E=%lld N=%d C=%d", name, (long long)E, N, C);
    if (E >= ((int64_t)1 << 31) - 1) return fail(ZS_ERR_INVALID_ARG, "%s: E=%lld exceeds the int32 index range", name, (long long)E);
    const int R = ladder_rows(lmax);
    if (cld < R || dld < R || cld > ((int64_t)1 << 24) || dld > ((int64_t)1 << 24))
        return fail(ZS_ERR_INVALID_ARG, "%s: row strides %lld / %lld below %d rows or too large", name, (long long)cld,
                    (long long)dld, R);
    if (E == 0) return ZS_OK;
    if (!coup || !rad || !dst || !d_coup || !d_rad) return fail(ZS_ERR_INVALID_ARG, "%s: NULL array with E > 0", name);
    if (N > 0 && !g) return fail(ZS_ERR_INVALID_ARG, "%s: g is NULL with N > 0", name);
    // coupling rows and d_coup may have any stride and 4-byte alignment on every path
    const bool fast = lmax == 3 && C == kC32 && aligned16(g) && aligned16(rad) && aligned16(d_rad);
    const bool rows = lmax != 3 && C == kC32 && aligned16(g) && aligned16(rad) && aligned16(d_rad);
    if (rows) {
        const int c = (int)cld, d = (int)dld;
        switch (lmax) {
            case 1: launch_edge_quad_auto<1>(g, coup, c, rad, dst, E, N, d_coup, d, d_rad, scale, s); break;
            case 2: launch_edge_quad_auto<2>(g, coup, c, rad, dst, E, N, d_coup, d, d_rad, scale, s); break;
            case 4: launch_edge_quad_auto<4>(g, coup, c, rad, dst, E, N, d_coup, d, d_rad, scale, s); break;
            default: launch_edge_quad_auto<5>(g, coup, c, rad, dst, E, N, d_coup, d, d_rad, scale, s); break;
        }
    } else if (fast) {
        // While the cotangent block is small enough to stay in L2 next to the
        // streams, more warps with one tile in flight each hide the gather
        // latency best; a larger block misses L2 more often and wants more
        // tiles in flight per warp.
        const bool small_g = (int64_t)N * 16 * kC32 * 4 <= kSmallCotangentBytes;
        if (small_g)
            launch_edge_quad<3, kEdgeWarpsSmall, kEdgeStagesSmall, kEdgeTileSmall>(g, coup, (int)cld, rad, dst, E, N, d_coup,
                                                                                    (int)dld, d_rad, scale, s);
        else
            launch_edge_quad<3, kEdgeWarpsLarge, 3, 4>(g, coup, (int)cld, rad, dst, E, N, d_coup, (int)dld, d_rad, scale, s);
    } else {
        const int c = (int)cld, d = (int)dld;
        switch (lmax) {
            case 1: launch_gen_edges<1>(g, coup, c, rad, dst, E, N, C, d_coup, d, d_rad, scale, s); break;
            case 2: launch_gen_edges<2>(g, coup, c, rad, dst, E, N, C, d_coup, d, d_rad, scale, s); break;
            case 3: launch_gen_edges<3>(g, coup, c, rad, dst, E, N, C, d_coup, d, d_rad, scale, s); break;
            case 4: launch_gen_edges<4>(g, coup, c, rad, dst, E, N, C, d_coup, d, d_rad, scale, s); break;
            default: launch_gen_edges<5>(g, coup, c, rad, dst, E, N, C, d_coup, d, d_rad, scale, s); break;
        }
    }
    return check_launch(name);
}

extern "C" zs_status zs_backward(const float* g, const float* coup, const float* rad,
                                 const int32_t* dst, int64_t E, int32_t N, int32_t C, int32_t lmax,
                                 float* d_coup, float* d_rad, zs_stream_t stream) {
    const int R = ladder_rows(lmax < 1 ? 1 : (lmax > kMaxLmax ? kMaxLmax : lmax));
    return backward_impl("zs_backward", g, coup, R, rad, dst, E, N, C, lmax, d_coup, R, d_rad, nullptr,
                         reinterpret_cast<cudaStream_t>(stream));
}

extern "C" zs_status zs_backward_ld(const float* g, const float* coup, int64_t coup_ld, const float* rad,
                                    const int32_t* dst, int64_t E, int32_t N, int32_t C, int32_t lmax,
                                    float* d_coup, int64_t d_coup_ld, float* d_rad, zs_stream_t stream) {
    return backward_impl("zs_backward_ld", g, coup, coup_ld, rad, dst, E, N, C, lmax, d_coup, d_coup_ld, d_rad,
                         nullptr, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" zs_status zs_backward_scaled(const float* g, const float* coup, const float* rad, const int32_t* dst,
                                        const float* node_scale, const float* out_raw,
                                        int64_t E, int32_t N, int32_t C, int32_t lmax,
                                        float* d_coup, float* d_rad, float* d_scale, zs_stream_t stream) {
    if (N > 0 && !node_scale) return fail(ZS_ERR_INVALID_ARG, "zs_backward_scaled: node_scale is NULL");
    if (N > 0 && d_scale && (!out_raw || !g))
        return fail(ZS_ERR_INVALID_ARG, "zs_backward_scaled: d_scale needs out_raw and g");
    if (lmax < 1 || lmax > kMaxLmax)
        return fail(ZS_ERR_UNSUPPORTED, "zs_backward_scaled: lmax=%d, supported ladders are lmax 1..%d", lmax, kMaxLmax);
    if (E < 0 || N < 0 || C < 1)
        return fail(ZS_ERR_INVALID_ARG, "zs_backward_scaled: bad sizes E=%lld N=%d C=%d", (long long)E, N, C);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (N > 0 && d_scale) {
        const int64_t node_floats = (int64_t)(lmax + 1) * (lmax + 1) * C;
        launch(bwd_scale_grad, (unsigned)((N + kBwdWarps - 1) / kBwdWarps), kBwdThreads, 0, s, g, out_raw, N,
               node_floats, (int)C, d_scale);
        const zs_status st = check_launch("zs_backward_scaled");
        if (st != ZS_OK) return st;
    }
    const int R = ladder_rows(lmax);
    return backward_impl("zs_backward_scaled", g, coup, R, rad, dst, E, N, C, lmax, d_coup, R, d_rad, node_scale, s);
}

extern "C" zs_status zs_backward_csr(const float* g, const float* coup, const float* rad,
                                     const int32_t* row_ptr, const int32_t* perm,
                                     int64_t E, int32_t N, int32_t C, int32_t lmax,
                                     float* d_coup, float* d_rad, zs_stream_t stream) {
    if (lmax < 1 || lmax > kMaxLmax)
        return fail(ZS_ERR_UNSUPPORTED, "zs_backward_csr: lmax=%d, supported ladders are lmax 1..%d", lmax, kMaxLmax);
    if (E < 0 || N < 0 || C < 1) return fail(ZS_ERR_INVALID_ARG, "zs_backward_csr: bad sizes E=%lld N=%d C=%d", (long long)E, N, C);
    if (E >= ((int64_t)1 << 31) - 1) return fail(ZS_ERR_INVALID_ARG, "zs_backward_csr: E=%lld exceeds the int32 index range", (long long)E);
    if (!row_ptr) return fail(ZS_ERR_INVALID_ARG, "zs_backward_csr: row_ptr is NULL");
    if (E == 0) return ZS_OK;
    if (!coup || !rad || !perm || !d_coup || !d_rad) return fail(ZS_ERR_INVALID_ARG, "zs_backward_csr: NULL array with E > 0");
    if (N > 0 && !g) return fail(ZS_ERR_INVALID_ARG, "zs_backward_csr: g is NULL with N > 0");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool fast = C == kC32 && aligned16(g) && aligned16(rad) && aligned16(d_rad) && aligned16(coup);
    if (fast) {
        constexpr int S = ZS_BWD_STAGES, T = ZS_BWD_TILE;
        switch (lmax) {
            case 1: launch_csr_quad<1, ZS_BWD_WARPS, S, T>(g, coup, rad, row_ptr, perm, E, N, d_coup, d_rad, s); break;
            case 2: launch_csr_quad<2, ZS_BWD_WARPS, S, T>(g, coup, rad, row_ptr, perm, E, N, d_coup, d_rad, s); break;
            case 3: launch_csr_quad<3, ZS_BWD_WARPS, S, T>(g, coup, rad, row_ptr, perm, E, N, d_coup, d_rad, s); break;
            case 4: launch_csr_quad<4, kCsrQuadWarps4, S, T>(g, coup, rad, row_ptr, perm, E, N, d_coup, d_rad, s); break;
            default:
                launch_csr_quad<5, kCsrQuadWarps5, S, kCsrQuadTile5>(g, coup, rad, row_ptr, perm, E, N, d_coup, d_rad, s);
                break;
        }
    } else {
        switch (lmax) {
            case 1: launch_gen_csr<1>(g, coup, rad, row_ptr, perm, E, N, C, d_coup, d_rad, s); break;
            case 2: launch_gen_csr<2>(g, coup, rad, row_ptr, perm, E, N, C, d_coup, d_rad, s); break;
            case 3: launch_gen_csr<3>(g, coup, rad, row_ptr, perm, E, N, C, d_coup, d_rad, s); break;
            case 4: launch_gen_csr<4>(g, coup, rad, row_ptr, perm, E, N, C, d_coup, d_rad, s); break;
            default: launch_gen_csr<5>(g, coup, rad, row_ptr, perm, E, N, C, d_coup, d_rad, s); break;
        }
    }
    return check_launch("zs_backward_csr");
}
