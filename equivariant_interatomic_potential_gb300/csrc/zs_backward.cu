// Backward of the zonal scatter, lmax = 3, one edge-parallel pass:
//   d_coup[e,r]  = sum_c g[dst[e],1+r,c] * rad[e,slot(r),c]
//   d_rad[e,s,c] = sum over rows r of slot s of g[dst[e],1+r,c] * coup[e,r]
// (deepmd-kit pull request "fused Triton zonal scatter for the GIE head",
// section "What", backward bullet: both operand gradients in a single
// edge-parallel kernel, no materialised message gradient).
//
// Edges are taken in their own order, 32 consecutive edges per warp step, so
// coup, rad, dst, d_coup and d_rad stream through HBM contiguously; the only
// gathered operand is g (N x 16 x C, a few MB, resident in L2).
#include "zs_common.cuh"
#include "zs_tma.cuh"

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
// C == 32 path.  Lane layout as in the forward: group g = lane/8 owns zonal
// rows 4g..4g+3 (row 15 padding), quad q = lane%8 owns channels 4q..4q+3.
// --------------------------------------------------------------------------
template <int U>
__global__ void __launch_bounds__(kBwdThreads, 2)
bwd_c32(const float* __restrict__ g, const float* __restrict__ coup, const float* __restrict__ rad,
        const int32_t* __restrict__ dst, int64_t E, int32_t N,
        float* __restrict__ d_coup, float* __restrict__ d_rad) {
    __shared__ __align__(16) float cs[kBwdWarps][32][16];
    __shared__ float dcs[kBwdWarps][32 * 15];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 3, q = lane & 7;
    const int slo = gq == 0 ? 0 : (gq == 1 ? 1 : 2);
    const int src_hi = gq == 0 ? lane + 8 : lane;
    const bool b2 = (lane & 4) != 0, b1 = (lane & 2) != 0;
    const int my_row = 4 * gq + (b2 ? 2 : 0) + (b1 ? 1 : 0);   // row this lane holds after the reduction
    const bool row_writer = (lane & 1) == 0 && my_row < 15;
    cs[warp][lane][15] = 0.f;
    __syncwarp();
    pdl_wait();
    pdl_trigger();

    const int64_t nbatch = (E + 31) / 32;
    for (int64_t bt = (int64_t)blockIdx.x * kBwdWarps + warp; bt < nbatch; bt += (int64_t)gridDim.x * kBwdWarps) {
        const int64_t e0 = bt * 32;
        const int cnt = (int)imin<int64_t>(32, E - e0);
        int d_l = -1;
        if (lane < cnt) {
            d_l = ld_stream_i(dst + e0 + lane);
            if (d_l < 0 || d_l >= N) d_l = -1;
        }
        const float* cblk = coup + e0 * 15;
#pragma unroll
        for (int it = 0; it < 15; ++it) {
            const int v = it * 32 + lane;
            const int j = v / 15;
            cs[warp][j][v - j * 15] = v < cnt * 15 ? ld_stream(cblk + v) : 0.f;
        }
        __syncwarp();

        for (int j0 = 0; j0 < cnt; j0 += U) {
            float4 gr[U][4], a[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + u;
                const int d = __shfl_sync(kFull, d_l, j & 31);
                const bool in = j < cnt;
                const float* gn = g + (int64_t)(d < 0 ? 0 : d) * (16 * kC32) + 4 * q;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = 4 * gq + i;
                    gr[u][i] = (in && d >= 0 && r < 15) ? ld_ro4(gn + (1 + r) * kC32)
                                                        : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                a[u] = in ? ld_stream4(rad + (e0 + j) * (3 * kC32) + slo * kC32 + 4 * q)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int j = j0 + u;
                const int d = __shfl_sync(kFull, d_l, j & 31);
                const bool ok = j < cnt && d >= 0;
                const float4 bb = f4_shfl(a[u], src_hi);
                const float4 c4 = *reinterpret_cast<const float4*>(&cs[warp][j & 31][4 * gq]);
                // d_coup: four row dot products over this lane's 4 channels,
                // then a transposed butterfly over the 8 lanes of the group.
                const float p0 = f4_dot(gr[u][0], a[u]);
                const float p1 = f4_dot(gr[u][1], a[u]);
                const float p2 = f4_dot(gr[u][2], a[u]);
                const float p3 = f4_dot(gr[u][3], bb);
                const float x0 = b2 ? p0 : p2, x1 = b2 ? p1 : p3;
                const float k0 = (b2 ? p2 : p0) + __shfl_xor_sync(kFull, x0, 4);
                const float k1 = (b2 ? p3 : p1) + __shfl_xor_sync(kFull, x1, 4);
                float m = (b1 ? k1 : k0) + __shfl_xor_sync(kFull, b1 ? k0 : k1, 2);
                m += __shfl_xor_sync(kFull, m, 1);
                if (row_writer && j < cnt) dcs[warp][(j & 31) * 15 + my_row] = ok ? m : 0.f;
                // d_rad: rows of the group weighted by their coupling, then the
                // degree-2 slot adds group 0's row 3 and the degree-3 slot adds group 3.
                float4 lo = make_float4(c4.x * gr[u][0].x, c4.x * gr[u][0].y, c4.x * gr[u][0].z, c4.x * gr[u][0].w);
                lo = f4_fma(c4.y, gr[u][1], lo);
                lo = f4_fma(c4.z, gr[u][2], lo);
                const float4 hi = make_float4(c4.w * gr[u][3].x, c4.w * gr[u][3].y, c4.w * gr[u][3].z, c4.w * gr[u][3].w);
                const float4 both = f4_add(lo, hi);
                const float4 y = f4_shfl_xor(gq == 0 ? hi : both, 8);
                if (gq < 3 && j < cnt) {
                    float4 res = gq == 0 ? lo : (gq == 1 ? f4_add(y, both) : f4_add(both, y));
                    if (!ok) res = make_float4(0.f, 0.f, 0.f, 0.f);
                    st_stream4(d_rad + (e0 + j) * (3 * kC32) + gq * kC32 + 4 * q, res);
                }
            }
        }
        __syncwarp();
        float* dblk = d_coup + e0 * 15;
#pragma unroll
        for (int it = 0; it < 15; ++it) {
            const int v = it * 32 + lane;
            if (v < cnt * 15) st_stream(dblk + v, dcs[warp][v]);
        }
        __syncwarp();
    }
}

// --------------------------------------------------------------------------
// Per-channel path (any C, any alignment): lane = channel within a chunk of
// 32; d_coup is reduced over the warp after the channel loop.
// --------------------------------------------------------------------------
// Gradients of one edge e whose destination is d (d < 0: no node, zero
// gradients), lane = channel within chunks of 32.
__device__ __forceinline__ void bwd_gen_edge(const float* __restrict__ g, const float* __restrict__ coup,
                                             const float* __restrict__ rad, int64_t e, int d, int C, int lane,
                                             float* __restrict__ d_coup, float* __restrict__ d_rad) {
    const bool ok = d >= 0;
    float cv[15];
#pragma unroll
    for (int r = 0; r < 15; ++r) cv[r] = __ldg(coup + e * 15 + r);
    float pc[15];
#pragma unroll
    for (int r = 0; r < 15; ++r) pc[r] = 0.f;
    const float* rp = rad + e * 3 * C;
    float* drp = d_rad + e * 3 * C;
    const float* gn = g + (int64_t)(ok ? d : 0) * 16 * C;
    for (int c = lane; c < C; c += 32) {
        if (!ok) {
            drp[c] = 0.f; drp[C + c] = 0.f; drp[2 * C + c] = 0.f;
            continue;
        }
        const float r0 = __ldg(rp + c), r1 = __ldg(rp + C + c), r2 = __ldg(rp + 2 * C + c);
        float s0 = 0.f, s1 = 0.f, s2 = 0.f;
#pragma unroll
        for (int r = 0; r < 15; ++r) {
            const float gv = __ldg(gn + (1 + r) * C + c);
            const float rv = r < 3 ? r0 : (r < 8 ? r1 : r2);
            pc[r] = fmaf(gv, rv, pc[r]);
            if (r < 3) s0 = fmaf(gv, cv[r], s0);
            else if (r < 8) s1 = fmaf(gv, cv[r], s1);
            else s2 = fmaf(gv, cv[r], s2);
        }
        drp[c] = s0; drp[C + c] = s1; drp[2 * C + c] = s2;
    }
#pragma unroll
    for (int r = 0; r < 15; ++r) {
        float v = pc[r];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
        pc[r] = v;
    }
    if (lane < 15) {
        float v = 0.f;
#pragma unroll
        for (int r = 0; r < 15; ++r) if (r == lane) v = pc[r];
        d_coup[e * 15 + lane] = ok ? v : 0.f;
    }
}

__global__ void __launch_bounds__(kBwdThreads)
bwd_gen(const float* __restrict__ g, const float* __restrict__ coup, const float* __restrict__ rad,
        const int32_t* __restrict__ dst, int64_t E, int32_t N, int C,
        float* __restrict__ d_coup, float* __restrict__ d_rad) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    for (int64_t e = (int64_t)blockIdx.x * kBwdWarps + warp; e < E; e += (int64_t)gridDim.x * kBwdWarps) {
        const int d = __ldg(dst + e);
        bwd_gen_edge(g, coup, rad, e, (d >= 0 && d < N) ? d : -1, C, lane, d_coup, d_rad);
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

__device__ __forceinline__ int first_node_b(const int32_t* __restrict__ row_ptr, int32_t N, int64_t p0) {
    const int n_lb = lower_bound_i32(row_ptr, N + 1, p0);
    if (n_lb >= 1 && n_lb <= N && (int64_t)__ldg(row_ptr + n_lb) > p0) return n_lb - 1;
    return n_lb;
}

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

// Sum of v over the 8 lanes of the group for 16 values at once: each lane
// ends with the totals of rows 8*b2 + 4*b1 + 2*b0 + {0, 1}.
__device__ __forceinline__ void group_reduce16(float v[16], const QuadLane& Q, float& r0, float& r1) {
    float w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float keep = Q.b2 ? v[k + 8] : v[k];
        const float send = Q.b2 ? v[k] : v[k + 8];
        w[k] = keep + __shfl_xor_sync(kFull, send, 4);
    }
    float x[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float keep = Q.b1 ? w[k + 4] : w[k];
        const float send = Q.b1 ? w[k] : w[k + 4];
        x[k] = keep + __shfl_xor_sync(kFull, send, 2);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const float keep = Q.b0 ? x[k + 2] : x[k];
        const float send = Q.b0 ? x[k] : x[k + 2];
        (k == 0 ? r0 : r1) = keep + __shfl_xor_sync(kFull, send, 1);
    }
}

template <int W, int S, int T>
__global__ void __launch_bounds__(W * 32, 1)
bwd_csr_c32_tma(const float* __restrict__ g, const float* __restrict__ coup, const float* __restrict__ rad,
                const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ perm,
                int E, int32_t N, int KW, int Wtot,
                float* __restrict__ d_coup, float* __restrict__ d_rad) {
    static_assert(T % 4 == 0, "tiles hold whole groups of four edges");
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const QuadLane Q(threadIdx.x & 31);
    const int gw = blockIdx.x * W + warp;
    const bool active = gw < Wtot;
    pdl_wait();
    pdl_trigger();
    const int p0 = active ? (int)imin<int64_t>((int64_t)gw * KW, E) : E;
    const int p1 = active ? (int)imin<int64_t>((int64_t)p0 + KW, E) : E;
    TileRing<S, T, true> ring;
    ring.init(smem + (size_t)warp * RingLayout<S, T>::kBytes, p0, p1, Q.lane);
    const uint64_t pol_first = l2_evict_first(), pol_last = l2_evict_last();
    if (active) {
        ring.prefetch_perm(perm, Q.lane);
#pragma unroll
        for (int i = 0; i < S; ++i) ring.issue(perm, coup, rad, E, Q.lane);
        const int vend = __ldg(row_ptr + N);
        // this group's node: n covers positions [.., b); G holds its rows 1..15
        int n = p0 < vend ? first_node_b(row_ptr, N, p0) : N;
        int b = n < N ? __ldg(row_ptr + n + 1) : 0;
        int c = 0;   // row_ptr[n + 2], fetched one node ahead
        float4 G[15];
        const float* gq = g + 4 * Q.q;
        auto load_g = [&]() {
            const float* gn = gq + (int64_t)n * (16 * kC32);
#pragma unroll
            for (int r = 0; r < 15; ++r) G[r] = ld_ro4(gn + (1 + r) * kC32);
        };
        if (p0 < vend) {
            while (b <= p0) b = __ldg(row_ptr + (++n) + 1);
            c = n + 2 <= N ? __ldg(row_ptr + n + 2) : 0;
            load_g();
        } else {
#pragma unroll
            for (int r = 0; r < 15; ++r) G[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int k = 0; k < ring.ntiles; ++k) {
            const int st = ring.acquire();
            const int tb = p0 + k * T;
            const int jt = imin(T, p1 - tb);
            const float* radst = ring.rad + st * T * 96 + 4 * Q.q;
            const float* coupst = ring.coup + st * T * kCoupSlotFloats;
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
                const float* rrow = radst + j * 96;
                const float4 a0 = *reinterpret_cast<const float4*>(rrow);
                const float4 a1 = *reinterpret_cast<const float4*>(rrow + kC32);
                const float4 a2 = *reinterpret_cast<const float4*>(rrow + 2 * kC32);
                const float* crow = coupst + j * kCoupSlotFloats + m.y;
                float c[15];
#pragma unroll
                for (int r = 0; r < 15; ++r) c[r] = crow[r];
                // radial gradient, one slot per degree group of rows
                float4 s0 = make_float4(c[0] * G[0].x, c[0] * G[0].y, c[0] * G[0].z, c[0] * G[0].w);
                s0 = f4_fma(c[1], G[1], s0);
                s0 = f4_fma(c[2], G[2], s0);
                float4 s1 = make_float4(c[3] * G[3].x, c[3] * G[3].y, c[3] * G[3].z, c[3] * G[3].w);
#pragma unroll
                for (int r = 4; r < 8; ++r) s1 = f4_fma(c[r], G[r], s1);
                float4 s2 = make_float4(c[8] * G[8].x, c[8] * G[8].y, c[8] * G[8].z, c[8] * G[8].w);
#pragma unroll
                for (int r = 9; r < 15; ++r) s2 = f4_fma(c[r], G[r], s2);
                // coupling gradient: per-row dot products over this lane's channels,
                // then summed over the group's 8 lanes
                float pr[16];
#pragma unroll
                for (int r = 0; r < 15; ++r) pr[r] = f4_dot(G[r], r < 3 ? a0 : (r < 8 ? a1 : a2));
                pr[15] = 0.f;
                float t0, t1;
                group_reduce16(pr, Q, t0, t1);
                const int e = m.x;
                if (in && e >= 0) {
                    const int row = 8 * Q.b2 + 4 * Q.b1 + 2 * Q.b0;
                    float* dc = d_coup + (int64_t)e * 15 + row;
                    float* dr = d_rad + (int64_t)e * (3 * kC32) + 4 * Q.q;
                    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                    // d_rad rows are whole lines: stream them out.  d_coup rows are 60 bytes in
                    // random order: keep their lines in L2 until neighbouring rows fill them
                    st_hint4(dr, has_node ? s0 : z, pol_first);
                    st_hint4(dr + kC32, has_node ? s1 : z, pol_first);
                    st_hint4(dr + 2 * kC32, has_node ? s2 : z, pol_first);
                    st_hint(dc, has_node ? t0 : 0.f, pol_last);
                    if (row + 1 < 15) st_hint(dc + 1, has_node ? t1 : 0.f, pol_last);
                }
            }
            ring.refill(perm, coup, rad, E, Q.lane);
        }
    }
    ring.drain();
}

// Per-channel CSR-order backward (any C, any alignment): same walk, no TMA.
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
    int n = p0 < vend ? first_node_b(row_ptr, N, p0) : N;
    for (int64_t pos = p0; pos < p1; ++pos) {
        int d = -1;
        if (pos < vend) {
            while ((int64_t)__ldg(row_ptr + n + 1) <= pos) ++n;
            d = n;
        }
        const int e = __ldg(perm + pos);
        if ((uint32_t)e >= (uint64_t)E) continue;
        bwd_gen_edge(g, coup, rad, e, d, C, lane, d_coup, d_rad);
    }
}

}  // namespace

unsigned int take_timeouts_backward() { return take_timeouts_local(); }

}  // namespace zs

using namespace zs;

extern "C" zs_status zs_backward(const float* g, const float* coup, const float* rad,
                                 const int32_t* dst, int64_t E, int32_t N, int32_t C, int32_t lmax,
                                 float* d_coup, float* d_rad, zs_stream_t stream) {
    if (lmax != 3) return fail(ZS_ERR_UNSUPPORTED, "zs_backward: lmax=%d, only lmax=3 (row groups 3/5/7) is supported", lmax);
    if (E < 0 || N < 0 || C < 1) return fail(ZS_ERR_INVALID_ARG, "zs_backward: bad sizes E=%lld N=%d C=%d", (long long)E, N, C);
    if (E >= ((int64_t)1 << 31) - 1) return fail(ZS_ERR_INVALID_ARG, "zs_backward: E=%lld exceeds the int32 index range", (long long)E);
    if (E == 0) return ZS_OK;
    if (!coup || !rad || !dst || !d_coup || !d_rad) return fail(ZS_ERR_INVALID_ARG, "zs_backward: NULL array with E > 0");
    if (N > 0 && !g) return fail(ZS_ERR_INVALID_ARG, "zs_backward: g is NULL with N > 0");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool fast = C == kC32 && aligned16(g) && aligned16(rad) && aligned16(d_rad);
    const int64_t nbatch = (E + 31) / 32;
    if (fast) {
        const int64_t want = (nbatch + kBwdWarps - 1) / kBwdWarps;
        const int grid = (int)imin<int64_t>(want, (int64_t)num_sms() * 2);
        launch(bwd_c32<4>, grid, kBwdThreads, 0, s, g, coup, rad, dst, E, N, d_coup, d_rad);
    } else {
        const int64_t want = (E + kBwdWarps - 1) / kBwdWarps;
        const int grid = (int)imin<int64_t>(want, (int64_t)num_sms() * 8);
        launch(bwd_gen, grid, kBwdThreads, 0, s, g, coup, rad, dst, E, N, C, d_coup, d_rad);
    }
    return check_launch("zs_backward");
}

extern "C" zs_status zs_backward_csr(const float* g, const float* coup, const float* rad,
                                     const int32_t* row_ptr, const int32_t* perm,
                                     int64_t E, int32_t N, int32_t C, int32_t lmax,
                                     float* d_coup, float* d_rad, zs_stream_t stream) {
    if (lmax != 3) return fail(ZS_ERR_UNSUPPORTED, "zs_backward_csr: lmax=%d, only lmax=3 (row groups 3/5/7) is supported", lmax);
    if (E < 0 || N < 0 || C < 1) return fail(ZS_ERR_INVALID_ARG, "zs_backward_csr: bad sizes E=%lld N=%d C=%d", (long long)E, N, C);
    if (E >= ((int64_t)1 << 31) - 1) return fail(ZS_ERR_INVALID_ARG, "zs_backward_csr: E=%lld exceeds the int32 index range", (long long)E);
    if (!row_ptr) return fail(ZS_ERR_INVALID_ARG, "zs_backward_csr: row_ptr is NULL");
    if (E == 0) return ZS_OK;
    if (!coup || !rad || !perm || !d_coup || !d_rad) return fail(ZS_ERR_INVALID_ARG, "zs_backward_csr: NULL array with E > 0");
    if (N > 0 && !g) return fail(ZS_ERR_INVALID_ARG, "zs_backward_csr: g is NULL with N > 0");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool fast = C == kC32 && aligned16(g) && aligned16(rad) && aligned16(d_rad) && aligned16(coup);
    if (fast) {
        constexpr int W = ZS_BWD_WARPS, S = ZS_BWD_STAGES, T = ZS_BWD_TILE;
        const int64_t warps_max = (int64_t)num_sms() * W;
        const int64_t KW = imax<int64_t>((E + warps_max - 1) / warps_max, T);
        const int64_t Wtot = imax<int64_t>((E + KW - 1) / KW, 1);
        const int64_t ctas = (Wtot + W - 1) / W;
        const int smem = W * RingLayout<S, T>::kBytes;
        static std::atomic<bool> attr_done[kMaxDevices];
        set_smem_limit_once(bwd_csr_c32_tma<W, S, T>, smem, attr_done);
        launch(bwd_csr_c32_tma<W, S, T>, (unsigned)ctas, W * 32, smem, s, g, coup, rad, row_ptr, perm, (int)E, N,
               (int)KW, (int)Wtot, d_coup, d_rad);
    } else {
        const int64_t KW = 64;
        const int64_t Wtot = (E + KW - 1) / KW;
        const int64_t ctas = (Wtot + kBwdWarps - 1) / kBwdWarps;
        launch(bwd_csr_gen, (unsigned)ctas, kBwdThreads, 0, s, g, coup, rad, row_ptr, perm, E, N, C, KW, (int)Wtot,
                                                            d_coup, d_rad);
    }
    return check_launch("zs_backward_csr");
}
