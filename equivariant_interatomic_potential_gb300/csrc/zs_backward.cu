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
#define ZS_BWD_WARPS 14
#endif
#ifndef ZS_BWD_STAGES
#define ZS_BWD_STAGES 2
#endif
#ifndef ZS_BWD_TILE
#define ZS_BWD_TILE 16
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

// Gradients of the edge at tile slot j, whose node's cotangent rows are in
// gr (rows 4g..4g+3 of this lane's group, channels 4q..4q+3).
struct BwdLane {
    int lane, gq, q, slo, shi, my_row;
    bool b2, b1, row_writer;
    __device__ __forceinline__ explicit BwdLane(int l) : lane(l), gq(l >> 3), q(l & 7) {
        slo = gq == 0 ? 0 : (gq == 1 ? 1 : 2);
        shi = gq == 0 ? 1 : slo;
        b2 = (lane & 4) != 0;
        b1 = (lane & 2) != 0;
        my_row = 4 * gq + (b2 ? 2 : 0) + (b1 ? 1 : 0);
        row_writer = (lane & 1) == 0 && my_row < 15;
    }
};

template <int S, int T>
__device__ __forceinline__ void bwd_edge32(const TileRing<S, T>& ring, int st, int j, const float4 gr[4],
                                           const BwdLane& B, float* __restrict__ d_coup, float* __restrict__ d_rad) {
    const int2 m = ring.meta[st * T + j];
    const float* rrow = ring.rad + (st * T + j) * 96;
    const float4 a = *reinterpret_cast<const float4*>(rrow + B.slo * kC32 + 4 * B.q);
    const float4 bb = *reinterpret_cast<const float4*>(rrow + B.shi * kC32 + 4 * B.q);
    const float* crow = ring.coup + (st * T + j) * kCoupSlotFloats + m.y + 4 * B.gq;
    const float4 c4 = make_float4(crow[0], crow[1], crow[2], B.gq == 3 ? 0.f : crow[3]);
    // d_coup: four row dot products over this lane's 4 channels, then a
    // transposed butterfly over the 8 lanes of the group
    const float p0v = f4_dot(gr[0], a);
    const float p1v = f4_dot(gr[1], a);
    const float p2v = f4_dot(gr[2], a);
    const float p3v = f4_dot(gr[3], bb);
    const float x0 = B.b2 ? p0v : p2v, x1 = B.b2 ? p1v : p3v;
    const float k0 = (B.b2 ? p2v : p0v) + __shfl_xor_sync(kFull, x0, 4);
    const float k1 = (B.b2 ? p3v : p1v) + __shfl_xor_sync(kFull, x1, 4);
    float mm = (B.b1 ? k1 : k0) + __shfl_xor_sync(kFull, B.b1 ? k0 : k1, 2);
    mm += __shfl_xor_sync(kFull, mm, 1);
    // d_rad: the group's rows weighted by their coupling; the degree-2 slot
    // adds group 0's row 3, the degree-3 slot adds group 3's rows
    float4 lo = make_float4(c4.x * gr[0].x, c4.x * gr[0].y, c4.x * gr[0].z, c4.x * gr[0].w);
    lo = f4_fma(c4.y, gr[1], lo);
    lo = f4_fma(c4.z, gr[2], lo);
    const float4 hi = make_float4(c4.w * gr[3].x, c4.w * gr[3].y, c4.w * gr[3].z, c4.w * gr[3].w);
    const float4 both = f4_add(lo, hi);
    const float4 y = f4_shfl_xor(B.gq == 0 ? hi : both, 8);
    if (m.x < 0) return;
    const int64_t e = m.x;
    if (B.row_writer) st_stream(d_coup + e * 15 + B.my_row, mm);
    if (B.gq < 3) {
        const float4 res = B.gq == 0 ? lo : (B.gq == 1 ? f4_add(y, both) : f4_add(both, y));
        st_stream4(d_rad + e * (3 * kC32) + B.gq * kC32 + 4 * B.q, res);
    }
}

template <int W, int S, int T>
__global__ void __launch_bounds__(W * 32, 1)
bwd_csr_c32_tma(const float* __restrict__ g, const float* __restrict__ coup, const float* __restrict__ rad,
                const int32_t* __restrict__ row_ptr, const int32_t* __restrict__ perm,
                int E, int32_t N, int KW, int Wtot,
                float* __restrict__ d_coup, float* __restrict__ d_rad) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int warp = threadIdx.x >> 5;
    const BwdLane B(threadIdx.x & 31);
    const int gw = blockIdx.x * W + warp;
    const bool active = gw < Wtot;
    pdl_wait();
    pdl_trigger();
    const int p0 = active ? (int)imin<int64_t>((int64_t)gw * KW, E) : E;
    const int p1 = active ? (int)imin<int64_t>((int64_t)p0 + KW, E) : E;
    TileRing<S, T> ring;
    ring.init(smem + (size_t)warp * RingLayout<S, T>::kBytes, p0, p1, B.lane);
    if (active) {
        ring.prefetch_perm(perm, B.lane);
#pragma unroll
        for (int i = 0; i < S; ++i) ring.issue(perm, coup, rad, E, B.lane);
        const int vend = __ldg(row_ptr + N);
        int n = p0 < vend ? first_node_b(row_ptr, N, p0) : N;
        int b = 0;
        float4 gr[4] = {};
        auto enter = [&](int pos) {   // make node n the one holding position pos < vend
            while ((b = __ldg(row_ptr + n + 1)) <= pos) ++n;
            const float* gn = g + (int64_t)n * (16 * kC32) + 4 * B.q;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = 4 * B.gq + i;
                gr[i] = r < 15 ? ld_ro4(gn + (1 + r) * kC32) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        };
        if (p0 < vend) enter(p0);
        for (int k = 0; k < ring.ntiles; ++k) {
            const int st = ring.acquire();
            const int tb = p0 + k * T;
            const int jt = imin(T, p1 - tb);
            int j = 0;
            while (j < jt) {
                if (tb + j >= vend) {              // edges without a node: zero gradients
                    for (int jj = j; jj < jt; ++jj) {
                        const int e = ring.meta[st * T + jj].x;
                        if (e < 0) continue;
                        if (B.lane < 24) st_stream4(d_rad + (int64_t)e * (3 * kC32) + 4 * B.lane,
                                                    make_float4(0.f, 0.f, 0.f, 0.f));
                        if (B.lane < 15) st_stream(d_coup + (int64_t)e * 15 + B.lane, 0.f);
                    }
                    break;
                }
                if (tb + j >= b) {
                    ++n;
                    enter(tb + j);
                }
                const int stop = imin(b - tb, jt);
                if (j == 0 && stop == T) {
#pragma unroll
                    for (int jj = 0; jj < T; ++jj) bwd_edge32(ring, st, jj, gr, B, d_coup, d_rad);
                } else {
#pragma unroll 2
                    for (int jj = j; jj < stop; ++jj) bwd_edge32(ring, st, jj, gr, B, d_coup, d_rad);
                }
                j = stop;
            }
            ring.refill(perm, coup, rad, E, B.lane);
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
        static bool attr_set = false;
        if (!attr_set) {
            cudaFuncSetAttribute(bwd_csr_c32_tma<W, S, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            attr_set = true;
        }
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
