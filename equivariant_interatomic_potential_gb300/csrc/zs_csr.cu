// Stable destination CSR for the zonal scatter (row_ptr, perm).
//
// The forward of the deepmd-kit pull request "fused Triton zonal scatter for
// the GIE head" walks a destination CSR whose within-node order is the edge
// order ("stable-sort CSR order", section "What").  Built here as an LSD
// radix sort of destination keys with 8-bit digits, each pass in three
// launches with no inter-CTA waiting:
//   upsweep   -- per tile of keys, a 256-bin digit histogram (shared atomics)
//   scan      -- per digit, exclusive scan of its histogram row over tiles
//   downsweep -- per tile, stable rank of every key among equal digits
//                (warp ballots + per-warp running counts), staged in shared
//                memory in digit order and written out run by run
// and a final pass that reads the sorted keys to write row_ptr.
// Every step is integer arithmetic in a fixed order, so perm is unique and
// bit-identical to a sequential counting sort.  Keys outside [0, N) sort as
// key N, after all valid ones.
#include "zs_common.cuh"

namespace zs {
namespace {

constexpr int kCsrWarps = 8;
constexpr int kCsrThreads = kCsrWarps * 32;
#ifndef ZS_CSR_ITEMS
#define ZS_CSR_ITEMS 8
#endif
constexpr int kCsrItems = ZS_CSR_ITEMS;
constexpr int kTile = kCsrWarps * kCsrItems * 32;  // keys per tile
constexpr int kRadix = 256;

__device__ __forceinline__ int32_t key_of(const int32_t* keys_in, int64_t idx, int32_t N, bool first) {
    int32_t k = __ldg(keys_in + idx);
    if (first) k = (k >= 0 && k < N) ? k : N;
    return k;
}

// Lanes of the warp holding the same 8-bit digit as this lane (valid lanes
// only), from one ballot per digit bit (cheaper here than a match instruction).
__device__ __forceinline__ unsigned digit_peers(int dig, bool valid) {
    unsigned peers = __ballot_sync(0xffffffffu, valid);
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const bool bit = (dig >> b) & 1;
        const unsigned bal = __ballot_sync(0xffffffffu, bit);
        peers &= bit ? bal : ~bal;
    }
    return peers;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

template <bool kFirst>
__global__ void __launch_bounds__(kCsrThreads)
csr_upsweep(const int32_t* __restrict__ keys_in, int64_t E, int32_t N, int shift,
            int32_t* __restrict__ hist, int T) {
    __shared__ int cnt[kRadix];
    const int tid = threadIdx.x;
    cnt[tid] = 0;   // kCsrThreads == kRadix
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    // counts do not depend on the order of the increments
    const int64_t base = (int64_t)blockIdx.x * kTile;
    for (int i = tid; i < kTile; i += kCsrThreads) {
        const int64_t idx = base + i;
        if (idx < E) atomicAdd(&cnt[(key_of(keys_in, idx, N, kFirst) >> shift) & (kRadix - 1)], 1);
    }
    __syncthreads();
    hist[(int64_t)tid * T + blockIdx.x] = cnt[tid];
}

// One warp per digit: exclusive scan of hist[d, 0..T) in place, total to tot[d].
__global__ void __launch_bounds__(kCsrThreads)
csr_scan(int32_t* __restrict__ hist, int T, int32_t* __restrict__ tot) {
    constexpr int R = 8;
    const int lane = threadIdx.x & 31;
    const int d = blockIdx.x * kCsrWarps + (threadIdx.x >> 5);
    pdl_wait();
    pdl_trigger();
    if (d >= kRadix) return;
    int32_t* row = hist + (int64_t)d * T;
    int carry = 0;
    for (int base = 0; base < T; base += 32 * R) {
        int v[R];
        int s = 0;
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const int i = base + lane * R + k;
            v[k] = i < T ? row[i] : 0;
            s += v[k];
        }
        int incl = s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        int run = carry + incl - s;
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const int i = base + lane * R + k;
            if (i < T) row[i] = run;
            run += v[k];
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) tot[d] = carry;
}

template <bool kFirst>
__global__ void __launch_bounds__(kCsrThreads)
csr_downsweep(const int32_t* __restrict__ keys_in, const int32_t* __restrict__ vals_in,
              int64_t E, int32_t N, int shift,
              const int32_t* __restrict__ hist, const int32_t* __restrict__ tot, int T,
              int32_t* __restrict__ keys_out, int32_t* __restrict__ vals_out) {
    __shared__ int cnt[kCsrWarps][kRadix];
    __shared__ int wsum[kCsrWarps];
    __shared__ int dbase[kRadix];
    __shared__ int32_t skey[kTile], sval[kTile];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < kCsrWarps * kRadix; i += kCsrThreads) (&cnt[0][0])[i] = 0;
    pdl_wait();
    pdl_trigger();

    // Exclusive scan of the 256 digit totals (kCsrThreads == kRadix).
    {
        const int v = tot[tid];
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        int pre = 0;
        for (int w = 0; w < warp; ++w) pre += wsum[w];
        dbase[tid] = pre + incl - v;
    }
    __syncthreads();

    const int64_t base = (int64_t)blockIdx.x * kTile + (int64_t)warp * kCsrItems * 32;
    int32_t key[kCsrItems], val[kCsrItems];
    int rank[kCsrItems], dig[kCsrItems];
    const unsigned lt = lanemask_lt();
#pragma unroll
    for (int i = 0; i < kCsrItems; ++i) {
        const int64_t idx = base + i * 32 + lane;
        const bool valid = idx < E;
        key[i] = valid ? key_of(keys_in, idx, N, kFirst) : 0;
        val[i] = valid ? (kFirst ? (int32_t)idx : __ldg(vals_in + idx)) : 0;
        dig[i] = valid ? ((key[i] >> shift) & (kRadix - 1)) : kRadix;
        const unsigned peers = digit_peers(dig[i] & (kRadix - 1), valid);
        rank[i] = valid ? cnt[warp][dig[i]] + __popc(peers & lt) : 0;
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1) cnt[warp][dig[i]] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    {
        // one thread per digit: per-warp offsets inside the tile, the tile's
        // count of the digit, and where the digit's run starts in the tile
        const int d = tid;
        int own = 0;
#pragma unroll
        for (int w = 0; w < kCsrWarps; ++w) {
            const int c = cnt[w][d];
            cnt[w][d] = own;
            own += c;
        }
        int incl = own;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        __syncthreads();                     // wsum is reused from the digit-total scan
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        int pre = 0;
        for (int w = 0; w < warp; ++w) pre += wsum[w];
        const int local = pre + incl - own;  // first tile slot of digit d
        // global position of the tile's first key of digit d, minus its tile slot
        dbase[d] = dbase[d] + hist[(int64_t)d * T + blockIdx.x] - local;
#pragma unroll
        for (int w = 0; w < kCsrWarps; ++w) cnt[w][d] += local;
    }
    __syncthreads();
    // stage the tile in digit order, then write each digit's run contiguously
#pragma unroll
    for (int i = 0; i < kCsrItems; ++i) {
        if (dig[i] < kRadix) {
            const int slot = cnt[warp][dig[i]] + rank[i];
            skey[slot] = key[i];
            sval[slot] = val[i];
        }
    }
    __syncthreads();
    const int n_in_tile = (int)imin<int64_t>(kTile, E - (int64_t)blockIdx.x * kTile);
    for (int slot = tid; slot < n_in_tile; slot += kCsrThreads) {
        const int32_t k = skey[slot];
        const int pos = dbase[(k >> shift) & (kRadix - 1)] + slot;
        keys_out[pos] = k;
        vals_out[pos] = sval[slot];
    }
}

// row_ptr from sorted keys: position j is the first of every node in
// (key[j-1], key[j]]; the count of keys equal to N (invalid) is E - row_ptr[N].
// Each thread looks at kRowPtrPer consecutive positions.
constexpr int kRowPtrPer = 4;

__global__ void __launch_bounds__(256)
csr_row_ptr(const int32_t* __restrict__ sorted, int64_t E, int32_t N,
            int32_t* __restrict__ row_ptr, int32_t* __restrict__ bad) {
    const int64_t j0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * kRowPtrPer;
    pdl_wait();
    pdl_trigger();
    if (j0 > E) return;
    int64_t kprev = j0 > 0 ? (int64_t)__ldg(sorted + j0 - 1) : -1;
#pragma unroll
    for (int i = 0; i < kRowPtrPer; ++i) {
        const int64_t j = j0 + i;
        if (j > E) break;
        const int64_t kcur = j < E ? (int64_t)__ldg(sorted + j) : (int64_t)N + 1;
        const int64_t hi = kcur < (int64_t)N ? kcur : (int64_t)N;
        for (int64_t n = kprev + 1; n <= hi; ++n) {
            row_ptr[n] = (int32_t)j;
            if (n == N && bad) *bad = (int32_t)(E - j);
        }
        kprev = kcur;
    }
}

struct CsrPlan {
    int T = 0;
    int passes = 0;
    size_t off_k[2] = {0, 0}, off_v[2] = {0, 0}, off_hist = 0, off_tot = 0, bytes = 0;
};

CsrPlan csr_plan(int64_t E, int32_t N) {
    CsrPlan p;
    if (E <= 0) return p;
    p.T = (int)((E + kTile - 1) / kTile);
    const uint32_t maxkey = (uint32_t)N;
    const int bits = maxkey == 0 ? 1 : 32 - __builtin_clz(maxkey);
    p.passes = (bits + 7) / 8;
    const size_t ebytes = align_up((size_t)E * 4, 256);
    size_t off = 0;
    p.off_k[0] = off; off += ebytes;
    p.off_v[0] = off; off += ebytes;
    p.off_k[1] = off; off += ebytes;
    p.off_v[1] = off; off += ebytes;
    p.off_hist = off; off += align_up((size_t)kRadix * p.T * 4, 256);
    p.off_tot = off; off += align_up((size_t)kRadix * 4, 256);
    p.bytes = off;
    return p;
}

}  // namespace
}  // namespace zs

using namespace zs;

extern "C" size_t zs_build_csr_workspace_bytes(int64_t E, int32_t N) {
    if (E < 0 || N < 0) return 0;
    return csr_plan(E, N).bytes;
}

extern "C" zs_status zs_build_csr(const int32_t* dst, int64_t E, int32_t N,
                                  int32_t* row_ptr, int32_t* perm, int32_t* bad_dst_count,
                                  void* workspace, size_t workspace_bytes, zs_stream_t stream) {
    if (E < 0 || N < 0) return fail(ZS_ERR_INVALID_ARG, "zs_build_csr: negative size (E=%lld, N=%d)", (long long)E, N);
    if (E >= ((int64_t)1 << 31) - 1) return fail(ZS_ERR_INVALID_ARG, "zs_build_csr: E=%lld exceeds the int32 index range", (long long)E);
    if (!row_ptr) return fail(ZS_ERR_INVALID_ARG, "zs_build_csr: row_ptr is NULL");
    if (E > 0 && (!dst || !perm)) return fail(ZS_ERR_INVALID_ARG, "zs_build_csr: dst or perm is NULL with E > 0");
    const CsrPlan p = csr_plan(E, N);
    if (workspace_bytes < p.bytes) return fail(ZS_ERR_INVALID_ARG, "zs_build_csr: workspace of %zu bytes, %zu needed", workspace_bytes, p.bytes);
    if (p.bytes > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return fail(ZS_ERR_INVALID_ARG, "zs_build_csr: workspace NULL or not 256-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    const int32_t* sorted = nullptr;
    if (E > 0) {
        int32_t* hist = reinterpret_cast<int32_t*>(ws + p.off_hist);
        int32_t* tot = reinterpret_cast<int32_t*>(ws + p.off_tot);
        const int32_t* kin = dst;
        const int32_t* vin = nullptr;
        for (int pass = 0; pass < p.passes; ++pass) {
            const bool first = pass == 0, last = pass == p.passes - 1;
            const int shift = 8 * pass;
            int32_t* kout = reinterpret_cast<int32_t*>(ws + p.off_k[pass & 1]);
            int32_t* vout = last ? perm : reinterpret_cast<int32_t*>(ws + p.off_v[pass & 1]);
            if (first) launch(csr_upsweep<true>, p.T, kCsrThreads, 0, s, kin, E, N, shift, hist, p.T);
            else launch(csr_upsweep<false>, p.T, kCsrThreads, 0, s, kin, E, N, shift, hist, p.T);
            launch(csr_scan, kRadix / kCsrWarps, kCsrThreads, 0, s, hist, p.T, tot);
            if (first) launch(csr_downsweep<true>, p.T, kCsrThreads, 0, s, kin, vin, E, N, shift, (const int32_t*)hist, (const int32_t*)tot, p.T, kout, vout);
            else launch(csr_downsweep<false>, p.T, kCsrThreads, 0, s, kin, vin, E, N, shift, (const int32_t*)hist, (const int32_t*)tot, p.T, kout, vout);
            kin = kout;
            vin = vout;
        }
        sorted = kin;
    }
    const int64_t threads = (E + 1 + kRowPtrPer - 1) / kRowPtrPer;
    launch(csr_row_ptr, (unsigned)((threads + 255) / 256), 256, 0, s, sorted, E, N, row_ptr, bad_dst_count);
    return check_launch("zs_build_csr");
}
