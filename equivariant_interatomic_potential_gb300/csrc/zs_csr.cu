// Stable destination CSR for the zonal scatter (row_ptr, perm).
//
// The forward of the deepmd-kit pull request "fused Triton zonal scatter for
// the GIE head" walks a destination CSR whose within-node order is the edge
// order ("stable-sort CSR order", section "What").  Two constructions, both
// integer-only in a fixed order, so perm is unique and bit-identical to a
// sequential counting sort; keys outside [0, N) count as key N, after all
// valid ones.
//
// Counting path (N + 1 <= kCntMaxKeys, every bench-sized graph but the
// largest): one pass, three launches with no inter-CTA waiting (one launch of
// one CTA, count_single, for up to kSingleMaxEdges edges):
//   count_rank    -- per tile of edges, each edge's stable rank among the
//                    tile's edges of the same node (warp match + per-warp
//                    running counts in shared memory, then a prefix over
//                    warps), and the tile's per-node counts M[tile][n]
//   scan_cols     -- per node, exclusive scan of M[.][n] over tiles
//   count_scatter -- per tile, node bases from a block scan of the node
//                    totals; perm[base[n] + M[tile][n] + rank] = edge
// Radix path (larger N): LSD radix sort with 8-bit digits, each pass in
// three launches:
//   upsweep   -- per tile of keys, a 256-bin digit histogram (shared atomics)
//   scan      -- per digit, exclusive scan of its histogram row over tiles
//   downsweep -- per tile, stable rank of every key among equal digits
//                (warp ballots + per-warp running counts), staged in shared
//                memory in digit order and written out run by run
// and a final pass that reads the sorted keys to write row_ptr.
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
    // counts do not depend on the order of the increments; the tile's keys
    // are all loaded before the first increment (one round trip, not eight)
    const int64_t base = (int64_t)blockIdx.x * kTile;
    int dig[kTile / kCsrThreads];
#pragma unroll
    for (int u = 0; u < kTile / kCsrThreads; ++u) {
        const int64_t idx = base + u * kCsrThreads + tid;
        dig[u] = idx < E ? (key_of(keys_in, idx, N, kFirst) >> shift) & (kRadix - 1) : -1;
    }
#pragma unroll
    for (int u = 0; u < kTile / kCsrThreads; ++u)
        if (dig[u] >= 0) atomicAdd(&cnt[dig[u]], 1);
    __syncthreads();
    hist[(int64_t)tid * T + blockIdx.x] = cnt[tid];
}

// One CTA per row: exclusive scan of hist[d, 0..T) in place, total to tot[d].
// Thread i takes the consecutive entries [i * per, (i + 1) * per), all loaded
// before they are added (a row is one round trip of loads, not one per
// 256 entries).
constexpr int kScanPer = 16;
__global__ void __launch_bounds__(kCsrThreads)
csr_scan(int32_t* __restrict__ hist, int T, int32_t* __restrict__ tot) {
    __shared__ int wsum[kCsrWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t* row = hist + (int64_t)blockIdx.x * T;
    pdl_wait();
    pdl_trigger();
    int carry = 0;
    for (int c0 = 0; c0 < T; c0 += kScanPer * kCsrThreads) {
        const int per = imin(kScanPer, (imin(T - c0, kScanPer * kCsrThreads) + kCsrThreads - 1) / kCsrThreads);
        const int i0 = c0 + tid * per;
        int v[kScanPer];
        int own = 0;
#pragma unroll
        for (int k = 0; k < kScanPer; ++k) {
            v[k] = (k < per && i0 + k < T) ? row[i0 + k] : 0;
            own += v[k];
        }
        int incl = own;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        int pre = carry;
        int all = carry;
#pragma unroll
        for (int w = 0; w < kCsrWarps; ++w) {
            if (w < warp) pre += wsum[w];
            all += wsum[w];
        }
        int run = pre + incl - own;
#pragma unroll
        for (int k = 0; k < kScanPer; ++k)
            if (k < per && i0 + k < T) {
                row[i0 + k] = run;
                run += v[k];
            }
        carry = all;
        __syncthreads();
    }
    if (tid == 0) tot[blockIdx.x] = carry;
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

    // this tile's offset within each digit, loaded now beside the totals
    const int hv = hist[(int64_t)tid * T + blockIdx.x];
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
    // every item's key and value are loaded before the ranking starts (its
    // warp synchronisations would otherwise hold each load back to its round)
#pragma unroll
    for (int i = 0; i < kCsrItems; ++i) {
        const int64_t idx = base + i * 32 + lane;
        const bool valid = idx < E;
        key[i] = valid ? key_of(keys_in, idx, N, kFirst) : 0;
        val[i] = valid ? (kFirst ? (int32_t)idx : __ldg(vals_in + idx)) : 0;
        dig[i] = valid ? ((key[i] >> shift) & (kRadix - 1)) : kRadix;
    }
#pragma unroll
    for (int i = 0; i < kCsrItems; ++i) {
        const bool valid = dig[i] < kRadix;
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
        dbase[d] = dbase[d] + hv - local;
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

// ---------------------------------------------------------------------------
// Counting path.  A tile is kCntWarps warps x `rounds` rounds of 32 edges;
// warp w of tile t owns the edges [t*TS + w*TW, t*TS + (w+1)*TW), TW = 32*rounds.
constexpr int kCntWarps = 16;
constexpr int kCntThreads = kCntWarps * 32;
#ifndef ZS_CNT_MAX_KEYS
#define ZS_CNT_MAX_KEYS 5120
#endif
constexpr int kCntMaxKeys = ZS_CNT_MAX_KEYS;   // N + 1 up to this takes the counting path
constexpr int kCntMaxRounds = 16;       // tile of at most 8192 edges
constexpr int kCntTargetTiles = 152;    // tiles sized so one wave covers 152 SMs

constexpr int kCntMaxPer = (kCntMaxKeys + kCntThreads - 1) / kCntThreads;   // keys per thread in a block scan

// Keys rounded up to even, so two keys' 16-bit counters share a 32-bit word.
__host__ __device__ __forceinline__ int count_pairs(int nkeys) { return (nkeys + 1) >> 1; }

// Shared memory of csr_count_rank: 16-bit counters [kCntWarps][keys, padded
// to even], then one 32-bit word per edge of the tile.
inline int count_rank_smem(int nkeys, int rounds) { return count_pairs(nkeys) * 4 * kCntWarps + rounds * kCntThreads * 4; }

// 4-byte asynchronous copy global -> shared (cp.async): a CTA issues all of
// a tile's copies, then waits once (cp_async_wait_all + a barrier).
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;"
                 :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))), "l"(gmem) : "memory");
}

// 8- and 16-byte copies (both addresses aligned to the size).
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;"
                 :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async16b(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem))), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// n int32 from global src to shared dst (16-byte aligned): 16-byte pieces
// when src is 16-byte aligned too, else 4-byte ones; CTA-cooperative.
__device__ __forceinline__ void copy_ints(int32_t* dst, const int32_t* src, int n, int tid, int nthreads) {
    if ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
        const int n4 = n >> 2;
        for (int j = tid; j < n4; j += nthreads) cp_async16b(dst + 4 * j, src + 4 * j);
        for (int i = 4 * n4 + tid; i < n; i += nthreads) cp_async4(dst + i, src + i);
    } else {
        for (int i = tid; i < n; i += nthreads) cp_async4(dst + i, src + i);
    }
}

__device__ __forceinline__ int32_t clamp_key(int32_t k, int32_t N) { return (uint32_t)k < (uint32_t)N ? k : N; }

// Ranks within each warp's run of a tile (warp w owns edges [w * 32 * rounds,
// (w + 1) * 32 * rounds) of the tile): packed[i] holds edge i's key on entry
// and key << 16 | (its rank among the warp's earlier edges of that key) on
// exit; wcnt (the warp's 16-bit counters, zeroed) ends with the warp's count
// of every key.  Per round of 32 edges, the lanes holding each key (peers)
// are found by claim and verify: every lane writes its lane id into bits
// 10..14 of its key's counter (count < 1024 stays in bits 0..9), reads the
// slot back, and lanes that lost the claim are grouped with the winner by
// one ballot per contested key.  Uncontested rounds cost no ballot loop.
__device__ __forceinline__ void rank_in_warp(uint32_t* packed, uint16_t* wcnt, int rounds, int n, int32_t N, int warp,
                                             int lane) {
    const unsigned lt = lanemask_lt();
    const int TW = rounds * 32;
    for (int r = 0; r < rounds; ++r) {
        const int i = warp * TW + r * 32 + lane;
        const bool valid = i < n;
        const int key = valid ? clamp_key((int32_t)packed[i], N) : 0;
        const uint32_t before = valid ? wcnt[key] : 0u;          // count so far, owner bits clear
        __syncwarp();
        if (valid) wcnt[key] = (uint16_t)(before | ((uint32_t)lane << 10));
        __syncwarp();
        const int owner = valid ? (int)(wcnt[key] >> 10) : lane;
        unsigned lost = __ballot_sync(0xffffffffu, valid && owner != lane);
        unsigned peers = 1u << lane;
        while (lost) {
            const int w = __shfl_sync(0xffffffffu, owner, __ffs(lost) - 1);
            const unsigned group = __ballot_sync(0xffffffffu, valid && owner == w);
            if (group & (1u << lane)) peers = group;
            lost &= ~group;
        }
        __syncwarp();
        if (valid) {
            if (lane == __ffs(peers) - 1) wcnt[key] = (uint16_t)(before + __popc(peers));
            packed[i] = ((uint32_t)key << 16) | (before + __popc(peers & lt));
        }
        __syncwarp();
    }
}

// Pair q of keys: the warps' counters turned into exclusive prefixes over the
// warps (both 16-bit halves at once: every partial sum is below 2^16); the
// tile's two counts are returned in the halves of the result.
__device__ __forceinline__ uint32_t prefix_over_warps(uint32_t* cnt_words, int npairs, int q) {
    uint32_t c[kCntWarps];
#pragma unroll
    for (int w = 0; w < kCntWarps; ++w) c[w] = cnt_words[w * npairs + q];
    uint32_t run = 0;
#pragma unroll
    for (int w = 0; w < kCntWarps; ++w) {
        cnt_words[w * npairs + q] = run;
        run += c[w];
    }
    return run;
}

// Node bases: an exclusive scan of the nkeys totals in tot (shared memory),
// thread tid taking keys [tid * per, (tid + 1) * per).  base[k] = first CSR
// position of key k plus off[k] (off may alias base; NULL: 0); with row_ptr,
// the positions go to row_ptr too and the total of key N (invalid keys) to
// *bad.  Every thread of the CTA must call it (it synchronises the CTA).
__device__ __forceinline__ void key_bases(const int32_t* tot, const int32_t* off, int32_t* base, int nkeys, int32_t N,
                                          int32_t* wsum, int32_t* __restrict__ row_ptr, int32_t* __restrict__ bad) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int per = (nkeys + kCntThreads - 1) / kCntThreads;
    const int k0 = tid * per;
    int32_t v[kCntMaxPer], o[kCntMaxPer];
    int32_t own = 0;
#pragma unroll
    for (int j = 0; j < kCntMaxPer; ++j) {
        const bool in = j < per && k0 + j < nkeys;
        v[j] = in ? tot[k0 + j] : 0;
        o[j] = (in && off) ? off[k0 + j] : 0;
        own += v[j];
    }
    int32_t incl = own;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int32_t run = incl - own;
    for (int w = 0; w < warp; ++w) run += wsum[w];
#pragma unroll
    for (int j = 0; j < kCntMaxPer; ++j) {
        const int k = k0 + j;
        if (j < per && k < nkeys) {
            if (row_ptr) {
                row_ptr[k] = run;
                if (k == N && bad) *bad = v[j];
            }
            base[k] = run + o[j];
            run += v[j];
        }
    }
}

// Per tile: each edge's stable rank among the tile's edges of the same key
// (to rank[]), and the tile's count of every key (to row `tile` of M, whose
// rows hold 2 * count_pairs(N + 1) counts).
__global__ void __launch_bounds__(kCntThreads, 1)
csr_count_rank(const int32_t* __restrict__ dst, int64_t E, int32_t N, int rounds,
               int32_t* __restrict__ M, uint16_t* __restrict__ rank) {
    extern __shared__ uint32_t cnt_words[];
    const int nkeys = N + 1;
    const int npairs = count_pairs(nkeys);
    // warp w's counter of key k is the 16-bit half (k & 1) of word w * npairs + k / 2
    uint16_t* cnt = reinterpret_cast<uint16_t*>(cnt_words);
    uint32_t* packed = cnt_words + kCntWarps * npairs;      // [TS]: key << 16 | rank in warp
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int TW = rounds * 32;
    const int64_t tbase = (int64_t)blockIdx.x * rounds * kCntThreads;
    const int n_in_tile = (int)imin<int64_t>((int64_t)rounds * kCntThreads, E - tbase);
    pdl_wait();
    pdl_trigger();
    // the tile's keys land in packed[] while the counters are cleared
    copy_ints(reinterpret_cast<int32_t*>(packed), dst + tbase, n_in_tile, tid, kCntThreads);
    // kCntWarps * npairs words, a multiple of four
    for (int i = tid; i < kCntWarps * npairs / 4; i += kCntThreads) reinterpret_cast<uint4*>(cnt_words)[i] = make_uint4(0u, 0u, 0u, 0u);
    cp_async_wait_all();
    __syncthreads();

    rank_in_warp(packed, cnt + 2 * warp * npairs, rounds, n_in_tile, N, warp, lane);
    __syncthreads();
    // per pair of keys: prefixes over the warps, tile counts to M
    for (int q = tid; q < npairs; q += kCntThreads) {
        const uint32_t run = prefix_over_warps(cnt_words, npairs, q);
        reinterpret_cast<int2*>(M + (int64_t)blockIdx.x * 2 * npairs)[q] = make_int2((int)(run & 0xffffu), (int)(run >> 16));
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kCntMaxRounds; ++u) {
        const int i = tid + u * kCntThreads;
        if (i >= n_in_tile) break;
        const uint32_t p = packed[i];
        const int w = i / TW;
        rank[tbase + i] = (uint16_t)((p & 0xffffu) + cnt[2 * w * npairs + (p >> 16)]);
    }
}

// Per key: exclusive scan over the tiles of its column of M (rows of S
// counts) in place, total to tot[key].  A CTA takes 32 keys, one per lane;
// its warps split the tiles into chunks and combine through shared memory.
__global__ void __launch_bounds__(kCntThreads)
csr_scan_cols(int32_t* __restrict__ M, int T, int S, int nkeys, int32_t* __restrict__ tot) {
    __shared__ int32_t part[kCntWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int key = blockIdx.x * 32 + lane;
    const int chunk = (T + kCntWarps - 1) / kCntWarps;
    const int t0 = imin(T, warp * chunk), t1 = imin(T, t0 + chunk);
    pdl_wait();
    pdl_trigger();
    constexpr int kRegs = 16;
    __shared__ int32_t stage[kCntWarps][kRegs][32];
    int32_t c[kRegs];
    int32_t sum = 0;
    const bool in_regs = chunk <= kRegs;
    if (in_regs) {
        // one batch of copies per lane, then the lane's own values from shared memory
        if (key < nkeys)
            for (int j = 0; j < t1 - t0; ++j) cp_async4(&stage[warp][j][lane], M + (int64_t)(t0 + j) * S + key);
        cp_async_wait_all();
#pragma unroll
        for (int j = 0; j < kRegs; ++j) {
            c[j] = (key < nkeys && j < t1 - t0) ? stage[warp][j][lane] : 0;
            sum += c[j];
        }
    } else if (key < nkeys) {
#pragma unroll 8
        for (int t = t0; t < t1; ++t) sum += M[(int64_t)t * S + key];
    }
    part[warp][lane] = sum;
    __syncthreads();
    int32_t run = 0;
    for (int w = 0; w < warp; ++w) run += part[w][lane];
    if (key >= nkeys) return;
    if (warp == kCntWarps - 1) tot[key] = run + sum;
    if (in_regs) {
#pragma unroll
        for (int j = 0; j < kRegs; ++j) {
            if (t0 + j < t1) M[(int64_t)(t0 + j) * S + key] = run;
            run += c[j];
        }
        return;
    }
    for (int t = t0; t < t1; ++t) {
        const int64_t i = (int64_t)t * S + key;
        const int32_t v = M[i];
        M[i] = run;
        run += v;
    }
}

// Shared memory of csr_count_scatter (int32 words, each array starting on a
// 16-byte boundary): the node totals, the tile's row of M, kCntWarps warp
// sums, the tile's keys, its ranks (two per word).
__host__ __device__ __forceinline__ int align4(int n) { return (n + 3) & ~3; }
inline int count_scatter_smem(int nkeys, int rounds) {
    return (align4(nkeys) + align4(2 * count_pairs(nkeys)) + kCntWarps + rounds * kCntThreads + rounds * kCntThreads / 2) * 4;
}

// Dynamic shared memory requested so that no two CTAs of a kernel share an SM
// (a kernel launched early behind its predecessor otherwise lands two CTAs
// on one SM while others idle, doubling the slowest CTA's time).
constexpr int kOneCtaPerSmSmem = 120 * 1024;

// Per tile: node bases from an exclusive scan of the key totals plus the
// tile's offset within each key, then every edge to its CSR position.  Tile 0
// also writes row_ptr and the count of invalid keys.
__global__ void __launch_bounds__(kCntThreads)
csr_count_scatter(const int32_t* __restrict__ dst, const uint16_t* __restrict__ rank,
                  const int32_t* __restrict__ M, const int32_t* __restrict__ tot,
                  int64_t E, int32_t N, int rounds,
                  int32_t* __restrict__ perm, int32_t* __restrict__ row_ptr, int32_t* __restrict__ bad) {
    extern __shared__ __align__(16) int32_t ktot[];
    const int nkeys = N + 1;
    const int S = 2 * count_pairs(nkeys);
    int32_t* kbase = ktot + align4(nkeys);
    int32_t* wsum = kbase + align4(S);
    int32_t* skey = wsum + kCntWarps;
    uint32_t* srank = reinterpret_cast<uint32_t*>(skey + rounds * kCntThreads);
    const int tid = threadIdx.x;
    const int64_t tbase = (int64_t)blockIdx.x * rounds * kCntThreads;
    const int n_in_tile = (int)imin<int64_t>((int64_t)rounds * kCntThreads, E - tbase);
    pdl_wait();
    pdl_trigger();
    // every input of the tile in one batch of asynchronous copies: the tile's
    // row of M, the node totals, the tile's keys and its ranks (in pairs; the
    // tile starts on an even edge, an odd last edge is read directly)
    // (rows of M are S = even counts long: 8-byte pieces; the rank array and
    // the tile start are 16-byte aligned: 16-byte pieces of eight ranks)
    const int32_t* mrow = M + (int64_t)blockIdx.x * S;
    for (int j = tid; j < S / 2; j += kCntThreads) cp_async8(kbase + 2 * j, mrow + 2 * j);
    copy_ints(ktot, tot, nkeys, tid, kCntThreads);
    copy_ints(skey, dst + tbase, n_in_tile, tid, kCntThreads);
    const int n8 = n_in_tile >> 3;
    for (int j = tid; j < n8; j += kCntThreads) cp_async16b(srank + 4 * j, rank + tbase + 8 * j);
    for (int j = 4 * n8 + tid; j < n_in_tile / 2; j += kCntThreads) cp_async4(srank + j, rank + tbase + 2 * j);
    if ((n_in_tile & 1) && tid == 0) srank[n_in_tile / 2] = __ldg(rank + tbase + n_in_tile - 1);
    cp_async_wait_all();
    __syncthreads();
    key_bases(ktot, kbase, kbase, nkeys, N, wsum, blockIdx.x == 0 ? row_ptr : nullptr, bad);
    __syncthreads();
#pragma unroll 4
    for (int i = tid; i < n_in_tile; i += kCntThreads) {
        const uint32_t rk = (srank[i >> 1] >> (16 * (i & 1))) & 0xffffu;
        perm[kbase[clamp_key(skey[i], N)] + (int32_t)rk] = (int32_t)(tbase + i);
    }
}

// Small graphs (E <= kCntMaxRounds * kCntThreads edges): the whole counting
// path in one CTA and one launch -- csr_count_rank's ranking and counts, then
// csr_count_scatter's node bases and scatter, the counts staying in shared
// memory (with one tile, every edge's offset within its key is its rank).
constexpr int kSingleMaxEdges = kCntMaxRounds * kCntThreads;
inline int count_single_smem(int nkeys, int rounds) {
    return count_rank_smem(nkeys, rounds) + 2 * count_pairs(nkeys) * 4;
}

__global__ void __launch_bounds__(kCntThreads, 1)
csr_count_single(const int32_t* __restrict__ dst, int64_t E, int32_t N, int rounds,
                 int32_t* __restrict__ perm, int32_t* __restrict__ row_ptr, int32_t* __restrict__ bad) {
    extern __shared__ uint32_t cnt_words[];
    __shared__ int32_t wsum[kCntWarps];
    const int nkeys = N + 1;
    const int npairs = count_pairs(nkeys);
    uint16_t* cnt = reinterpret_cast<uint16_t*>(cnt_words);
    uint32_t* packed = cnt_words + kCntWarps * npairs;                          // [TS]: key << 16 | rank
    int32_t* ktot = reinterpret_cast<int32_t*>(packed + rounds * kCntThreads);   // [2 * npairs]: key totals, then bases
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int TW = rounds * 32;
    const int n = (int)E;
    pdl_wait();
    pdl_trigger();
    copy_ints(reinterpret_cast<int32_t*>(packed), dst, n, tid, kCntThreads);
    for (int i = tid; i < kCntWarps * npairs / 4; i += kCntThreads) reinterpret_cast<uint4*>(cnt_words)[i] = make_uint4(0u, 0u, 0u, 0u);
    cp_async_wait_all();
    __syncthreads();
    rank_in_warp(packed, cnt + 2 * warp * npairs, rounds, n, N, warp, lane);
    __syncthreads();
    // per pair of keys: exclusive prefix over the warps, and the key totals
    for (int q = tid; q < npairs; q += kCntThreads) {
        const uint32_t run = prefix_over_warps(cnt_words, npairs, q);
        ktot[2 * q] = (int32_t)(run & 0xffffu);
        ktot[2 * q + 1] = (int32_t)(run >> 16);
    }
    __syncthreads();
    for (int i = tid; i < n; i += kCntThreads) {
        const uint32_t p = packed[i];
        const int w = i / TW;
        packed[i] = (p & 0xffff0000u) | ((p & 0xffffu) + cnt[2 * w * npairs + (p >> 16)]);
    }
    // node bases (one tile: an edge's offset within its key is its rank)
    key_bases(ktot, nullptr, ktot, nkeys, N, wsum, row_ptr, bad);
    __syncthreads();
#pragma unroll 4
    for (int i = tid; i < n; i += kCntThreads) {
        const uint32_t p = packed[i];
        perm[ktot[p >> 16] + (int32_t)(p & 0xffffu)] = i;
    }
}

struct CsrPlan {
    bool counting = false;
    int T = 0;
    int passes = 0;
    int rounds = 0;     // counting path: rounds of 32 edges per warp in a tile
    size_t off_k[2] = {0, 0}, off_v[2] = {0, 0}, off_hist = 0, off_tot = 0, off_rank = 0, bytes = 0;
};

CsrPlan csr_plan(int64_t E, int32_t N) {
    CsrPlan p;
    if (E <= 0) return p;
    const size_t ebytes = align_up((size_t)E * 4, 256);
    size_t off = 0;
    if ((int64_t)N + 1 <= kCntMaxKeys) {
        p.counting = true;
        const int64_t per_tile = (E + kCntTargetTiles - 1) / kCntTargetTiles;
        p.rounds = (int)imax<int64_t>(1, imin<int64_t>(kCntMaxRounds, (per_tile + kCntThreads - 1) / kCntThreads));
        const int64_t ts = (int64_t)p.rounds * kCntThreads;
        p.T = (int)((E + ts - 1) / ts);
        const int nkeys = N + 1;
        p.off_hist = off; off += align_up((size_t)2 * count_pairs(nkeys) * p.T * 4, 256);
        p.off_tot = off; off += align_up((size_t)nkeys * 4, 256);
        p.off_rank = off; off += align_up((size_t)E * 2, 256);
        p.bytes = off;
        return p;
    }
    p.T = (int)((E + kTile - 1) / kTile);
    const uint32_t maxkey = (uint32_t)N;
    const int bits = maxkey == 0 ? 1 : 32 - __builtin_clz(maxkey);
    p.passes = (bits + 7) / 8;
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
    if (p.counting) {
        static std::atomic<uint64_t> rank_smem_set[kMaxDevices];
        int32_t* M = reinterpret_cast<int32_t*>(ws + p.off_hist);
        int32_t* tot = reinterpret_cast<int32_t*>(ws + p.off_tot);
        uint16_t* rank = reinterpret_cast<uint16_t*>(ws + p.off_rank);
        if (E <= kSingleMaxEdges) {
            static std::atomic<uint64_t> single_smem_set[kMaxDevices];
            set_smem_limit_once(csr_count_single, count_single_smem(kCntMaxKeys, kCntMaxRounds), single_smem_set);
            const int rounds = (int)((E + kCntThreads - 1) / kCntThreads);
            launch(csr_count_single, 1, kCntThreads, count_single_smem(N + 1, rounds), s, dst, E, N, rounds, perm,
                   row_ptr, bad_dst_count);
            return check_launch("zs_build_csr");
        }
        const int smem = count_rank_smem(kCntMaxKeys, kCntMaxRounds);
        set_smem_limit_once(csr_count_rank, smem, rank_smem_set);
        const int S = 2 * count_pairs(N + 1);
        launch(csr_count_rank, p.T, kCntThreads, count_rank_smem(N + 1, p.rounds), s, dst, E, N, p.rounds, M, rank);
        static std::atomic<uint64_t> scan_smem_set[kMaxDevices];
        set_smem_limit_once(csr_scan_cols, kOneCtaPerSmSmem, scan_smem_set);
        launch(csr_scan_cols, (N + 1 + 31) / 32, kCntThreads, kOneCtaPerSmSmem, s, M, p.T, S, N + 1, tot);
        static std::atomic<uint64_t> scatter_smem_set[kMaxDevices];
        set_smem_limit_once(csr_count_scatter, imax(kOneCtaPerSmSmem, count_scatter_smem(kCntMaxKeys, kCntMaxRounds)), scatter_smem_set);
        launch(csr_count_scatter, p.T, kCntThreads, imax(kOneCtaPerSmSmem, count_scatter_smem(N + 1, p.rounds)), s, dst, (const uint16_t*)rank,
               (const int32_t*)M, (const int32_t*)tot, E, N, p.rounds, perm, row_ptr, bad_dst_count);
        return check_launch("zs_build_csr");
    }
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
            launch(csr_scan, kRadix, kCsrThreads, 0, s, hist, p.T, tot);
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
