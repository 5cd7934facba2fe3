// Shared definitions of libzs's CUDA sources (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "zs.h"

namespace zs {

constexpr int kRows = 15;   // zonal rows of the lmax = 3 ladder (3 + 5 + 7)
constexpr int kSlots = 3;   // radial slots, one per degree 1..3
constexpr int kD = 16;      // node rows: scalar row + 15

// Degree group of zonal row r as a radial slot (row groups 3/5/7).
__host__ __device__ __forceinline__ int slot_of_row(int r) { return r < 3 ? 0 : (r < 8 ? 1 : 2); }

// The ladder of degree L (1..kMaxLmax): D = (L+1)^2 node rows, the scalar row
// then degree groups of 2l+1 zonal rows for l = 1..L (3/5/7 at L = 3), radial
// slot l - 1 for the rows of degree l.
constexpr int kMaxLmax = 5;
template <int L>
struct Ladder {
    static_assert(L >= 1 && L <= kMaxLmax, "ladder degree 1..5");
    static constexpr int D = (L + 1) * (L + 1);
    static constexpr int R = D - 1;
    static constexpr int S = L;
};

// Radial slot of zonal row r: degree l holds rows [l^2 - 1, (l+1)^2 - 1).
__host__ __device__ constexpr int ladder_slot(int r) {
    int l = 1;
    while ((l + 1) * (l + 1) - 1 <= r) ++l;
    return l - 1;
}

inline int ladder_rows(int lmax) { return (lmax + 1) * (lmax + 1) - 1; }

// Record a message for zs_last_error() and return the status.
zs_status fail(zs_status st, const char* fmt, ...);
// Check the last launch on this thread; ZS_ERR_CUDA with a message on failure.
zs_status check_launch(const char* what);

__host__ __device__ __forceinline__ bool aligned16(const void* p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Streaming loads: data read once, kept out of L1.
__device__ __forceinline__ float4 ld_stream4(const float* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_stream(const float* p) {
    float v;
    asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ int ld_stream_i(const int32_t* p) {
    int v;
    asm volatile("ld.global.nc.L1::no_allocate.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
// Read-only load that may be cached in L1 (gathered, reused data).
__device__ __forceinline__ float4 ld_ro4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

// Streaming stores (written once, not re-read by this kernel).
__device__ __forceinline__ void st_stream4(float* p, float4 v) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" :: "l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}
__device__ __forceinline__ void st_stream(float* p, float v) {
    asm volatile("st.global.cs.f32 [%0], %1;" :: "l"(p), "f"(v) : "memory");
}

// L2 eviction-priority policies.  Read-once streams are marked evict-first so
// that the small, reused or partially written arrays stay in L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// Ring copies name their L2 policy at compile time.
enum : int { kL2Normal = 0, kL2EvictFirst = 1, kL2EvictLast = 2 };
__device__ __forceinline__ uint64_t l2_policy(int hint) {
    return hint == kL2EvictFirst ? l2_evict_first() : hint == kL2EvictLast ? l2_evict_last() : l2_evict_normal();
}
__device__ __forceinline__ void st_hint4(float* p, float4 v, uint64_t pol) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.f32 [%0], {%1,%2,%3,%4}, %5;"
                 :: "l"(p), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_hint(float* p, float v, uint64_t pol) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.f32 [%0], %1, %2;" :: "l"(p), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ int ld_hint_i(const int32_t* p, uint64_t pol) {
    int v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.s32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ float4 f4_fma(float s, float4 a, float4 acc) {
    acc.x = fmaf(s, a.x, acc.x);
    acc.y = fmaf(s, a.y, acc.y);
    acc.z = fmaf(s, a.z, acc.z);
    acc.w = fmaf(s, a.w, acc.w);
    return acc;
}
__device__ __forceinline__ float4 f4_add(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ __forceinline__ float4 f4_shfl(float4 v, int src) {
    v.x = __shfl_sync(0xffffffffu, v.x, src);
    v.y = __shfl_sync(0xffffffffu, v.y, src);
    v.z = __shfl_sync(0xffffffffu, v.z, src);
    v.w = __shfl_sync(0xffffffffu, v.w, src);
    return v;
}
__device__ __forceinline__ float4 f4_shfl_xor(float4 v, int m) {
    v.x = __shfl_xor_sync(0xffffffffu, v.x, m);
    v.y = __shfl_xor_sync(0xffffffffu, v.y, m);
    v.z = __shfl_xor_sync(0xffffffffu, v.z, m);
    v.w = __shfl_xor_sync(0xffffffffu, v.w, m);
    return v;
}
__device__ __forceinline__ float f4_dot(float4 a, float4 b) {
    return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, a.x * b.x)));
}

// First index i in [0, n) with a[i] >= key (n if none), for a non-decreasing
// a, found by the whole warp (every lane gets the same answer; all 32 lanes
// must call it together).  Each round samples 32 evenly spaced entries at
// once and keeps the one interval that holds the answer: ceil(log32(n)) + 1
// rounds of dependent global loads instead of log2(n) for a binary search,
// at several hundred nanoseconds of latency each.
__device__ __forceinline__ int lower_bound_warp(const int32_t* a, int n, int64_t key, int lane) {
    int lo = 0, hi = n;   // a[i] < key for i < lo; a[i] >= key for i >= hi (a[n] counts as infinite)
    while (lo < hi) {
        const int step = ((hi - lo) + 31) >> 5;
        const int idx = lo + lane * step;
        const bool ge = idx >= hi || (int64_t)__ldg(a + idx) >= key;
        const unsigned m = __ballot_sync(0xffffffffu, ge);
        if (m == 0) {
            lo += 31 * step + 1;                    // every sample is below key
        } else {
            const int f = __ffs(m) - 1;             // first sample at or above key
            const int nhi = lo + f * step < hi ? lo + f * step : hi;
            if (f > 0) lo += (f - 1) * step + 1;
            hi = nhi;
        }
    }
    return lo;
}

// lower_bound_warp split into rounds, so that a kernel can interleave the
// search's dependent loads with other start-up loads: begin() issues the
// first round's loads, resolve() consumes a round and load() issues the
// next, until done().
struct WarpSearch {
    int lo, hi, step, idx, v;
    int64_t key;
    __device__ __forceinline__ void begin(const int32_t* a, int n, int64_t key_, int lane) {
        lo = 0;
        hi = n;
        key = key_;
        load(a, lane);
    }
    __device__ __forceinline__ void load(const int32_t* a, int lane) {
        if (lo >= hi) return;
        step = ((hi - lo) + 31) >> 5;
        idx = lo + lane * step;
        v = idx < hi ? __ldg(a + idx) : 0;
    }
    __device__ __forceinline__ bool done() const { return lo >= hi; }
    __device__ __forceinline__ void resolve() {
        if (lo >= hi) return;
        const bool ge = idx >= hi || (int64_t)v >= key;
        const unsigned m = __ballot_sync(0xffffffffu, ge);
        if (m == 0) {
            lo += 31 * step + 1;
        } else {
            const int f = __ffs(m) - 1;
            const int nhi = lo + f * step < hi ? lo + f * step : hi;
            if (f > 0) lo += (f - 1) * step + 1;
            hi = nhi;
        }
    }
};

// The first CSR node a window of positions starting at p0 visits: the node
// containing p0 when it starts before p0, else the first node starting at or
// after p0 (which may be empty).  Whole warp, as lower_bound_warp.
__device__ __forceinline__ int first_node_warp(const int32_t* __restrict__ row_ptr, int32_t N, int64_t p0, int lane) {
    const int n_lb = lower_bound_warp(row_ptr, N + 1, p0, lane);
    if (n_lb >= 1 && n_lb <= N && (int64_t)__ldg(row_ptr + n_lb) > p0) return n_lb - 1;
    return n_lb;
}

constexpr int kMaxDevices = 128;

inline int current_device() {
    int dev = 0;
    cudaGetDevice(&dev);
    return (dev >= 0 && dev < kMaxDevices) ? dev : 0;
}

// Number of SMs of the current device (looked up once per device).
inline int num_sms() {
    static std::atomic<int> cached[kMaxDevices];
    const int dev = current_device();
    int v = cached[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (v <= 0) v = 1;
        cached[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// Unique id (never 0) of the calling thread's current CUDA context, 0 when
// there is none or the driver cannot say.  A setting made in one context (a
// kernel attribute, a device symbol's address) does not outlive it: after
// cudaDeviceReset the device's primary context is a new one, with a new id.
uint64_t current_context_id();

// Raise a kernel's dynamic shared-memory limit once per context (again after
// a cudaDeviceReset).  done[dev] holds the id of the context it was set in.
template <typename K>
inline void set_smem_limit_once(K kernel, int bytes, std::atomic<uint64_t>* done) {
    const int dev = current_device();
    const uint64_t ctx = current_context_id();
    if (ctx == 0 || done[dev].load(std::memory_order_acquire) != ctx) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        done[dev].store(current_context_id(), std::memory_order_release);
    }
}

// Per-call value mixed into the launch tags of kernels whose CTAs signal one
// another through tagged flags (see launch_tag).
inline uint64_t next_salt() {
    static std::atomic<uint64_t> counter{0x2545F4914F6CDD1Dull};
    return counter.fetch_add(0x9E3779B97F4A7C15ull, std::memory_order_relaxed);
}

template <class T>
__host__ __device__ __forceinline__ constexpr T imin(T a, T b) { return a < b ? a : b; }
template <class T>
__host__ __device__ __forceinline__ constexpr T imax(T a, T b) { return a < b ? b : a; }

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Programmatic dependent launch.  Every kernel of this library is launched
// with programmatic stream serialisation, so it may be scheduled while the
// previous kernel in the stream is still finishing; pdl_wait() blocks until
// that kernel has completed and its memory is visible, and must come before
// the first global-memory access (read or write).  pdl_trigger() lets the
// next kernel start being scheduled.  Both are no-ops when the kernel was
// not launched as a dependent.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" :::); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace zs
