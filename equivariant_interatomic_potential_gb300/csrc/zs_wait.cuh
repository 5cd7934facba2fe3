// Bounded waits of libzs's kernels and how a wait that runs out is reported.
//
// No kernel of this library waits without a limit: a wait gives up after
// kMaxSpins unsuccessful tries, counts a timeout in g_zs_timeouts (one
// counter per translation unit that includes this header) and sets the
// caller's flag word when one is registered, and the kernel carries on to
// its end instead of hanging the GPU (its outputs are then undefined).
// zs_check_timeouts() reads and clears the counters; zs_set_timeout_flag()
// registers the flag word.
#pragma once

#include "zs_common.cuh"

namespace zs {

constexpr uint32_t kMaxSpins = 1u << 22;

// Count of bounded waits that ran out in this translation unit's kernels.
static __device__ unsigned int g_zs_timeouts;
// Caller-registered word (device memory or host memory the device can reach)
// set to 1 when a bounded wait runs out; NULL when none is registered.
static __device__ unsigned int* g_zs_timeout_flag;

// Host: read and clear this translation unit's count (synchronises the device).
static inline unsigned int take_timeouts_local() {
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_zs_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
    if (v) cudaMemcpyToSymbol(g_zs_timeouts, &zero, sizeof(zero));
    return v;
}

// Host: register the flag word of the current device for this translation
// unit's kernels (synchronous copy to the device symbol).
static inline cudaError_t set_timeout_flag_local(unsigned int* flag) {
    return cudaMemcpyToSymbol(g_zs_timeout_flag, &flag, sizeof(flag));
}

// Device: record one bounded wait that ran out.
__device__ __forceinline__ void note_timeout() {
    atomicAdd(&g_zs_timeouts, 1u);
    unsigned int* f = g_zs_timeout_flag;
    if (f) {
        *reinterpret_cast<volatile unsigned int*>(f) = 1u;
        __threadfence_system();
    }
}

__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// 64-bit mixing function (the finaliser of Steele, Lea and Flood's SplitMix64).
__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Value that marks a flag as written by this launch: %gridid (the launch's
// number in its context) mixed with a per-call value from the host.  Unique
// for launches from the host, but NOT for the replays of one CUDA graph: a
// graph replays its kernel nodes with the same arguments and, as measured,
// the same tag.  Protocols built on it must therefore leave no flag set
// when the launch ends (see the forward), or take their tag from device
// memory instead (an epoch word that every launch advances).
__device__ __forceinline__ uint64_t launch_tag(uint64_t salt) {
    uint64_t id;
    asm volatile("mov.u64 %0, %%gridid;" : "=l"(id));
    return mix64(id ^ salt);
}

// A flag value is never 0, the value of a flag that was reset.
__device__ __forceinline__ uint64_t flag_tag(uint64_t t) { return t ? t : 1ull; }

// Bounded wait until flags[k] == tag, with a pause of backoff_ns between
// tries (0: none); false (and one timeout noted) if it never comes.
__device__ __forceinline__ bool wait_flag(const uint64_t* flags, int k, uint64_t tag, unsigned backoff_ns = 0) {
    for (uint32_t i = 0; i < kMaxSpins; ++i) {
        if (ld_acquire_u64(flags + k) == tag) return true;
        if (backoff_ns) __nanosleep(backoff_ns);
    }
    note_timeout();
    return false;
}

}  // namespace zs
