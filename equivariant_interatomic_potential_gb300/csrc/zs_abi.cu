// Status strings and the per-thread error message of libzs.
#include <stdarg.h>
#include <stdio.h>

#include "zs_common.cuh"

namespace {
thread_local char g_last_error[512] = {0};
}

namespace zs {

zs_status fail(zs_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

zs_status check_launch(const char* what) {
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) {
        return fail(ZS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(err), cudaGetErrorName(err));
    }
    return ZS_OK;
}

unsigned int take_timeouts_forward();
unsigned int take_timeouts_backward();
cudaError_t set_timeout_flag_forward(unsigned int* flag);
cudaError_t set_timeout_flag_backward(unsigned int* flag);
zs_status selftest_bounded_wait(uint32_t max_spins, cudaStream_t s);

// The driver's cuCtxGetCurrent and cuCtxGetId, resolved once through the
// runtime (no link against the driver library).
namespace {
using CtxGetCurrentFn = int (*)(void**);
using CtxGetIdFn = int (*)(void*, unsigned long long*);
struct CtxFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
    CtxFns() {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(f);
        cudaGetLastError();
    }
};
}  // namespace

uint64_t current_context_id() {
    static const CtxFns fns;
    if (!fns.get_current || !fns.get_id) return 0;
    void* ctx = nullptr;
    if (fns.get_current(&ctx) != 0 || ctx == nullptr) return 0;
    unsigned long long id = 0;
    if (fns.get_id(ctx, &id) != 0) return 0;
    return (uint64_t)id + 1;   // never 0 for a live context
}

}  // namespace zs

extern "C" {

zs_status zs_check_timeouts(void) {
    const unsigned int f = zs::take_timeouts_forward();
    const unsigned int b = zs::take_timeouts_backward();
    if (f == 0xffffffffu || b == 0xffffffffu)
        return zs::fail(ZS_ERR_CUDA, "zs_check_timeouts: %s", cudaGetErrorString(cudaGetLastError()));
    if (f + b) return zs::fail(ZS_ERR_TIMEOUT, "zs_check_timeouts: %u bounded waits ran out", f + b);
    return ZS_OK;
}


zs_status zs_set_timeout_flag(uint32_t* flag) {
    if (flag) {
        cudaPointerAttributes attr;
        const cudaError_t err = cudaPointerGetAttributes(&attr, flag);
        if (err != cudaSuccess) {
            cudaGetLastError();
            return zs::fail(ZS_ERR_INVALID_ARG, "zs_set_timeout_flag: %s", cudaGetErrorString(err));
        }
        const bool reachable = (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged ||
                                attr.type == cudaMemoryTypeHost) && attr.devicePointer == flag;
        if (!reachable)
            return zs::fail(ZS_ERR_INVALID_ARG,
                            "zs_set_timeout_flag: the word is not device memory or page-locked host memory that "
                            "the device reaches at the same address");
        if (reinterpret_cast<uintptr_t>(flag) & 3u)
            return zs::fail(ZS_ERR_INVALID_ARG, "zs_set_timeout_flag: the word is not 4-byte aligned");
    }
    unsigned int* f = reinterpret_cast<unsigned int*>(flag);
    cudaError_t err = zs::set_timeout_flag_forward(f);
    if (err == cudaSuccess) err = zs::set_timeout_flag_backward(f);
    if (err != cudaSuccess) return zs::fail(ZS_ERR_CUDA, "zs_set_timeout_flag: %s", cudaGetErrorString(err));
    return ZS_OK;
}

zs_status zs_selftest_bounded_wait(uint32_t max_spins, zs_stream_t stream) {
    if (max_spins == 0 || max_spins > (1u << 16))
        return zs::fail(ZS_ERR_INVALID_ARG, "zs_selftest_bounded_wait: max_spins=%u outside [1, 2^16]", max_spins);
    return zs::selftest_bounded_wait(max_spins, reinterpret_cast<cudaStream_t>(stream));
}

const char* zs_status_string(int status) {
    switch (status) {
        case ZS_OK: return "ZS_OK";
        case ZS_ERR_INVALID_ARG: return "ZS_ERR_INVALID_ARG";
        case ZS_ERR_UNSUPPORTED: return "ZS_ERR_UNSUPPORTED";
        case ZS_ERR_CUDA: return "ZS_ERR_CUDA";
        case ZS_ERR_TIMEOUT: return "ZS_ERR_TIMEOUT";
        default: return "ZS_ERR_UNKNOWN";
    }
}

const char* zs_last_error(void) { return g_last_error; }

int zs_version(void) { return 10000; }

}  // extern "C"
