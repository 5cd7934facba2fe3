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
zs_status selftest_bounded_wait(uint32_t max_spins, cudaStream_t s);

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
