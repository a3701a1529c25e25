#include "streams.h"

namespace gdn {

namespace {
constexpr int kMaxDevices = 64;
LibStreams g_streams[kMaxDevices];
}  // namespace

std::mutex& lib_streams_mutex() {
    static std::mutex mu;
    return mu;
}

cudaError_t lib_streams(LibStreams** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    LibStreams& s = g_streams[dev];
    if (!s.ev_b) {
        int least = 0, greatest = 0;
        if ((e = cudaDeviceGetStreamPriorityRange(&least, &greatest)) != cudaSuccess) return e;
        if (!s.lo && (e = cudaStreamCreateWithPriority(&s.lo, cudaStreamNonBlocking, least)) != cudaSuccess) return e;
        if (!s.hi && (e = cudaStreamCreateWithPriority(&s.hi, cudaStreamNonBlocking, greatest)) != cudaSuccess) return e;
        if (!s.ev_a && (e = cudaEventCreateWithFlags(&s.ev_a, cudaEventDisableTiming)) != cudaSuccess) return e;
        for (int i = 0; i < LIB_EVENT_POOL; ++i)
            if (!s.pool[i] && (e = cudaEventCreateWithFlags(&s.pool[i], cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&s.ev_b, cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    *out = &s;
    return cudaSuccess;
}

namespace {
CopyStreams g_copy[kMaxDevices];
bool g_copy_ready[kMaxDevices] = {};
}  // namespace

std::mutex& copy_streams_mutex() {
    static std::mutex mu;
    return mu;
}

cudaError_t copy_streams(CopyStreams** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    CopyStreams& s = g_copy[dev];
    if (!g_copy_ready[dev]) {
        auto ev = [&](cudaEvent_t* x) {
            return *x ? cudaSuccess : cudaEventCreateWithFlags(x, cudaEventDisableTiming);
        };
        if (!s.h2d && (e = cudaStreamCreateWithFlags(&s.h2d, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if (!s.d2h && (e = cudaStreamCreateWithFlags(&s.d2h, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = ev(&s.fork)) != cudaSuccess || (e = ev(&s.join_h2d)) != cudaSuccess ||
            (e = ev(&s.join_d2h)) != cudaSuccess)
            return e;
        for (int i = 0; i < 2; ++i)
            if ((e = ev(&s.in_ready[i])) != cudaSuccess || (e = ev(&s.pass_done[i])) != cudaSuccess ||
                (e = ev(&s.out_free[i])) != cudaSuccess)
                return e;
        g_copy_ready[dev] = true;
    }
    *out = &s;
    return cudaSuccess;
}

}  // namespace gdn
