// Two streams and two events of the library per device, for work that runs
// beside the caller's stream within one call: forked from the caller's stream
// and joined back to it before the call returns, so the call stays ordered on
// that stream and a stream capture records it.
#pragma once

#include <cuda_runtime.h>

#include <stdint.h>

#include <functional>
#include <mutex>

namespace gdn {

// Work over the token range [t_begin, t_end) enqueued on a given stream.
using TokenRangeHook = std::function<cudaError_t(int64_t t_begin, int64_t t_end, cudaStream_t)>;

constexpr int LIB_EVENT_POOL = 64;

struct LibStreams {
    cudaStream_t lo = nullptr;   // least priority
    cudaStream_t hi = nullptr;   // greatest priority
    cudaEvent_t ev_a = nullptr, ev_b = nullptr;   // timing disabled
    cudaEvent_t pool[LIB_EVENT_POOL] = {};         // one per pending dependency of a call
};

// Guards the table and every enqueue sequence that uses the streams and events.
std::mutex& lib_streams_mutex();

// The current device's streams and events, created on first use (call with
// lib_streams_mutex() held).
cudaError_t lib_streams(LibStreams** out);

// Copy streams of a host-fed prefill: one for host-to-device copies, one for
// device-to-host copies, and the events that pace two staging slots between
// them and the compute stream (timing disabled).
struct CopyStreams {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t fork = nullptr, join_h2d = nullptr, join_d2h = nullptr;
    cudaEvent_t in_ready[2] = {}, pass_done[2] = {}, out_free[2] = {};
};

// Guards the copy-stream table and every enqueue sequence that uses it.
std::mutex& copy_streams_mutex();

// The current device's copy streams and events, created on first use (call
// with copy_streams_mutex() held).
cudaError_t copy_streams(CopyStreams** out);

}  // namespace gdn
