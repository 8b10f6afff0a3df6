// Shared host-side helpers of libradixattn.so: error reporting and argument checks.
#pragma once

#include <cstdarg>
#include <cstdio>
#include <string>

#include "radix_attn.h"

#include <atomic>

namespace rx {

// Thread-local message for rx_last_error(); defined in radix_tree.cpp.
void set_error(const char* fmt, ...);
void clear_error();

// Tracing: an NVTX range named after the entry point around every ABI call that does work,
// for a profiler's timeline.  Off by default (rx_set_tracing, or RX_NVTX=1 in the environment
// when the library loads): when off a call pays one relaxed load and a branch.  The ranges go
// through NVTX's own dispatch, which does nothing unless a profiler is attached.
extern std::atomic<int> g_trace;                 // radix_tree.cpp
void trace_push(const char* name);               // step_runtime.cu (NVTX)
void trace_pop();
struct TraceRange {
    bool on;
    explicit TraceRange(const char* name) : on(g_trace.load(std::memory_order_relaxed) != 0) {
        if (on) trace_push(name);
    }
    ~TraceRange() {
        if (on) trace_pop();
    }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace rx

#define RX_TRACE(name) ::rx::TraceRange rx_trace_range_(name)

#define RX_REQUIRE(cond, ...)          \
    do {                               \
        if (!(cond)) {                 \
            ::rx::set_error(__VA_ARGS__); \
            return RX_EINVAL;          \
        }                              \
    } while (0)
