// trace.h -- internal hooks of the optional per-kernel timing (trace.cu).
#pragma once

#include <cuda_runtime.h>

namespace moe {

// Record the start event of `kernel` on `st` if tracing is on and the name
// matches the filter; trace_end records the matching stop event.
void trace_begin(const char *kernel, cudaStream_t st);
void trace_end(cudaStream_t st);

// Launch helper: brackets one <<<>>> launch with the trace hooks.
#define MOE_TRACED_LAUNCH(name, st, ...) \
    do {                                 \
        ::moe::trace_begin(name, st);    \
        __VA_ARGS__;                     \
        ::moe::trace_end(st);            \
    } while (0)

}  // namespace moe
