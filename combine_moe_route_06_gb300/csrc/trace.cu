// trace.cu -- optional per-kernel timing: CUDA events around each launch.
//
// Off by default.  moe_trace_enable(filter, max_records) creates 2*max_records
// events (host handles; no device memory); while enabled, every launch whose
// kernel name contains `filter` (all launches if NULL/empty) is bracketed by an
// event pair recorded on the launch's own stream.  Records beyond max_records
// are not taken.  moe_trace_get waits for a record's stop event and returns its
// duration.  A launch captured into a CUDA graph gets event nodes in the graph:
// every replay re-records them, and moe_trace_get returns the latest replay.
#include <string.h>

#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "launch.h"
#include "trace.h"

namespace moe {

namespace {

struct Record {
    const char *name;
    int idx;  // event pair index
};

struct TraceState {
    std::mutex mu;
    bool on = false;
    std::string filter;
    std::vector<cudaEvent_t> ev;  // 2 per record
    std::vector<Record> rec;
    int pending = -1;             // pair opened by trace_begin, not yet closed
};

TraceState &state()
{
    static TraceState s;
    return s;
}

// Record `ev` on `st`; inside a stream capture the record becomes an event node
// of the graph (re-recorded on every replay).
cudaError_t record(cudaEvent_t ev, cudaStream_t st)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
        return cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
    return cudaEventRecord(ev, st);
}

void destroy_events(TraceState &s)
{
    for (cudaEvent_t e : s.ev) cudaEventDestroy(e);
    s.ev.clear();
    s.rec.clear();
    s.pending = -1;
}

}  // namespace

void trace_begin(const char *kernel, cudaStream_t st)
{
    TraceState &s = state();
    std::lock_guard<std::mutex> lock(s.mu);
    s.pending = -1;
    if (!s.on) return;
    if (!s.filter.empty() && strstr(kernel, s.filter.c_str()) == nullptr) return;
    const int idx = (int)s.rec.size();
    if (2 * idx + 1 >= (int)s.ev.size()) return;
    if (record(s.ev[2 * idx], st) != cudaSuccess) return;
    s.rec.push_back({kernel, idx});
    s.pending = idx;
}

void trace_end(cudaStream_t st)
{
    TraceState &s = state();
    std::lock_guard<std::mutex> lock(s.mu);
    if (s.pending < 0) return;
    record(s.ev[2 * s.pending + 1], st);
    s.pending = -1;
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_trace_enable(const char *kernel_filter, int max_records)
{
    if (max_records < 1 || max_records > (1 << 20)) return MOE_ERR_INVALID_ARG;
    TraceState &s = state();
    std::lock_guard<std::mutex> lock(s.mu);
    destroy_events(s);
    s.filter = kernel_filter ? kernel_filter : "";
    s.ev.resize(2 * (size_t)max_records);
    for (size_t i = 0; i < s.ev.size(); i++) {
        if (cudaEventCreate(&s.ev[i]) != cudaSuccess) {
            s.ev.resize(i);
            destroy_events(s);
            s.on = false;
            return MOE_ERR_CUDA;
        }
    }
    s.on = true;
    return MOE_OK;
}

void moe_trace_disable(void)
{
    TraceState &s = state();
    std::lock_guard<std::mutex> lock(s.mu);
    s.on = false;
    destroy_events(s);
}

void moe_trace_reset(void)
{
    TraceState &s = state();
    std::lock_guard<std::mutex> lock(s.mu);
    s.rec.clear();
    s.pending = -1;
}

int moe_trace_count(void)
{
    TraceState &s = state();
    std::lock_guard<std::mutex> lock(s.mu);
    return (int)s.rec.size();
}

moe_status_t moe_trace_get(int i, const char **kernel_name, float *ms)
{
    TraceState &s = state();
    std::lock_guard<std::mutex> lock(s.mu);
    if (i < 0 || i >= (int)s.rec.size() || !kernel_name || !ms) return MOE_ERR_INVALID_ARG;
    const Record &r = s.rec[i];
    if (cudaEventSynchronize(s.ev[2 * r.idx + 1]) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaEventElapsedTime(ms, s.ev[2 * r.idx], s.ev[2 * r.idx + 1]) != cudaSuccess)
        return MOE_ERR_CUDA;
    *kernel_name = r.name;
    return MOE_OK;
}

}  // extern "C"
