// layout_static.cu -- moe_dispatch_layout_static: the dispatch layout for
// callers that cannot allocate device memory themselves.
//
// The layout's two kernels exchange per-chunk counts through scratch memory.
// Here that scratch is one array of fixed size compiled into the library (a
// file-scope __device__ array: every GPU that loads the library holds it until
// the process exits), so the caller passes only inputs and outputs.
//
// Host code cannot use the array's name as a device address (on the host it
// names a stand-in object), so the device address is looked up once per
// device with cudaGetSymbolAddress, with that device current, and cached.
#include <stdio.h>

#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "launch.h"

namespace moe {

namespace {

constexpr size_t kStaticScratchBytes = (size_t)4 << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_layout_scratch[kStaticScratchBytes];

// Device address of g_layout_scratch on the current device (looked up once).
cudaError_t static_scratch(void **out)
{
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_layout_scratch);
        if (e != cudaSuccess) return e;
        if (p == nullptr) return cudaErrorInvalidSymbol;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_dispatch_layout_static(const int32_t *topk_ids, int S, int T, int k,
                                                   int E, int P, int32_t *expert_counts,
                                                   int32_t *expert_rank, int32_t *part_counts,
                                                   int32_t *part_offsets, int32_t *token_slot,
                                                   uint32_t *dev_status, cudaStream_t stream)
{
    // one NVTX range per call, as for the other entry points
    struct Range {
        Range() { nvtxRangePushA("moe_dispatch_layout_static"); }
        ~Range() { nvtxRangePop(); }
    } range;
    // Sizes first (no CUDA call yet): invalid sizes give moe_workspace_bytes == 0
    // and are reported by moe_dispatch_layout below with its own message.
    const size_t need = moe_workspace_bytes(S, T, k, E, P);
    if (need > kStaticScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "moe_dispatch_layout_static: S=%d T=%d E=%d P=%d needs %zu bytes of scratch, "
                 "more than the %zu bytes built into the library; use moe_dispatch_layout "
                 "with a caller-provided workspace",
                 S, T, E, P, need, kStaticScratchBytes);
        return report(MOE_ERR_INVALID_ARG, msg);
    }
    void *scratch = nullptr;
    if (need > 0) {
        const cudaError_t e = static_scratch(&scratch);
        if (e != cudaSuccess) {
            char msg[256];
            snprintf(msg, sizeof msg,
                     "moe_dispatch_layout_static: device address of the built-in scratch: %s",
                     cudaGetErrorString(e));
            return report(MOE_ERR_CUDA, msg);
        }
    }
    // The count kernel writes every scratch entry that the rank kernel reads,
    // so nothing in the array has to start at zero.
    return moe_dispatch_layout(topk_ids, S, T, k, E, P, expert_counts, expert_rank, part_counts,
                               part_offsets, token_slot, scratch, kStaticScratchBytes, dev_status,
                               stream);
}
