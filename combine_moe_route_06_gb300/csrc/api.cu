// api.cu -- the extern "C" entry points of libmoeroute.so: argument checks,
// error reporting, then the launchers of the kernel families.
//
// Nothing here allocates, frees or synchronises; a rejected call enqueues
// nothing on the stream.
#include <stdarg.h>
#include <stdio.h>

#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "launch.h"

namespace {
// One NVTX range per library call (host side: argument checks and enqueue), so a
// profiler's timeline shows which call launched which kernels.  A push/pop costs
// a branch when no tool is attached.
struct CallRange {
    explicit CallRange(const char *name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
};
}  // namespace
#define MOE_CALL_RANGE() CallRange moe_call_range_(__func__)

namespace moe {

namespace {

thread_local char g_msg[512] = "";

moe_status_t fail(moe_status_t code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return code;
}

moe_status_t cuda_status(cudaError_t e, const char *where)
{
    if (e == cudaSuccess) {
        g_msg[0] = '\0';
        return MOE_OK;
    }
    return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

#define REQUIRE(cond, ...)                                         \
    do {                                                           \
        if (!(cond)) return fail(MOE_ERR_INVALID_ARG, __VA_ARGS__); \
    } while (0)

// An array of `count` elements: non-null and aligned unless it is empty.
#define REQUIRE_ARR(p, count, a)                                                             \
    do {                                                                                     \
        if ((int64_t)(count) > 0) {                                                          \
            REQUIRE((p) != nullptr, "%s: null pointer `%s`", __func__, #p);                  \
            REQUIRE(aligned((p), (a)), "%s: `%s` is not %d-byte aligned", __func__, #p, (int)(a)); \
        }                                                                                    \
    } while (0)
// The optional device status word.
#define REQUIRE_STATUS(p) \
    REQUIRE(aligned((p), 4), "%s: `%s` is not 4-byte aligned", __func__, #p)

moe_status_t check_sizes(const char *fn, int S, int T, int k, int E, int P)
{
    REQUIRE(S >= 1, "%s: S=%d must be >= 1", fn, S);
    REQUIRE(T >= 0, "%s: T=%d must be >= 0", fn, T);
    REQUIRE(k >= 1 && k <= kMaxK, "%s: k=%d must be in [1, %d]", fn, k, kMaxK);
    REQUIRE(E >= k && E <= kMaxE, "%s: E=%d must be in [k=%d, %d]", fn, E, k, kMaxE);
    REQUIRE(P >= 1 && P <= kMaxP, "%s: P=%d must be in [1, %d]", fn, P, kMaxP);
    REQUIRE(E % P == 0, "%s: E=%d must be a multiple of P=%d", fn, E, P);
    REQUIRE((int64_t)S * T * k < ((int64_t)1 << 31), "%s: S*T*k must be < 2^31", fn);
    REQUIRE((int64_t)S * T * P < ((int64_t)1 << 31), "%s: S*T*P must be < 2^31", fn);
    return MOE_OK;
}

}  // namespace

int resident_grid(const void *kernel, int threads, size_t smem)
{
    struct Key {
        const void *k;
        int dev, threads;
        size_t smem;
    };
    static std::mutex mu;
    static Key keys[64];
    static int vals[64];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; i++)
        if (keys[i].k == kernel && keys[i].dev == dev && keys[i].threads == threads &&
            keys[i].smem == smem)
            return vals[i];
    DeviceInfo di;
    int per_sm = 0;
    if (device_info(&di) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess)
        return 0;
    const int v = (per_sm > 0 ? per_sm : 1) * di.sm_count;
    if (used < 64) {
        keys[used] = {kernel, dev, threads, smem};
        vals[used] = v;
        used++;
    }
    return v;
}

moe_status_t report(moe_status_t code, const char *message)
{
    return fail(code, "%s", message);
}

cudaError_t device_info(DeviceInfo *out)
{
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        DeviceInfo d{};
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) !=
            cudaSuccess)
            return e;
        if ((e = cudaDeviceGetAttribute(&d.max_smem_optin,
                                        cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
            cudaSuccess)
            return e;
        cache[dev] = d;
        have[dev] = true;
    }
    *out = cache[dev];
    return cudaSuccess;
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_version(void) { return 10000; }

const char *moe_status_string(moe_status_t code)
{
    switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_CAPACITY: return "capacity exceeded";
    case MOE_ERR_BAD_EXPERT_ID: return "expert id out of range";
    case MOE_ERR_TIMEOUT: return "timeout";
    case MOE_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

const char *moe_last_error_message(void) { return g_msg; }

size_t moe_workspace_bytes(int S, int T, int k, int E, int P)
{
    if (check_sizes("moe_workspace_bytes", S, T, k, E, P) != MOE_OK) return 0;
    const size_t a = layout_ws_bytes(S, T, E, P);
    const size_t b = permute_ws_bytes(S, T, E);
    return a > b ? a : b;
}

int moe_dispatch_layout_kernels(int S, int T, int k, int E, int P)
{
    if (check_sizes("moe_dispatch_layout_kernels", S, T, k, E, P) != MOE_OK) return -1;
    int n = 0;
    if (layout_kernel_count(T, k, E, P, &n) != cudaSuccess) return -1;
    return n;
}

int moe_permute_to_experts_kernels(int S, int T, int k, int E, int P)
{
    if (check_sizes("moe_permute_to_experts_kernels", S, T, k, E, P) != MOE_OK) return -1;
    return permute_map_fused(S, E) ? 1 : 2;
}

moe_status_t moe_route_topk(const float *logits, int S, int T, int E, int k, int32_t *topk_ids,
                            float *topk_w, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, k, E, 1);
    if (st != MOE_OK) return st;
    REQUIRE((int64_t)S * T * E < ((int64_t)1 << 40), "%s: S*T*E too large", __func__);
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(logits, NT * E, 4);
    REQUIRE_ARR(topk_ids, NT * k, 4);
    REQUIRE_ARR(topk_w, NT * k, 4);
    return cuda_status(launch_route_topk(logits, (int64_t)S * T, E, k, topk_ids, topk_w, stream),
                       __func__);
}

moe_status_t moe_dispatch_layout(const int32_t *topk_ids, int S, int T, int k, int E, int P,
                                 int32_t *expert_counts, int32_t *expert_rank,
                                 int32_t *part_counts, int32_t *part_offsets, int32_t *token_slot,
                                 void *ws, size_t ws_bytes, uint32_t *dev_status,
                                 cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, k, E, P);
    if (st != MOE_OK) return st;
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(topk_ids, NT * k, 4);
    REQUIRE_ARR(expert_counts, (int64_t)S * E, 4);
    REQUIRE_ARR(expert_rank, NT * k, 4);
    REQUIRE_ARR(part_counts, (int64_t)S * P, 4);
    REQUIRE_ARR(part_offsets, (int64_t)S * (P + 1), 4);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_STATUS(dev_status);
    const size_t need = moe_workspace_bytes(S, T, k, E, P);
    REQUIRE_ARR(ws, need, 256);
    REQUIRE(ws_bytes >= need, "%s: ws_bytes=%zu < required %zu", __func__, ws_bytes, need);
    return cuda_status(launch_dispatch_layout(topk_ids, S, T, k, E, P, expert_counts, expert_rank,
                                              part_counts, part_offsets, token_slot, ws,
                                              dev_status, stream),
                       __func__);
}

moe_status_t moe_dispatch_pack(const uint16_t *x, int S, int T, int H, int P,
                               const int32_t *token_slot, const int32_t *part_offsets,
                               int cap_send, uint16_t *send, int32_t *send_src,
                               uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, 1, P, P);
    if (st != MOE_OK) return st;
    REQUIRE(H >= 8 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", __func__, H);
    REQUIRE(cap_send >= 0, "%s: cap_send=%d must be >= 0", __func__, cap_send);
    REQUIRE((int64_t)S * cap_send < ((int64_t)1 << 31), "%s: S*cap_send must be < 2^31", __func__);
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(x, NT * H, 16);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_ARR(part_offsets, (int64_t)S * (P + 1), 4);
    REQUIRE_ARR(send, (int64_t)S * cap_send * H, 16);
    REQUIRE_ARR(send_src, (int64_t)S * cap_send, 4);
    REQUIRE_STATUS(dev_status);
    return cuda_status(launch_dispatch_pack(x, S, T, H, P, token_slot, part_offsets, cap_send,
                                            send, send_src, dev_status, stream),
                       __func__);
}

moe_status_t moe_dispatch_pack_mxfp8(const uint16_t *x, int S, int T, int H, int P,
                                     const int32_t *token_slot, const int32_t *part_offsets,
                                     int cap_send, uint8_t *send_q, int32_t *send_src,
                                     uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, 1, P, P);
    if (st != MOE_OK) return st;
    REQUIRE(H >= 256 && H % 256 == 0, "%s: H=%d must be a positive multiple of 256", __func__, H);
    REQUIRE(cap_send >= 0, "%s: cap_send=%d must be >= 0", __func__, cap_send);
    REQUIRE((int64_t)S * cap_send < ((int64_t)1 << 31), "%s: S*cap_send must be < 2^31", __func__);
    const int64_t NT = (int64_t)S * T;
    const int64_t rb = (int64_t)H + H / 32;
    REQUIRE_ARR(x, NT * H, 16);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_ARR(part_offsets, (int64_t)S * (P + 1), 4);
    REQUIRE_ARR(send_q, (int64_t)S * cap_send * rb, 8);
    REQUIRE_ARR(send_src, (int64_t)S * cap_send, 4);
    REQUIRE_STATUS(dev_status);
    return cuda_status(launch_dispatch_pack_mxfp8(x, S, T, H, P, token_slot, part_offsets,
                                                  cap_send, send_q, send_src, dev_status, stream),
                       __func__);
}

moe_status_t moe_permute_to_experts(const uint16_t *send, const int32_t *token_slot,
                                    const int32_t *topk_ids, const int32_t *expert_counts,
                                    const int32_t *expert_rank, int S, int T, int k, int E, int P,
                                    int H, int recv_part, int align, int cap_send, int cap_recv,
                                    uint16_t *recv, int32_t *expert_offsets, int32_t *pair_row,
                                    int32_t *recv_pair, void *ws, size_t ws_bytes,
                                    uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, k, E, P);
    if (st != MOE_OK) return st;
    REQUIRE(H >= 8 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", __func__, H);
    REQUIRE(recv_part >= -1 && recv_part < P, "%s: recv_part=%d must be in [-1, P)", __func__,
            recv_part);
    REQUIRE(align >= 1 && align <= 1024, "%s: align=%d must be in [1, 1024]", __func__, align);
    REQUIRE(cap_send >= 0 && cap_recv >= 0, "%s: capacities must be >= 0", __func__);
    REQUIRE((int64_t)S * cap_send < ((int64_t)1 << 31), "%s: S*cap_send must be < 2^31", __func__);
    REQUIRE((int64_t)S * T * k + (int64_t)E * (align - 1) < ((int64_t)1 << 31),
            "%s: S*T*k + E*(align-1) must be < 2^31", __func__);
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(send, (int64_t)S * cap_send * H, 16);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_ARR(topk_ids, NT * k, 4);
    REQUIRE_ARR(expert_counts, (int64_t)S * E, 4);
    REQUIRE_ARR(expert_rank, NT * k, 4);
    REQUIRE_ARR(recv, (int64_t)cap_recv * H, 16);
    REQUIRE_ARR(expert_offsets, E + 1, 4);
    REQUIRE_ARR(pair_row, NT * k, 4);
    REQUIRE_ARR(recv_pair, cap_recv, 4);
    REQUIRE_STATUS(dev_status);
    const size_t need = moe_workspace_bytes(S, T, k, E, P);
    REQUIRE_ARR(ws, need, 256);
    REQUIRE(ws_bytes >= need, "%s: ws_bytes=%zu < required %zu", __func__, ws_bytes, need);
    return cuda_status(launch_permute(send, token_slot, topk_ids, expert_counts, expert_rank, S, T,
                                      k, E, P, H, recv_part, align, cap_send, cap_recv, recv,
                                      expert_offsets, pair_row, recv_pair, ws, dev_status, stream),
                       __func__);
}

int moe_dispatch_kernels(int S, int T, int k, int E, int P)
{
    if (check_sizes("moe_dispatch_kernels", S, T, k, E, P) != MOE_OK) return -1;
    int n = 0;
    if (dispatch_kernel_count(S, T, k, E, P, &n) != cudaSuccess) return -1;
    return n;
}

moe_status_t moe_dispatch(const float *logits, const uint16_t *x, int S, int T, int H, int E,
                          int k, int P, int recv_part, int align, int cap_send, int cap_recv,
                          int32_t *topk_ids, float *topk_w, int32_t *expert_counts,
                          int32_t *expert_rank, int32_t *part_counts, int32_t *part_offsets,
                          int32_t *token_slot, uint16_t *send, int32_t *send_src, uint16_t *recv,
                          int32_t *expert_offsets, int32_t *pair_row, int32_t *recv_pair,
                          void *ws, size_t ws_bytes, uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, k, E, P);
    if (st != MOE_OK) return st;
    REQUIRE((int64_t)S * T * E < ((int64_t)1 << 40), "%s: S*T*E too large", __func__);
    REQUIRE(H >= 8 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", __func__, H);
    REQUIRE(recv_part >= -1 && recv_part < P, "%s: recv_part=%d must be in [-1, P)", __func__,
            recv_part);
    REQUIRE(align >= 1 && align <= 1024, "%s: align=%d must be in [1, 1024]", __func__, align);
    REQUIRE(cap_send >= 0 && cap_recv >= 0, "%s: capacities must be >= 0", __func__);
    REQUIRE((int64_t)S * cap_send < ((int64_t)1 << 31), "%s: S*cap_send must be < 2^31", __func__);
    REQUIRE((int64_t)S * T * k + (int64_t)E * (align - 1) < ((int64_t)1 << 31),
            "%s: S*T*k + E*(align-1) must be < 2^31", __func__);
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(logits, NT * E, 4);
    REQUIRE_ARR(x, NT * H, 16);
    REQUIRE_ARR(topk_ids, NT * k, 4);
    REQUIRE_ARR(topk_w, NT * k, 4);
    REQUIRE_ARR(expert_counts, (int64_t)S * E, 4);
    REQUIRE_ARR(expert_rank, NT * k, 4);
    REQUIRE_ARR(part_counts, (int64_t)S * P, 4);
    REQUIRE_ARR(part_offsets, (int64_t)S * (P + 1), 4);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_ARR(send, (int64_t)S * cap_send * H, 16);
    REQUIRE_ARR(send_src, (int64_t)S * cap_send, 4);
    REQUIRE_ARR(recv, (int64_t)cap_recv * H, 16);
    REQUIRE_ARR(expert_offsets, E + 1, 4);
    REQUIRE_ARR(pair_row, NT * k, 4);
    REQUIRE_ARR(recv_pair, cap_recv, 4);
    REQUIRE_STATUS(dev_status);
    const size_t need = moe_workspace_bytes(S, T, k, E, P);
    REQUIRE_ARR(ws, need, 256);
    REQUIRE(ws_bytes >= need, "%s: ws_bytes=%zu < required %zu", __func__, ws_bytes, need);
    return cuda_status(launch_dispatch(logits, x, S, T, H, E, k, P, recv_part, align, cap_send,
                                       cap_recv, topk_ids, topk_w, expert_counts, expert_rank,
                                       part_counts, part_offsets, token_slot, send, send_src, recv,
                                       expert_offsets, pair_row, recv_pair, ws, dev_status, stream),
                       __func__);
}

int moe_dispatch_pack_permute_kernels(int S, int T, int k, int E, int P)
{
    if (check_sizes("moe_dispatch_pack_permute_kernels", S, T, k, E, P) != MOE_OK) return -1;
    return pack_permute_kernel_count(S, T, E);
}

moe_status_t moe_dispatch_pack_permute(const uint16_t *x, const int32_t *token_slot,
                                       const int32_t *part_offsets, const int32_t *topk_ids,
                                       const int32_t *expert_counts, const int32_t *expert_rank,
                                       int S, int T, int k, int E, int P, int H, int recv_part,
                                       int align, int cap_send, int cap_recv, uint16_t *send,
                                       int32_t *send_src, uint16_t *recv,
                                       int32_t *expert_offsets, int32_t *pair_row,
                                       int32_t *recv_pair, void *ws, size_t ws_bytes,
                                       uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, k, E, P);
    if (st != MOE_OK) return st;
    REQUIRE(H >= 8 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", __func__, H);
    REQUIRE(recv_part >= -1 && recv_part < P, "%s: recv_part=%d must be in [-1, P)", __func__,
            recv_part);
    REQUIRE(align >= 1 && align <= 1024, "%s: align=%d must be in [1, 1024]", __func__, align);
    REQUIRE(cap_send >= 0 && cap_recv >= 0, "%s: capacities must be >= 0", __func__);
    REQUIRE((int64_t)S * cap_send < ((int64_t)1 << 31), "%s: S*cap_send must be < 2^31", __func__);
    REQUIRE((int64_t)S * T * k + (int64_t)E * (align - 1) < ((int64_t)1 << 31),
            "%s: S*T*k + E*(align-1) must be < 2^31", __func__);
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(x, NT * H, 16);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_ARR(part_offsets, (int64_t)S * (P + 1), 4);
    REQUIRE_ARR(topk_ids, NT * k, 4);
    REQUIRE_ARR(expert_counts, (int64_t)S * E, 4);
    REQUIRE_ARR(expert_rank, NT * k, 4);
    REQUIRE_ARR(send, (int64_t)S * cap_send * H, 16);
    REQUIRE_ARR(send_src, (int64_t)S * cap_send, 4);
    REQUIRE_ARR(recv, (int64_t)cap_recv * H, 16);
    REQUIRE_ARR(expert_offsets, E + 1, 4);
    REQUIRE_ARR(pair_row, NT * k, 4);
    REQUIRE_ARR(recv_pair, cap_recv, 4);
    REQUIRE_STATUS(dev_status);
    const size_t need = moe_workspace_bytes(S, T, k, E, P);
    REQUIRE_ARR(ws, need, 256);
    REQUIRE(ws_bytes >= need, "%s: ws_bytes=%zu < required %zu", __func__, ws_bytes, need);
    return cuda_status(launch_pack_permute(x, token_slot, part_offsets, topk_ids, expert_counts,
                                           expert_rank, S, T, k, E, P, H, recv_part, align,
                                           cap_send, cap_recv, send, send_src, recv,
                                           expert_offsets, pair_row, recv_pair, ws, dev_status,
                                           stream, false),
                       __func__);
}

int moe_dispatch_pack_permute_masked_kernels(int S, int T, int k, int E, int P, int recv_part)
{
    if (check_sizes("moe_dispatch_pack_permute_masked_kernels", S, T, k, E, P) != MOE_OK) return -1;
    if (recv_part < -1 || recv_part >= P) return -1;
    return pack_permute_masked_kernel_count(S, T, E, P, recv_part);
}

moe_status_t moe_dispatch_pack_permute_masked(const uint16_t *x, const int32_t *token_slot,
                                              const int32_t *part_offsets,
                                              const int32_t *topk_ids,
                                              const int32_t *expert_counts,
                                              const int32_t *expert_rank, int S, int T, int k,
                                              int E, int P, int H, int recv_part, int block_rows,
                                              int cap_send, uint16_t *send, int32_t *send_src,
                                              uint16_t *recv, int32_t *masked_counts,
                                              int32_t *pair_row, int32_t *recv_pair,
                                              uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, k, E, P);
    if (st != MOE_OK) return st;
    REQUIRE(H >= 8 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", __func__, H);
    REQUIRE(recv_part >= -1 && recv_part < P, "%s: recv_part=%d must be in [-1, P)", __func__,
            recv_part);
    REQUIRE(block_rows >= 0, "%s: block_rows=%d must be >= 0", __func__, block_rows);
    REQUIRE(cap_send >= 0, "%s: cap_send=%d must be >= 0", __func__, cap_send);
    REQUIRE((int64_t)S * cap_send < ((int64_t)1 << 31), "%s: S*cap_send must be < 2^31", __func__);
    const int64_t nb = recv_part < 0 ? E : E / P;
    REQUIRE(nb * block_rows < ((int64_t)1 << 31), "%s: blocks*block_rows must be < 2^31",
            __func__);
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(x, NT * H, 16);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_ARR(part_offsets, (int64_t)S * (P + 1), 4);
    REQUIRE_ARR(topk_ids, NT * k, 4);
    REQUIRE_ARR(expert_counts, (int64_t)S * E, 4);
    REQUIRE_ARR(expert_rank, NT * k, 4);
    REQUIRE_ARR(send, (int64_t)S * cap_send * H, 16);
    REQUIRE_ARR(send_src, (int64_t)S * cap_send, 4);
    REQUIRE_ARR(recv, nb * block_rows * H, 16);
    REQUIRE_ARR(masked_counts, nb, 4);
    REQUIRE_ARR(pair_row, NT * k, 4);
    REQUIRE_ARR(recv_pair, nb * block_rows, 4);
    REQUIRE_STATUS(dev_status);
    return cuda_status(launch_pack_permute_masked(x, token_slot, part_offsets, topk_ids,
                                                  expert_counts, expert_rank, S, T, k, E, P, H,
                                                  recv_part, block_rows, cap_send, send, send_src,
                                                  recv, masked_counts, pair_row, recv_pair,
                                                  dev_status, stream, false),
                       __func__);
}

int moe_dispatch_masked_kernels(int S, int T, int k, int E, int P, int recv_part)
{
    if (check_sizes("moe_dispatch_masked_kernels", S, T, k, E, P) != MOE_OK) return -1;
    if (recv_part < -1 || recv_part >= P) return -1;
    return dispatch_masked_kernel_count(S, T, k, E, P, recv_part);
}

moe_status_t moe_dispatch_masked(const float *logits, const uint16_t *x, int S, int T, int H,
                                 int E, int k, int P, int recv_part, int block_rows,
                                 int cap_send, int32_t *topk_ids, float *topk_w,
                                 int32_t *expert_counts, int32_t *expert_rank,
                                 int32_t *part_counts, int32_t *part_offsets,
                                 int32_t *token_slot, uint16_t *send, int32_t *send_src,
                                 uint16_t *recv, int32_t *masked_counts, int32_t *pair_row,
                                 int32_t *recv_pair, void *ws, size_t ws_bytes,
                                 uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, k, E, P);
    if (st != MOE_OK) return st;
    REQUIRE((int64_t)S * T * E < ((int64_t)1 << 40), "%s: S*T*E too large", __func__);
    REQUIRE(H >= 8 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", __func__, H);
    REQUIRE(recv_part >= -1 && recv_part < P, "%s: recv_part=%d must be in [-1, P)", __func__,
            recv_part);
    REQUIRE(block_rows >= 0, "%s: block_rows=%d must be >= 0", __func__, block_rows);
    REQUIRE(cap_send >= 0, "%s: cap_send=%d must be >= 0", __func__, cap_send);
    REQUIRE((int64_t)S * cap_send < ((int64_t)1 << 31), "%s: S*cap_send must be < 2^31", __func__);
    const int64_t nb = recv_part < 0 ? E : E / P;
    REQUIRE(nb * block_rows < ((int64_t)1 << 31), "%s: blocks*block_rows must be < 2^31",
            __func__);
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(logits, NT * E, 4);
    REQUIRE_ARR(x, NT * H, 16);
    REQUIRE_ARR(topk_ids, NT * k, 4);
    REQUIRE_ARR(topk_w, NT * k, 4);
    REQUIRE_ARR(expert_counts, (int64_t)S * E, 4);
    REQUIRE_ARR(expert_rank, NT * k, 4);
    REQUIRE_ARR(part_counts, (int64_t)S * P, 4);
    REQUIRE_ARR(part_offsets, (int64_t)S * (P + 1), 4);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_ARR(send, (int64_t)S * cap_send * H, 16);
    REQUIRE_ARR(send_src, (int64_t)S * cap_send, 4);
    REQUIRE_ARR(recv, nb * block_rows * H, 16);
    REQUIRE_ARR(masked_counts, nb, 4);
    REQUIRE_ARR(pair_row, NT * k, 4);
    REQUIRE_ARR(recv_pair, nb * block_rows, 4);
    REQUIRE_STATUS(dev_status);
    const size_t need = moe_workspace_bytes(S, T, k, E, P);
    REQUIRE_ARR(ws, need, 256);
    REQUIRE(ws_bytes >= need, "%s: ws_bytes=%zu < required %zu", __func__, ws_bytes, need);
    return cuda_status(launch_dispatch_masked(logits, x, S, T, H, E, k, P, recv_part, block_rows,
                                              cap_send, topk_ids, topk_w, expert_counts,
                                              expert_rank, part_counts, part_offsets, token_slot,
                                              send, send_src, recv, masked_counts, pair_row,
                                              recv_pair, ws, dev_status, stream),
                       __func__);
}

int moe_dispatch_quantized_kernels(int S, int T, int k, int E, int P)
{
    if (check_sizes("moe_dispatch_quantized_kernels", S, T, k, E, P) != MOE_OK) return -1;
    int n = 0;
    if (dispatch_quantized_kernel_count(S, T, k, E, P, &n) != cudaSuccess) return -1;
    return n;
}

moe_status_t moe_dispatch_quantized(const float *logits, const uint16_t *x, int S, int T, int H,
                                    int E, int k, int P, int format, float global_scale,
                                    int recv_part, int align, int cap_send, int cap_recv,
                                    int32_t *topk_ids, float *topk_w, int32_t *expert_counts,
                                    int32_t *expert_rank, int32_t *part_counts,
                                    int32_t *part_offsets, int32_t *token_slot, uint8_t *send_q,
                                    int32_t *send_src, uint8_t *recv_q, int32_t *expert_offsets,
                                    int32_t *pair_row, int32_t *recv_pair, void *ws,
                                    size_t ws_bytes, uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, k, E, P);
    if (st != MOE_OK) return st;
    REQUIRE(format == MOE_FORMAT_MXFP8 || format == MOE_FORMAT_NVFP4,
            "%s: format=%d must be MOE_FORMAT_MXFP8 (1) or MOE_FORMAT_NVFP4 (2)", __func__, format);
    if (format == MOE_FORMAT_MXFP8)
        REQUIRE(H >= 512 && H % 512 == 0, "%s: H=%d must be a positive multiple of 512 for MXFP8",
                __func__, H);
    else
        REQUIRE(H >= 256 && H % 256 == 0, "%s: H=%d must be a positive multiple of 256 for NVFP4",
                __func__, H);
    REQUIRE(format != MOE_FORMAT_NVFP4 || (global_scale > 0.f && global_scale < 3.0e38f),
            "%s: global_scale must be positive and finite", __func__);
    REQUIRE((int64_t)S * T * E < ((int64_t)1 << 40), "%s: S*T*E too large", __func__);
    REQUIRE(recv_part >= -1 && recv_part < P, "%s: recv_part=%d must be in [-1, P)", __func__,
            recv_part);
    REQUIRE(align >= 1 && align <= 1024, "%s: align=%d must be in [1, 1024]", __func__, align);
    REQUIRE(cap_send >= 0 && cap_recv >= 0, "%s: capacities must be >= 0", __func__);
    REQUIRE((int64_t)S * cap_send < ((int64_t)1 << 31), "%s: S*cap_send must be < 2^31", __func__);
    REQUIRE((int64_t)S * T * k + (int64_t)E * (align - 1) < ((int64_t)1 << 31),
            "%s: S*T*k + E*(align-1) must be < 2^31", __func__);
    const int64_t NT = (int64_t)S * T;
    const int64_t rb = format == MOE_FORMAT_MXFP8 ? (int64_t)H + H / 32 : (int64_t)H / 2 + H / 16;
    REQUIRE_ARR(logits, NT * E, 4);
    REQUIRE_ARR(x, NT * H, 16);
    REQUIRE_ARR(topk_ids, NT * k, 4);
    REQUIRE_ARR(topk_w, NT * k, 4);
    REQUIRE_ARR(expert_counts, (int64_t)S * E, 4);
    REQUIRE_ARR(expert_rank, NT * k, 4);
    REQUIRE_ARR(part_counts, (int64_t)S * P, 4);
    REQUIRE_ARR(part_offsets, (int64_t)S * (P + 1), 4);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_ARR(send_q, (int64_t)S * cap_send * rb, 16);
    REQUIRE_ARR(send_src, (int64_t)S * cap_send, 4);
    REQUIRE_ARR(recv_q, (int64_t)cap_recv * rb, 16);
    REQUIRE_ARR(expert_offsets, E + 1, 4);
    REQUIRE_ARR(pair_row, NT * k, 4);
    REQUIRE_ARR(recv_pair, cap_recv, 4);
    REQUIRE_STATUS(dev_status);
    const size_t need = moe_workspace_bytes(S, T, k, E, P);
    REQUIRE_ARR(ws, need, 256);
    REQUIRE(ws_bytes >= need, "%s: ws_bytes=%zu < required %zu", __func__, ws_bytes, need);
    return cuda_status(launch_dispatch_quantized(logits, x, S, T, H, E, k, P, format, global_scale,
                                                 recv_part, align, cap_send, cap_recv, topk_ids,
                                                 topk_w, expert_counts, expert_rank, part_counts,
                                                 part_offsets, token_slot, send_q, send_src,
                                                 recv_q, expert_offsets, pair_row, recv_pair, ws,
                                                 dev_status, stream),
                       __func__);
}

moe_status_t moe_permute_to_experts_masked(const uint16_t *send, const int32_t *token_slot,
                                           const int32_t *topk_ids, const int32_t *expert_counts,
                                           const int32_t *expert_rank, int S, int T, int k,
                                           int E, int P, int H, int recv_part, int block_rows,
                                           int cap_send, uint16_t *recv, int32_t *masked_counts,
                                           int32_t *pair_row, int32_t *recv_pair,
                                           uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, k, E, P);
    if (st != MOE_OK) return st;
    REQUIRE(H >= 8 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", __func__, H);
    REQUIRE(recv_part >= -1 && recv_part < P, "%s: recv_part=%d must be in [-1, P)", __func__,
            recv_part);
    REQUIRE(block_rows >= 0, "%s: block_rows=%d must be >= 0", __func__, block_rows);
    REQUIRE(cap_send >= 0, "%s: cap_send=%d must be >= 0", __func__, cap_send);
    REQUIRE((int64_t)S * cap_send < ((int64_t)1 << 31), "%s: S*cap_send must be < 2^31", __func__);
    const int64_t nb = recv_part < 0 ? E : E / P;
    REQUIRE(nb * block_rows < ((int64_t)1 << 31), "%s: blocks*block_rows must be < 2^31",
            __func__);
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(send, (int64_t)S * cap_send * H, 16);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_ARR(topk_ids, NT * k, 4);
    REQUIRE_ARR(expert_counts, (int64_t)S * E, 4);
    REQUIRE_ARR(expert_rank, NT * k, 4);
    REQUIRE_ARR(recv, nb * block_rows * H, 16);
    REQUIRE_ARR(masked_counts, nb, 4);
    REQUIRE_ARR(pair_row, NT * k, 4);
    REQUIRE_ARR(recv_pair, nb * block_rows, 4);
    REQUIRE_STATUS(dev_status);
    return cuda_status(launch_permute_masked(send, token_slot, topk_ids, expert_counts, expert_rank,
                                             S, T, k, E, P, H, recv_part, block_rows, cap_send,
                                             recv, masked_counts, pair_row, recv_pair, dev_status,
                                             stream),
                       __func__);
}

moe_status_t moe_combine(const uint16_t *y, int y_rows, const int32_t *pair_row,
                         const float *topk_w, int S, int T, int k, int H, uint16_t *out,
                         uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, k, k, 1);
    if (st != MOE_OK) return st;
    REQUIRE(H >= 8 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", __func__, H);
    REQUIRE(y_rows >= 0, "%s: y_rows=%d must be >= 0", __func__, y_rows);
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(y, (int64_t)y_rows * H, 16);
    REQUIRE_ARR(pair_row, NT * k, 4);
    REQUIRE_ARR(topk_w, NT * k, 4);
    REQUIRE_ARR(out, NT * H, 16);
    REQUIRE_STATUS(dev_status);
    return cuda_status(
        launch_combine(y, y_rows, pair_row, topk_w, NT, k, H, out, dev_status, stream), __func__);
}

moe_status_t moe_combine_stage1(const uint16_t *y, int y_rows, const int32_t *pair_row,
                                const float *topk_w, const int32_t *topk_ids,
                                const int32_t *token_slot, int S, int T, int k, int E, int P,
                                int H, int recv_part, int cap_send, uint16_t *ret,
                                uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, k, E, P);
    if (st != MOE_OK) return st;
    REQUIRE(H >= 8 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", __func__, H);
    REQUIRE(recv_part >= -1 && recv_part < P, "%s: recv_part=%d must be in [-1, P)", __func__,
            recv_part);
    REQUIRE(y_rows >= 0 && cap_send >= 0, "%s: y_rows and cap_send must be >= 0", __func__);
    REQUIRE((int64_t)S * cap_send < ((int64_t)1 << 31), "%s: S*cap_send must be < 2^31", __func__);
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(y, (int64_t)y_rows * H, 16);
    REQUIRE_ARR(pair_row, NT * k, 4);
    REQUIRE_ARR(topk_w, NT * k, 4);
    REQUIRE_ARR(topk_ids, NT * k, 4);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_ARR(ret, (int64_t)S * cap_send * H, 16);
    REQUIRE_STATUS(dev_status);
    return cuda_status(launch_combine_stage1(y, y_rows, pair_row, topk_w, topk_ids, token_slot, S,
                                             T, k, E, P, H, recv_part, cap_send, ret, dev_status,
                                             stream),
                       __func__);
}

moe_status_t moe_combine_stage2(const uint16_t *ret, const int32_t *token_slot, int S, int T,
                                int P, int H, int recv_part, int cap_send, uint16_t *out,
                                uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, 1, P, P);
    if (st != MOE_OK) return st;
    REQUIRE(recv_part >= -1 && recv_part < P, "%s: recv_part=%d must be in [-1, %d)", __func__,
            recv_part, P);
    REQUIRE(H >= 8 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", __func__, H);
    REQUIRE(cap_send >= 0, "%s: cap_send=%d must be >= 0", __func__, cap_send);
    REQUIRE((int64_t)S * cap_send < ((int64_t)1 << 31), "%s: S*cap_send must be < 2^31", __func__);
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(ret, (int64_t)S * cap_send * H, 16);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_ARR(out, NT * H, 16);
    REQUIRE_STATUS(dev_status);
    return cuda_status(
        launch_combine_stage2(ret, token_slot, S, T, P, H, recv_part, cap_send, out, dev_status,
                              stream),
        __func__);
}

moe_status_t moe_expert_scale(const uint16_t *recv, const int32_t *expert_offsets,
                              const float *scale, int E, int H, int cap_recv, uint16_t *y,
                              cudaStream_t stream)
{
    MOE_CALL_RANGE();
    REQUIRE(E >= 1 && E <= kMaxE, "%s: E=%d must be in [1, %d]", __func__, E, kMaxE);
    REQUIRE(H >= 8 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", __func__, H);
    REQUIRE(cap_recv >= 0, "%s: cap_recv=%d must be >= 0", __func__, cap_recv);
    REQUIRE_ARR(recv, (int64_t)cap_recv * H, 16);
    REQUIRE_ARR(expert_offsets, E + 1, 4);
    REQUIRE_ARR(scale, E, 4);
    REQUIRE_ARR(y, (int64_t)cap_recv * H, 16);
    return cuda_status(
        launch_expert_scale(recv, expert_offsets, scale, E, H, cap_recv, y, stream), __func__);
}

moe_status_t moe_expert_scale_mxfp8(const uint8_t *recv_q, const int32_t *expert_offsets,
                                    const float *scale, int E, int H, int cap_recv, uint16_t *y,
                                    cudaStream_t stream)
{
    MOE_CALL_RANGE();
    REQUIRE(E >= 1 && E <= kMaxE, "%s: E=%d must be in [1, %d]", __func__, E, kMaxE);
    REQUIRE(H >= 256 && H % 256 == 0, "%s: H=%d must be a positive multiple of 256", __func__, H);
    REQUIRE(cap_recv >= 0, "%s: cap_recv=%d must be >= 0", __func__, cap_recv);
    REQUIRE_ARR(recv_q, (int64_t)cap_recv * (H + H / 32), 8);
    REQUIRE_ARR(expert_offsets, E + 1, 4);
    REQUIRE_ARR(scale, E, 4);
    REQUIRE_ARR(y, (int64_t)cap_recv * H, 16);
    return cuda_status(
        launch_expert_scale_mxfp8(recv_q, expert_offsets, scale, E, H, cap_recv, y, stream),
        __func__);
}

moe_status_t moe_plan_placement(const int64_t *load, int E, int P, int R, int32_t *copy_offsets,
                                int32_t *copy_slots, int32_t *slot_expert, int64_t *part_load)
{
    REQUIRE(E >= 1 && E <= kMaxE, "%s: E=%d must be in [1, %d]", __func__, E, kMaxE);
    REQUIRE(P >= 1 && P <= kMaxP, "%s: P=%d must be in [1, %d]", __func__, P, kMaxP);
    REQUIRE(E % P == 0, "%s: E=%d must be a multiple of P=%d", __func__, E, P);
    REQUIRE(R >= 0 && (int64_t)P * (E / P + R) <= kMaxE,
            "%s: R=%d: P*(E/P+R) slots must be at most %d", __func__, R, kMaxE);
    REQUIRE(load && copy_offsets && copy_slots && slot_expert && part_load,
            "%s: null pointer", __func__);
    for (int e = 0; e < E; e++)
        REQUIRE(load[e] >= 0, "%s: load[%d] < 0", __func__, e);
    plan_placement(load, E, P, R, copy_offsets, copy_slots, slot_expert, part_load);
    return MOE_OK;
}

size_t moe_workspace_bytes_mapped(int S, int T, int k, int E, int P, int Lp)
{
    if (check_sizes("moe_workspace_bytes_mapped", S, T, k, E, P) != MOE_OK) return 0;
    if (Lp < E / P || (int64_t)P * Lp > kMaxE) return 0;
    return mapped_ws_bytes(S, T, k, E, P, P * Lp);
}

moe_status_t moe_dispatch_layout_mapped(const int32_t *topk_ids, int S, int T, int k, int E,
                                        int P, int Lp, const int32_t *copy_offsets,
                                        const int32_t *copy_slots, int n_copies,
                                        int32_t *phys_ids, int32_t *expert_counts,
                                        int32_t *expert_rank, int32_t *part_counts,
                                        int32_t *part_offsets, int32_t *token_slot, void *ws,
                                        size_t ws_bytes, uint32_t *dev_status,
                                        cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, k, E, P);
    if (st != MOE_OK) return st;
    REQUIRE(Lp >= E / P && (int64_t)P * Lp <= kMaxE,
            "%s: Lp=%d must be in [E/P, %d/P]", __func__, Lp, kMaxE);
    REQUIRE(n_copies >= E && n_copies <= P * Lp, "%s: n_copies=%d must be in [E, P*Lp]",
            __func__, n_copies);
    const int E_phys = P * Lp;
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(topk_ids, NT * k, 4);
    REQUIRE_ARR(copy_offsets, E + 1, 4);
    REQUIRE_ARR(copy_slots, n_copies, 4);
    REQUIRE_ARR(phys_ids, NT * k, 4);
    REQUIRE_ARR(expert_counts, (int64_t)S * E_phys, 4);
    REQUIRE_ARR(expert_rank, NT * k, 4);
    REQUIRE_ARR(part_counts, (int64_t)S * P, 4);
    REQUIRE_ARR(part_offsets, (int64_t)S * (P + 1), 4);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_STATUS(dev_status);
    const size_t need = mapped_ws_bytes(S, T, k, E, P, E_phys);
    REQUIRE_ARR(ws, need, 256);
    REQUIRE(ws_bytes >= need, "%s: ws_bytes=%zu < required %zu", __func__, ws_bytes, need);
    return cuda_status(launch_dispatch_layout_mapped(topk_ids, S, T, k, E, P, E_phys,
                                                     copy_offsets, copy_slots, n_copies, phys_ids,
                                                     expert_counts, expert_rank, part_counts,
                                                     part_offsets, token_slot, ws, dev_status,
                                                     stream),
                       __func__);
}

moe_status_t moe_dispatch_pack_routed(const uint16_t *x, const int32_t *topk_ids,
                                      const float *topk_w, int S, int T, int H, int k, int P,
                                      const int32_t *token_slot, const int32_t *part_offsets,
                                      int cap_send, uint16_t *send, int32_t *send_src,
                                      int32_t *send_ids, float *send_w, uint32_t *dev_status,
                                      cudaStream_t stream)
{
    MOE_CALL_RANGE();
    REQUIRE(S >= 1 && T >= 0, "%s: S=%d, T=%d", __func__, S, T);
    REQUIRE(k >= 1 && k <= kMaxK, "%s: k=%d must be in [1, %d]", __func__, k, kMaxK);
    REQUIRE(P >= 1 && P <= kMaxP, "%s: P=%d must be in [1, %d]", __func__, P, kMaxP);
    REQUIRE((int64_t)S * T * (k > P ? k : P) < ((int64_t)1 << 31), "%s: S*T*max(k,P) too large",
            __func__);
    REQUIRE(H >= 8 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", __func__, H);
    REQUIRE(cap_send >= 0, "%s: cap_send=%d must be >= 0", __func__, cap_send);
    REQUIRE((int64_t)S * cap_send * k < ((int64_t)1 << 31), "%s: S*cap_send*k must be < 2^31",
            __func__);
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(x, NT * H, 16);
    REQUIRE_ARR(topk_ids, NT * k, 4);
    REQUIRE_ARR(topk_w, NT * k, 4);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_ARR(part_offsets, (int64_t)S * (P + 1), 4);
    REQUIRE_ARR(send, (int64_t)S * cap_send * H, 16);
    REQUIRE_ARR(send_src, (int64_t)S * cap_send, 4);
    REQUIRE_ARR(send_ids, (int64_t)S * cap_send * k, 4);
    REQUIRE_ARR(send_w, (int64_t)S * cap_send * k, 4);
    REQUIRE_STATUS(dev_status);
    return cuda_status(launch_dispatch_pack(x, S, T, H, P, token_slot, part_offsets, cap_send, send,
                                            send_src, dev_status, stream, topk_ids, topk_w, k,
                                            send_ids, send_w),
                       __func__);
}

moe_status_t moe_routed_expert_stage1(const uint16_t *send, const int32_t *send_ids,
                                      const float *send_w, const int32_t *part_offsets, int S,
                                      int T, int cap_send, int k, int E, int P, int H,
                                      int recv_part, const float *scale, uint16_t *ret,
                                      uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, k, E, P);
    if (st != MOE_OK) return st;
    REQUIRE(H >= 8 && H % 8 == 0, "%s: H=%d must be a positive multiple of 8", __func__, H);
    REQUIRE(cap_send >= 0, "%s: cap_send=%d must be >= 0", __func__, cap_send);
    REQUIRE((int64_t)S * cap_send < ((int64_t)1 << 31), "%s: S*cap_send must be < 2^31", __func__);
    REQUIRE(recv_part >= -1 && recv_part < P, "%s: recv_part=%d must be in [-1, %d)", __func__,
            recv_part, P);
    const int64_t rows = (int64_t)S * cap_send;
    REQUIRE_ARR(send, rows * H, 16);
    REQUIRE_ARR(send_ids, rows * k, 4);
    REQUIRE_ARR(send_w, rows * k, 4);
    REQUIRE_ARR(part_offsets, (int64_t)S * (P + 1), 4);
    if (scale) REQUIRE_ARR(scale, E, 4);
    REQUIRE_ARR(ret, rows * H, 16);
    REQUIRE_STATUS(dev_status);
    return cuda_status(launch_routed_stage1(send, send_ids, send_w, part_offsets, S, T, cap_send, k,
                                            E, P, H, recv_part, scale, ret, dev_status, stream),
                       __func__);
}

moe_status_t moe_dispatch_pack_nvfp4(const uint16_t *x, int S, int T, int H, int P,
                                     float global_scale, const int32_t *token_slot,
                                     const int32_t *part_offsets, int cap_send, uint8_t *send_q,
                                     int32_t *send_src, uint32_t *dev_status, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    moe_status_t st = check_sizes(__func__, S, T, 1, P, P);
    if (st != MOE_OK) return st;
    REQUIRE(H >= 256 && H % 256 == 0, "%s: H=%d must be a positive multiple of 256", __func__, H);
    REQUIRE(global_scale > 0.f && global_scale < 3.0e38f, "%s: global_scale must be positive and finite",
            __func__);
    REQUIRE(cap_send >= 0, "%s: cap_send=%d must be >= 0", __func__, cap_send);
    REQUIRE((int64_t)S * cap_send < ((int64_t)1 << 31), "%s: S*cap_send must be < 2^31", __func__);
    const int64_t NT = (int64_t)S * T;
    REQUIRE_ARR(x, NT * H, 16);
    REQUIRE_ARR(token_slot, NT * P, 4);
    REQUIRE_ARR(part_offsets, (int64_t)S * (P + 1), 4);
    REQUIRE_ARR(send_q, (int64_t)S * cap_send * (H / 2 + H / 16), 16);
    REQUIRE_ARR(send_src, (int64_t)S * cap_send, 4);
    REQUIRE_STATUS(dev_status);
    return cuda_status(launch_dispatch_pack_nvfp4(x, S, T, H, P, global_scale, token_slot,
                                                  part_offsets, cap_send, send_q, send_src,
                                                  dev_status, stream),
                       __func__);
}

moe_status_t moe_expert_scale_nvfp4(const uint8_t *recv_q, const int32_t *expert_offsets,
                                    const float *scale, int E, int H, float global_scale,
                                    int cap_recv, uint16_t *y, cudaStream_t stream)
{
    MOE_CALL_RANGE();
    REQUIRE(E >= 1 && E <= kMaxE, "%s: E=%d must be in [1, %d]", __func__, E, kMaxE);
    REQUIRE(H >= 256 && H % 256 == 0, "%s: H=%d must be a positive multiple of 256", __func__, H);
    REQUIRE(global_scale > 0.f && global_scale < 3.0e38f, "%s: global_scale must be positive and finite",
            __func__);
    REQUIRE(cap_recv >= 0, "%s: cap_recv=%d must be >= 0", __func__, cap_recv);
    REQUIRE_ARR(recv_q, (int64_t)cap_recv * (H / 2 + H / 16), 16);
    REQUIRE_ARR(expert_offsets, E + 1, 4);
    REQUIRE_ARR(scale, E, 4);
    REQUIRE_ARR(y, (int64_t)cap_recv * H, 16);
    return cuda_status(launch_expert_scale_nvfp4(recv_q, expert_offsets, scale, E, H, global_scale,
                                                 cap_recv, y, stream),
                       __func__);
}

}  // extern "C"
