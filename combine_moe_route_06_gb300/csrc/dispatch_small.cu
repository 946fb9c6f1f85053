// dispatch_small.cu -- moe_dispatch and moe_dispatch_masked in one launch for
// one source of at most 256 tokens (a decode step) with bf16 rows: the launcher
// of the one-launch kernel (dispatch_small.cuh) for bf16 rows, and the test
// that picks the one-launch form.
#include "dispatch_small.cuh"
#include "launch.h"
#include "trace.h"

namespace moe {

namespace {

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Whether the one-launch form runs for these sizes on the current device:
// one source of 1..256 tokens whose shared memory fits in one CTA.  (Only
// cached device attributes are queried, so the answer is the same inside a
// stream capture.)
cudaError_t use_small_form(int S, int T, int k, int E, int P, bool *out)
{
    *out = false;
    if (S != 1 || T < 1 || T > kSmallMaxT) return cudaSuccess;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    *out = small_smem(T, k, E, P) + kSmallStaticBound <= (size_t)di.max_smem_optin;
    return cudaSuccess;
}

template <int VPL>
cudaError_t launch_small(const float *logits, const uint16_t *x, int T, int H, int E, int k,
                         int P, int recv_part, int align, int cap_send, int cap_recv,
                         int32_t *topk_ids, float *topk_w, int32_t *expert_counts,
                         int32_t *expert_rank, int32_t *part_counts, int32_t *part_offsets,
                         int32_t *token_slot, uint16_t *send, int32_t *send_src, uint16_t *recv,
                         int32_t *expert_offsets, int32_t *pair_row, int32_t *recv_pair,
                         uint32_t *dev_status, int32_t *masked_counts, int block_rows,
                         cudaStream_t st)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const size_t smem = small_smem(T, k, E, P);
    // the 48 KB default covers static and dynamic shared memory together
    if (smem + kSmallStaticBound > 48 * 1024) {
        e = cudaFuncSetAttribute(k_dispatch_small<VPL, kSmallBf16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    // clusters: about kSmallTasksPerCta row tasks per CTA (six of its eight
    // warps: spreading the rows over more SMs measured faster than one task per
    // warp, 10.48 -> 10.37 us per decode layer), at most what fits at once
    const int V = H / 8;
    const int nseg = (V + kSmallSegVec - 1) / kSmallSegVec;
    int64_t ctas = div_up((int64_t)T * nseg, kSmallTasksPerCta);
    const int resident =
        resident_grid((const void *)k_dispatch_small<VPL, kSmallBf16>, kSmallThreads, smem);
    const int64_t cap = (resident > 0 ? resident : di.sm_count) / kSmallCluster * kSmallCluster;
    ctas = div_up(ctas, kSmallCluster) * kSmallCluster;
    if (ctas > cap) ctas = cap;
    if (ctas < kSmallCluster) ctas = kSmallCluster;
    // multiply-high divisors: pair index / k (< 2^13), expert / L (< 2^10) always
    // fit div_small; task / nseg does while T * nseg < 2^16
    const unsigned long long m_k = div_small_magic(k), m_L = div_small_magic(E / P);
    const unsigned long long m_seg = (int64_t)T * nseg < 65536 ? div_small_magic(nseg) : 0ull;
    MOE_TRACED_LAUNCH("k_dispatch_small", st,
                      e = launch_pdl_cluster(k_dispatch_small<VPL, kSmallBf16>, dim3((unsigned)ctas),
                                             dim3(kSmallThreads), smem, kSmallCluster, st, logits,
                                             (const int4 *)x, T, E, k, P, V, recv_part, align,
                                             cap_send, cap_recv, 0.0f, m_k, m_L, m_seg, topk_ids,
                                             topk_w, expert_counts, expert_rank, part_counts,
                                             part_offsets, token_slot, (void *)send, send_src,
                                             (void *)recv, expert_offsets, pair_row, recv_pair,
                                             dev_status, masked_counts, block_rows));
    return e;
}

}  // namespace

cudaError_t dispatch_small_form(int S, int T, int k, int E, int P, bool *out)
{
    return use_small_form(S, T, k, E, P, out);
}

cudaError_t launch_dispatch_small(const float *logits, const uint16_t *x, int T, int H, int E,
                                  int k, int P, int recv_part, int align, int cap_send,
                                  int cap_recv, int32_t *topk_ids, float *topk_w,
                                  int32_t *expert_counts, int32_t *expert_rank,
                                  int32_t *part_counts, int32_t *part_offsets,
                                  int32_t *token_slot, uint16_t *send, int32_t *send_src,
                                  uint16_t *recv, int32_t *expert_offsets, int32_t *pair_row,
                                  int32_t *recv_pair, uint32_t *dev_status,
                                  int32_t *masked_counts, int block_rows, cudaStream_t st)
{
    // logits per lane of the routing warp, rounded up to an instantiated width
    const int vpl = (E + 31) / 32;
#define MOE_SMALL_CASE(VV)                                                                        \
    if (vpl <= VV)                                                                                \
        return launch_small<VV>(logits, x, T, H, E, k, P, recv_part, align, cap_send, cap_recv,   \
                                topk_ids, topk_w, expert_counts, expert_rank, part_counts,        \
                                part_offsets, token_slot, send, send_src, recv, expert_offsets,   \
                                pair_row, recv_pair, dev_status, masked_counts, block_rows, st);
    MOE_SMALL_CASE(1)
    MOE_SMALL_CASE(2)
    MOE_SMALL_CASE(4)
    MOE_SMALL_CASE(8)
    MOE_SMALL_CASE(12)
    MOE_SMALL_CASE(16)
    MOE_SMALL_CASE(24)
    MOE_SMALL_CASE(32)
#undef MOE_SMALL_CASE
    return cudaErrorInvalidValue;
}

}  // namespace moe
