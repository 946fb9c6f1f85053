// dispatch_small_q.cu -- moe_dispatch_quantized in one launch for one source
// of at most 256 tokens (a decode step): the launcher of the one-launch kernel
// (dispatch_small.cuh) for MXFP8 or NVFP4 records.
#include "dispatch_small.cuh"
#include "launch.h"
#include "trace.h"

namespace moe {

namespace {

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <int VPL, int FMT>
cudaError_t launch_small_q(const float *logits, const uint16_t *x, int T, int H, int E, int k,
                           int P, float g, int recv_part, int align, int cap_send, int cap_recv,
                           int32_t *topk_ids, float *topk_w, int32_t *expert_counts,
                           int32_t *expert_rank, int32_t *part_counts, int32_t *part_offsets,
                           int32_t *token_slot, uint8_t *send_q, int32_t *send_src,
                           uint8_t *recv_q, int32_t *expert_offsets, int32_t *pair_row,
                           int32_t *recv_pair, uint32_t *dev_status, cudaStream_t st)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const size_t smem = small_smem(T, k, E, P);
    // the 48 KB default covers static and dynamic shared memory together
    if (smem + kSmallStaticBound > 48 * 1024) {
        e = cudaFuncSetAttribute(k_dispatch_small<VPL, FMT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    // clusters: about kSmallTasksPerCta row tasks per CTA, at most what fits at once
    const int V = H / 8;
    const int nseg = (V + kQSegVec - 1) / kQSegVec;
    int64_t ctas = div_up((int64_t)T * nseg, kSmallTasksPerCta);
    const int resident =
        resident_grid((const void *)k_dispatch_small<VPL, FMT>, kSmallThreads, smem);
    const int64_t cap = (resident > 0 ? resident : di.sm_count) / kSmallCluster * kSmallCluster;
    ctas = div_up(ctas, kSmallCluster) * kSmallCluster;
    if (ctas > cap) ctas = cap;
    if (ctas < kSmallCluster) ctas = kSmallCluster;
    // multiply-high divisors: pair index / k (< 2^13), expert / L (< 2^10) always
    // fit div_small; task / nseg does while T * nseg < 2^16
    const unsigned long long m_k = div_small_magic(k), m_L = div_small_magic(E / P);
    const unsigned long long m_seg = (int64_t)T * nseg < 65536 ? div_small_magic(nseg) : 0ull;
    MOE_TRACED_LAUNCH(FMT == kQFmtMxfp8 ? "k_dispatch_small_mxfp8" : "k_dispatch_small_nvfp4", st,
                      e = launch_pdl_cluster(k_dispatch_small<VPL, FMT>, dim3((unsigned)ctas),
                                             dim3(kSmallThreads), smem, kSmallCluster, st, logits,
                                             (const int4 *)x, T, E, k, P, V, recv_part, align,
                                             cap_send, cap_recv, g, m_k, m_L, m_seg, topk_ids,
                                             topk_w, expert_counts, expert_rank, part_counts,
                                             part_offsets, token_slot, (void *)send_q, send_src,
                                             (void *)recv_q, expert_offsets, pair_row, recv_pair,
                                             dev_status, (int32_t *)nullptr, 0));
    return e;
}

}  // namespace

cudaError_t launch_dispatch_small_q(const float *logits, const uint16_t *x, int T, int H, int E,
                                    int k, int P, int format, float g, int recv_part, int align,
                                    int cap_send, int cap_recv, int32_t *topk_ids, float *topk_w,
                                    int32_t *expert_counts, int32_t *expert_rank,
                                    int32_t *part_counts, int32_t *part_offsets,
                                    int32_t *token_slot, uint8_t *send_q, int32_t *send_src,
                                    uint8_t *recv_q, int32_t *expert_offsets, int32_t *pair_row,
                                    int32_t *recv_pair, uint32_t *dev_status, cudaStream_t st)
{
    // logits per lane of the routing warp, rounded up to an instantiated width
    const int vpl = (E + 31) / 32;
#define MOE_SMALL_Q_CASE(VV)                                                                      \
    if (vpl <= VV) {                                                                              \
        if (format == kQFmtMxfp8)                                                                 \
            return launch_small_q<VV, kQFmtMxfp8>(logits, x, T, H, E, k, P, g, recv_part, align,  \
                                                  cap_send, cap_recv, topk_ids, topk_w,           \
                                                  expert_counts, expert_rank, part_counts,        \
                                                  part_offsets, token_slot, send_q, send_src,     \
                                                  recv_q, expert_offsets, pair_row, recv_pair,    \
                                                  dev_status, st);                                \
        return launch_small_q<VV, kQFmtNvfp4>(logits, x, T, H, E, k, P, g, recv_part, align,      \
                                              cap_send, cap_recv, topk_ids, topk_w,               \
                                              expert_counts, expert_rank, part_counts,            \
                                              part_offsets, token_slot, send_q, send_src, recv_q, \
                                              expert_offsets, pair_row, recv_pair, dev_status,    \
                                              st);                                                \
    }
    MOE_SMALL_Q_CASE(1)
    MOE_SMALL_Q_CASE(2)
    MOE_SMALL_Q_CASE(4)
    MOE_SMALL_Q_CASE(8)
    MOE_SMALL_Q_CASE(12)
    MOE_SMALL_Q_CASE(16)
    MOE_SMALL_Q_CASE(24)
    MOE_SMALL_Q_CASE(32)
#undef MOE_SMALL_Q_CASE
    return cudaErrorInvalidValue;
}

}  // namespace moe
