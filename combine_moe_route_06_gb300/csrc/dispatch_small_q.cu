// dispatch_small_q.cu -- moe_dispatch_quantized in one launch for one source
// of at most 256 tokens (a decode step): route -> layout -> pack of quantized
// records -> receiver permute.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends): section 1.4 (a
// decode step's fixed cost is launches and latency chains) and section 7.2
// (rows are converted to a low-precision format before they are sent).
// k_dispatch_small_q runs the routing and the layout (small_head.cuh), then
// the grid's warps move the records, one (token, 1,024-value segment) per task:
// the segment is quantized once (qrow.cuh) and its piece stored to the token's
// send records, then the receiving partitions' pieces are read back, up to
// eight partitions at once, and stored to their pair records.  The outputs are
// the bytes moe_route_topk, moe_dispatch_layout, the quantized pack and
// moe_permute_to_experts of the records give one after the other.
#include "common.cuh"
#include "launch.h"
#include "qrow.cuh"
#include "small_head.cuh"
#include "trace.h"

namespace moe {

namespace {

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int kSmallQBatch = 8;            // partitions whose pieces are read back together

template <int VPL, int FMT>
__global__ void __launch_bounds__(kSmallThreads) k_dispatch_small_q(
    const float *__restrict__ logits, const int4 *__restrict__ x, int T, int E, int k, int P,
    int V, int recv_part, int align, int cap_send, int cap_recv, float g,
    unsigned long long m_k, unsigned long long m_L, unsigned long long m_seg,
    int32_t *__restrict__ topk_ids, float *__restrict__ topk_w,
    int32_t *__restrict__ expert_counts, int32_t *__restrict__ expert_rank,
    int32_t *__restrict__ part_counts, int32_t *__restrict__ part_offsets,
    int32_t *__restrict__ token_slot, uint8_t *__restrict__ send_q,
    int32_t *__restrict__ send_src, uint8_t *__restrict__ recv_q,
    int32_t *__restrict__ expert_offsets, int32_t *__restrict__ pair_row,
    int32_t *__restrict__ recv_pair, uint32_t *dev_status)
{
    using QL = QLayout<FMT>;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = E / P;
    extern __shared__ __align__(16) int sm[];
    __shared__ int ptot[kMaxP], poff[kMaxP + 1];
    __shared__ int wsum[kSmallWarps];
    const SmallLayout l = small_layout(sm, T, k, E, P, ptot, poff);
    small_head<VPL>(logits, T, E, k, P, recv_part, align, 0, m_k, m_L, topk_ids, topk_w,
                    expert_counts, part_counts, part_offsets, expert_offsets, nullptr, l, wsum,
                    []() {});

    const int64_t rb = (int64_t)V * QL::kCodePerVec + V / QL::kVecPerScale;
    const float d = __fmul_rn(6.0f, g);
    const int nseg = (V + kQSegVec - 1) / kQSegVec;
    const int gw = w * (int)gridDim.x + (int)blockIdx.x, nw = (int)gridDim.x * kSmallWarps;
    bool cap_flag = false, bad_slot = false, dropped = false;
    for (int task = gw; task < T * nseg; task += nw) {
        const int t = div_by(task, nseg, m_seg), gs = task - t * nseg;
        int ts = -1, pr = -1, pp = -1, rk = -1;
        if (lane < P) ts = small_slot(l, P, t, lane);
        if (lane < k) {
            const int e = l.ids_s[t * k + lane];
            rk = small_rank(l, E, t, e);
            if (in_recv(e, E, L, recv_part)) {
                pr = l.off[e] + rk;
                if (pr >= cap_recv) {
                    dropped = true;
                    pr = -1;
                }
            }
            if (pr >= 0) pp = div_small(e, m_L);
        }
        if (gs == 0) {
            if (lane < P) {
                token_slot[t * P + lane] = ts;
                if (ts >= cap_send) cap_flag = true;
                else if (ts >= 0) send_src[ts] = t;
            }
            if (lane < k) {
                expert_rank[t * k + lane] = rk;
                pair_row[t * k + lane] = pr;
                if (pr >= 0) recv_pair[pr] = t * k + lane;
            }
        }
        // quantize the segment once (every lane takes part in the block shuffles)
        const int vb = gs * kQSegVec;
        const QPiece q = quantize_piece<FMT>(x + (int64_t)t * V, V, vb, g, d);
        unsigned smask = __ballot_sync(kFull, lane < P && ts >= 0 && ts < cap_send);
        while (smask) {
            const int p = __ffs(smask) - 1;
            smask &= smask - 1;
            const int sl = __shfl_sync(kFull, ts, p);
            store_piece<FMT>(send_q + (int64_t)sl * rb, V, vb, q);
        }
        // read back the pieces of up to kSmallQBatch receiving partitions, then
        // store each to its pairs' records
        unsigned rmask = __ballot_sync(kFull, pr >= 0);
        while (rmask) {
            QPiece r[kSmallQBatch];
            unsigned gm[kSmallQBatch];
#pragma unroll
            for (int b = 0; b < kSmallQBatch; b++) {
                gm[b] = 0u;
                r[b].code[0] = r[b].code[1] = make_uint4(0u, 0u, 0u, 0u);
                r[b].sw = 0u;
                if (rmask) {
                    const int j0 = __ffs(rmask) - 1;
                    const int p0 = __shfl_sync(kFull, pp, j0);
                    const unsigned gmask = __ballot_sync(kFull, pr >= 0 && pp == p0);
                    rmask &= ~gmask;
                    gm[b] = gmask;
                    const int sl = __shfl_sync(kFull, ts, p0);
                    const bool ok = sl >= 0 && sl < cap_send;
                    if (!ok && gs == 0 && lane == 0) {
                        if (sl < 0) bad_slot = true;
                        else cap_flag = true;
                    }
                    if (ok) r[b] = load_piece<FMT>(send_q + (int64_t)sl * rb, V, vb);
                }
            }
#pragma unroll
            for (int b = 0; b < kSmallQBatch; b++) {
                unsigned dm = gm[b];
                while (dm) {
                    const int j = __ffs(dm) - 1;
                    dm &= dm - 1;
                    const int row = __shfl_sync(kFull, pr, j);
                    store_piece<FMT>(recv_q + (int64_t)row * rb, V, vb, r[b]);
                }
            }
        }
    }

    // padding records of the receiving runs: a warp per (expert, padding row),
    // zeroed in 16-byte vectors
    if (align > 1) {
        const int rbv = (int)(rb / 16);
        const int64_t ptask = (int64_t)E * (align - 1);
        for (int64_t task = gw; task < ptask; task += nw) {
            const int e = (int)(task / (align - 1));
            const int i = (int)(task - (int64_t)e * (align - 1));
            const int row = l.off[e] + l.cnt[e] + i;
            if (!in_recv(e, E, L, recv_part) || row >= l.off[e + 1] || row >= cap_recv) continue;
            int4 *dst = reinterpret_cast<int4 *>(recv_q + (int64_t)row * rb);
            for (int vi = lane; vi < rbv; vi += 32) st_cg(dst + vi, make_int4(0, 0, 0, 0));
            if (lane == 0) recv_pair[row] = -1;
        }
    }
    // unused receive rows and send rows
    const int gtid = (int)blockIdx.x * kSmallThreads + threadIdx.x;
    const int gthreads = (int)gridDim.x * kSmallThreads;
    for (int rr = l.off[E] + gtid; rr < cap_recv; rr += gthreads) recv_pair[rr] = -1;
    for (int rr = l.poff[P] + gtid; rr < cap_send; rr += gthreads) send_src[rr] = -1;

    if (cap_flag || dropped) flag_status(dev_status, MOE_ERR_CAPACITY);
    if (bad_slot) flag_status(dev_status, MOE_ERR_INVALID_ARG);
}

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
        e = cudaFuncSetAttribute(k_dispatch_small_q<VPL, FMT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    // clusters: about kSmallTasksPerCta row tasks per CTA, at most what fits at once
    const int V = H / 8;
    const int nseg = (V + kQSegVec - 1) / kQSegVec;
    int64_t ctas = div_up((int64_t)T * nseg, kSmallTasksPerCta);
    const int resident =
        resident_grid((const void *)k_dispatch_small_q<VPL, FMT>, kSmallThreads, smem);
    const int64_t cap = (resident > 0 ? resident : di.sm_count) / kSmallCluster * kSmallCluster;
    ctas = div_up(ctas, kSmallCluster) * kSmallCluster;
    if (ctas > cap) ctas = cap;
    if (ctas < kSmallCluster) ctas = kSmallCluster;
    // multiply-high divisors: pair index / k (< 2^13), expert / L (< 2^10) always
    // fit div_small; task / nseg does while T * nseg < 2^16
    const unsigned long long m_k = div_small_magic(k), m_L = div_small_magic(E / P);
    const unsigned long long m_seg = (int64_t)T * nseg < 65536 ? div_small_magic(nseg) : 0ull;
    MOE_TRACED_LAUNCH(FMT == kQFmtMxfp8 ? "k_dispatch_small_mxfp8" : "k_dispatch_small_nvfp4", st,
                      e = launch_pdl_cluster(k_dispatch_small_q<VPL, FMT>, dim3((unsigned)ctas),
                                             dim3(kSmallThreads), smem, kSmallCluster, st, logits,
                                             (const int4 *)x, T, E, k, P, V, recv_part, align,
                                             cap_send, cap_recv, g, m_k, m_L, m_seg, topk_ids,
                                             topk_w, expert_counts, expert_rank, part_counts,
                                             part_offsets, token_slot, send_q, send_src, recv_q,
                                             expert_offsets, pair_row, recv_pair, dev_status));
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
