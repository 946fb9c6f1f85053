// dispatch_small.cu -- moe_dispatch (and moe_dispatch_masked) in one launch
// for one source of at most 256 tokens (a decode step) with bf16 rows: route
// -> layout -> pack -> receiver permute.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 1.4: a
// decode step makes ~40 such round trips, so their fixed cost is launches and
// latency chains, not bytes.  k_dispatch_small runs the routing and the layout
// (small_head.cuh), then the grid's warps move the rows, one (token, 1 KiB
// column segment) per task (row_move.cuh).  The outputs are the bytes
// moe_route_topk, moe_dispatch_layout, moe_dispatch_pack and
// moe_permute_to_experts (or moe_permute_to_experts_masked) give one after the
// other.
#include "common.cuh"
#include "launch.h"
#include "row_move.cuh"
#include "small_head.cuh"
#include "trace.h"

namespace moe {

namespace {

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int kSmallU = 2;                 // int4 per lane per column segment (1 KiB)
constexpr int kSmallSegVec = 32 * kSmallU;
constexpr int kSmallBatch = 8;             // partitions whose rows are read back together

// grid = clusters of kSmallCluster CTAs; small_head routes and lays out the
// batch, then the row tasks (token, segment) go to the CTAs round robin (warp
// w of CTA b starts at task w * grid + b), so each SM's share of the row
// traffic stays small.  With masked_counts the receive rows take the masked
// layout (pair row = block of the expert + rank, dropped past block_rows).
template <int VPL>
__global__ void __launch_bounds__(kSmallThreads) k_dispatch_small(
    const float *__restrict__ logits, const int4 *__restrict__ x, int T, int E, int k, int P,
    int V, int recv_part, int align, int cap_send, int cap_recv, unsigned long long m_k,
    unsigned long long m_L, unsigned long long m_seg, int32_t *__restrict__ topk_ids,
    float *__restrict__ topk_w, int32_t *__restrict__ expert_counts,
    int32_t *__restrict__ expert_rank, int32_t *__restrict__ part_counts,
    int32_t *__restrict__ part_offsets, int32_t *__restrict__ token_slot, int4 *__restrict__ send,
    int32_t *__restrict__ send_src, int4 *__restrict__ recv, int32_t *__restrict__ expert_offsets,
    int32_t *__restrict__ pair_row, int32_t *__restrict__ recv_pair, uint32_t *dev_status,
    int32_t *__restrict__ masked_counts, int block_rows)
{
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = E / P;
    extern __shared__ __align__(16) int sm[];
    __shared__ int ptot[kMaxP], poff[kMaxP + 1];
    __shared__ int wsum[kSmallWarps];
    const SmallLayout l = small_layout(sm, T, k, E, P, ptot, poff);
    const int gw = w * (int)gridDim.x + (int)blockIdx.x, nw = (int)gridDim.x * kSmallWarps;
    const int nseg = (V + kSmallSegVec - 1) / kSmallSegVec;
    // this warp's first row task is fixed by its index: its x segment is loaded
    // right after the grid-dependency wait, so the load overlaps the routing and
    // the layout
    int4 xpre[kSmallU];
    small_head<VPL>(logits, T, E, k, P, recv_part, align, block_rows, m_k, m_L, topk_ids, topk_w,
                    expert_counts, part_counts, part_offsets, expert_offsets, masked_counts, l,
                    wsum, [&]() {
#pragma unroll
                        for (int u = 0; u < kSmallU; u++) {
                            xpre[u] = make_int4(0, 0, 0, 0);
                            if (gw < T * nseg) {
                                const int t0 = div_by(gw, nseg, m_seg);
                                const int vi = (gw - t0 * nseg) * kSmallSegVec + lane + 32 * u;
                                if (vi < V) xpre[u] = ld_stream(x + (int64_t)t0 * V + vi);
                            }
                        }
                    });
    const bool masked = masked_counts != nullptr;
    const int e0 = recv_part < 0 ? 0 : recv_part * L, nb = recv_part < 0 ? E : L;

    // 3. rows: warp task (token, 1 KiB column segment) over the whole grid
    bool cap_flag = false, bad_slot = false, dropped = false;
    for (int task = gw; task < T * nseg; task += nw) {
        const int t = div_by(task, nseg, m_seg), g = task - t * nseg;
        int ts = -1, pr = -1, pp = -1, rk = -1;
        if (lane < P) ts = small_slot(l, P, t, lane);
        if (lane < k) {
            const int e = l.ids_s[t * k + lane];
            rk = small_rank(l, E, t, e);
            if (in_recv(e, E, L, recv_part)) {
                if (masked) {
                    if (rk < block_rows) pr = (e - e0) * block_rows + rk;
                    else dropped = true;
                } else {
                    pr = l.off[e] + rk;
                    if (pr >= cap_recv) {
                        dropped = true;
                        pr = -1;
                    }
                }
            }
            if (pr >= 0) pp = div_small(e, m_L);
        }
        if (g == 0) {
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
        move_token_segment<kSmallU, kSmallBatch>(x + (int64_t)t * V, send, recv, V, g * kSmallSegVec + lane,
                                    ts, pr, pp, P, cap_send, bad_slot, cap_flag, g == 0,
                                    task == gw ? xpre : nullptr);
    }

    // 4. padding rows of the receiving runs: warp task (expert, row, segment)
    if (align > 1 && !masked) {
        const int64_t ptask = (int64_t)E * (align - 1) * nseg;
        for (int64_t task = gw; task < ptask; task += nw) {
            const int g = (int)(task % nseg);
            const int64_t ei = task / nseg;
            const int e = (int)(ei / (align - 1));
            const int i = (int)(ei - (int64_t)e * (align - 1));
            const int row = l.off[e] + l.cnt[e] + i;
            if (!in_recv(e, E, L, recv_part) || row >= l.off[e + 1] || row >= cap_recv) continue;
            int4 *dst = recv + (int64_t)row * V;
            const int v0 = g * kSmallSegVec + lane;
#pragma unroll
            for (int u = 0; u < kSmallU; u++) {
                const int vi = v0 + 32 * u;
                if (vi < V) st_cg(dst + vi, make_int4(0, 0, 0, 0));
            }
            if (g == 0 && lane == 0) recv_pair[row] = -1;
        }
    }
    // 5. unused receive rows and send rows
    const int gtid = (int)blockIdx.x * kSmallThreads + threadIdx.x;
    const int gthreads = (int)gridDim.x * kSmallThreads;
    if (masked) {
        const int rows = nb * block_rows;
        for (int rr = gtid; rr < rows; rr += gthreads) {
            const int b = rr / block_rows;
            if (rr - b * block_rows >= min(l.cnt[e0 + b], block_rows)) recv_pair[rr] = -1;
        }
    } else {
        for (int rr = l.off[E] + gtid; rr < cap_recv; rr += gthreads) recv_pair[rr] = -1;
    }
    for (int rr = l.poff[P] + gtid; rr < cap_send; rr += gthreads) send_src[rr] = -1;

    if (cap_flag || dropped) flag_status(dev_status, MOE_ERR_CAPACITY);
    if (bad_slot) flag_status(dev_status, MOE_ERR_INVALID_ARG);
}

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
        e = cudaFuncSetAttribute(k_dispatch_small<VPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
    }
    // clusters: about kSmallTasksPerCta row tasks per CTA (six of its eight
    // warps: spreading the rows over more SMs measured faster than one task per
    // warp, 10.48 -> 10.37 us per decode layer), at most what fits at once
    const int V = H / 8;
    const int nseg = (V + kSmallSegVec - 1) / kSmallSegVec;
    int64_t ctas = div_up((int64_t)T * nseg, kSmallTasksPerCta);
    const int resident = resident_grid((const void *)k_dispatch_small<VPL>, kSmallThreads, smem);
    const int64_t cap = (resident > 0 ? resident : di.sm_count) / kSmallCluster * kSmallCluster;
    ctas = div_up(ctas, kSmallCluster) * kSmallCluster;
    if (ctas > cap) ctas = cap;
    if (ctas < kSmallCluster) ctas = kSmallCluster;
    // multiply-high divisors: pair index / k (< 2^13), expert / L (< 2^10) always
    // fit div_small; task / nseg does while T * nseg < 2^16
    const unsigned long long m_k = div_small_magic(k), m_L = div_small_magic(E / P);
    const unsigned long long m_seg = (int64_t)T * nseg < 65536 ? div_small_magic(nseg) : 0ull;
    MOE_TRACED_LAUNCH("k_dispatch_small", st,
                      e = launch_pdl_cluster(k_dispatch_small<VPL>, dim3((unsigned)ctas),
                                             dim3(kSmallThreads), smem, kSmallCluster, st, logits,
                                             (const int4 *)x, T, E, k, P, V, recv_part, align,
                                             cap_send, cap_recv, m_k, m_L, m_seg, topk_ids, topk_w,
                                             expert_counts,
                                             expert_rank, part_counts, part_offsets, token_slot,
                                             (int4 *)send, send_src, (int4 *)recv, expert_offsets,
                                             pair_row, recv_pair, dev_status, masked_counts,
                                             block_rows));
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
