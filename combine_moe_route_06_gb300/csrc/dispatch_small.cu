// dispatch_small.cu -- moe_dispatch in one launch for one source of at most
// 256 tokens (a decode step): route -> layout -> pack -> receiver permute.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 1.4: a
// decode step makes ~40 such round trips, so their fixed cost is launches and
// latency chains, not bytes.  k_dispatch_small: thread-block clusters of 8
// CTAs; the CTAs of a cluster route a share of the tokens each (section 1.1)
// and broadcast the ids into every CTA's shared memory (distributed shared
// memory, between two cluster barriers).  Every CTA then builds the whole
// layout of the batch in its own shared memory (one bit per token in words
// per expert and per partition: popcounts give the counts, the slots of
// sections 1.3 and 3.2 and the ranks; a scan gives the receiving experts' run
// starts of sections 1.5 and 3.3), so no CTA waits on another outside its
// cluster.  Finally the grid's warps move the rows, one (token, 1 KiB column
// segment) per task (row_move.cuh).  The outputs are the
// bytes moe_route_topk, moe_dispatch_layout, moe_dispatch_pack and
// moe_permute_to_experts give one after the other.
#include <cooperative_groups.h>

#include "common.cuh"
#include "launch.h"
#include "route_warp.cuh"
#include "row_move.cuh"
#include "trace.h"

namespace cg = cooperative_groups;

namespace moe {

namespace {

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int kSmallMaxT = 256;            // tokens (at most 8 words of token bits per expert)
constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallCluster = 8;           // CTAs that share one batch's routing
constexpr int kSmallU = 2;                 // int4 per lane per column segment (1 KiB)
constexpr int kSmallSegVec = 32 * kSmallU;
constexpr int kSmallBatch = 8;             // partitions whose rows are read back together
constexpr int kSmallTasksPerCta = 6;       // row tasks per CTA the grid is sized for

// Dynamic shared memory of k_dispatch_small: the batch's ids, one bit per
// (token, expert) and per (token, partition) in words of 32 tokens, expert
// counts and run starts.
inline size_t small_smem(int T, int k, int E, int P)
{
    const int nw = (T + 31) / 32;
    return (size_t)(T * k + nw * (E + P) + E + (E + 1)) * sizeof(int);
}

__device__ __forceinline__ void cl_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// An arrival that orders no memory operation (the CTA only announces that it
// has started).
__device__ __forceinline__ void cl_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

// floor(n / d) for 0 <= n < 2^16, 1 <= d < 2^16, given m = ceil(2^32 / d):
// n m / 2^32 exceeds n / d by less than n / 2^32 < 2^-16, and the fractional
// part of n / d is at most 1 - 1/d, so the floor is unchanged.
__device__ __forceinline__ int div_small(int n, unsigned long long m)
{
    return (int)(((unsigned long long)(unsigned)n * m) >> 32);
}
inline unsigned long long div_small_magic(int d)
{
    return ((1ull << 32) + (unsigned long long)d - 1) / (unsigned long long)d;
}
// n / d, by div_small where the launcher passed m (its operands fit), else by division.
__device__ __forceinline__ int div_by(int n, int d, unsigned long long m)
{
    return m ? div_small(n, m) : n / d;
}
__device__ __forceinline__ void cl_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// One launch for one source of T <= 256 tokens.  grid = clusters of
// kSmallCluster CTAs; warp w of CTA r of a cluster routes tokens r + 8w,
// r + 8w + 64, ... and writes their ids into every CTA of the cluster; the
// first cluster also stores ids and weights.  Needs E <= 1024 (four experts
// per thread in the scan), k, P <= 32.
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
    cg::cluster_group cluster = cg::this_cluster();
    const int G = (int)cluster.num_blocks();
    const int r = (int)cluster.block_rank();
    const bool first_cluster = (int)blockIdx.x < G;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = E / P;

    const int NW = (T + 31) >> 5;                                // words of token bits
    extern __shared__ __align__(16) int sm[];
    int *ids_s = sm;                                             // [T][k]
    unsigned *ebits = (unsigned *)(ids_s + T * k);               // [NW][E] tokens choosing e
    unsigned *pbits = ebits + NW * E;                            // [NW][P] tokens sent to p
    int *cnt = (int *)(pbits + NW * P);                          // [E] pairs of expert e
    int *off = cnt + E;                                          // [E + 1] run starts
    __shared__ int ptot[kMaxP], poff[kMaxP + 1];
    __shared__ int wsum[kSmallWarps];

    // Ask L2 for the logits row this warp routes first.  A prefetch returns no
    // value to the program, so it may run before the grid-dependency wait
    // whatever the previous kernel writes (L2 is coherent for every SM); when
    // the logits sit in HBM their fetch overlaps the wait.
    {
        const int tr = r + G * w;
        if (tr < T && lane * 32 < E)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(logits + (int64_t)tr * E + lane * 32));
    }
    // this CTA has started: the others may write into its shared memory once
    // every CTA has arrived here
    cl_arrive_relaxed();
    for (int i = threadIdx.x; i < NW * (E + P); i += blockDim.x) ebits[i] = 0u;
    pdl_wait();
    pdl_trigger();
    // this warp's first row task, (token, segment), is fixed by its index: load
    // its x segment now so the load overlaps the routing and the layout.  Row
    // tasks go to the CTAs round robin (warp w of CTA b starts at task
    // w * grid + b), so each SM's share of the row traffic stays small.
    const int nseg0 = (V + kSmallSegVec - 1) / kSmallSegVec;
    const int task0 = w * (int)gridDim.x + (int)blockIdx.x;
    int4 xpre[kSmallU];
#pragma unroll
    for (int u = 0; u < kSmallU; u++) {
        xpre[u] = make_int4(0, 0, 0, 0);
        if (task0 < T * nseg0) {
            const int t0 = div_by(task0, nseg0, m_seg), vi = (task0 - t0 * nseg0) * kSmallSegVec + lane + 32 * u;
            if (vi < V) xpre[u] = ld_stream(x + (int64_t)t0 * V + vi);
        }
    }

    cl_wait();                                  // every CTA of the cluster has started

    // 1. route this CTA's tokens (a warp per token) and write each token's ids
    // into every CTA of the cluster.  (The loop is kept rolled: one copy of the
    // routing code is fetched, which measured faster than unrolled copies.)
#pragma unroll 1
    for (int t = r + G * w; t < T; t += G * kSmallWarps) {
        int id;
        float wt;
        route_token_warp<VPL>(logits + (int64_t)t * E, E, k, id, wt);
        if (first_cluster && lane < k) {
            topk_ids[t * k + lane] = id;
            topk_w[t * k + lane] = wt;
        }
        if (lane < k)
            for (int c = 0; c < G; c++) *cluster.map_shared_rank(ids_s + t * k + lane, c) = id;
    }
    cl_arrive();                                // this CTA's remote writes are done
    cl_wait();                                  // every CTA holds every token's ids

    // 2. the layout of the batch.  Token t sets bit t of its experts' and its
    // partitions' words (thread per pair; the ids of a token are distinct
    // experts < E: they come from the routing above).  An expert's count is the
    // popcount of its words, a partition's likewise; the rank of a pair, or a
    // token's slot in a partition, is the popcount of the earlier tokens' bits,
    // taken below by the warp that moves the token.
    for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
        const int t = div_small(i, m_k), e = ids_s[i];
        const unsigned bit = 1u << (t & 31);
        atomicOr(ebits + (t >> 5) * E + e, bit);
        atomicOr(pbits + (t >> 5) * P + div_small(e, m_L), bit);
    }
    __syncthreads();
    // counts and padded run lengths, thread tid taking experts 4 tid .. 4 tid + 3
    // (E <= 1024), then their exclusive scan: warp scans, then the warp sums
    int v[4], local = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int e = (int)threadIdx.x * 4 + i;
        int c = 0;
        if (e < E) {
            for (int q = 0; q < NW; q++) c += __popc(ebits[q * E + e]);
            cnt[e] = c;
        }
        if (align > 1) c = (c + align - 1) / align * align;
        v[i] = (e < E && in_recv(e, E, L, recv_part)) ? c : 0;
        local += v[i];
    }
    const int inc = warp_inclusive_scan(local);
    if (lane == 31) wsum[w] = inc;
    if (w == kSmallWarps - 1) {                 // partition totals and offsets, P <= 32
        int c = 0;
        if (lane < P)
            for (int q = 0; q < NW; q++) c += __popc(pbits[q * P + lane]);
        const int pinc = warp_inclusive_scan(c);
        if (lane < P) {
            ptot[lane] = c;
            poff[lane] = pinc - c;
        }
        if (lane == 31) poff[P] = pinc;
    }
    __syncthreads();
    {
        int base = 0, used = 0;
#pragma unroll
        for (int q = 0; q < kSmallWarps; q++) {
            const int sq = wsum[q];
            base += (q < w) ? sq : 0;
            used += sq;
        }
        int run = base + inc - local;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int e = (int)threadIdx.x * 4 + i;
            if (e < E) off[e] = run;
            run += v[i];
        }
        if (threadIdx.x == 0) off[E] = used;
    }
    __syncthreads();
    // masked receive layout (masked_counts given): expert e0 + b of the receiving
    // set owns rows b * block_rows .. (b + 1) * block_rows - 1
    const bool masked = masked_counts != nullptr;
    const int e0 = recv_part < 0 ? 0 : recv_part * L, nb = recv_part < 0 ? E : L;
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e <= E; e += blockDim.x) {
            if (!masked) expert_offsets[e] = off[e];
            if (e < E) expert_counts[e] = cnt[e];
        }
        if (masked)
            for (int b = threadIdx.x; b < nb; b += blockDim.x)
                masked_counts[b] = min(cnt[e0 + b], block_rows);
        if ((int)threadIdx.x < P) part_counts[threadIdx.x] = ptot[threadIdx.x];
        if ((int)threadIdx.x <= P) part_offsets[threadIdx.x] = poff[threadIdx.x];
    }

    // 3. rows: warp task (token, 1 KiB column segment) over the whole grid
    const int gw = w * (int)gridDim.x + (int)blockIdx.x, nw = (int)gridDim.x * kSmallWarps;
    const int nseg = (V + kSmallSegVec - 1) / kSmallSegVec;
    bool cap_flag = false, bad_slot = false, dropped = false;
    for (int task = gw; task < T * nseg; task += nw) {
        const int t = div_by(task, nseg, m_seg), g = task - t * nseg;
        int ts = -1, pr = -1, pp = -1, rk = -1;
        const int tq = t >> 5;
        const unsigned tbit = 1u << (t & 31), before = tbit - 1u;
        if (lane < P) {
            const unsigned m = pbits[tq * P + lane];
            if (m & tbit) {
                ts = poff[lane] + __popc(m & before);
                for (int q = 0; q < tq; q++) ts += __popc(pbits[q * P + lane]);
            }
        }
        if (lane < k) {
            const int e = ids_s[t * k + lane];
            rk = __popc(ebits[tq * E + e] & before);
            for (int q = 0; q < tq; q++) rk += __popc(ebits[q * E + e]);
            if (in_recv(e, E, L, recv_part)) {
                if (masked) {
                    if (rk < block_rows) pr = (e - e0) * block_rows + rk;
                    else dropped = true;
                } else {
                    pr = off[e] + rk;
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
            const int row = off[e] + cnt[e] + i;
            if (!in_recv(e, E, L, recv_part) || row >= off[e + 1] || row >= cap_recv) continue;
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
            if (rr - b * block_rows >= min(cnt[e0 + b], block_rows)) recv_pair[rr] = -1;
        }
    } else {
        for (int rr = off[E] + gtid; rr < cap_recv; rr += gthreads) recv_pair[rr] = -1;
    }
    for (int rr = poff[P] + gtid; rr < cap_send; rr += gthreads) send_src[rr] = -1;

    if (cap_flag || dropped) flag_status(dev_status, MOE_ERR_CAPACITY);
    if (bad_slot) flag_status(dev_status, MOE_ERR_INVALID_ARG);
}

// Static shared memory of k_dispatch_small is about 0.3 KB (partition totals
// and offsets, warp sums of the scan); the dynamic part must leave this much
// of the per-CTA limit.
constexpr size_t kSmallStaticBound = 4096;

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
