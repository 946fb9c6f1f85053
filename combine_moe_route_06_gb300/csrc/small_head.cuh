// small_head.cuh -- the routing and layout steps of the one-launch dispatch
// (one source of at most 256 tokens, a decode step), shared by the bf16 kernel
// (dispatch_small.cu) and the quantized one (dispatch_small_q.cu).
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 1.4: a
// decode step makes ~40 round trips, so their fixed cost is launches and
// latency chains, not bytes.  Thread-block clusters of 8 CTAs; the CTAs of a
// cluster route a share of the tokens each (section 1.1) and broadcast the ids
// into every CTA's shared memory (distributed shared memory, between two
// cluster barriers).  Every CTA then builds the whole layout of the batch in
// its own shared memory (one bit per token in words per expert and per
// partition: popcounts give the counts, the slots of sections 1.3 and 3.2 and
// the ranks; a scan gives the receiving experts' run starts of sections 1.5 and
// 3.3), so no CTA waits on another outside its cluster.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "route_warp.cuh"

namespace moe {

constexpr int kSmallMaxT = 256;            // tokens (at most 8 words of token bits per expert)
constexpr int kSmallThreads = 256;
constexpr int kSmallWarps = kSmallThreads / 32;
constexpr int kSmallCluster = 8;           // CTAs that share one batch's routing
constexpr int kSmallTasksPerCta = 6;       // row tasks per CTA the grids are sized for
// Static shared memory of the one-launch kernels is about 0.3 KB (partition
// totals and offsets, warp sums of the scan); the dynamic part must leave this
// much of the per-CTA limit.
constexpr size_t kSmallStaticBound = 4096;

// Dynamic shared memory of the one-launch kernels: the batch's ids, one bit
// per (token, expert) and per (token, partition) in words of 32 tokens, expert
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
__device__ __forceinline__ void cl_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
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

// The batch's layout in one CTA's shared memory.
struct SmallLayout {
    int NW;            // words of token bits
    int *ids_s;        // [T][k]
    unsigned *ebits;   // [NW][E] tokens choosing expert e
    unsigned *pbits;   // [NW][P] tokens sent to partition p
    int *cnt;          // [E] pairs of expert e
    int *off;          // [E + 1] run starts of the receiving experts
    int *ptot;         // [P] tokens sent to partition p
    int *poff;         // [P + 1] partition offsets
};

__device__ __forceinline__ SmallLayout small_layout(int *sm, int T, int k, int E, int P, int *ptot,
                                                    int *poff)
{
    SmallLayout l;
    l.NW = (T + 31) >> 5;
    l.ids_s = sm;
    l.ebits = (unsigned *)(l.ids_s + T * k);
    l.pbits = l.ebits + l.NW * E;
    l.cnt = (int *)(l.pbits + l.NW * P);
    l.off = l.cnt + E;
    l.ptot = ptot;
    l.poff = poff;
    return l;
}

// Token t's slot in partition p (lane p < P) or -1, and the rank of its pair
// with expert e among the batch's pairs of e: popcounts of the earlier tokens'
// bits.
__device__ __forceinline__ int small_slot(const SmallLayout &l, int P, int t, int p)
{
    const int tq = t >> 5;
    const unsigned tbit = 1u << (t & 31);
    const unsigned m = l.pbits[tq * P + p];
    if (!(m & tbit)) return -1;
    int ts = l.poff[p] + __popc(m & (tbit - 1u));
    for (int q = 0; q < tq; q++) ts += __popc(l.pbits[q * P + p]);
    return ts;
}
__device__ __forceinline__ int small_rank(const SmallLayout &l, int E, int t, int e)
{
    const int tq = t >> 5;
    const unsigned tbit = 1u << (t & 31);
    int rk = __popc(l.ebits[tq * E + e] & (tbit - 1u));
    for (int q = 0; q < tq; q++) rk += __popc(l.ebits[q * E + e]);
    return rk;
}

// The steps before the rows move, every thread of every CTA: the grid-dependency
// wait (after_wait() runs right after it, for loads that may start then), the
// routing of this CTA's tokens with their ids broadcast to the cluster, and the
// layout of the whole batch in this CTA's shared memory.  The first cluster
// stores ids and weights; CTA 0 stores the counts and offsets (and, with
// masked_counts, the rows in use per block of the masked layout instead of the
// run starts).  Needs E <= 1024 (four experts per thread in the scan), k, P <=
// 32.  m_k and m_L are div_small's divisors for k and E / P.
template <int VPL, class AfterWait>
__device__ __forceinline__ void small_head(
    const float *__restrict__ logits, int T, int E, int k, int P, int recv_part, int align,
    int block_rows, unsigned long long m_k, unsigned long long m_L, int32_t *__restrict__ topk_ids,
    float *__restrict__ topk_w, int32_t *__restrict__ expert_counts,
    int32_t *__restrict__ part_counts, int32_t *__restrict__ part_offsets,
    int32_t *__restrict__ expert_offsets, int32_t *__restrict__ masked_counts,
    const SmallLayout &l, int *wsum, AfterWait &&after_wait)
{
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int G = (int)cluster.num_blocks();
    const int r = (int)cluster.block_rank();
    const bool first_cluster = (int)blockIdx.x < G;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = E / P;

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
    for (int i = threadIdx.x; i < l.NW * (E + P); i += blockDim.x) l.ebits[i] = 0u;
    pdl_wait();
    pdl_trigger();
    after_wait();
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
            for (int c = 0; c < G; c++) *cluster.map_shared_rank(l.ids_s + t * k + lane, c) = id;
    }
    cl_arrive();                                // this CTA's remote writes are done
    cl_wait();                                  // every CTA holds every token's ids

    // 2. the layout of the batch.  Token t sets bit t of its experts' and its
    // partitions' words (thread per pair; the ids of a token are distinct
    // experts < E: they come from the routing above).  An expert's count is the
    // popcount of its words, a partition's likewise; the rank of a pair, or a
    // token's slot in a partition, is the popcount of the earlier tokens' bits,
    // taken by the warp that moves the token (small_slot, small_rank).
    for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
        const int t = div_small(i, m_k), e = l.ids_s[i];
        const unsigned bit = 1u << (t & 31);
        atomicOr(l.ebits + (t >> 5) * E + e, bit);
        atomicOr(l.pbits + (t >> 5) * P + div_small(e, m_L), bit);
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
            for (int q = 0; q < l.NW; q++) c += __popc(l.ebits[q * E + e]);
            l.cnt[e] = c;
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
            for (int q = 0; q < l.NW; q++) c += __popc(l.pbits[q * P + lane]);
        const int pinc = warp_inclusive_scan(c);
        if (lane < P) {
            l.ptot[lane] = c;
            l.poff[lane] = pinc - c;
        }
        if (lane == 31) l.poff[P] = pinc;
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
            if (e < E) l.off[e] = run;
            run += v[i];
        }
        if (threadIdx.x == 0) l.off[E] = used;
    }
    __syncthreads();
    // masked receive layout (masked_counts given): expert e0 + b of the receiving
    // set owns rows b * block_rows .. (b + 1) * block_rows - 1
    const bool masked = masked_counts != nullptr;
    const int e0 = recv_part < 0 ? 0 : recv_part * L, nb = recv_part < 0 ? E : L;
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e <= E; e += blockDim.x) {
            if (!masked) expert_offsets[e] = l.off[e];
            if (e < E) expert_counts[e] = l.cnt[e];
        }
        if (masked)
            for (int b = threadIdx.x; b < nb; b += blockDim.x)
                masked_counts[b] = min(l.cnt[e0 + b], block_rows);
        if ((int)threadIdx.x < P) part_counts[threadIdx.x] = l.ptot[threadIdx.x];
        if ((int)threadIdx.x <= P) part_offsets[threadIdx.x] = l.poff[threadIdx.x];
    }
}

}  // namespace moe
