// dispatch_small.cuh -- moe_dispatch (bf16 rows, contiguous or masked receive
// layout) and moe_dispatch_quantized (MXFP8 or NVFP4 records) in one launch for
// one source of at most 256 tokens (a decode step): route -> layout -> pack ->
// receiver permute.  The kernel template is instantiated for bf16 rows in
// dispatch_small.cu and for quantized records in dispatch_small_q.cu.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 1.4: a
// decode step makes ~40 round trips, so their fixed cost is launches and
// latency chains, not bytes; section 7.2 for the quantized records.
// Thread-block clusters of 8 CTAs; the CTAs of a cluster route a share of the
// tokens each (section 1.1) and broadcast the ids into every CTA's shared memory
// (distributed shared memory, between two cluster barriers).  Every CTA then
// builds the whole layout of the batch in its own shared memory (one bit per
// token in words per expert and per partition: popcounts give the counts, the
// slots of sections 1.3 and 3.2 and the ranks; a scan gives the receiving
// experts' run starts of sections 1.5 and 3.3), so no CTA waits on another
// outside its cluster.  Finally the grid's warps move the rows (row_move.cuh)
// or the record pieces (qrow.cuh).  The outputs are the bytes the separate
// calls give one after the other.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "qrow.cuh"
#include "route_warp.cuh"
#include "row_move.cuh"

namespace moe {

namespace {

namespace cg = cooperative_groups;

constexpr int kSmallBf16 = 0;              // FMT of bf16 rows (kQFmtMxfp8 / kQFmtNvfp4: records)
constexpr int kSmallU = 2;                 // int4 per lane per bf16 column segment (1 KiB)
constexpr int kSmallSegVec = 32 * kSmallU;
constexpr int kSmallBatch = 8;             // partitions whose rows are read back together
constexpr int kSmallQBatch = 8;            // partitions whose record pieces are read back together
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

// One launch for one source of T <= 256 tokens.  grid = clusters of
// kSmallCluster CTAs; warp w of CTA r of a cluster routes tokens r + 8w,
// r + 8w + 64, ... and writes their ids into every CTA of the cluster; the
// first cluster also stores ids and weights.  Every CTA lays out the whole
// batch, then the row tasks go to the CTAs round robin.  FMT kSmallBf16: bf16
// rows, (token, 1 KiB segment) tasks, with masked_counts the masked receive
// layout; kQFmtMxfp8 / kQFmtNvfp4: quantized records (g the NVFP4 tensor
// scale), (token, 1,024-value segment) tasks, each segment quantized once.
// Needs E <= 1024 (four experts per thread in the scan), k, P <= 32.
template <int VPL, int FMT>
__global__ void __launch_bounds__(kSmallThreads) k_dispatch_small(
    const float *__restrict__ logits, const int4 *__restrict__ x, int T, int E, int k, int P,
    int V, int recv_part, int align, int cap_send, int cap_recv, float g, unsigned long long m_k,
    unsigned long long m_L, unsigned long long m_seg, int32_t *__restrict__ topk_ids,
    float *__restrict__ topk_w, int32_t *__restrict__ expert_counts,
    int32_t *__restrict__ expert_rank, int32_t *__restrict__ part_counts,
    int32_t *__restrict__ part_offsets, int32_t *__restrict__ token_slot,
    void *__restrict__ send_v, int32_t *__restrict__ send_src, void *__restrict__ recv_v,
    int32_t *__restrict__ expert_offsets, int32_t *__restrict__ pair_row,
    int32_t *__restrict__ recv_pair, uint32_t *dev_status, int32_t *__restrict__ masked_counts,
    int block_rows)
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
    int4 xpre[kSmallU];
    if constexpr (FMT == kSmallBf16) {
        const int nseg0 = (V + kSmallSegVec - 1) / kSmallSegVec;
        const int task0 = w * (int)gridDim.x + (int)blockIdx.x;
#pragma unroll
        for (int u = 0; u < kSmallU; u++) {
            xpre[u] = make_int4(0, 0, 0, 0);
            if (task0 < T * nseg0) {
                const int t0 = div_by(task0, nseg0, m_seg);
                const int vi = (task0 - t0 * nseg0) * kSmallSegVec + lane + 32 * u;
                if (vi < V) xpre[u] = ld_stream(x + (int64_t)t0 * V + vi);
            }
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

    const int gw = w * (int)gridDim.x + (int)blockIdx.x, nw = (int)gridDim.x * kSmallWarps;
    bool cap_flag = false, bad_slot = false, dropped = false;
    if constexpr (FMT == kSmallBf16) {
        int4 *send = reinterpret_cast<int4 *>(send_v);
        int4 *recv = reinterpret_cast<int4 *>(recv_v);
        // 3. rows: warp task (token, 1 KiB column segment) over the whole grid
        const int nseg = (V + kSmallSegVec - 1) / kSmallSegVec;
        for (int task = gw; task < T * nseg; task += nw) {
            const int t = div_by(task, nseg, m_seg), gs = task - t * nseg;
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
            move_token_segment<kSmallU, kSmallBatch>(x + (int64_t)t * V, send, recv, V, gs * kSmallSegVec + lane,
                                        ts, pr, pp, P, cap_send, bad_slot, cap_flag, gs == 0,
                                        task == gw ? xpre : nullptr);
        }

        // 4. padding rows of the receiving runs: warp task (expert, row, segment)
        if (align > 1 && !masked) {
            const int64_t ptask = (int64_t)E * (align - 1) * nseg;
            for (int64_t task = gw; task < ptask; task += nw) {
                const int gs = (int)(task % nseg);
                const int64_t ei = task / nseg;
                const int e = (int)(ei / (align - 1));
                const int i = (int)(ei - (int64_t)e * (align - 1));
                const int row = off[e] + cnt[e] + i;
                if (!in_recv(e, E, L, recv_part) || row >= off[e + 1] || row >= cap_recv) continue;
                int4 *dst = recv + (int64_t)row * V;
                const int v0 = gs * kSmallSegVec + lane;
#pragma unroll
                for (int u = 0; u < kSmallU; u++) {
                    const int vi = v0 + 32 * u;
                    if (vi < V) st_cg(dst + vi, make_int4(0, 0, 0, 0));
                }
                if (gs == 0 && lane == 0) recv_pair[row] = -1;
            }
        }
    } else {
        using QL = QLayout<FMT>;
        uint8_t *send_q = reinterpret_cast<uint8_t *>(send_v);
        uint8_t *recv_q = reinterpret_cast<uint8_t *>(recv_v);
        const int64_t rb = (int64_t)V * QL::kCodePerVec + V / QL::kVecPerScale;
        const float d = __fmul_rn(6.0f, g);
        const int nseg = (V + kQSegVec - 1) / kQSegVec;
        for (int task = gw; task < T * nseg; task += nw) {
            const int t = div_by(task, nseg, m_seg), gs = task - t * nseg;
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
                    pr = off[e] + rk;
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
                const int row = off[e] + cnt[e] + i;
                if (!in_recv(e, E, L, recv_part) || row >= off[e + 1] || row >= cap_recv) continue;
                int4 *dst = reinterpret_cast<int4 *>(recv_q + (int64_t)row * rb);
                for (int vi = lane; vi < rbv; vi += 32) st_cg(dst + vi, make_int4(0, 0, 0, 0));
                if (lane == 0) recv_pair[row] = -1;
            }
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

}  // namespace

}  // namespace moe
