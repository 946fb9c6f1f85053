// layout.cu -- dispatch layout: de-duplicated per-partition copies and their
// prefix-sum layout.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 1.3 (third
// answer: one copy per GPU holding at least one of the token's experts) and
// section 3.2 (first step: per-token GPU set and per-GPU row counts).  The
// counts stay on the device (section 1.4): nothing here needs the host.
//
// The work is cut into 256-token chunks, one CTA each.  Every form does the
// same chunk step: the chunk's ids are staged in shared memory with coalesced
// loads; a block-wide ballot scan gives each token its rank among the chunk's
// tokens that need partition p; per-warp expert counts and lane masks
// (shared-memory adds and ORs) and, when a token repeats an expert, warp match
// groups give each pair its rank in its expert's run inside the chunk (pairs
// in (token, slot) order).  The forms differ in how the chunks learn the
// counts of the chunks before them:
//   - one chunk per source (a decode step): nothing to learn; k_layout_local
//     adds the partition offsets and stores final values;
//   - 2 to 16 chunks per source: one thread-block cluster per source
//     (k_layout_cluster).  The chunks exchange their counts through
//     distributed shared memory between two cluster barriers and store final
//     values: one launch, no counts through global memory.  A source of up to
//     16 chunks of 1,024 tokens takes the same kernel with 1,024-token chunks
//     (and threads) where their shared memory fits;
//   - more chunks: k_layout_local stores chunk-local values and the chunk's
//     counts in the workspace; k_layout_fix sums the earlier chunks' counts
//     and adds them.
// Chunk 0 publishes part_counts / part_offsets; expert_counts come from the
// last chunk (or, in a cluster, from the CTA that scans each expert).
// All counting is order-independent integer addition and the ranks follow the
// fixed (token, slot) order, so the outputs are the same bytes on every run.
#include <cooperative_groups.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "trace.h"

namespace cg = cooperative_groups;

namespace moe {

namespace {

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int kBatch = 8;  // global loads issued together before they are used

// dst[i] = src[i] for i < cnt: every thread issues kBatch loads before its
// first store, so the loads' latencies overlap.
__device__ __forceinline__ void stage_batched(const int32_t *__restrict__ src, int cnt, int *dst)
{
    for (int i0 = threadIdx.x; i0 < cnt; i0 += kBatch * blockDim.x) {
        int v[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; b++) {
            const int i = i0 + b * blockDim.x;
            v[b] = (i < cnt) ? __ldg(src + i) : 0;
        }
#pragma unroll
        for (int b = 0; b < kBatch; b++) {
            const int i = i0 + b * blockDim.x;
            if (i < cnt) dst[i] = v[b];
        }
    }
}

// Shared memory of the local kernel: staged ids, warp histograms, warp lane
// masks per expert, the partition of every expert.
inline size_t local_smem(int k, int E)
{
    return (size_t)(kChunk * k + 2 * kChunkWarps * E + E) * sizeof(int);
}

// Chunk-local layout of 256 tokens.  Writes chunk-local slots (rank among the
// chunk's tokens that need partition p) and chunk-local expert ranks into the
// outputs, and the chunk's partition and expert counts into the workspace.
// With one chunk per source (C == 1, e.g. a decode step) the chunk-local values
// are already final: the kernel then adds the partition offsets itself and
// publishes the counts, and no fix-up kernel runs.
__global__ void __launch_bounds__(kChunk) k_layout_local(const int32_t *__restrict__ ids, int T,
                                                         int k, int E, int P, int C,
                                                         int32_t *__restrict__ ws_pc,
                                                         int32_t *__restrict__ ws_ec,
                                                         int32_t *__restrict__ expert_rank,
                                                         int32_t *__restrict__ token_slot,
                                                         int32_t *__restrict__ expert_counts,
                                                         int32_t *__restrict__ part_counts,
                                                         int32_t *__restrict__ part_offsets,
                                                         uint32_t *dev_status)
{
    const bool single = (C == 1);
    extern __shared__ int sm[];
    int *ids_s = sm;                          // [kChunk * k] the chunk's ids, (token, slot) order
    int *whist = sm + kChunk * k;             // [kChunkWarps][E] per-warp expert counts
    unsigned *wmask = (unsigned *)(whist + kChunkWarps * E);  // [kChunkWarps][E] lanes with e
    int *part_s = (int *)(wmask + kChunkWarps * E);           // [E] partition of each expert
    __shared__ int wpart[kChunkWarps][kMaxP]; // per-warp partition counts, then bases
    __shared__ int ptot[kMaxP], poff[kMaxP + 1];
    const int s = blockIdx.x / C, c = blockIdx.x % C;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = E / P;
    const int t0 = c * kChunk;
    const int n = min(kChunk, T - t0);
    for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) {
        whist[i] = 0;
        wmask[i] = 0u;
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) part_s[e] = e / L;
    pdl_wait();
    pdl_trigger();
    stage_batched(ids + ((int64_t)s * T + t0) * k, n * k, ids_s);
    __syncthreads();

    // partition bitmask of this thread's token
    const bool valid_t = threadIdx.x < n;
    unsigned mask = 0;
    bool bad = false;
    if (valid_t) {
        const int *it_ids = ids_s + threadIdx.x * k;
        for (int j = 0; j < k; j++) {
            const int e = it_ids[j];
            if (e >= E) bad = true;
            if (e >= 0 && e < E) mask |= 1u << part_s[e];
        }
    }
    for (int p = 0; p < P; p++) {
        const unsigned b = __ballot_sync(kFull, (mask >> p) & 1u);
        if (lane == 0) wpart[w][p] = __popc(b);
    }
    // per-warp expert counts and the set of the warp's lanes (tokens) that
    // route to each expert.  Counting and OR-ing are order-free, so shared-
    // memory atomics keep the result exact and deterministic.
    const int *my_ids = ids_s + threadIdx.x * k;
    bool dup = false;                          // a token that lists one expert twice
    if (valid_t) {
        for (int j = 0; j < k; j++) {
            const int e = my_ids[j];
            if (e < 0 || e >= E) continue;
            atomicAdd(whist + w * E + e, 1);
            // only this lane sets its bit: set already means e came up before
            dup |= (atomicOr(wmask + w * E + e, 1u << lane) >> lane) & 1u;
        }
    }
    const bool any_dup = __syncthreads_or(dup);
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(dev_status, MOE_ERR_BAD_EXPERT_ID);

    // warp bases inside the chunk; chunk totals to the workspace
    if (threadIdx.x < P) {
        const int p = threadIdx.x;
        int run = 0;
#pragma unroll
        for (int ww = 0; ww < kChunkWarps; ww++) {
            const int v = wpart[ww][p];
            wpart[ww][p] = run;
            run += v;
        }
        ws_pc[((int64_t)s * P + p) * C + c] = run;
        ptot[p] = run;
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int ww = 0; ww < kChunkWarps; ww++) {
            const int v = whist[ww * E + e];
            whist[ww * E + e] = run;
            run += v;
        }
        ws_ec[((int64_t)s * C + c) * E + e] = run;
        if (single) expert_counts[(int64_t)s * E + e] = run;
    }
    __syncthreads();
    if (single) {
        if (threadIdx.x == 0) {
            int run = 0;
            for (int p = 0; p < P; p++) {
                poff[p] = run;
                run += ptot[p];
            }
            poff[P] = run;
        }
        __syncthreads();
        if (threadIdx.x < P) part_counts[(int64_t)s * P + threadIdx.x] = ptot[threadIdx.x];
        if (threadIdx.x <= P) part_offsets[(int64_t)s * (P + 1) + threadIdx.x] = poff[threadIdx.x];
    }

    // chunk-local slots
    const unsigned lt = lanemask_lt();
    int32_t *slot = token_slot + ((int64_t)s * T + t0 + threadIdx.x) * P;
    for (int p = 0; p < P; p++) {
        const unsigned b = __ballot_sync(kFull, (mask >> p) & 1u);
        if (valid_t)
            slot[p] = ((mask >> p) & 1u) ? (single ? poff[p] : 0) + wpart[w][p] + __popc(b & lt) : -1;
    }

    // chunk-local expert ranks, pairs in (token, slot) order: warp base +
    // earlier lanes of the warp with the same expert (each lists it once when no
    // token repeats an expert) + earlier slots of the same token
    int *base = whist + w * E;
    if (!any_dup) {
        if (valid_t) {
            int32_t *rk_t = expert_rank + ((int64_t)s * T + t0 + threadIdx.x) * k;
            for (int j = 0; j < k; j++) {
                const int e = my_ids[j];
                int r = -1;
                if (e >= 0 && e < E) r = base[e] + __popc(wmask[w * E + e] & lt);
                rk_t[j] = r;
            }
        }
        return;
    }
    // a token lists an expert twice: rank inside the warp's match groups instead
    const int *wids = ids_s + w * 32 * k;      // the warp's 32 tokens
    const int wpairs = max(0, min(32, n - w * 32)) * k;
    int32_t *rk = expert_rank + ((int64_t)s * T + t0 + w * 32) * k;
    for (int it = 0; it < k; it++) {
        const int qi = it * 32 + lane;
        const int e = (qi < wpairs) ? wids[qi] : -1;
        const bool ok = e >= 0 && e < E;
        const unsigned grp = __match_any_sync(kFull, ok ? e : -1);
        const int r = ok ? base[e] + __popc(grp & lt) : -1;
        __syncwarp();
        if (ok && lane == __ffs(grp) - 1) base[e] += __popc(grp);
        __syncwarp();
        if (qi < wpairs) rk[qi] = r;
    }
}

// Adds the chunk's global bases to the chunk-local slots and ranks; publishes
// part_counts / part_offsets (chunk 0) and expert_counts (last chunk).
__global__ void __launch_bounds__(kChunk) k_layout_fix(const int32_t *__restrict__ ids, int T,
                                                       int k, int E, int P, int C,
                                                       const int32_t *__restrict__ ws_pc,
                                                       const int32_t *__restrict__ ws_ec,
                                                       int32_t *__restrict__ expert_counts,
                                                       int32_t *__restrict__ expert_rank,
                                                       int32_t *__restrict__ part_counts,
                                                       int32_t *__restrict__ part_offsets,
                                                       int32_t *__restrict__ token_slot)
{
    extern __shared__ int ebase[];            // [E] pairs of expert e in chunks before c
    __shared__ int tot[kMaxP], pre[kMaxP], poff[kMaxP + 1];
    const int s = blockIdx.x / C, c = blockIdx.x % C;
    const int t0 = c * kChunk;
    const int n = min(kChunk, T - t0);
    const bool last = (c == C - 1);   // the last chunk also publishes expert totals
    pdl_wait();
    pdl_trigger();

    // sums over chunks (every load of a thread issued before its adds)
    const int32_t *pc = ws_pc + (int64_t)s * P * C;
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        int all = 0, before = 0;
        for (int c0 = 0; c0 < C; c0 += kBatch) {
            int v[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; b++) v[b] = (c0 + b < C) ? __ldg(pc + p * C + c0 + b) : 0;
#pragma unroll
            for (int b = 0; b < kBatch; b++) {
                all += v[b];
                before += (c0 + b < c) ? v[b] : 0;
            }
        }
        tot[p] = all;
        pre[p] = before;
    }
    const int32_t *ec = ws_ec + (int64_t)s * C * E;
    const int nc = last ? c + 1 : c;          // the last chunk also adds its own counts
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int before = 0, mine = 0;
        for (int c0 = 0; c0 < nc; c0 += kBatch) {
            int v[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; b++)
                v[b] = (c0 + b < nc) ? __ldg(ec + (int64_t)(c0 + b) * E + e) : 0;
#pragma unroll
            for (int b = 0; b < kBatch; b++) {
                if (c0 + b < c) before += v[b];
                else if (c0 + b == c) mine = v[b];
            }
        }
        ebase[e] = before;
        if (last) expert_counts[(int64_t)s * E + e] = before + mine;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int p = 0; p < P; p++) {
            poff[p] = run;
            run += tot[p];
        }
        poff[P] = run;
    }
    __syncthreads();
    if (c == 0) {
        if (threadIdx.x < P) part_counts[(int64_t)s * P + threadIdx.x] = tot[threadIdx.x];
        if (threadIdx.x <= P) part_offsets[(int64_t)s * (P + 1) + threadIdx.x] = poff[threadIdx.x];
    }

    // elementwise fix-up of the chunk's slots and ranks (coalesced; each thread
    // loads kBatch values before it stores any)
    int32_t *slot = token_slot + ((int64_t)s * T + t0) * P;
    for (int i0 = threadIdx.x; i0 < n * P; i0 += kBatch * blockDim.x) {
        int v[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; b++) {
            const int i = i0 + b * blockDim.x;
            v[b] = (i < n * P) ? slot[i] : -1;
        }
#pragma unroll
        for (int b = 0; b < kBatch; b++) {
            const int i = i0 + b * blockDim.x;
            if (v[b] >= 0) slot[i] = v[b] + poff[i % P] + pre[i % P];
        }
    }
    const int32_t *cid = ids + ((int64_t)s * T + t0) * k;
    int32_t *rk = expert_rank + ((int64_t)s * T + t0) * k;
    for (int i0 = threadIdx.x; i0 < n * k; i0 += kBatch * blockDim.x) {
        int r[kBatch], e[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; b++) {
            const int i = i0 + b * blockDim.x;
            r[b] = (i < n * k) ? rk[i] : -1;
            e[b] = (i < n * k) ? __ldg(cid + i) : 0;
        }
#pragma unroll
        for (int b = 0; b < kBatch; b++) {
            const int i = i0 + b * blockDim.x;
            if (r[b] >= 0) rk[i] = r[b] + ebase[e[b]];
        }
    }
}

// Counts and offsets of an empty batch (T == 0).
__global__ void k_layout_empty(int S, int E, int P, int32_t *__restrict__ expert_counts,
                               int32_t *__restrict__ part_counts,
                               int32_t *__restrict__ part_offsets)
{
    pdl_wait();
    for (int i = threadIdx.x; i < S * E; i += blockDim.x) expert_counts[i] = 0;
    for (int i = threadIdx.x; i < S * P; i += blockDim.x) part_counts[i] = 0;
    for (int i = threadIdx.x; i < S * (P + 1); i += blockDim.x) part_offsets[i] = 0;
}

// ---------------------------------------------------------------- cluster form
//
// One thread-block cluster per source, one CTA per 256-token chunk (up to
// kMaxCluster chunks).  Each CTA lays out its chunk in shared memory counted
// from the chunk's start.  After the cluster barrier, CTA j scans a slice of
// the experts across the cluster (reading every CTA's chunk counts through
// distributed shared memory) and writes each CTA's earlier-chunk counts into
// that CTA's shared memory; after a second barrier every CTA adds them and the
// partition offsets and stores final slots and ranks, coalesced.  Clusters are
// scheduled as a whole, so the barriers need no time limit, and no counts go
// through global memory.

constexpr int kMaxCluster = 16;
constexpr int kChunkWide = 1024;  // tokens (and threads) per CTA of the wide cluster form

// Dynamic shared memory of k_layout_cluster<CHUNK>: ids (16-byte aligned,
// offset 0), slots, ranks, warp histograms and lane masks, the partition of
// each expert, this chunk's and the earlier chunks' expert counts.
template <int CHUNK>
inline size_t cluster_smem(int k, int E, int P)
{
    const size_t ids_pad = ((size_t)CHUNK * k + 3) / 4 * 4;
    return (ids_pad + (size_t)CHUNK * ((P | 1) + (k | 1)) + 2 * (CHUNK / 32) * E + 3 * E) *
           sizeof(int);
}

// Split cluster barrier: arrive (release: this thread's earlier writes) when
// the data the other CTAs need is ready, wait (acquire) before reading theirs;
// work in between overlaps the barrier.
__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

template <int CHUNK>
__global__ void __launch_bounds__(CHUNK) k_layout_cluster(const int32_t *__restrict__ ids, int T,
                                                           int k, int E, int P, int G,
                                                           int32_t *__restrict__ expert_counts,
                                                           int32_t *__restrict__ expert_rank,
                                                           int32_t *__restrict__ part_counts,
                                                           int32_t *__restrict__ part_offsets,
                                                           int32_t *__restrict__ token_slot,
                                                           uint32_t *dev_status)
{
    cg::cluster_group cluster = cg::this_cluster();
    const int j = (int)cluster.block_rank();         // chunk of the source
    const int s = blockIdx.x / G;
    const int t0 = j * CHUNK;
    const int n = min(CHUNK, T - t0);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = E / P;
    const int sp = P | 1, sk = k | 1;                // odd row strides: no bank conflicts

    extern __shared__ __align__(16) int sm[];
    int *ids_s = sm;                                                  // [CHUNK][k]
    int *slot_s = ids_s + ((CHUNK * k + 3) & ~3);                    // [CHUNK][sp]
    int *rank_s = slot_s + CHUNK * sp;                               // [CHUNK][sk]
    int *whist = rank_s + CHUNK * sk;                                // [CHUNK / 32][E]
    unsigned *wmask = (unsigned *)(whist + (CHUNK / 32) * E);          // [CHUNK / 32][E]
    int *part_s = (int *)(wmask + (CHUNK / 32) * E);                   // [E]
    int *own_e = part_s + E;     // [E] pairs of expert e in this chunk
    int *ebase = own_e + E;      // [E] pairs of expert e in the earlier chunks (written remotely)
    __shared__ int wpart[(CHUNK / 32)][kMaxP];
    __shared__ int own_p[kMaxP];  // tokens of this chunk that need partition p
    __shared__ int tot[kMaxP], pre[kMaxP], poff[kMaxP + 1], padd[kMaxP];

    for (int i = threadIdx.x; i < (CHUNK / 32) * E; i += blockDim.x) {
        whist[i] = 0;
        wmask[i] = 0u;
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) part_s[e] = e / L;
    pdl_wait();
    pdl_trigger();

    // the chunk's ids, 16-byte loads when the source row allows
    const int32_t *src = ids + ((int64_t)s * T + t0) * k;
    const int cnt = n * k;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        const int n4 = cnt >> 2;
        const int4 *s4 = reinterpret_cast<const int4 *>(src);
        int4 *d4 = reinterpret_cast<int4 *>(ids_s);
        for (int i0 = threadIdx.x; i0 < n4; i0 += kBatch * blockDim.x) {
            int4 v[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; b++) {
                const int i = i0 + b * blockDim.x;
                if (i < n4) v[b] = __ldg(s4 + i);
            }
#pragma unroll
            for (int b = 0; b < kBatch; b++) {
                const int i = i0 + b * blockDim.x;
                if (i < n4) d4[i] = v[b];
            }
        }
        for (int i = (n4 << 2) + threadIdx.x; i < cnt; i += blockDim.x) ids_s[i] = __ldg(src + i);
    } else {
        stage_batched(src, cnt, ids_s);
    }
    __syncthreads();

    // partitions of this thread's token; per-warp expert counts and lane masks
    const bool valid_t = threadIdx.x < n;
    const int *my_ids = ids_s + threadIdx.x * k;
    unsigned mask = 0;
    bool bad = false, dup = false;                   // an id >= E; a token lists one expert twice
    if (valid_t) {
        for (int jj = 0; jj < k; jj++) {
            const int e = my_ids[jj];
            if (e >= E) bad = true;
            if (e < 0 || e >= E) continue;
            mask |= 1u << part_s[e];
            atomicAdd(whist + w * E + e, 1);
            // only this lane sets its bit: set already means e came up before
            dup |= (atomicOr(wmask + w * E + e, 1u << lane) >> lane) & 1u;
        }
    }
    for (int p = 0; p < P; p++) {
        const unsigned b = __ballot_sync(kFull, (mask >> p) & 1u);
        if (lane == 0) wpart[w][p] = __popc(b);
    }
    const bool any_dup = __syncthreads_or(dup);
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(dev_status, MOE_ERR_BAD_EXPERT_ID);

    // warp bases inside the chunk; chunk totals
    if (threadIdx.x < P) {
        const int p = threadIdx.x;
        int run = 0;
#pragma unroll
        for (int ww = 0; ww < (CHUNK / 32); ww++) {
            const int v = wpart[ww][p];
            wpart[ww][p] = run;
            run += v;
        }
        own_p[p] = run;
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int ww = 0; ww < (CHUNK / 32); ww++) {
            const int v = whist[ww * E + e];
            whist[ww * E + e] = run;
            run += v;
        }
        own_e[e] = run;
    }
    __syncthreads();
    cluster_arrive();                                // this chunk's counts are final

    // chunk-local slots and ranks into shared memory (overlaps the barrier)
    const unsigned lt = lanemask_lt();
    for (int p = 0; p < P; p++) {
        const unsigned b = __ballot_sync(kFull, (mask >> p) & 1u);
        slot_s[threadIdx.x * sp + p] = ((mask >> p) & 1u) ? wpart[w][p] + __popc(b & lt) : -1;
    }
    // ranks in (token, slot) order: warp base + earlier lanes of the warp with
    // the same expert (+ earlier slots of the same token when a token repeats
    // an expert: warp match groups then)
    int *base = whist + w * E;
    if (!any_dup) {
        for (int jj = 0; jj < k; jj++) {
            const int e = my_ids[jj];
            int r = -1;
            if (valid_t && e >= 0 && e < E) r = base[e] + __popc(wmask[w * E + e] & lt);
            rank_s[threadIdx.x * sk + jj] = r;
        }
    } else {
        const int *wids = ids_s + w * 32 * k;         // the warp's 32 tokens
        const int wpairs = max(0, min(32, n - w * 32)) * k;
        for (int it = 0; it < k; it++) {
            const int qi = it * 32 + lane;
            const int e = (qi < wpairs) ? wids[qi] : -1;
            const bool ok = e >= 0 && e < E;
            const unsigned grp = __match_any_sync(kFull, ok ? e : -1);
            const int r = ok ? base[e] + __popc(grp & lt) : -1;
            __syncwarp();
            if (ok && lane == __ffs(grp) - 1) base[e] += __popc(grp);
            __syncwarp();
            if (qi < wpairs) rank_s[(w * 32 + qi / k) * sk + (qi - (qi / k) * k)] = r;
        }
    }

    cluster_wait();                                  // every chunk's counts are final
    if (threadIdx.x < P) {                           // partition totals and earlier chunks
        const int p = threadIdx.x;
        int v[kMaxCluster];
#pragma unroll
        for (int jj = 0; jj < kMaxCluster; jj++)
            v[jj] = (jj < G) ? *cluster.map_shared_rank(own_p + p, jj) : 0;
        int all = 0, before = 0;
#pragma unroll
        for (int jj = 0; jj < kMaxCluster; jj++) {
            all += v[jj];
            before += (jj < j) ? v[jj] : 0;
        }
        tot[p] = all;
        pre[p] = before;
    }
    // this CTA's slice of the experts: exclusive scan over the chunks, each
    // prefix written into its chunk's CTA; the total is the expert's count
    const int e_lo = (int)((int64_t)j * E / G), e_hi = (int)((int64_t)(j + 1) * E / G);
    for (int e = e_lo + threadIdx.x; e < e_hi; e += blockDim.x) {
        int v[kMaxCluster];
#pragma unroll
        for (int jj = 0; jj < kMaxCluster; jj++)
            v[jj] = (jj < G) ? *cluster.map_shared_rank(own_e + e, jj) : 0;
        int run = 0;
#pragma unroll
        for (int jj = 0; jj < kMaxCluster; jj++) {
            if (jj < G) *cluster.map_shared_rank(ebase + e, jj) = run;
            run += v[jj];
        }
        expert_counts[(int64_t)s * E + e] = run;
    }
    // this CTA's remote reads and writes are done; the slots need only local
    // values, so they are stored while the other CTAs finish theirs
    cluster_arrive();
    __syncthreads();
    if (w == 0) {                                   // partition offsets: warp scan, P <= 32
        const int v = (lane < P) ? tot[lane] : 0;
        const int inc = warp_inclusive_scan(v);
        if (lane < P) {
            poff[lane] = inc - v;
            padd[lane] = inc - v + pre[lane];
        }
        if (lane == 31) poff[P] = inc;
    }
    __syncthreads();
    if (j == 0) {
        if (threadIdx.x < P) part_counts[(int64_t)s * P + threadIdx.x] = tot[threadIdx.x];
        if (threadIdx.x <= P) part_offsets[(int64_t)s * (P + 1) + threadIdx.x] = poff[threadIdx.x];
    }
    // coalesced copies out of shared memory; element i is (token i / P, slot
    // i % P), kept up to date by steps of blockDim.x instead of a division each
    int32_t *slot_g = token_slot + ((int64_t)s * T + t0) * P;
    {
        const int dt = CHUNK / P, dp = CHUNK % P;
        int t = threadIdx.x / P, p = threadIdx.x % P;
        for (int i = threadIdx.x; i < n * P; i += CHUNK) {
            const int v = slot_s[t * sp + p];
            slot_g[i] = v >= 0 ? v + padd[p] : -1;
            t += dt;
            p += dp;
            if (p >= P) {
                p -= P;
                t++;
            }
        }
    }
    // every CTA has written this CTA's ebase, and no shared memory is accessed
    // remotely after this
    cluster_wait();
    int32_t *rank_g = expert_rank + ((int64_t)s * T + t0) * k;
    {
        const int dt = CHUNK / k, dj = CHUNK % k;
        int t = threadIdx.x / k, jj = threadIdx.x % k;
        for (int i = threadIdx.x; i < n * k; i += CHUNK) {
            const int r = rank_s[t * sk + jj];
            rank_g[i] = r >= 0 ? r + ebase[ids_s[t * k + jj]] : -1;
            t += dt;
            jj += dj;
            if (jj >= k) {
                jj -= k;
                t++;
            }
        }
    }
}

// Largest cluster (16, 8, 4, 2 or 1 CTAs) of k_layout_cluster<CHUNK> that the
// current device can schedule with `smem` bytes of dynamic shared memory per
// CTA, and the most dynamic shared memory a CTA of it may have (the opt-in
// limit less the kernel's static shared memory); looked up once per device.
template <int CHUNK>
cudaError_t cluster_size_limit(size_t smem, int *out, size_t *max_dyn)
{
    static std::mutex mu;
    static int cache[64] = {};
    static size_t dyn[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        DeviceInfo di;
        if ((e = device_info(&di)) != cudaSuccess) return e;
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, k_layout_cluster<CHUNK>)) != cudaSuccess) return e;
        const size_t limit = (size_t)di.max_smem_optin - fa.sharedSizeBytes;
        if ((e = cudaFuncSetAttribute(k_layout_cluster<CHUNK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)limit)) != cudaSuccess)
            return e;
        dyn[dev] = limit;
        // clusters of 16 need the non-portable size; a device that refuses it
        // gets the portable limit of 8
        int g = kMaxCluster;
        if (cudaFuncSetAttribute(k_layout_cluster<CHUNK>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                 1) != cudaSuccess) {
            (void)cudaGetLastError();
            g = 8;
        }
        // Cached only once the occupancy query itself answered: a query that
        // errors (e.g. refused while a stream is being captured) is asked
        // again on the next call, which meanwhile takes the two-launch form.
        bool answered = false;
        for (; g > 1; g /= 2) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)g);
            cfg.blockDim = dim3(CHUNK);
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = (unsigned)g;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, k_layout_cluster<CHUNK>, &cfg) == cudaSuccess) {
                answered = true;
                if (n > 0) break;
            } else {
                (void)cudaGetLastError();      // a refused size is not an error here
            }
        }
        if (!answered) {
            *out = 1;
            *max_dyn = limit;
            return cudaSuccess;
        }
        cache[dev] = g;
    }
    *out = cache[dev];
    *max_dyn = dyn[dev];
    return cudaSuccess;
}

// The cluster form runs when a source has 2 to kMaxCluster chunks, the device
// schedules clusters of that many CTAs with one CTA per SM, and a chunk's
// shared memory fits.  Chunks are 256 tokens; a source too long for 16 of
// them takes chunks of 1,024 tokens (and threads) where 16 of those hold it
// and their shared memory fits.  *chunk is the chunk size, 0 for no cluster.
cudaError_t use_cluster_form(int T, int k, int E, int P, int *chunk)
{
    *chunk = 0;
    const int C = (int)div_up(T, kChunk);
    if (C < 2) return cudaSuccess;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const size_t one_per_sm = (size_t)di.max_smem_optin / 2 + 1024;
    int gmax = 0;
    size_t max_dyn = 0;
    if ((e = cluster_size_limit<kChunk>(one_per_sm, &gmax, &max_dyn)) != cudaSuccess) return e;
    if (C <= gmax) {
        if (cluster_smem<kChunk>(k, E, P) <= max_dyn) *chunk = kChunk;
        return cudaSuccess;
    }
    const int Cw = (int)div_up(T, kChunkWide);
    if ((e = cluster_size_limit<kChunkWide>(one_per_sm, &gmax, &max_dyn)) != cudaSuccess) return e;
    if (Cw <= gmax && cluster_smem<kChunkWide>(k, E, P) <= max_dyn) *chunk = kChunkWide;
    return cudaSuccess;
}

}  // namespace

cudaError_t layout_kernel_count(int T, int k, int E, int P, int *n)
{
    int chunk = 0;
    const cudaError_t e = use_cluster_form(T, k, E, P, &chunk);
    if (e != cudaSuccess) return e;
    *n = (T <= kChunk || chunk > 0) ? 1 : 2;
    return cudaSuccess;
}

size_t layout_ws_bytes(int S, int T, int E, int P)
{
    const int64_t C = div_up(T, kChunk);
    const int64_t pc = (int64_t)S * P * C * 4, ec = (int64_t)S * E * C * 4;
    return (size_t)(div_up(pc, 256) * 256 + div_up(ec, 256) * 256);
}

cudaError_t launch_dispatch_layout(const int32_t *ids, int S, int T, int k, int E, int P,
                                   int32_t *expert_counts, int32_t *expert_rank, int32_t *part_counts,
                                   int32_t *part_offsets, int32_t *token_slot, void *ws,
                                   uint32_t *dev_status, cudaStream_t st)
{
    cudaError_t e = cudaSuccess;
    if (T == 0) {
        MOE_TRACED_LAUNCH("k_layout_empty", st,
                          e = launch_pdl(k_layout_empty, dim3(1), dim3(256), 0, st, S, E, P,
                                         expert_counts, part_counts, part_offsets));
        return e;
    }
    const int C = (int)div_up(T, kChunk);
    DeviceInfo di;
    if ((e = device_info(&di)) != cudaSuccess) return e;
    // These CTAs are few and latency-bound: reserve enough shared memory that
    // the block scheduler gives each its own SM instead of stacking them.
    const size_t one_per_sm = (size_t)di.max_smem_optin / 2 + 1024;

    // Cluster form: one cluster per source, one CTA per chunk.
    int chunk = 0;
    if ((e = use_cluster_form(T, k, E, P, &chunk)) != cudaSuccess) return e;
    if (chunk == kChunk) {
        const size_t smc = cluster_smem<kChunk>(k, E, P);
        const size_t smem = smc > one_per_sm ? smc : one_per_sm;
        MOE_TRACED_LAUNCH("k_layout_cluster", st,
                          e = launch_pdl_cluster(k_layout_cluster<kChunk>, dim3((unsigned)(S * C)),
                                                 dim3(kChunk), smem, (unsigned)C, st, ids, T, k, E,
                                                 P, C, expert_counts, expert_rank, part_counts,
                                                 part_offsets, token_slot, dev_status));
        return e;
    }
    if (chunk == kChunkWide) {
        const int Cw = (int)div_up(T, kChunkWide);
        const size_t smc = cluster_smem<kChunkWide>(k, E, P);
        const size_t smem = smc > one_per_sm ? smc : one_per_sm;
        MOE_TRACED_LAUNCH("k_layout_cluster", st,
                          e = launch_pdl_cluster(k_layout_cluster<kChunkWide>,
                                                 dim3((unsigned)(S * Cw)), dim3(kChunkWide), smem,
                                                 (unsigned)Cw, st, ids, T, k, E, P, Cw,
                                                 expert_counts, expert_rank, part_counts,
                                                 part_offsets, token_slot, dev_status));
        return e;
    }

    // One chunk per source: the local kernel alone (its values are final).
    // More chunks per source than a cluster holds: chunk-local layout, counts
    // through the workspace, then the fix-up.
    const int64_t pc_bytes = div_up((int64_t)S * P * C * 4, 256) * 256;
    int32_t *ws_pc = (int32_t *)ws;
    int32_t *ws_ec = (int32_t *)((char *)ws + pc_bytes);
    size_t smem1 = local_smem(k, E);
    size_t smem2 = (size_t)E * sizeof(int);
    if ((int64_t)S * C <= di.sm_count) {
        if (smem1 < one_per_sm) smem1 = one_per_sm;
        if (smem2 < one_per_sm) smem2 = one_per_sm;
    }
    if (smem1 > 48 * 1024) {
        e = cudaFuncSetAttribute(k_layout_local, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem1);
        if (e != cudaSuccess) return e;
    }
    if (smem2 > 48 * 1024) {
        e = cudaFuncSetAttribute(k_layout_fix, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem2);
        if (e != cudaSuccess) return e;
    }
    MOE_TRACED_LAUNCH("k_layout_local", st,
                      e = launch_pdl(k_layout_local, dim3((unsigned)(S * C)), dim3(kChunk), smem1,
                                     st, ids, T, k, E, P, C, ws_pc, ws_ec, expert_rank,
                                     token_slot, expert_counts, part_counts, part_offsets,
                                     dev_status));
    if (e != cudaSuccess || C == 1) return e;
    MOE_TRACED_LAUNCH("k_layout_fix", st,
                      e = launch_pdl(k_layout_fix, dim3((unsigned)(S * C)), dim3(kChunk), smem2,
                                     st, ids, T, k, E, P, C, (const int32_t *)ws_pc,
                                     (const int32_t *)ws_ec, expert_counts, expert_rank,
                                     part_counts, part_offsets, token_slot));
    return e;
}

}  // namespace moe
