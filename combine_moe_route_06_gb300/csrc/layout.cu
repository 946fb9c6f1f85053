// layout.cu -- dispatch layout: de-duplicated per-partition copies and their
// prefix-sum layout.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 1.3 (third
// answer: one copy per GPU holding at least one of the token's experts) and
// section 3.2 (first step: per-token GPU set and per-GPU row counts).  The
// counts stay on the device (section 1.4): nothing here needs the host.
//
// Two launches over 256-token chunks:
//   1. local: the chunk's ids are staged in shared memory with coalesced
//      loads.  A block-wide ballot scan gives each token its rank among the
//      chunk's tokens that need partition p; per-warp expert counts
//      (shared-memory adds) and warp match groups give each pair its rank in
//      its expert's run inside the chunk (pairs in (token, slot) order).  These
//      chunk-local values go straight into token_slot / expert_rank; the
//      chunk's counts go to the workspace.
//   2. fix: every CTA sums the counts of the chunks before its own (flat,
//      coalesced loads) and adds them, plus the partition offsets, to its
//      chunk's slots and ranks.  Chunk 0 publishes part_counts / part_offsets,
//      the last chunk expert_counts.
// All counting is order-independent integer addition and the ranks follow the
// fixed (token, slot) order, so the outputs are the same bytes on every run.
#include "common.cuh"
#include "launch.h"
#include "trace.h"

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
            atomicOr(wmask + w * E + e, 1u << lane);
            for (int j2 = 0; j2 < j; j2++) dup |= (my_ids[j2] == e);
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

}  // namespace

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
    const int64_t pc_bytes = div_up((int64_t)S * P * C * 4, 256) * 256;
    int32_t *ws_pc = (int32_t *)ws;
    int32_t *ws_ec = (int32_t *)((char *)ws + pc_bytes);
    size_t smem1 = local_smem(k, E);
    size_t smem2 = (size_t)E * sizeof(int);
    // These CTAs are few and latency-bound: when the grid fits on the device
    // with one CTA per SM, reserve enough shared memory that the block
    // scheduler cannot stack two of them on one SM.
    DeviceInfo di;
    if ((e = device_info(&di)) != cudaSuccess) return e;
    if ((int64_t)S * C <= di.sm_count) {
        const size_t one_per_sm = (size_t)di.max_smem_optin / 2 + 1024;
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
