// layout.cu -- dispatch layout: de-duplicated per-partition copies and their
// prefix-sum layout.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 1.3 (third
// answer: one copy per GPU holding at least one of the token's experts) and
// section 3.2 (first step: per-token GPU set and per-GPU row counts).  The
// counts stay on the device (section 1.4): nothing here needs the host.
//
// Two launches over 256-token chunks, both atomic-free in the counting:
//   1. count: the chunk's ids are staged in shared memory with coalesced
//      loads; per-token partition bitmask; partition counts by warp ballot +
//      popc; expert histogram by warp match groups into warp-private
//      shared-memory rows.  Per-chunk counts go to the workspace.
//   2. rank: every CTA reduces the per-chunk counts of its source itself
//      (partition totals -> part_offsets, partition and expert prefixes before
//      its chunk; the last chunk's CTA publishes the expert totals).  A
//      block-wide ballot scan gives each token its slot in every partition it
//      needs, and warp match groups give each pair its rank in its expert's
//      run (pairs in (token, slot) order).
#include "common.cuh"
#include "launch.h"
#include "trace.h"

namespace moe {

namespace {

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Stage the ids of tokens [t0, t0 + n) of source s into shared memory
// (coalesced: consecutive threads read consecutive ids).
__device__ __forceinline__ void stage_ids(const int32_t *__restrict__ ids, int64_t first_token,
                                          int n, int k, int *ids_s)
{
    const int64_t base = first_token * k;
    const int cnt = n * k;
    for (int i = threadIdx.x; i < cnt; i += blockDim.x) ids_s[i] = __ldg(ids + base + i);
}

// Partition bitmask of this thread's token (k ids in shared memory);
// optionally adds its experts to the warp's private histogram row.
template <bool kHist>
__device__ __forceinline__ unsigned token_mask(const int *ids_t, bool valid_t, int k, int E, int L,
                                               int *whist_row, bool &bad)
{
    unsigned mask = 0;
    const int lane = threadIdx.x & 31;
    for (int j = 0; j < k; j++) {
        const int e = valid_t ? ids_t[j] : -1;
        const bool ok = (e >= 0) && (e < E);
        if (e >= E) bad = true;
        if (ok) mask |= 1u << (e / L);
        if (kHist) {
            const unsigned grp = __match_any_sync(kFull, ok ? e : -1);
            if (ok && lane == __ffs(grp) - 1) whist_row[e] += __popc(grp);
            __syncwarp();
        }
    }
    return mask;
}

// Shared memory of the count kernel: staged ids, then warp histograms.
inline size_t count_smem(int k, int E)
{
    return (size_t)(kChunk * k + kChunkWarps * E) * sizeof(int);
}

__global__ void __launch_bounds__(kChunk) k_layout_count(const int32_t *__restrict__ ids, int T,
                                                         int k, int E, int P, int C,
                                                         int32_t *__restrict__ ws_pc,
                                                         int32_t *__restrict__ ws_ec,
                                                         uint32_t *dev_status)
{
    extern __shared__ int smem[];
    int *ids_s = smem;                        // [kChunk * k]
    int *whist = smem + kChunk * k;           // [kChunkWarps][E]
    __shared__ int wpc[kChunkWarps][kMaxP];   // per-warp partition counts
    const int s = blockIdx.x / C, c = blockIdx.x % C;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = E / P;
    const int t0 = c * kChunk;
    const int n = min(kChunk, T - t0);
    for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) whist[i] = 0;
    pdl_wait();
    pdl_trigger();
    stage_ids(ids, (int64_t)s * T + t0, n, k, ids_s);
    __syncthreads();

    bool bad = false;
    const bool valid_t = threadIdx.x < n;
    const unsigned mask =
        token_mask<true>(ids_s + threadIdx.x * k, valid_t, k, E, L, whist + w * E, bad);
    for (int p = 0; p < P; p++) {
        const unsigned b = __ballot_sync(kFull, (mask >> p) & 1u);
        if (lane == 0) wpc[w][p] = __popc(b);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(dev_status, MOE_ERR_BAD_EXPERT_ID);
    if (threadIdx.x < P) {
        int sum = 0;
#pragma unroll
        for (int ww = 0; ww < kChunkWarps; ww++) sum += wpc[ww][threadIdx.x];
        ws_pc[((int64_t)s * P + threadIdx.x) * C + c] = sum;
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int sum = 0;
#pragma unroll
        for (int ww = 0; ww < kChunkWarps; ww++) sum += whist[ww * E + e];
        ws_ec[((int64_t)s * C + c) * E + e] = sum;
    }
}

// Shared memory of the rank kernel: staged ids, warp histograms, expert bases.
inline size_t rank_smem(int k, int E)
{
    return (size_t)(kChunk * k + kChunkWarps * E + E) * sizeof(int);
}

__global__ void __launch_bounds__(kChunk) k_layout_rank(const int32_t *__restrict__ ids, int T,
                                                        int k, int E, int P, int C,
                                                        const int32_t *__restrict__ ws_pc,
                                                        const int32_t *__restrict__ ws_ec,
                                                        int32_t *__restrict__ expert_counts,
                                                        int32_t *__restrict__ expert_rank,
                                                        int32_t *__restrict__ part_counts,
                                                        int32_t *__restrict__ part_offsets,
                                                        int32_t *__restrict__ token_slot)
{
    extern __shared__ int sm[];
    int *ids_s = sm;                          // [kChunk * k]
    int *whist = sm + kChunk * k;             // [kChunkWarps][E]
    int *ebase = whist + kChunkWarps * E;     // [E] pairs of expert e in earlier chunks
    __shared__ int tot[kMaxP], pre[kMaxP], poff[kMaxP + 1];
    __shared__ int wbase[kChunkWarps][kMaxP];
    const int s = blockIdx.x / C, c = blockIdx.x % C;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = E / P;
    const int t0 = c * kChunk;
    const int n = min(kChunk, T - t0);
    for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) whist[i] = 0;
    pdl_wait();
    pdl_trigger();
    stage_ids(ids, (int64_t)s * T + t0, n, k, ids_s);

    // per partition: total over the source's chunks and the prefix before c
    for (int p = w; p < P; p += kChunkWarps) {
        const int32_t *row = ws_pc + ((int64_t)s * P + p) * C;
        int all = 0, before = 0;
        for (int c0 = 0; c0 < C; c0 += 32) {
            const int cc = c0 + lane;
            const int v = (cc < C) ? __ldg(row + cc) : 0;
            all += v;
            before += (cc < c) ? v : 0;
        }
        all = warp_sum(all);
        before = warp_sum(before);
        if (lane == 0) {
            tot[p] = all;
            pre[p] = before;
        }
    }
    // per expert: pairs in the chunks before c (and the total, in the last chunk)
    const int32_t *ec = ws_ec + (int64_t)s * C * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int before = 0;
#pragma unroll 8
        for (int cc = 0; cc < c; cc++) before += __ldg(ec + (int64_t)cc * E + e);
        ebase[e] = before;
        if (c == C - 1) expert_counts[(int64_t)s * E + e] = before + __ldg(ec + (int64_t)c * E + e);
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

    // ---- expert ranks: pass A (warp totals per expert) -------------------
    const int *wids = ids_s + w * 32 * k;      // the warp's 32 tokens, (token, slot) order
    const int wpairs = max(0, min(32, n - w * 32)) * k;
    for (int it = 0; it < k; it++) {
        const int qi = it * 32 + lane;
        const int e = (qi < wpairs) ? wids[qi] : -1;
        const bool ok = e >= 0 && e < E;
        const unsigned grp = __match_any_sync(kFull, ok ? e : -1);
        if (ok && lane == __ffs(grp) - 1) whist[w * E + e] += __popc(grp);
        __syncwarp();
    }
    __syncthreads();
    if (c == 0) {
        if (threadIdx.x < P) part_counts[(int64_t)s * P + threadIdx.x] = tot[threadIdx.x];
        if (threadIdx.x <= P) part_offsets[(int64_t)s * (P + 1) + threadIdx.x] = poff[threadIdx.x];
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = ebase[e];
#pragma unroll
        for (int ww = 0; ww < kChunkWarps; ww++) {
            const int v = whist[ww * E + e];
            whist[ww * E + e] = run;
            run += v;
        }
    }

    // ---- token slots: ballot scan per partition ---------------------------
    bool bad = false;
    const bool valid_t = threadIdx.x < n;
    const unsigned mask = token_mask<false>(ids_s + threadIdx.x * k, valid_t, k, E, L, nullptr, bad);
    for (int p = 0; p < P; p++) {
        const unsigned b = __ballot_sync(kFull, (mask >> p) & 1u);
        if (lane == 0) wbase[w][p] = __popc(b);
    }
    __syncthreads();
    if (threadIdx.x < P) {
        const int p = threadIdx.x;
        int run = poff[p] + pre[p];
#pragma unroll
        for (int ww = 0; ww < kChunkWarps; ww++) {
            const int v = wbase[ww][p];
            wbase[ww][p] = run;
            run += v;
        }
    }
    __syncthreads();
    const unsigned lt = lanemask_lt();
    int32_t *out = token_slot + ((int64_t)s * T + t0 + threadIdx.x) * P;
    for (int p = 0; p < P; p++) {
        const unsigned b = __ballot_sync(kFull, (mask >> p) & 1u);
        if (valid_t) out[p] = ((mask >> p) & 1u) ? wbase[w][p] + __popc(b & lt) : -1;
    }

    // ---- expert ranks: pass B (rank inside the warp's match group) --------
    int *base = whist + w * E;
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
    const size_t smem1 = count_smem(k, E);
    const size_t smem2 = rank_smem(k, E);
    if (smem1 > 48 * 1024) {
        e = cudaFuncSetAttribute(k_layout_count, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem1);
        if (e != cudaSuccess) return e;
    }
    if (smem2 > 48 * 1024) {
        e = cudaFuncSetAttribute(k_layout_rank, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem2);
        if (e != cudaSuccess) return e;
    }
    MOE_TRACED_LAUNCH("k_layout_count", st,
                      e = launch_pdl(k_layout_count, dim3((unsigned)(S * C)), dim3(kChunk), smem1,
                                     st, ids, T, k, E, P, C, ws_pc, ws_ec, dev_status));
    if (e != cudaSuccess) return e;
    MOE_TRACED_LAUNCH("k_layout_rank", st,
                      e = launch_pdl(k_layout_rank, dim3((unsigned)(S * C)), dim3(kChunk), smem2,
                                     st, ids, T, k, E, P, C, (const int32_t *)ws_pc,
                                     (const int32_t *)ws_ec, expert_counts, expert_rank,
                                     part_counts, part_offsets, token_slot));
    return e;
}

}  // namespace moe
