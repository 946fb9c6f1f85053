// layout.cu -- dispatch layout: de-duplicated per-partition copies and their
// prefix-sum layout.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 1.3 (third
// answer: one copy per GPU holding at least one of the token's experts) and
// section 3.2 (first step: per-token GPU set and per-GPU row counts).  The
// counts stay on the device (section 1.4): nothing here needs the host.
//
// Three launches, all atomic-free in the counting:
//   1. count  (one CTA per 256-token chunk): per-token partition bitmask;
//      partition counts by warp ballot + popc; expert histogram by warp match
//      groups into warp-private shared-memory rows.
//   2. scan   (one CTA per source): exclusive scan of the chunk counts per
//      partition, part_counts / part_offsets, expert_counts.
//   3. slots  (one CTA per chunk): block-wide ballot scan gives every token its
//      rank among the chunk's tokens that need partition p.
#include "common.cuh"
#include "launch.h"
#include "trace.h"

namespace moe {

namespace {

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Partition bitmask of one token; expert histogram (optional) into whist.
template <bool kHist>
__device__ __forceinline__ unsigned token_mask(const int32_t *__restrict__ ids, int64_t tok,
                                               bool valid_t, int k, int E, int L,
                                               int *whist_row, bool &bad)
{
    unsigned mask = 0;
    const int lane = threadIdx.x & 31;
    for (int j = 0; j < k; j++) {
        int e = valid_t ? __ldg(ids + tok * k + j) : -1;
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

__global__ void __launch_bounds__(kChunk) k_layout_count(const int32_t *__restrict__ ids, int T,
                                                         int k, int E, int P, int C,
                                                         int32_t *__restrict__ ws_pc,
                                                         int32_t *__restrict__ ws_ec,
                                                         uint32_t *dev_status)
{
    extern __shared__ int smem[];
    int *whist = smem;                       // [kChunkWarps][E]
    __shared__ int wpc[kChunkWarps][kMaxP];  // per-warp partition counts
    const int s = blockIdx.x / C, c = blockIdx.x % C;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = E / P;
    for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) whist[i] = 0;
    __syncthreads();

    const int t = c * kChunk + threadIdx.x;
    const bool valid_t = t < T;
    bool bad = false;
    const unsigned mask =
        token_mask<true>(ids, (int64_t)s * T + t, valid_t, k, E, L, whist + w * E, bad);
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
        ws_ec[((int64_t)s * E + e) * C + c] = sum;
    }
}

// One CTA (32 warps) per source.
__global__ void __launch_bounds__(1024) k_layout_scan(int E, int P, int C,
                                                      int32_t *__restrict__ ws_pc,
                                                      const int32_t *__restrict__ ws_ec,
                                                      int32_t *__restrict__ expert_counts,
                                                      int32_t *__restrict__ part_counts,
                                                      int32_t *__restrict__ part_offsets)
{
    __shared__ int tot[kMaxP];
    const int s = blockIdx.x;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    // warp p: exclusive scan over the chunks of partition p, in place
    for (int p = w; p < P; p += nw) {
        int32_t *row = ws_pc + ((int64_t)s * P + p) * C;
        int carry = 0;
        for (int c0 = 0; c0 < C; c0 += 32) {
            const int c = c0 + lane;
            const int v = (c < C) ? row[c] : 0;
            const int inc = warp_inclusive_scan(v);
            if (c < C) row[c] = carry + inc - v;
            carry += __shfl_sync(kFull, inc, 31);
        }
        if (lane == 0) tot[p] = carry;
    }
    // expert totals over the chunks
    for (int e = w; e < E; e += nw) {
        const int32_t *row = ws_ec + ((int64_t)s * E + e) * C;
        int sum = 0;
        for (int c = lane; c < C; c += 32) sum += row[c];
        sum = warp_sum(sum);
        if (lane == 0) expert_counts[(int64_t)s * E + e] = sum;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        part_offsets[(int64_t)s * (P + 1)] = 0;
        for (int p = 0; p < P; p++) {
            part_counts[(int64_t)s * P + p] = tot[p];
            run += tot[p];
            part_offsets[(int64_t)s * (P + 1) + p + 1] = run;
        }
    }
}

__global__ void __launch_bounds__(kChunk) k_layout_slots(const int32_t *__restrict__ ids, int T,
                                                         int k, int E, int P, int C,
                                                         const int32_t *__restrict__ ws_pc,
                                                         const int32_t *__restrict__ part_offsets,
                                                         int32_t *__restrict__ token_slot)
{
    __shared__ int wbase[kChunkWarps][kMaxP];
    const int s = blockIdx.x / C, c = blockIdx.x % C;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = E / P;
    const int t = c * kChunk + threadIdx.x;
    const bool valid_t = t < T;
    bool bad = false;
    const unsigned mask = token_mask<false>(ids, (int64_t)s * T + t, valid_t, k, E, L, nullptr, bad);
    for (int p = 0; p < P; p++) {
        const unsigned b = __ballot_sync(kFull, (mask >> p) & 1u);
        if (lane == 0) wbase[w][p] = __popc(b);
    }
    __syncthreads();
    if (threadIdx.x < P) {
        const int p = threadIdx.x;
        int run = part_offsets[(int64_t)s * (P + 1) + p] + ws_pc[((int64_t)s * P + p) * C + c];
#pragma unroll
        for (int ww = 0; ww < kChunkWarps; ww++) {
            const int v = wbase[ww][p];
            wbase[ww][p] = run;
            run += v;
        }
    }
    __syncthreads();
    const unsigned lt = lanemask_lt();
    int32_t *out = token_slot + ((int64_t)s * T + t) * P;
    for (int p = 0; p < P; p++) {
        const unsigned b = __ballot_sync(kFull, (mask >> p) & 1u);
        if (valid_t) out[p] = ((mask >> p) & 1u) ? wbase[w][p] + __popc(b & lt) : -1;
    }
}

}  // namespace

size_t layout_ws_bytes(int S, int T, int E, int P)
{
    const int64_t C = div_up(T, kChunk);
    const int64_t pc = (int64_t)S * P * C * 4, ec = (int64_t)S * E * C * 4;
    return (size_t)(div_up(pc, 256) * 256 + div_up(ec, 256) * 256);
}

cudaError_t launch_dispatch_layout(const int32_t *ids, int S, int T, int k, int E, int P,
                                   int32_t *expert_counts, int32_t *part_counts,
                                   int32_t *part_offsets, int32_t *token_slot, void *ws,
                                   uint32_t *dev_status, cudaStream_t st)
{
    const int C = (int)div_up(T, kChunk);
    const int64_t pc_bytes = div_up((int64_t)S * P * C * 4, 256) * 256;
    int32_t *ws_pc = (int32_t *)ws;
    int32_t *ws_ec = (int32_t *)((char *)ws + pc_bytes);
    const size_t hist_smem = (size_t)kChunkWarps * E * sizeof(int);
    if (C > 0) {
        if (hist_smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(k_layout_count,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)hist_smem);
            if (e != cudaSuccess) return e;
        }
        MOE_TRACED_LAUNCH("k_layout_count", st,
                          k_layout_count<<<(unsigned)(S * C), kChunk, hist_smem, st>>>(
                              ids, T, k, E, P, C, ws_pc, ws_ec, dev_status));
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    MOE_TRACED_LAUNCH("k_layout_scan", st,
                      k_layout_scan<<<(unsigned)S, 1024, 0, st>>>(E, P, C, ws_pc, ws_ec, expert_counts,
                                                                  part_counts, part_offsets));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (C > 0) {
        MOE_TRACED_LAUNCH("k_layout_slots", st,
                          k_layout_slots<<<(unsigned)(S * C), kChunk, 0, st>>>(
                              ids, T, k, E, P, C, ws_pc, part_offsets, token_slot));
        e = cudaGetLastError();
    }
    return e;
}

}  // namespace moe
