// permute.cu -- receiver side: rows into expert-contiguous runs.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends): section 1.5 (the
// contiguous layout; runs padded to a multiple of `align`, DeepGEMM wants 128),
// section 3.3 (one row per (token, local expert): "5 rows become 7") and
// section 5.1 (DeepEP v2's copy epilogue with do_expand and device offsets).
//
// The run order is a stable counting sort of the pairs (s, t, j) by expert id
// over the receiving partition(s).  Four launches:
//   1. count (one CTA per 256-token chunk): per-chunk expert histogram from
//      warp match groups (no atomics), written expert-major [E][G].
//   2. scan  (one warp per expert): exclusive scan over the chunks, in place;
//      expert totals.
//   3. rank  (one CTA per chunk): padded run offsets (every CTA scans the E
//      totals itself, CTA 0 publishes expert_offsets), then each pair's row =
//      run start + chunk base + earlier warps + rank inside the warp's match
//      group.  Writes pair_row and recv_pair.
//   4. copy  (grid-stride over warps): per (token, 2 KiB column segment) read
//      each received row of the token once and store it to every local pair
//      row; then zero padding rows and mark unused recv_pair entries.
#include "common.cuh"
#include "launch.h"
#include "trace.h"

namespace moe {

namespace {

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int kCopyUnroll = 4;
constexpr int kCopySegVec = 32 * kCopyUnroll;
constexpr int kCopyThreads = 256;

__device__ __forceinline__ bool in_recv(int e, int E, int L, int recv_part)
{
    return e >= 0 && e < E && (recv_part < 0 || e / L == recv_part);
}

// Warp-private histogram of the warp's pairs.  Pairs are visited in
// lexicographic (token, j) order, 32 at a time: q = it*32 + lane.
__device__ __forceinline__ void warp_pair_hist(const int32_t *__restrict__ ids, int64_t pair0,
                                               int64_t npairs, int k, int E, int L, int recv_part,
                                               int *whist_row, bool &bad)
{
    const int lane = threadIdx.x & 31;
    for (int it = 0; it < k; it++) {
        const int64_t q = pair0 + it * 32 + lane;
        const int e = (q < npairs) ? __ldg(ids + q) : -1;
        if (e >= E) bad = true;
        const bool ok = in_recv(e, E, L, recv_part);
        const unsigned grp = __match_any_sync(kFull, ok ? e : -1);
        if (ok && lane == __ffs(grp) - 1) whist_row[e] += __popc(grp);
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kChunk) k_perm_count(const int32_t *__restrict__ ids,
                                                       int64_t npairs, int k, int E, int L,
                                                       int recv_part, int G,
                                                       int32_t *__restrict__ ws_hist,
                                                       uint32_t *dev_status)
{
    extern __shared__ int whist[];  // [kChunkWarps][E]
    const int w = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) whist[i] = 0;
    __syncthreads();
    const int64_t pair0 = ((int64_t)blockIdx.x * kChunk + w * 32) * k;
    bool bad = false;
    warp_pair_hist(ids, pair0, npairs, k, E, L, recv_part, whist + w * E, bad);
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(dev_status, MOE_ERR_BAD_EXPERT_ID);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int sum = 0;
#pragma unroll
        for (int ww = 0; ww < kChunkWarps; ww++) sum += whist[ww * E + e];
        ws_hist[(int64_t)e * G + blockIdx.x] = sum;
    }
}

// One warp per expert: in-place exclusive scan of its G chunk counts.
__global__ void __launch_bounds__(256) k_perm_scan(int E, int G, int32_t *__restrict__ ws_hist,
                                                   int32_t *__restrict__ ws_tot)
{
    const int lane = threadIdx.x & 31;
    const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (e >= E) return;
    int32_t *row = ws_hist + (int64_t)e * G;
    int carry = 0;
    for (int g0 = 0; g0 < G; g0 += 32) {
        const int g = g0 + lane;
        const int v = (g < G) ? row[g] : 0;
        const int inc = warp_inclusive_scan(v);
        if (g < G) row[g] = carry + inc - v;
        carry += __shfl_sync(kFull, inc, 31);
    }
    if (lane == 0) ws_tot[e] = carry;
}

// Exclusive scan of n <= 1024 values in shared memory by a 256-thread CTA;
// returns the total.  `a` is overwritten with the exclusive prefix.
__device__ int block_exclusive_scan_1024(int *a, int n)
{
    __shared__ int wsum[8];
    __shared__ int total;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    int v[4];
    int local = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int idx = tid * 4 + i;
        v[i] = (idx < n) ? a[idx] : 0;
        local += v[i];
    }
    const int inc = warp_inclusive_scan(local);
    if (lane == 31) wsum[w] = inc;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int i = 0; i < 8; i++) {
            const int t = wsum[i];
            wsum[i] = run;
            run += t;
        }
        total = run;
    }
    __syncthreads();
    int run = wsum[w] + inc - local;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int idx = tid * 4 + i;
        if (idx < n) a[idx] = run;
        run += v[i];
    }
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(kChunk) k_perm_rank(const int32_t *__restrict__ ids,
                                                      int64_t npairs, int k, int E, int L,
                                                      int recv_part, int align, int G,
                                                      const int32_t *__restrict__ ws_base,
                                                      const int32_t *__restrict__ ws_tot,
                                                      int cap_recv,
                                                      int32_t *__restrict__ expert_offsets,
                                                      int32_t *__restrict__ pair_row,
                                                      int32_t *__restrict__ recv_pair,
                                                      uint32_t *dev_status)
{
    extern __shared__ int sm[];
    int *off = sm;                 // [E + 1] padded run starts
    int *whist = sm + (E + 1);     // [kChunkWarps][E]
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // padded run lengths -> run starts (redundantly in every CTA)
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const bool r = (recv_part < 0) || (e / L == recv_part);
        const int c = __ldg(ws_tot + e);
        off[e] = r ? (c + align - 1) / align * align : 0;
    }
    for (int i = threadIdx.x; i < kChunkWarps * E; i += blockDim.x) whist[i] = 0;
    __syncthreads();
    const int total = block_exclusive_scan_1024(off, E);
    if (threadIdx.x == 0) off[E] = total;
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e <= E; e += blockDim.x) expert_offsets[e] = off[e];
    }
    if (npairs == 0) return;

    // pass A: warp totals per expert
    const int64_t pair0 = ((int64_t)blockIdx.x * kChunk + w * 32) * k;
    bool bad = false;
    warp_pair_hist(ids, pair0, npairs, k, E, L, recv_part, whist + w * E, bad);
    __syncthreads();
    // warp bases: run start + chunk base + earlier warps of this chunk
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = off[e] + __ldg(ws_base + (int64_t)e * G + blockIdx.x);
#pragma unroll
        for (int ww = 0; ww < kChunkWarps; ww++) {
            const int v = whist[ww * E + e];
            whist[ww * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    // pass B: ranks inside the warp, in (token, j) order
    int *base = whist + w * E;
    const unsigned lt = lanemask_lt();
    bool dropped = false;
    for (int it = 0; it < k; it++) {
        const int64_t q = pair0 + it * 32 + lane;
        const int e = (q < npairs) ? __ldg(ids + q) : -1;
        const bool ok = in_recv(e, E, L, recv_part);
        const unsigned grp = __match_any_sync(kFull, ok ? e : -1);
        int row = -1;
        if (ok) row = base[e] + __popc(grp & lt);
        __syncwarp();
        if (ok && lane == __ffs(grp) - 1) base[e] += __popc(grp);
        __syncwarp();
        if (q < npairs) {
            if (ok && row < cap_recv) {
                pair_row[q] = row;
                recv_pair[row] = (int32_t)q;
            } else {
                pair_row[q] = -1;
                if (ok) dropped = true;
            }
        }
    }
    (void)bad;  // flagged by the count kernel
    if (__syncthreads_or(dropped) && threadIdx.x == 0) flag_status(dev_status, MOE_ERR_CAPACITY);
}

__global__ void __launch_bounds__(kCopyThreads) k_perm_copy(
    const int4 *__restrict__ send, const int32_t *__restrict__ token_slot,
    const int32_t *__restrict__ ids, const int32_t *__restrict__ pair_row, int64_t NT, int k,
    int E, int L, int P, int T, int V, int recv_part, int align, int cap_send, int cap_recv,
    const int32_t *__restrict__ expert_offsets, const int32_t *__restrict__ ws_tot,
    int4 *__restrict__ recv, int32_t *__restrict__ recv_pair, uint32_t *dev_status)
{
    const int lane = threadIdx.x & 31;
    const int64_t gthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t gwarps = gthreads >> 5;
    const int nseg = (V + kCopySegVec - 1) / kCopySegVec;
    bool cap_flag = false, bad_slot = false;

    // 1. pair rows, one warp per (token, column segment)
    const int64_t ntask = NT * nseg;
    for (int64_t task = gtid >> 5; task < ntask; task += gwarps) {
        const int64_t n = task / nseg;
        const int g = (int)(task - n * nseg);
        int pr = -1, p = -1;
        if (lane < k) {
            pr = __ldg(pair_row + n * k + lane);
            if (pr >= 0) p = __ldg(ids + n * k + lane) / L;
        }
        unsigned vmask = __ballot_sync(kFull, pr >= 0);
        const int s = (int)(n / T);
        const int v0 = g * kCopySegVec + lane;
        while (vmask) {
            const int j0 = __ffs(vmask) - 1;
            const int p0 = __shfl_sync(kFull, p, j0);
            const unsigned gmask = __ballot_sync(kFull, pr >= 0 && p == p0);
            vmask &= ~gmask;
            const int slot = __ldg(token_slot + n * P + p0);
            const bool src_ok = slot >= 0 && slot < cap_send;
            if (!src_ok && g == 0 && lane == 0) {
                if (slot < 0) bad_slot = true;
                else cap_flag = true;
            }
            int4 r[kCopyUnroll];
            const int4 *src = send + ((int64_t)s * cap_send + (src_ok ? slot : 0)) * V;
#pragma unroll
            for (int u = 0; u < kCopyUnroll; u++) {
                const int vi = v0 + 32 * u;
                r[u] = make_int4(0, 0, 0, 0);
                if (src_ok && vi < V) r[u] = ld_stream(src + vi);
            }
            unsigned dm = gmask;
            while (dm) {
                const int j = __ffs(dm) - 1;
                dm &= dm - 1;
                const int row = __shfl_sync(kFull, pr, j);
                int4 *dst = recv + (int64_t)row * V;
#pragma unroll
                for (int u = 0; u < kCopyUnroll; u++) {
                    const int vi = v0 + 32 * u;
                    if (vi < V) st_cg(dst + vi, r[u]);
                }
            }
        }
    }

    // 2. padding rows: warp task (expert, padding row index, segment)
    if (align > 1) {
        const int64_t ptask = (int64_t)E * (align - 1) * nseg;
        for (int64_t task = gtid >> 5; task < ptask; task += gwarps) {
            const int g = (int)(task % nseg);
            const int64_t ei = task / nseg;
            const int e = (int)(ei / (align - 1));
            const int i = (int)(ei - (int64_t)e * (align - 1));
            const int start = __ldg(expert_offsets + e) + __ldg(ws_tot + e);
            const int row = start + i;
            if (row >= __ldg(expert_offsets + e + 1) || row >= cap_recv) continue;
            if (recv_part >= 0 && e / L != recv_part) continue;
            int4 *dst = recv + (int64_t)row * V;
            const int v0 = g * kCopySegVec + lane;
#pragma unroll
            for (int u = 0; u < kCopyUnroll; u++) {
                const int vi = v0 + 32 * u;
                if (vi < V) st_cg(dst + vi, make_int4(0, 0, 0, 0));
            }
            if (g == 0 && lane == 0) recv_pair[row] = -1;
        }
    }

    // 3. recv_pair entries past the used rows
    const int used = __ldg(expert_offsets + E);
    for (int64_t r = (int64_t)used + gtid; r < cap_recv; r += gthreads) recv_pair[r] = -1;

    if (cap_flag) flag_status(dev_status, MOE_ERR_CAPACITY);
    if (bad_slot) flag_status(dev_status, MOE_ERR_INVALID_ARG);
}

}  // namespace

size_t permute_ws_bytes(int S, int T, int E)
{
    const int64_t G = div_up((int64_t)S * T, kChunk);
    const int64_t h = (int64_t)E * (G > 0 ? G : 1) * 4, t = (int64_t)E * 4;
    return (size_t)(div_up(h, 256) * 256 + div_up(t, 256) * 256);
}

cudaError_t launch_permute(const uint16_t *send, const int32_t *token_slot, const int32_t *ids,
                           int S, int T, int k, int E, int P, int H, int recv_part, int align,
                           int cap_send, int cap_recv, uint16_t *recv, int32_t *expert_offsets,
                           int32_t *pair_row, int32_t *recv_pair, void *ws,
                           uint32_t *dev_status, cudaStream_t st)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int64_t NT = (int64_t)S * T;
    const int64_t npairs = NT * k;
    const int G = (int)div_up(NT, kChunk);
    const int L = E / P;
    const int64_t h_bytes = div_up((int64_t)E * (G > 0 ? G : 1) * 4, 256) * 256;
    int32_t *ws_hist = (int32_t *)ws;
    int32_t *ws_tot = (int32_t *)((char *)ws + h_bytes);

    const size_t hist_smem = (size_t)kChunkWarps * E * sizeof(int);
    if (G > 0) {
        if (hist_smem > 48 * 1024) {
            e = cudaFuncSetAttribute(k_perm_count, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)hist_smem);
            if (e != cudaSuccess) return e;
        }
        MOE_TRACED_LAUNCH("k_perm_count", st,
                          k_perm_count<<<(unsigned)G, kChunk, hist_smem, st>>>(
                              ids, npairs, k, E, L, recv_part, G, ws_hist, dev_status));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    MOE_TRACED_LAUNCH("k_perm_scan", st,
                      k_perm_scan<<<(unsigned)div_up(E, 8), 256, 0, st>>>(E, G, ws_hist, ws_tot));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    const size_t rank_smem = (size_t)(E + 1 + kChunkWarps * E) * sizeof(int);
    if (rank_smem > 48 * 1024) {
        e = cudaFuncSetAttribute(k_perm_rank, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)rank_smem);
        if (e != cudaSuccess) return e;
    }
    MOE_TRACED_LAUNCH("k_perm_rank", st,
                      k_perm_rank<<<(unsigned)(G > 0 ? G : 1), kChunk, rank_smem, st>>>(
                          ids, npairs, k, E, L, recv_part, align, G, ws_hist, ws_tot, cap_recv,
                          expert_offsets, pair_row, recv_pair, dev_status));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    const int V = H / 8;
    const int nseg = (V + kCopySegVec - 1) / kCopySegVec;
    const int64_t warps = NT * nseg + (align > 1 ? (int64_t)E * (align - 1) * nseg : 0);
    // persistent grid: at most one full wave; at least enough threads for the
    // recv_pair tail (capped at one CTA per SM)
    const int64_t wave = (int64_t)di.sm_count * (2048 / kCopyThreads);
    int64_t blocks = div_up(warps, kCopyThreads / 32);
    const int64_t tail = div_up(cap_recv, kCopyThreads);
    const int64_t tail_blocks = tail < di.sm_count ? tail : di.sm_count;
    if (blocks < tail_blocks) blocks = tail_blocks;
    if (blocks > wave) blocks = wave;
    if (blocks < 1) blocks = 1;
    MOE_TRACED_LAUNCH("k_perm_copy", st,
                      k_perm_copy<<<(unsigned)blocks, kCopyThreads, 0, st>>>(
                          (const int4 *)send, token_slot, ids, pair_row, NT, k, E, L, P, T, V,
                          recv_part, align, cap_send, cap_recv, expert_offsets, ws_tot,
                          (int4 *)recv, recv_pair, dev_status));
    return cudaGetLastError();
}

}  // namespace moe
