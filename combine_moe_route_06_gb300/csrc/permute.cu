// permute.cu -- receiver side: rows into expert-contiguous runs.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends): section 1.5 (the
// contiguous layout; runs padded to a multiple of `align`, DeepGEMM wants 128),
// section 3.3 (one row per (token, local expert): "5 rows become 7") and
// section 5.1 (DeepEP v2's copy epilogue with do_expand and device offsets).
//
// The run order is a stable counting sort of the pairs (s, t, j) by expert id
// over the receiving partition(s).  The layout call already ranked every pair
// inside its source's run of its expert (expert_rank) and counted the runs
// (expert_counts), so the permute needs no scan over the pairs:
//   map:  run starts from the expert counts (padded run lengths, exclusive
//         scan over the experts), then
//           row = run start + pairs of the expert in earlier sources + rank;
//         pair_row and recv_pair record the result.
//   copy: per (token, 2 KiB column segment) read each received row of the
//         token once and store it to every local pair row; then zero padding
//         rows and mark unused recv_pair entries.
// One kernel does both when the counts' prefix sums fit in shared memory: every
// CTA of the persistent copy grid builds the run starts itself, each warp
// derives its token's rows, and the warp of segment 0 stores them, so the rows
// are never written and read back and no launch sits between the pack and the
// copy.  Otherwise (many sources) k_perm_map runs first, one CTA per 1,024
// pairs.  The masked form always uses its own map kernel.
#include "common.cuh"
#include "launch.h"
#include "trace.h"

namespace moe {

namespace {

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int kCopyUnroll = 4;
constexpr int kCopySegVec = 32 * kCopyUnroll;
constexpr int kCopyThreads = 256;

constexpr int kMapThreads = 256;
constexpr int kMapPairs = 4 * kMapThreads;      // pairs per CTA
constexpr size_t kFusedMapSmem = 48 * 1024;     // map step inside the copy up to this smem

// grid = S * B CTAs; CTA (s, b) maps pairs [b*kMapPairs, (b+1)*kMapPairs) of source s.
// Every global load is issued before the first barrier so their latencies overlap.
__global__ void __launch_bounds__(kMapThreads) k_perm_map(
    const int32_t *__restrict__ ids, const int32_t *__restrict__ expert_counts,
    const int32_t *__restrict__ expert_rank, int S, int T, int k, int E, int L, int recv_part,
    int align, int B, int cap_recv, int32_t *__restrict__ expert_offsets,
    int32_t *__restrict__ ws_tot, int32_t *__restrict__ pair_row,
    int32_t *__restrict__ recv_pair, uint32_t *dev_status)
{
    extern __shared__ int sm[];
    int *off = sm;              // [E + 1] padded run starts
    int *sb = sm + E + 1;       // [E] pairs of expert e in sources before s
    int *own = sb + E;          // [E] pairs of expert e in source s
    constexpr int kPer = kMapPairs / kMapThreads;
    const int s = blockIdx.x / B, b = blockIdx.x % B;
    const int64_t per_src = (int64_t)T * k;
    const int64_t q0 = (int64_t)s * per_src + (int64_t)b * kMapPairs;
    const int64_t q1 = min((int64_t)s * per_src + per_src, q0 + kMapPairs);
    pdl_wait();
    pdl_trigger();

    int e_[kPer], r_[kPer];
#pragma unroll
    for (int i = 0; i < kPer; i++) {
        const int64_t q = q0 + threadIdx.x + i * kMapThreads;
        e_[i] = (q < q1) ? __ldg(ids + q) : -1;
        r_[i] = (q < q1) ? __ldg(expert_rank + q) : -1;
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const bool r = (recv_part < 0) || (e / L == recv_part);
        int cnt = 0, before = 0, mine = 0;
        for (int s2 = 0; s2 < S; s2++) {
            const int c = __ldg(expert_counts + (int64_t)s2 * E + e);
            cnt += c;
            before += (s2 < s) ? c : 0;
            mine = (s2 == s) ? c : mine;
        }
        off[e] = r ? (cnt + align - 1) / align * align : 0;
        sb[e] = before;
        own[e] = mine;
        if (blockIdx.x == 0) ws_tot[e] = r ? cnt : 0;
    }
    __syncthreads();
    const int total = block_exclusive_scan_1024(off, E);
    if (threadIdx.x == 0) off[E] = total;
    __syncthreads();
    if (blockIdx.x == 0)
        for (int e = threadIdx.x; e <= E; e += blockDim.x) expert_offsets[e] = off[e];

    bool dropped = false, bad = false, bad_id = false;
#pragma unroll
    for (int i = 0; i < kPer; i++) {
        const int64_t q = q0 + threadIdx.x + i * kMapThreads;
        if (q >= q1) continue;
        const int e = e_[i];
        if (e >= E) bad_id = true;
        int row = -1;
        if (in_recv(e, E, L, recv_part)) {
            const int r = r_[i];
            if (r < 0 || r >= own[e]) {
                bad = true;             // rank inconsistent with the counts
            } else {
                row = off[e] + sb[e] + r;
                if (row >= cap_recv) {
                    dropped = true;
                    row = -1;
                }
            }
        }
        pair_row[q] = row;
        if (row >= 0) recv_pair[row] = (int32_t)q;
    }
    if (__syncthreads_or(dropped) && threadIdx.x == 0) flag_status(dev_status, MOE_ERR_CAPACITY);
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(dev_status, MOE_ERR_INVALID_ARG);
    if (__syncthreads_or(bad_id) && threadIdx.x == 0) flag_status(dev_status, MOE_ERR_BAD_EXPERT_ID);
}

// Masked layout map (DeepEP low-latency style, fixed block per expert): the
// first S * B CTAs map pairs as in k_perm_map; block b holds expert e0 + b.
// Every CTA (including extra ones launched for large blocks) marks a share of
// the unused block rows in recv_pair.
__global__ void __launch_bounds__(kMapThreads) k_perm_map_masked(
    const int32_t *__restrict__ ids, const int32_t *__restrict__ expert_counts,
    const int32_t *__restrict__ expert_rank, int S, int T, int k, int E, int e0, int nb,
    int B, int block_rows, int32_t *__restrict__ masked_counts, int32_t *__restrict__ pair_row,
    int32_t *__restrict__ recv_pair, uint32_t *dev_status)
{
    extern __shared__ int sm[];
    int *cnt = sm;           // [nb] rows of block b in use
    int *sb = sm + nb;       // [nb] pairs of its expert in sources before s
    int *own = sb + nb;      // [nb] pairs of its expert in source s
    constexpr int kPer = kMapPairs / kMapThreads;
    const bool mapper = blockIdx.x < S * B;       // extra CTAs only mark unused rows
    const int s = mapper ? blockIdx.x / B : 0, b = mapper ? blockIdx.x % B : 0;
    const int64_t per_src = (int64_t)T * k;
    const int64_t q0 = (int64_t)s * per_src + (int64_t)b * kMapPairs;
    const int64_t q1 = mapper ? min((int64_t)s * per_src + per_src, q0 + kMapPairs) : q0;
    pdl_wait();
    pdl_trigger();

    int e_[kPer], r_[kPer];
#pragma unroll
    for (int i = 0; i < kPer; i++) {
        const int64_t q = q0 + threadIdx.x + i * kMapThreads;
        e_[i] = (q < q1) ? __ldg(ids + q) : -1;
        r_[i] = (q < q1) ? __ldg(expert_rank + q) : -1;
    }
    for (int bb = threadIdx.x; bb < nb; bb += blockDim.x) {
        const int e = e0 + bb;
        int total = 0, before = 0, mine = 0;
        for (int s2 = 0; s2 < S; s2++) {
            const int c = __ldg(expert_counts + (int64_t)s2 * E + e);
            total += c;
            before += (s2 < s) ? c : 0;
            mine = (s2 == s) ? c : mine;
        }
        cnt[bb] = min(total, block_rows);
        sb[bb] = before;
        own[bb] = mine;
        if (blockIdx.x == 0) masked_counts[bb] = cnt[bb];
    }
    __syncthreads();

    bool dropped = false, bad = false, bad_id = false;
#pragma unroll
    for (int i = 0; i < kPer; i++) {
        const int64_t q = q0 + threadIdx.x + i * kMapThreads;
        if (q >= q1) continue;
        const int e = e_[i];
        if (e >= E) bad_id = true;
        int row = -1;
        if (e >= e0 && e < e0 + nb) {
            const int bb = e - e0, r = r_[i];
            if (r < 0 || r >= own[bb]) {
                bad = true;
            } else if (sb[bb] + r >= block_rows) {
                dropped = true;
            } else {
                row = bb * block_rows + sb[bb] + r;
            }
        }
        pair_row[q] = row;
        if (row >= 0) recv_pair[row] = (int32_t)q;
    }
    // unused rows of every block: recv_pair = -1 (spread over all CTAs)
    const int64_t rows = (int64_t)nb * block_rows;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows;
         r += (int64_t)gridDim.x * blockDim.x) {
        const int bb = (int)(r / block_rows);
        if (r - (int64_t)bb * block_rows >= cnt[bb]) recv_pair[r] = -1;
    }
    if (__syncthreads_or(dropped) && threadIdx.x == 0) flag_status(dev_status, MOE_ERR_CAPACITY);
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(dev_status, MOE_ERR_INVALID_ARG);
    if (__syncthreads_or(bad_id) && threadIdx.x == 0) flag_status(dev_status, MOE_ERR_BAD_EXPERT_ID);
}

// Row copy, and with MAP the map step as well: every CTA first builds the run
// starts (off) from the expert counts in shared memory, and each warp derives
// its token's pair rows from the ids and ranks (the warp of column segment 0
// stores them in pair_row / recv_pair).  Without MAP the rows come from
// pair_row and the starts from expert_offsets / ws_tot (k_perm_map ran first).
template <bool MAP>
__global__ void __launch_bounds__(kCopyThreads) k_perm_copy(
    const int4 *__restrict__ send, const int32_t *__restrict__ token_slot,
    const int32_t *__restrict__ ids, int32_t *__restrict__ pair_row,
    const int32_t *__restrict__ expert_counts, const int32_t *__restrict__ expert_rank, int S,
    int64_t NT, int k, int E, int L, int P, int T, int V, int recv_part, int align, int fill,
    int cap_send, int cap_recv, int32_t *__restrict__ expert_offsets,
    const int32_t *__restrict__ ws_tot, int4 *__restrict__ recv, int32_t *__restrict__ recv_pair,
    uint32_t *dev_status)
{
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t gthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t gwarps = gthreads >> 5;
    const int nseg = (V + kCopySegVec - 1) / kCopySegVec;
    bool cap_flag = false, bad_slot = false;
    bool dropped = false, bad_rank = false, bad_id = false;

    // Phase 1 walks warp tasks (token, column segment), tokens last to first:
    // the pack kernel wrote the send rows of the last tokens most recently, so
    // those reads still hit L2; the rows written here last (first tokens) are
    // the ones the combine reads first.  Each warp loads the index data of its
    // next task (ids, ranks or pair rows, the token's send slots) one task
    // ahead, the first before the run starts below are built.
    const int64_t ntask = NT * nseg;
    int64_t rtask = gtid >> 5;
    int e_nx = -1, x_nx = -1, ts_nx = -1;
    auto fetch = [&](int64_t rt) {
        const int64_t n = (ntask - 1 - rt) / nseg;
        if (lane < k) {
            e_nx = __ldg(ids + n * k + lane);
            x_nx = __ldg((MAP ? expert_rank : pair_row) + n * k + lane);
        }
        if (lane < P) ts_nx = __ldg(token_slot + n * P + lane);
    };
    if (rtask < ntask) fetch(rtask);

    // run starts: off[e] = padded pairs of the receiving experts before e,
    // cnt[e] = pairs of e, sb[s][e] = pairs of e in the sources before s
    extern __shared__ int smp[];
    int *off = smp;              // [E + 1]
    int *cnt = off + E + 1;      // [E]
    int *sb = cnt + E;           // [S][E]
    if (MAP) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            int run = 0;
            for (int s2 = 0; s2 < S; s2++) {
                sb[s2 * E + e] = run;
                run += __ldg(expert_counts + (int64_t)s2 * E + e);
            }
            cnt[e] = run;
            off[e] = in_recv(e, E, L, recv_part) ? (run + align - 1) / align * align : 0;
        }
        __syncthreads();
        const int total = block_exclusive_scan_1024(off, E);
        if (threadIdx.x == 0) off[E] = total;
        __syncthreads();
        if (blockIdx.x == 0)
            for (int e = threadIdx.x; e <= E; e += blockDim.x) expert_offsets[e] = off[e];
    }

    // 1. pair rows, one warp per (token, column segment)
    for (; rtask < ntask; rtask += gwarps) {
        const int64_t task = ntask - 1 - rtask;
        const int64_t n = task / nseg;
        const int g = (int)(task - n * nseg);
        const int e_c = e_nx, x_c = x_nx, ts_c = ts_nx;
        if (rtask + gwarps < ntask) fetch(rtask + gwarps);
        const int s = (int)(n / T);
        int pr = -1, p = -1;
        if (lane < k) {
            const int64_t q = n * k + lane;
            if (MAP) {
                // row = run start + pairs of e in earlier sources + rank
                const int e = e_c;
                if (e >= E) bad_id = true;
                if (in_recv(e, E, L, recv_part)) {
                    const int r = x_c;
                    const int before = sb[s * E + e];
                    const int own = (s + 1 < S ? sb[(s + 1) * E + e] : cnt[e]) - before;
                    if (r < 0 || r >= own) {
                        bad_rank = true;            // rank inconsistent with the counts
                    } else {
                        pr = off[e] + before + r;
                        if (pr >= cap_recv) {
                            dropped = true;
                            pr = -1;
                        }
                    }
                }
                if (g == 0) {
                    pair_row[q] = pr;
                    if (pr >= 0) recv_pair[pr] = (int32_t)q;
                }
                if (pr >= 0) p = e / L;
            } else {
                pr = x_c;
                if (pr >= 0) p = e_c / L;
            }
        }
        unsigned vmask = __ballot_sync(kFull, pr >= 0);
        const int v0 = g * kCopySegVec + lane;
        while (vmask) {
            const int j0 = __ffs(vmask) - 1;
            const int p0 = __shfl_sync(kFull, p, j0);
            const unsigned gmask = __ballot_sync(kFull, pr >= 0 && p == p0);
            vmask &= ~gmask;
            const int slot = __shfl_sync(kFull, ts_c, p0);
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
    if (fill && align > 1) {
        const int64_t ptask = (int64_t)E * (align - 1) * nseg;
        for (int64_t task = gtid >> 5; task < ptask; task += gwarps) {
            const int g = (int)(task % nseg);
            const int64_t ei = task / nseg;
            const int e = (int)(ei / (align - 1));
            const int i = (int)(ei - (int64_t)e * (align - 1));
            const int start = MAP ? off[e] + cnt[e] : __ldg(expert_offsets + e) + __ldg(ws_tot + e);
            const int end = MAP ? off[e + 1] : __ldg(expert_offsets + e + 1);
            const int row = start + i;
            if (row >= end || row >= cap_recv) continue;
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
    if (fill) {
        const int used = MAP ? off[E] : __ldg(expert_offsets + E);
        for (int64_t r = (int64_t)used + gtid; r < cap_recv; r += gthreads) recv_pair[r] = -1;
    }

    if (cap_flag || dropped) flag_status(dev_status, MOE_ERR_CAPACITY);
    if (bad_slot || bad_rank) flag_status(dev_status, MOE_ERR_INVALID_ARG);
    if (bad_id) flag_status(dev_status, MOE_ERR_BAD_EXPERT_ID);
}

}  // namespace

bool permute_map_fused(int S, int E)
{
    return (size_t)(2 * E + 1 + (int64_t)S * E) * sizeof(int) <= kFusedMapSmem;
}

size_t permute_ws_bytes(int S, int T, int E)
{
    (void)S;
    (void)T;
    return (size_t)(div_up((int64_t)E * 4, 256) * 256);
}

cudaError_t launch_permute(const uint16_t *send, const int32_t *token_slot, const int32_t *ids,
                           const int32_t *expert_counts, const int32_t *expert_rank,
                           int S, int T, int k, int E, int P, int H, int recv_part, int align,
                           int cap_send, int cap_recv, uint16_t *recv, int32_t *expert_offsets,
                           int32_t *pair_row, int32_t *recv_pair, void *ws,
                           uint32_t *dev_status, cudaStream_t st)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int64_t NT = (int64_t)S * T;
    const int L = E / P;
    int32_t *ws_tot = (int32_t *)ws;

    const int V = H / 8;
    const int nseg = (V + kCopySegVec - 1) / kCopySegVec;
    const int64_t warps = NT * nseg + (align > 1 ? (int64_t)E * (align - 1) * nseg : 0);
    // The map step runs inside the copy kernel when every CTA can hold the
    // counts' prefix sums (off, cnt, sb) in shared memory; otherwise as
    // k_perm_map before it.
    const size_t fused_smem = (size_t)(2 * E + 1 + (int64_t)S * E) * sizeof(int);
    const bool fused = permute_map_fused(S, E);
    const void *copy_fn = fused ? (const void *)k_perm_copy<true> : (const void *)k_perm_copy<false>;
    const size_t copy_smem = fused ? fused_smem : 0;
    if (!fused) {
        const int B = (int)(div_up((int64_t)T * k, kMapPairs) > 0 ? div_up((int64_t)T * k, kMapPairs) : 1);
        const size_t map_smem = (size_t)(3 * E + 1) * sizeof(int);
        MOE_TRACED_LAUNCH("k_perm_map", st,
                          e = launch_pdl(k_perm_map, dim3((unsigned)(S * B)), dim3(kMapThreads),
                                         map_smem, st, ids, expert_counts, expert_rank, S, T, k, E,
                                         L, recv_part, align, B, cap_recv, expert_offsets, ws_tot,
                                         pair_row, recv_pair, dev_status));
        if (e != cudaSuccess) return e;
    }

    // persistent grid: at most the CTAs that fit at once; at least enough
    // threads for the recv_pair tail (capped at one CTA per SM)
    const int resident = resident_grid(copy_fn, kCopyThreads, copy_smem);
    const int64_t wave = resident > 0 ? resident : (int64_t)di.sm_count * (2048 / kCopyThreads);
    int64_t blocks = div_up(warps, kCopyThreads / 32);
    const int64_t tail = div_up(cap_recv, kCopyThreads);
    const int64_t tail_blocks = tail < di.sm_count ? tail : di.sm_count;
    if (blocks < tail_blocks) blocks = tail_blocks;
    if (blocks > wave) blocks = wave;
    if (blocks < 1) blocks = 1;
    if (fused) {
        MOE_TRACED_LAUNCH("k_perm_copy", st,
                          e = launch_pdl(k_perm_copy<true>, dim3((unsigned)blocks),
                                         dim3(kCopyThreads), copy_smem, st, (const int4 *)send,
                                         token_slot, ids, pair_row, expert_counts, expert_rank, S,
                                         NT, k, E, L, P, T, V, recv_part, align, 1, cap_send,
                                         cap_recv, expert_offsets, (const int32_t *)nullptr,
                                         (int4 *)recv, recv_pair, dev_status));
    } else {
        MOE_TRACED_LAUNCH("k_perm_copy", st,
                          e = launch_pdl(k_perm_copy<false>, dim3((unsigned)blocks),
                                         dim3(kCopyThreads), 0, st, (const int4 *)send, token_slot,
                                         ids, pair_row, (const int32_t *)nullptr,
                                         (const int32_t *)nullptr, S, NT, k, E, L, P, T, V,
                                         recv_part, align, 1, cap_send, cap_recv, expert_offsets,
                                         (const int32_t *)ws_tot, (int4 *)recv, recv_pair,
                                         dev_status));
    }
    return e;
}

cudaError_t launch_permute_masked(const uint16_t *send, const int32_t *token_slot,
                                  const int32_t *ids, const int32_t *expert_counts,
                                  const int32_t *expert_rank, int S, int T, int k, int E, int P,
                                  int H, int recv_part, int block_rows, int cap_send,
                                  uint16_t *recv, int32_t *masked_counts, int32_t *pair_row,
                                  int32_t *recv_pair, uint32_t *dev_status, cudaStream_t st)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int64_t NT = (int64_t)S * T;
    const int L = E / P;
    const int nb = recv_part < 0 ? E : L;
    const int e0 = recv_part < 0 ? 0 : recv_part * L;
    const int B = (int)(div_up((int64_t)T * k, kMapPairs) > 0 ? div_up((int64_t)T * k, kMapPairs) : 1);
    const size_t smem = (size_t)(3 * nb) * sizeof(int);
    // enough CTAs that each marks at most ~2,048 unused block rows
    int64_t grid = (int64_t)S * B;
    const int64_t mark = div_up((int64_t)nb * block_rows, 8 * kMapThreads);
    if (grid < mark) grid = mark < di.sm_count ? mark : di.sm_count;
    MOE_TRACED_LAUNCH("k_perm_map_masked", st,
                      e = launch_pdl(k_perm_map_masked, dim3((unsigned)grid), dim3(kMapThreads),
                                     smem, st, ids, expert_counts, expert_rank, S, T, k, E, e0, nb,
                                     B, block_rows, masked_counts, pair_row, recv_pair, dev_status));
    if (e != cudaSuccess || NT == 0) return e;
    const int V = H / 8;
    const int nseg = (V + kCopySegVec - 1) / kCopySegVec;
    const int resident = resident_grid((const void *)k_perm_copy<false>, kCopyThreads, 0);
    int64_t blocks = div_up(NT * nseg, kCopyThreads / 32);
    const int64_t wave = resident > 0 ? resident : (int64_t)di.sm_count * (2048 / kCopyThreads);
    if (blocks > wave) blocks = wave;
    if (blocks < 1) blocks = 1;
    const int cap_recv = nb * block_rows;
    MOE_TRACED_LAUNCH("k_perm_copy", st,
                      e = launch_pdl(k_perm_copy<false>, dim3((unsigned)blocks), dim3(kCopyThreads),
                                     0, st, (const int4 *)send, token_slot, ids, pair_row,
                                     (const int32_t *)nullptr, (const int32_t *)nullptr, S, NT, k,
                                     E, L, P, T, V, recv_part, 1, 0, cap_send, cap_recv,
                                     (int32_t *)nullptr, (const int32_t *)nullptr, (int4 *)recv,
                                     recv_pair, dev_status));
    return e;
}

}  // namespace moe
