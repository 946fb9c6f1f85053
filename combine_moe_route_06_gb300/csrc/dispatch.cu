// dispatch.cu -- the one-pass pack + receiver permute and the whole dispatch
// side in one call for batches larger than one launch takes (moe_dispatch,
// moe_dispatch_quantized, moe_dispatch_pack_permute, _masked).
//
// a2a-backends page (vincentzed.com/writing/a2a-backends): the router's ids
// and weights (section 1.1), one copy per partition that holds one of the
// token's experts with prefix-sum slots (sections 1.3, 3.2), rows packed into
// per-partition send regions (sections 3.2, 5.1, 6.1) and the receiver's
// expert-contiguous runs (sections 1.5, 3.3, 5.1).  The outputs are the bytes
// moe_route_topk, moe_dispatch_layout, moe_dispatch_pack and
// moe_permute_to_experts give one after the other.
//
// moe_dispatch, moe_dispatch_masked and moe_dispatch_quantized for one source
// of at most 256 tokens (a decode step) are one launch (dispatch_small.cuh,
// launched from dispatch_small.cu and dispatch_small_q.cu; their launchers
// below pick that form).  Larger batches run the routing kernel, the
// layout (moe_dispatch_layout's kernels), then k_pack_permute: pack and
// permute in one pass.  A row task reads the token's segment of x once,
// stores it to every send slot of the token, then reads back the segment of
// the send row of each receiving partition and stores it to that partition's
// pair rows (row_move.cuh).  The read-back is the receiver reading the row
// that just landed in its receive region (the emulated all-to-all: partition
// p's region of the send buffer); the warp that landed it issues the read, so
// it is served from L2 and the send rows are not read from HBM a second time.
#include "common.cuh"
#include "launch.h"
#include "qrow.cuh"
#include "row_move.cuh"
#include "trace.h"

namespace moe {

namespace {

inline int64_t div_up(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------ pack + permute --

constexpr int kPPUnroll = 4;                       // int4 per lane per segment (2 KiB)
constexpr int kPPSegVec = 32 * kPPUnroll;
constexpr int kPPThreads = 256;
constexpr int kPPBatch = 1;                        // one partition's row read back at a time
constexpr int kPPStageMax = 3;                     // tasks per warp whose x is staged early
constexpr size_t kPPStageBytes = (size_t)(kPPThreads / 32) * kPPSegVec * sizeof(int4);  // per task

// 16-byte asynchronous copy global -> shared (no register staging).  The
// copying thread sees the bytes after cp_async_wait_all.
__device__ __forceinline__ void cp_async16(int4 *smem_dst, const int4 *gmem_src)
{
    const unsigned d = static_cast<unsigned>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

static_assert(kPPSegVec == kQSegVec, "bf16 and record segments cover the same x vectors");

// x vector of this lane's u-th 16-byte piece of the segment starting at vb:
// bf16 rows (FMT 0) take vectors lane + 32 u, record pieces their
// quantizer's order (piece_vec).
template <int FMT>
__device__ __forceinline__ int seg_piece(int vb, int u)
{
    if constexpr (FMT == 0) return vb + (threadIdx.x & 31) + 32 * u;
    else return piece_vec<FMT>(vb, u);
}

// The early x reads of the one-pass kernels (tasks last to first, task rt of
// warp w = rt0 + j * gwarps at its j-th iteration).  With REG0 the segment of
// the warp's first task goes to registers (x0) and those of its next `stage`
// tasks to shared memory; without, its first `stage` tasks' segments go to
// shared memory and x0 stays unused.  stg: this warp's slots, [slot][kPPUnroll]
// [32 lanes] int4, each lane's pieces in seg_piece<FMT> order.  Each lane
// copies the 16-byte pieces it will use itself, so no barrier orders the
// copies with their use, only cp_async_wait_all.  Every lane must call (the
// copy group is committed even when empty).
template <int FMT, bool REG0>
__device__ __forceinline__ void stage_x(const int4 *__restrict__ x, int64_t ntask, int nseg, int V,
                                        int64_t rt0, int64_t gwarps, int stage,
                                        int4 (&x0)[kPPUnroll], int4 *stg)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int u = 0; u < kPPUnroll; u++) x0[u] = make_int4(0, 0, 0, 0);
    const int last = REG0 ? stage : stage - 1;
    for (int j = 0; j <= last; j++) {
        const int64_t rt = rt0 + (int64_t)j * gwarps;
        if (rt >= ntask) break;
        const int64_t t = ntask - 1 - rt;
        const int64_t n = t / nseg;
        const int g = (int)(t - n * nseg);
        const int slot = REG0 ? j - 1 : j;
#pragma unroll
        for (int u = 0; u < kPPUnroll; u++) {
            const int vi = seg_piece<FMT>(g * kPPSegVec, u);
            if (vi >= V) continue;
            if (REG0 && j == 0) x0[u] = ld_stream(x + n * V + vi);
            else cp_async16(stg + (slot * kPPUnroll + u) * 32 + lane, x + n * V + vi);
        }
    }
    cp_async_commit();
}

// The x segment of the warp's it-th task if stage_x fetched it (into xs, and
// true), else false.  Call after cp_async_wait_all.
template <bool REG0>
__device__ __forceinline__ bool staged_x(int it, int stage, const int4 (&x0)[kPPUnroll],
                                         const int4 *stg, int4 (&xs)[kPPUnroll])
{
    const int lane = threadIdx.x & 31;
    const int slot = REG0 ? it - 1 : it;
    const bool have = REG0 ? it <= stage : it < stage;
#pragma unroll
    for (int u = 0; u < kPPUnroll; u++)
        xs[u] = (REG0 && it == 0) ? x0[u]
                                  : (have ? stg[(slot * kPPUnroll + u) * 32 + lane]
                                          : make_int4(0, 0, 0, 0));
    return have;
}

// Run starts of the receiving experts, built by every CTA in shared memory
// from the expert counts (as the permute's map step does): off[e] = padded
// pairs of the receiving experts before e (off[E] = rows used), cnt[e] = pairs
// of e, sb[s][e] = pairs of e in the sources before s.  CTA 0 also stores
// expert_offsets.  Every thread of the CTA must call; synchronises the CTA.
__device__ __forceinline__ void build_run_starts(const int32_t *__restrict__ expert_counts, int S,
                                                 int E, int L, int recv_part, int align, int *off,
                                                 int *cnt, int *sb,
                                                 int32_t *__restrict__ expert_offsets)
{
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

// Receive row of a pair (expert e, rank r within source s's run of e): run
// start + pairs of e in earlier sources + rank; -1 if e is not received, the
// rank is inconsistent with the counts (bad_rank) or the row is past cap_recv
// (dropped).  An id >= E sets bad_id.
__device__ __forceinline__ int pair_row_of(int e, int r, int s, int S, int E, int L, int recv_part,
                                           int cap_recv, const int *off, const int *cnt,
                                           const int *sb, bool &bad_id, bool &bad_rank,
                                           bool &dropped)
{
    if (e >= E) bad_id = true;
    if (!in_recv(e, E, L, recv_part)) return -1;
    const int before = sb[s * E + e];
    const int own = (s + 1 < S ? sb[(s + 1) * E + e] : cnt[e]) - before;
    if (r < 0 || r >= own) {
        bad_rank = true;
        return -1;
    }
    const int row = off[e] + before + r;
    if (row >= cap_recv) {
        dropped = true;
        return -1;
    }
    return row;
}

// recv_pair = -1 for receive rows past the used ones; send_src = -1 for send
// rows past each source's last copy.  Grid-stride over every thread.
__device__ __forceinline__ void mark_unused_rows(int used, int cap_recv, int S, int P, int cap_send,
                                                 const int32_t *__restrict__ part_offsets,
                                                 int32_t *__restrict__ recv_pair,
                                                 int32_t *__restrict__ send_src)
{
    const int64_t gthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t rr = (int64_t)used + gtid; rr < cap_recv; rr += gthreads) recv_pair[rr] = -1;
    for (int64_t i = gtid; i < (int64_t)S * cap_send; i += gthreads) {
        const int s = (int)(i / cap_send);
        const int rr = (int)(i - (int64_t)s * cap_send);
        if (rr >= __ldg(part_offsets + (int64_t)s * (P + 1) + P)) send_src[i] = -1;
    }
}

// Pack and permute in one pass over warp tasks (token, 2 KiB column segment),
// tokens last to first (the receive rows written last, those of the first
// tokens, are the ones the combine reads first).  Every CTA first builds the
// run starts from the expert counts in shared memory (as the permute's map
// step does); each warp derives its token's pair rows from the ids and ranks;
// the warp of segment 0 stores pair_row, recv_pair and send_src.  Inside
// moe_dispatch each warp loads its first task's x segment into registers and
// copies the next `stage` tasks' segments into shared memory before the
// grid-dependency wait, while the layout kernel still runs.
__global__ void __launch_bounds__(kPPThreads, 3) k_pack_permute(
    const int4 *__restrict__ x, const int32_t *__restrict__ token_slot,
    const int32_t *__restrict__ part_offsets, const int32_t *__restrict__ ids,
    const int32_t *__restrict__ expert_counts, const int32_t *__restrict__ expert_rank, int S,
    int64_t NT, int k, int E, int L, int P, int T, int V, int recv_part, int align, int cap_send,
    int cap_recv, int4 *__restrict__ send, int32_t *__restrict__ send_src,
    int4 *__restrict__ recv, int32_t *__restrict__ expert_offsets, int32_t *__restrict__ pair_row,
    int32_t *__restrict__ recv_pair, uint32_t *dev_status, bool x_before_wait, int stage)
{
    const int lane = threadIdx.x & 31;
    const int64_t gthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t gwarps = gthreads >> 5;
    const int nseg = (V + kPPSegVec - 1) / kPPSegVec;
    extern __shared__ int smp[];
    int *off = smp;              // [E + 1]
    int *cnt = off + E + 1;      // [E]
    int *sb = cnt + E;           // [S][E]
    // [warp][stage][kPPUnroll][32 lanes]: x segments of this warp's tasks 1..stage
    int4 *stg = reinterpret_cast<int4 *>(smp + ((2 * E + 1 + S * E + 3) & ~3)) +
                (threadIdx.x >> 5) * stage * kPPSegVec;
    // With x_before_wait the first task's x segment is loaded before the
    // grid-dependency wait, so its HBM latency passes while the layout finishes.
    // moe_dispatch sets it: x was complete before its routing kernel ran, this
    // kernel is launched only once the layout kernel has passed its own wait (it
    // waits, then lets dependents launch), and the layout's wait returns only
    // after the routing kernel, which waited for everything before it, has
    // completed.  Nothing here reads what the layout writes before pdl_wait().
    // Called on its own (moe_dispatch_pack_permute) the kernel does not know
    // what ran before it, so it waits first.
    if (!x_before_wait) pdl_wait();
    const int64_t rt0 = gtid >> 5;
    // Tasks 1..stage: their x segments are copied into shared memory now, so
    // that while the layout finishes HBM reads x instead of idling and the row
    // phase that follows is left almost only writes.
    int4 x0[kPPUnroll];
    stage_x<0, true>(x, NT * nseg, nseg, V, rt0, gwarps, stage, x0, stg);
    if (x_before_wait) pdl_wait();
    pdl_trigger();
    bool cap_flag = false, bad_slot = false, dropped = false, bad_rank = false, bad_id = false;
    bool pack_overflow = false;

    const int64_t ntask = NT * nseg;
    int64_t rtask = gtid >> 5;
    int e_nx = -1, r_nx = -1, ts_nx = -1;
    auto fetch = [&](int64_t rt) {
        const int64_t n = (ntask - 1 - rt) / nseg;
        if (lane < k) {
            e_nx = __ldg(ids + n * k + lane);
            r_nx = __ldg(expert_rank + n * k + lane);
        }
        if (lane < P) ts_nx = __ldg(token_slot + n * P + lane);
    };
    if (rtask < ntask) fetch(rtask);

    build_run_starts(expert_counts, S, E, L, recv_part, align, off, cnt, sb, expert_offsets);
    cp_async_wait_all();

    for (int it = 0; rtask < ntask; rtask += gwarps, it++) {
        const int64_t task = ntask - 1 - rtask;
        const int64_t n = task / nseg;
        const int g = (int)(task - n * nseg);
        const int e_c = e_nx, r_c = r_nx, ts_c = ts_nx;
        if (rtask + gwarps < ntask) fetch(rtask + gwarps);
        const int s = (int)(n / T);
        int pr = -1, pp = -1;
        if (lane < k) {
            pr = pair_row_of(e_c, r_c, s, S, E, L, recv_part, cap_recv, off, cnt, sb, bad_id,
                             bad_rank, dropped);
            if (g == 0) {
                const int64_t q = n * k + lane;
                pair_row[q] = pr;
                if (pr >= 0) recv_pair[pr] = (int32_t)q;
            }
            if (pr >= 0) pp = e_c / L;
        }
        if (g == 0 && lane < P) {
            if (ts_c >= cap_send) pack_overflow = true;
            else if (ts_c >= 0) send_src[(int64_t)s * cap_send + ts_c] = (int32_t)(n - (int64_t)s * T);
        }
        // x0 (task 0) and the staged segments pass through one register
        // array, so the row task sees one array or none
        int4 xs[kPPUnroll];
        const bool have = staged_x<true>(it, stage, x0, stg, xs);
        move_token_segment<kPPUnroll, kPPBatch>(x + n * V, send + (int64_t)s * cap_send * V, recv, V,
                                      g * kPPSegVec + lane, ts_c, pr, pp, P, cap_send, bad_slot,
                                      cap_flag, g == 0, have ? xs : nullptr);
    }

    // padding rows: warp task (expert, padding row index, segment)
    if (align > 1) {
        const int64_t ptask = (int64_t)E * (align - 1) * nseg;
        for (int64_t task = gtid >> 5; task < ptask; task += gwarps) {
            const int g = (int)(task % nseg);
            const int64_t ei = task / nseg;
            const int e = (int)(ei / (align - 1));
            const int i = (int)(ei - (int64_t)e * (align - 1));
            const int row = off[e] + cnt[e] + i;
            if (!in_recv(e, E, L, recv_part) || row >= off[e + 1] || row >= cap_recv) continue;
            int4 *dst = recv + (int64_t)row * V;
            const int v0 = g * kPPSegVec + lane;
#pragma unroll
            for (int u = 0; u < kPPUnroll; u++) {
                const int vi = v0 + 32 * u;
                if (vi < V) st_cg(dst + vi, make_int4(0, 0, 0, 0));
            }
            if (g == 0 && lane == 0) recv_pair[row] = -1;
        }
    }
    mark_unused_rows(off[E], cap_recv, S, P, cap_send, part_offsets, recv_pair, send_src);

    if (cap_flag || dropped || pack_overflow) flag_status(dev_status, MOE_ERR_CAPACITY);
    if (bad_slot || bad_rank) flag_status(dev_status, MOE_ERR_INVALID_ARG);
    if (bad_id) flag_status(dev_status, MOE_ERR_BAD_EXPERT_ID);
}

// ---------------------------------------- pack + permute, masked layout --

// Pack and the masked receive layout in one pass: as k_pack_permute, but the
// receiving set's nb experts (e0 .. e0 + nb - 1) own fixed blocks of
// block_rows rows, a pair's row is its block base + pairs of its expert in
// earlier sources + its rank (dropped past the block), and every CTA marks a
// share of the blocks' unused rows; CTA 0 stores the rows in use per block.
// Shared memory: per block the rows in use, the pairs in all sources, and the
// pairs in the sources before each s.
__global__ void __launch_bounds__(kPPThreads, 3) k_pack_permute_masked(
    const int4 *__restrict__ x, const int32_t *__restrict__ token_slot,
    const int32_t *__restrict__ part_offsets, const int32_t *__restrict__ ids,
    const int32_t *__restrict__ expert_counts, const int32_t *__restrict__ expert_rank, int S,
    int64_t NT, int k, int E, int L, int P, int T, int V, int e0, int nb, int block_rows,
    int cap_send, int4 *__restrict__ send, int32_t *__restrict__ send_src,
    int4 *__restrict__ recv, int32_t *__restrict__ masked_counts, int32_t *__restrict__ pair_row,
    int32_t *__restrict__ recv_pair, uint32_t *dev_status, bool x_before_wait, int stage)
{
    const int lane = threadIdx.x & 31;
    const int64_t gthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t gwarps = gthreads >> 5;
    const int nseg = (V + kPPSegVec - 1) / kPPSegVec;
    bool cap_flag = false, bad_slot = false, dropped = false, bad_rank = false, bad_id = false;
    bool pack_overflow = false;

    extern __shared__ int smm[];
    int *bcnt = smm;             // [nb] rows of block b in use
    int *btot = bcnt + nb;       // [nb] pairs of its expert in all sources
    int *bsb = btot + nb;        // [S][nb] pairs of its expert in the sources before s
    // [warp][stage][kPPUnroll][32 lanes]: x segments of this warp's tasks 1..stage
    int4 *stg = reinterpret_cast<int4 *>(smm + ((2 * nb + S * nb + 3) & ~3)) +
                (threadIdx.x >> 5) * stage * kPPSegVec;
    // x before the grid-dependency wait only inside moe_dispatch_masked (the
    // same ordering argument as k_pack_permute); called on its own the kernel
    // waits first.
    if (!x_before_wait) pdl_wait();
    const int64_t rt0 = gtid >> 5;
    int4 x0[kPPUnroll];
    stage_x<0, true>(x, NT * nseg, nseg, V, rt0, gwarps, stage, x0, stg);
    if (x_before_wait) pdl_wait();
    pdl_trigger();
    for (int bb = threadIdx.x; bb < nb; bb += blockDim.x) {
        int run = 0;
        for (int s2 = 0; s2 < S; s2++) {
            bsb[s2 * nb + bb] = run;
            run += __ldg(expert_counts + (int64_t)s2 * E + e0 + bb);
        }
        btot[bb] = run;
        bcnt[bb] = min(run, block_rows);
        if (blockIdx.x == 0) masked_counts[bb] = bcnt[bb];
    }
    __syncthreads();
    cp_async_wait_all();
    // unused rows of every block
    const int64_t rows = (int64_t)nb * block_rows;
    for (int64_t r = gtid; r < rows; r += gthreads) {
        const int bb = (int)(r / block_rows);
        if (r - (int64_t)bb * block_rows >= bcnt[bb]) recv_pair[r] = -1;
    }

    const int64_t ntask = NT * nseg;
    int it = 0;
    for (int64_t rtask = rt0; rtask < ntask; rtask += gwarps, it++) {
        const int64_t task = ntask - 1 - rtask;       // tokens last to first
        const int64_t n = task / nseg;
        const int g = (int)(task - n * nseg);
        const int s = (int)(n / T);
        int ts = -1, pr = -1, pp = -1;
        if (lane < P) ts = __ldg(token_slot + n * P + lane);
        if (lane < k) {
            const int e = __ldg(ids + n * k + lane);
            if (e >= E) bad_id = true;
            if (e >= e0 && e < e0 + nb) {
                const int bb = e - e0, r = __ldg(expert_rank + n * k + lane);
                const int before = bsb[s * nb + bb];
                const int own = (s + 1 < S ? bsb[(s + 1) * nb + bb] : btot[bb]) - before;
                if (r < 0 || r >= own) bad_rank = true;          // rank inconsistent with the counts
                else if (before + r >= block_rows) dropped = true;
                else pr = bb * block_rows + before + r;
            }
            if (g == 0) {
                const int64_t q = n * k + lane;
                pair_row[q] = pr;
                if (pr >= 0) recv_pair[pr] = (int32_t)q;
            }
            if (pr >= 0) pp = e / L;
        }
        if (g == 0 && lane < P) {
            if (ts >= cap_send) pack_overflow = true;
            else if (ts >= 0) send_src[(int64_t)s * cap_send + ts] = (int32_t)(n - (int64_t)s * T);
        }
        int4 xs[kPPUnroll];
        const bool have = staged_x<true>(it, stage, x0, stg, xs);
        move_token_segment<kPPUnroll, kPPBatch>(x + n * V, send + (int64_t)s * cap_send * V, recv, V,
                                                g * kPPSegVec + lane, ts, pr, pp, P, cap_send,
                                                bad_slot, cap_flag, g == 0, have ? xs : nullptr);
    }
    for (int64_t i = gtid; i < (int64_t)S * cap_send; i += gthreads) {
        const int s = (int)(i / cap_send);
        const int rr = (int)(i - (int64_t)s * cap_send);
        if (rr >= __ldg(part_offsets + (int64_t)s * (P + 1) + P)) send_src[i] = -1;
    }
    if (cap_flag || dropped || pack_overflow) flag_status(dev_status, MOE_ERR_CAPACITY);
    if (bad_slot || bad_rank) flag_status(dev_status, MOE_ERR_INVALID_ARG);
    if (bad_id) flag_status(dev_status, MOE_ERR_BAD_EXPERT_ID);
}

// ------------------------------------------- pack + permute, quantized --

// moe_dispatch's pack + permute pass with quantized rows: as k_pack_permute,
// but each warp task (token, 1,024-value segment) quantizes the segment once
// (MXFP8 or NVFP4, quant.cuh) into its record piece (QPiece: codes, and the
// block scale bytes at the record's tail), stores it to every send slot, reads
// the piece back from each receiving partition's send record and stores it to
// that partition's pair records.  Records are rb = V * kCodePerVec +
// V / kVecPerScale bytes; padding records are zero.  g is the NVFP4 tensor
// scale.
template <int FMT>
__global__ void __launch_bounds__(kPPThreads) k_pack_permute_q(
    const int4 *__restrict__ x, const int32_t *__restrict__ token_slot,
    const int32_t *__restrict__ part_offsets, const int32_t *__restrict__ ids,
    const int32_t *__restrict__ expert_counts, const int32_t *__restrict__ expert_rank, int S,
    int64_t NT, int k, int E, int L, int P, int T, int V, int recv_part, int align, int cap_send,
    int cap_recv, float g, uint8_t *__restrict__ send_q, int32_t *__restrict__ send_src,
    uint8_t *__restrict__ recv_q, int32_t *__restrict__ expert_offsets,
    int32_t *__restrict__ pair_row, int32_t *__restrict__ recv_pair, uint32_t *dev_status,
    int stage)
{
    using QL = QLayout<FMT>;
    const int lane = threadIdx.x & 31;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t gwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t rb = (int64_t)V * QL::kCodePerVec + V / QL::kVecPerScale;
    const float d = __fmul_rn(6.0f, g);
    const int nseg = (V + kQSegVec - 1) / kQSegVec;
    bool cap_flag = false, bad_slot = false, dropped = false, bad_rank = false, bad_id = false;
    bool pack_overflow = false;

    extern __shared__ int smq[];
    int *off = smq;              // [E + 1]
    int *cnt = off + E + 1;      // [E]
    int *sb = cnt + E;           // [S][E]
    // [warp][stage][4 pieces][32 lanes]: x segments of this warp's tasks 0..stage-1
    int4 *stg = reinterpret_cast<int4 *>(smq + ((2 * E + 1 + S * E + 3) & ~3)) +
                (threadIdx.x >> 5) * stage * kPPSegVec;
    // Only moe_dispatch_quantized launches this kernel, right after the layout:
    // x is read before the grid-dependency wait as in k_pack_permute.
    const int64_t rt0 = gtid >> 5;
    int4 x0[kPPUnroll];
    stage_x<FMT, false>(x, NT * nseg, nseg, V, rt0, gwarps, stage, x0, stg);
    pdl_wait();
    pdl_trigger();
    build_run_starts(expert_counts, S, E, L, recv_part, align, off, cnt, sb, expert_offsets);
    cp_async_wait_all();

    const int64_t ntask = NT * nseg;
    int it = 0;
    for (int64_t rtask = rt0; rtask < ntask; rtask += gwarps, it++) {
        const int64_t task = ntask - 1 - rtask;       // tokens last to first
        const int64_t n = task / nseg;
        const int gs = (int)(task - n * nseg);
        const int s = (int)(n / T);
        int ts = -1, pr = -1, pp = -1;
        if (lane < P) ts = __ldg(token_slot + n * P + lane);
        if (lane < k) {
            const int e = __ldg(ids + n * k + lane);
            pr = pair_row_of(e, __ldg(expert_rank + n * k + lane), s, S, E, L, recv_part, cap_recv,
                             off, cnt, sb, bad_id, bad_rank, dropped);
            if (gs == 0) {
                const int64_t q = n * k + lane;
                pair_row[q] = pr;
                if (pr >= 0) recv_pair[pr] = (int32_t)q;
            }
            if (pr >= 0) pp = e / L;
        }
        if (gs == 0 && lane < P) {
            if (ts >= cap_send) pack_overflow = true;
            else if (ts >= 0) send_src[(int64_t)s * cap_send + ts] = (int32_t)(n - (int64_t)s * T);
        }
        // quantize the segment once (every lane takes part in the block shuffles)
        const int vb = gs * kQSegVec;
        int4 xs[kPPUnroll];
        if (!staged_x<false>(it, stage, x0, stg, xs)) {
#pragma unroll
            for (int u = 0; u < kPPUnroll; u++) {
                const int vi = piece_vec<FMT>(vb, u);
                xs[u] = (vi < V) ? ld_stream(x + n * V + vi) : make_int4(0, 0, 0, 0);
            }
        }
        const QPiece q = quantize_loaded<FMT>(xs, g, d);
        uint8_t *send_s = send_q + (int64_t)s * cap_send * rb;
        unsigned smask = __ballot_sync(kFull, lane < P && ts >= 0 && ts < cap_send);
        while (smask) {
            const int p = __ffs(smask) - 1;
            smask &= smask - 1;
            const int sl = __shfl_sync(kFull, ts, p);
            store_piece<FMT>(send_s + (int64_t)sl * rb, V, vb, q);
        }
        unsigned rmask = __ballot_sync(kFull, pr >= 0);
        while (rmask) {
            const int j0 = __ffs(rmask) - 1;
            const int p0 = __shfl_sync(kFull, pp, j0);
            const unsigned gmask = __ballot_sync(kFull, pr >= 0 && pp == p0);
            rmask &= ~gmask;
            const int sl = __shfl_sync(kFull, ts, p0);
            const bool ok = sl >= 0 && sl < cap_send;
            if (!ok && gs == 0 && lane == 0) {
                if (sl < 0) bad_slot = true;
                else cap_flag = true;
            }
            QPiece r;
            if (ok) {
                r = load_piece<FMT>(send_s + (int64_t)sl * rb, V, vb);
            } else {
                r.code[0] = r.code[1] = make_uint4(0u, 0u, 0u, 0u);
                r.sw = 0u;
            }
            unsigned dm = gmask;
            while (dm) {
                const int j = __ffs(dm) - 1;
                dm &= dm - 1;
                const int row = __shfl_sync(kFull, pr, j);
                store_piece<FMT>(recv_q + (int64_t)row * rb, V, vb, r);
            }
        }
    }

    // padding records: a warp per (expert, padding row), zeroed in 16-byte vectors
    if (align > 1) {
        const int rbv = (int)(rb / 16);
        const int64_t ptask = (int64_t)E * (align - 1);
        for (int64_t task = gtid >> 5; task < ptask; task += gwarps) {
            const int e = (int)(task / (align - 1));
            const int i = (int)(task - (int64_t)e * (align - 1));
            const int row = off[e] + cnt[e] + i;
            if (!in_recv(e, E, L, recv_part) || row >= off[e + 1] || row >= cap_recv) continue;
            int4 *dst = reinterpret_cast<int4 *>(recv_q + (int64_t)row * rb);
            for (int vi = lane; vi < rbv; vi += 32) st_cg(dst + vi, make_int4(0, 0, 0, 0));
            if (lane == 0) recv_pair[row] = -1;
        }
    }
    mark_unused_rows(off[E], cap_recv, S, P, cap_send, part_offsets, recv_pair, send_src);

    if (cap_flag || dropped || pack_overflow) flag_status(dev_status, MOE_ERR_CAPACITY);
    if (bad_slot || bad_rank) flag_status(dev_status, MOE_ERR_INVALID_ARG);
    if (bad_id) flag_status(dev_status, MOE_ERR_BAD_EXPERT_ID);
}

}  // namespace

int pack_permute_kernel_count(int S, int T, int E)
{
    if (T == 0) return 2;                    // the separate pack and permute
    return permute_map_fused(S, E) ? 1 : 3;  // else pack, map and copy
}

namespace {

// Shared memory per SM the staged kernels may take together (bytes, with the
// 1 KiB each CTA reserves): the SM's remaining 256 KiB - 164 KiB stay L1 for
// the kernel that follows under programmatic launch (the combine reads its
// pair rows and weights through L1; 64 KiB staged per CTA, 212 KiB per SM,
// made the 16,384-token step 12 us slower).
constexpr size_t kStageSmemPerSm = (size_t)164 * 1024;

// Staged tasks per warp for a one-pass kernel whose own shared memory is
// `base` bytes: as many (at most kPPStageMax) as fit beside the CTAs that its
// registers allow per SM within kStageSmemPerSm, none unless `want`.  Sets the
// kernel's dynamic shared memory limit when it stages.  resident: CTAs of the
// kernel that fit on the device with `base` bytes (the grid's cap either way).
template <typename Kern>
cudaError_t pick_stage(Kern kernel, size_t base, bool want, const DeviceInfo &di, int *stage,
                       size_t *smem, int *resident)
{
    *stage = 0;
    *smem = base;
    *resident = resident_grid((const void *)kernel, kPPThreads, base);
    if (!want || *resident <= 0) return cudaSuccess;
    const int per_sm = (*resident + di.sm_count - 1) / di.sm_count;
    // the opt-in limit covers static shared memory too (48 bytes here)
    const size_t max_dyn = (size_t)di.max_smem_optin - 1024;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_dyn);
    if (e != cudaSuccess) return e;
    const size_t base16 = (base + 15) / 16 * 16;
    for (int m = kPPStageMax; m >= 1; m--) {
        const size_t sm = base16 + (size_t)m * kPPStageBytes;
        if ((size_t)per_sm * (sm + 1024) > kStageSmemPerSm) continue;
        if (sm <= max_dyn && resident_grid((const void *)kernel, kPPThreads, sm) >= *resident) {
            *stage = m;
            *smem = sm;
            break;
        }
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_pack_permute(const uint16_t *x, const int32_t *token_slot,
                                const int32_t *part_offsets, const int32_t *topk_ids,
                                const int32_t *expert_counts, const int32_t *expert_rank, int S,
                                int T, int k, int E, int P, int H, int recv_part, int align,
                                int cap_send, int cap_recv, uint16_t *send, int32_t *send_src,
                                uint16_t *recv, int32_t *expert_offsets, int32_t *pair_row,
                                int32_t *recv_pair, void *ws, uint32_t *dev_status,
                                cudaStream_t st, bool x_before_wait)
{
    cudaError_t e;
    if (T == 0 || !permute_map_fused(S, E)) {
        // empty batch, or run starts too large for one CTA's shared memory:
        // the separate pack and permute
        if ((e = launch_dispatch_pack(x, S, T, H, P, token_slot, part_offsets, cap_send, send,
                                      send_src, dev_status, st)) != cudaSuccess)
            return e;
        return launch_permute(send, token_slot, topk_ids, expert_counts, expert_rank, S, T, k, E, P,
                              H, recv_part, align, cap_send, cap_recv, recv, expert_offsets,
                              pair_row, recv_pair, ws, dev_status, st);
    }
    DeviceInfo di;
    if ((e = device_info(&di)) != cudaSuccess) return e;
    const int64_t NT = (int64_t)S * T;
    const int V = H / 8;
    const int L = E / P;
    const int nseg = (V + kPPSegVec - 1) / kPPSegVec;
    const size_t base = (size_t)(2 * E + 1 + (int64_t)S * E) * sizeof(int);
    // Staged x segments, for one source only (measured on GB300, step through
    // moe_dispatch: 4,096-token prefill 139.8 -> 134.4 us with three tasks per
    // warp, 136.1 with two; four took 48 KB more shared memory per CTA and made
    // the 16,384-token step 12 us slower, the combine that follows it under
    // programmatic launch landing on SMs left with little L1; eight sources of
    // 4,096 tokens were 3.6 us slower with three tasks, so several sources
    // stage nothing).
    int stage = 0, resident = 0;
    size_t smem = base;
    if ((e = pick_stage(k_pack_permute, base, x_before_wait && S == 1, di, &stage, &smem,
                        &resident)) != cudaSuccess)
        return e;
    const int64_t wave = resident > 0 ? resident : (int64_t)di.sm_count * (2048 / kPPThreads);
    const int64_t warps = NT * nseg + (align > 1 ? (int64_t)E * (align - 1) * nseg : 0);
    int64_t blocks = div_up(warps, kPPThreads / 32);
    const int64_t tail = div_up((int64_t)cap_recv > (int64_t)S * cap_send ? cap_recv
                                                                          : (int64_t)S * cap_send,
                                kPPThreads);
    const int64_t tail_blocks = tail < di.sm_count ? tail : di.sm_count;
    if (blocks < tail_blocks) blocks = tail_blocks;
    if (blocks > wave) blocks = wave;
    if (blocks < 1) blocks = 1;
    MOE_TRACED_LAUNCH("k_pack_permute", st,
                      e = launch_pdl(k_pack_permute, dim3((unsigned)blocks), dim3(kPPThreads), smem,
                                     st, (const int4 *)x, token_slot, part_offsets, topk_ids,
                                     expert_counts, expert_rank, S, NT, k, E, L, P, T, V,
                                     recv_part, align, cap_send, cap_recv, (int4 *)send, send_src,
                                     (int4 *)recv, expert_offsets, pair_row, recv_pair,
                                     dev_status, x_before_wait, stage));
    return e;
}

cudaError_t dispatch_kernel_count(int S, int T, int k, int E, int P, int *n)
{
    bool small = false;
    cudaError_t e = dispatch_small_form(S, T, k, E, P, &small);
    if (e != cudaSuccess) return e;
    if (small) {
        *n = 1;
        return cudaSuccess;
    }
    int nl = 1;                             // an empty batch: one layout kernel
    if (T > 0 && (e = layout_kernel_count(T, k, E, P, &nl)) != cudaSuccess) return e;
    *n = (T > 0 ? 1 : 0) + nl + pack_permute_kernel_count(S, T, E);
    return cudaSuccess;
}

cudaError_t launch_dispatch(const float *logits, const uint16_t *x, int S, int T, int H, int E,
                            int k, int P, int recv_part, int align, int cap_send, int cap_recv,
                            int32_t *topk_ids, float *topk_w, int32_t *expert_counts,
                            int32_t *expert_rank, int32_t *part_counts, int32_t *part_offsets,
                            int32_t *token_slot, uint16_t *send, int32_t *send_src,
                            uint16_t *recv, int32_t *expert_offsets, int32_t *pair_row,
                            int32_t *recv_pair, void *ws, uint32_t *dev_status, cudaStream_t st)
{
    bool small = false;
    cudaError_t e = dispatch_small_form(S, T, k, E, P, &small);
    if (e != cudaSuccess) return e;
    if (small)
        return launch_dispatch_small(logits, x, T, H, E, k, P, recv_part, align, cap_send,
                                     cap_recv, topk_ids, topk_w, expert_counts, expert_rank,
                                     part_counts, part_offsets, token_slot, send, send_src, recv,
                                     expert_offsets, pair_row, recv_pair, dev_status, nullptr, 0,
                                     st);
    const int64_t NT = (int64_t)S * T;
    if ((e = launch_route_topk(logits, NT, E, k, topk_ids, topk_w, st)) != cudaSuccess) return e;
    if ((e = launch_dispatch_layout(topk_ids, S, T, k, E, P, expert_counts, expert_rank,
                                    part_counts, part_offsets, token_slot, ws, dev_status, st)) !=
        cudaSuccess)
        return e;
    return launch_pack_permute(x, token_slot, part_offsets, topk_ids, expert_counts, expert_rank,
                               S, T, k, E, P, H, recv_part, align, cap_send, cap_recv, send,
                               send_src, recv, expert_offsets, pair_row, recv_pair, ws, dev_status,
                               st, true);
}

namespace {
inline bool masked_fits(int S, int nb) { return (size_t)(2 + S) * nb * sizeof(int) <= 48 * 1024; }
}  // namespace

int pack_permute_masked_kernel_count(int S, int T, int E, int P, int recv_part)
{
    const int nb = recv_part < 0 ? E : E / P;
    if (T == 0) return 2;                       // the pack, then the masked map alone
    return masked_fits(S, nb) ? 1 : 3;          // else pack, map and copy
}

cudaError_t launch_pack_permute_masked(const uint16_t *x, const int32_t *token_slot,
                                       const int32_t *part_offsets, const int32_t *topk_ids,
                                       const int32_t *expert_counts, const int32_t *expert_rank,
                                       int S, int T, int k, int E, int P, int H, int recv_part,
                                       int block_rows, int cap_send, uint16_t *send,
                                       int32_t *send_src, uint16_t *recv, int32_t *masked_counts,
                                       int32_t *pair_row, int32_t *recv_pair,
                                       uint32_t *dev_status, cudaStream_t st, bool x_before_wait)
{
    cudaError_t e;
    const int L = E / P;
    const int nb = recv_part < 0 ? E : L;
    const int e0 = recv_part < 0 ? 0 : recv_part * L;
    if (T == 0 || !masked_fits(S, nb)) {
        if ((e = launch_dispatch_pack(x, S, T, H, P, token_slot, part_offsets, cap_send, send,
                                      send_src, dev_status, st)) != cudaSuccess)
            return e;
        return launch_permute_masked(send, token_slot, topk_ids, expert_counts, expert_rank, S, T, k,
                                     E, P, H, recv_part, block_rows, cap_send, recv, masked_counts,
                                     pair_row, recv_pair, dev_status, st);
    }
    DeviceInfo di;
    if ((e = device_info(&di)) != cudaSuccess) return e;
    const int64_t NT = (int64_t)S * T;
    const int V = H / 8;
    const int nseg = (V + kPPSegVec - 1) / kPPSegVec;
    const size_t base = (size_t)(2 + S) * nb * sizeof(int);
    // staged x segments as in k_pack_permute: one source, x read before the wait
    int stage = 0, resident = 0;
    size_t smem = base;
    if ((e = pick_stage(k_pack_permute_masked, base, x_before_wait && S == 1, di, &stage, &smem,
                        &resident)) != cudaSuccess)
        return e;
    const int64_t wave = resident > 0 ? resident : (int64_t)di.sm_count * (2048 / kPPThreads);
    int64_t blocks = div_up(NT * nseg, kPPThreads / 32);
    const int64_t rows = (int64_t)nb * block_rows;
    const int64_t big = rows > (int64_t)S * cap_send ? rows : (int64_t)S * cap_send;
    const int64_t tail = div_up(big, kPPThreads);
    const int64_t tail_blocks = tail < di.sm_count ? tail : di.sm_count;
    if (blocks < tail_blocks) blocks = tail_blocks;
    if (blocks > wave) blocks = wave;
    if (blocks < 1) blocks = 1;
    MOE_TRACED_LAUNCH("k_pack_permute_masked", st,
                      e = launch_pdl(k_pack_permute_masked, dim3((unsigned)blocks),
                                     dim3(kPPThreads), smem, st, (const int4 *)x, token_slot,
                                     part_offsets, topk_ids, expert_counts, expert_rank, S, NT, k,
                                     E, L, P, T, V, e0, nb, block_rows, cap_send, (int4 *)send,
                                     send_src, (int4 *)recv, masked_counts, pair_row, recv_pair,
                                     dev_status, x_before_wait, stage));
    return e;
}

int dispatch_masked_kernel_count(int S, int T, int k, int E, int P, int recv_part)
{
    bool small = false;
    if (dispatch_small_form(S, T, k, E, P, &small) != cudaSuccess) return -1;
    if (small) return 1;
    int nl = 1;                             // an empty batch: one layout kernel
    if (T > 0 && layout_kernel_count(T, k, E, P, &nl) != cudaSuccess) return -1;
    return (T > 0 ? 1 : 0) + nl + pack_permute_masked_kernel_count(S, T, E, P, recv_part);
}

cudaError_t launch_dispatch_masked(const float *logits, const uint16_t *x, int S, int T, int H,
                                   int E, int k, int P, int recv_part, int block_rows,
                                   int cap_send, int32_t *topk_ids, float *topk_w,
                                   int32_t *expert_counts, int32_t *expert_rank,
                                   int32_t *part_counts, int32_t *part_offsets,
                                   int32_t *token_slot, uint16_t *send, int32_t *send_src,
                                   uint16_t *recv, int32_t *masked_counts, int32_t *pair_row,
                                   int32_t *recv_pair, void *ws, uint32_t *dev_status,
                                   cudaStream_t st)
{
    bool small = false;
    cudaError_t e = dispatch_small_form(S, T, k, E, P, &small);
    if (e != cudaSuccess) return e;
    if (small) {
        const int nb = recv_part < 0 ? E : E / P;
        return launch_dispatch_small(logits, x, T, H, E, k, P, recv_part, 1, cap_send,
                                     nb * block_rows, topk_ids, topk_w, expert_counts,
                                     expert_rank, part_counts, part_offsets, token_slot, send,
                                     send_src, recv, nullptr, pair_row, recv_pair, dev_status,
                                     masked_counts, block_rows, st);
    }
    const int64_t NT = (int64_t)S * T;
    if ((e = launch_route_topk(logits, NT, E, k, topk_ids, topk_w, st)) != cudaSuccess) return e;
    if ((e = launch_dispatch_layout(topk_ids, S, T, k, E, P, expert_counts, expert_rank,
                                    part_counts, part_offsets, token_slot, ws, dev_status, st)) !=
        cudaSuccess)
        return e;
    return launch_pack_permute_masked(x, token_slot, part_offsets, topk_ids, expert_counts,
                                      expert_rank, S, T, k, E, P, H, recv_part, block_rows,
                                      cap_send, send, send_src, recv, masked_counts, pair_row,
                                      recv_pair, dev_status, st, true);
}

cudaError_t dispatch_quantized_kernel_count(int S, int T, int k, int E, int P, int *n)
{
    bool small = false;
    const cudaError_t es = dispatch_small_form(S, T, k, E, P, &small);
    if (es != cudaSuccess) return es;
    if (small) {                            // one launch (dispatch_small_q.cu)
        *n = 1;
        return cudaSuccess;
    }
    if (T == 0) {                           // layout, pack and permute of an empty batch
        *n = 3;
        return cudaSuccess;
    }
    int nl = 0;
    const cudaError_t e = layout_kernel_count(T, k, E, P, &nl);
    if (e != cudaSuccess) return e;
    *n = 1 + nl + (permute_map_fused(S, E) ? 1 : 3);
    return cudaSuccess;
}

cudaError_t launch_dispatch_quantized(const float *logits, const uint16_t *x, int S, int T, int H,
                                      int E, int k, int P, int format, float g, int recv_part,
                                      int align, int cap_send, int cap_recv, int32_t *topk_ids,
                                      float *topk_w, int32_t *expert_counts, int32_t *expert_rank,
                                      int32_t *part_counts, int32_t *part_offsets,
                                      int32_t *token_slot, uint8_t *send_q, int32_t *send_src,
                                      uint8_t *recv_q, int32_t *expert_offsets, int32_t *pair_row,
                                      int32_t *recv_pair, void *ws, uint32_t *dev_status,
                                      cudaStream_t st)
{
    bool small = false;
    cudaError_t e = dispatch_small_form(S, T, k, E, P, &small);
    if (e != cudaSuccess) return e;
    if (small)
        return launch_dispatch_small_q(logits, x, T, H, E, k, P, format, g, recv_part, align,
                                       cap_send, cap_recv, topk_ids, topk_w, expert_counts,
                                       expert_rank, part_counts, part_offsets, token_slot, send_q,
                                       send_src, recv_q, expert_offsets, pair_row, recv_pair,
                                       dev_status, st);
    const int64_t NT = (int64_t)S * T;
    if ((e = launch_route_topk(logits, NT, E, k, topk_ids, topk_w, st)) != cudaSuccess) return e;
    if ((e = launch_dispatch_layout(topk_ids, S, T, k, E, P, expert_counts, expert_rank,
                                    part_counts, part_offsets, token_slot, ws, dev_status, st)) !=
        cudaSuccess)
        return e;
    const int V = H / 8;
    const int64_t rb = format == kQFmtMxfp8 ? (int64_t)V * 8 + V / 4 : (int64_t)V * 4 + V / 2;
    if (T == 0 || !permute_map_fused(S, E)) {
        // empty batch, or run starts too large for one CTA's shared memory:
        // the separate quantized pack and the permute of records as opaque rows
        e = format == kQFmtMxfp8
                ? launch_dispatch_pack_mxfp8(x, S, T, H, P, token_slot, part_offsets, cap_send,
                                             send_q, send_src, dev_status, st)
                : launch_dispatch_pack_nvfp4(x, S, T, H, P, g, token_slot, part_offsets, cap_send,
                                             send_q, send_src, dev_status, st);
        if (e != cudaSuccess) return e;
        return launch_permute((const uint16_t *)send_q, token_slot, topk_ids, expert_counts,
                              expert_rank, S, T, k, E, P, (int)(rb / 2), recv_part, align,
                              cap_send, cap_recv, (uint16_t *)recv_q, expert_offsets, pair_row,
                              recv_pair, ws, dev_status, st);
    }
    DeviceInfo di;
    if ((e = device_info(&di)) != cudaSuccess) return e;
    const int L = E / P;
    const int nseg = (V + kQSegVec - 1) / kQSegVec;
    const size_t base = (size_t)(2 * E + 1 + (int64_t)S * E) * sizeof(int);
    // staged x segments as in k_pack_permute (one source)
    int stage = 0, resident = 0;
    size_t smem = base;
    e = format == kQFmtMxfp8 ? pick_stage(k_pack_permute_q<kQFmtMxfp8>, base, S == 1, di, &stage,
                                          &smem, &resident)
                             : pick_stage(k_pack_permute_q<kQFmtNvfp4>, base, S == 1, di, &stage,
                                          &smem, &resident);
    if (e != cudaSuccess) return e;
    const int64_t wave = resident > 0 ? resident : (int64_t)di.sm_count * (2048 / kPPThreads);
    const int64_t warps = NT * nseg + (align > 1 ? (int64_t)E * (align - 1) : 0);
    int64_t blocks = div_up(warps, kPPThreads / 32);
    const int64_t tail = div_up((int64_t)cap_recv > (int64_t)S * cap_send ? cap_recv
                                                                          : (int64_t)S * cap_send,
                                kPPThreads);
    const int64_t tail_blocks = tail < di.sm_count ? tail : di.sm_count;
    if (blocks < tail_blocks) blocks = tail_blocks;
    if (blocks > wave) blocks = wave;
    if (blocks < 1) blocks = 1;
    if (format == kQFmtMxfp8) {
        MOE_TRACED_LAUNCH("k_pack_permute_mxfp8", st,
                          e = launch_pdl(k_pack_permute_q<kQFmtMxfp8>, dim3((unsigned)blocks),
                                         dim3(kPPThreads), smem, st, (const int4 *)x, token_slot,
                                         (const int32_t *)part_offsets, (const int32_t *)topk_ids,
                                         (const int32_t *)expert_counts,
                                         (const int32_t *)expert_rank, S, NT, k, E, L, P, T, V,
                                         recv_part, align, cap_send, cap_recv, g, send_q, send_src,
                                         recv_q, expert_offsets, pair_row, recv_pair, dev_status,
                                         stage));
    } else {
        MOE_TRACED_LAUNCH("k_pack_permute_nvfp4", st,
                          e = launch_pdl(k_pack_permute_q<kQFmtNvfp4>, dim3((unsigned)blocks),
                                         dim3(kPPThreads), smem, st, (const int4 *)x, token_slot,
                                         (const int32_t *)part_offsets, (const int32_t *)topk_ids,
                                         (const int32_t *)expert_counts,
                                         (const int32_t *)expert_rank, S, NT, k, E, L, P, T, V,
                                         recv_part, align, cap_send, cap_recv, g, send_q, send_src,
                                         recv_q, expert_offsets, pair_row, recv_pair, dev_status,
                                         stage));
    }
    return e;
}

}  // namespace moe
