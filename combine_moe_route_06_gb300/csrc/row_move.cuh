// row_move.cuh -- the row work of the one-pass dispatch kernels: one
// (token, column segment) task stores x's segment to the token's send rows and
// copies each receiving partition's send row to that partition's pair rows.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends): one copy of a row
// per partition that holds one of the token's experts, at its prefix-sum slot
// (sections 1.3, 3.2), and the receiver's expert-contiguous runs (sections
// 1.5, 3.3).  The read-back is the receiver reading the row that just landed
// in its receive region (on one GPU, partition p's region of the send buffer);
// the warp that landed it issues the read, so it is served from L2.
#pragma once

#include "common.cuh"

namespace moe {

// Stores the row segment r (U int4 per lane, vector v0 + 32u) at dst.
template <int U>
__device__ __forceinline__ void store_seg(int4 *dst, const int4 *r, int v0, int V)
{
#pragma unroll
    for (int u = 0; u < U; u++) {
        const int vi = v0 + 32 * u;
        if (vi < V) st_cg(dst + vi, r[u]);
    }
}

// The row work of one (token, column segment) task, shared by both forms.
//   ts    lane p < P: the token's slot in partition p (or -1)
//   pr    lane j < k: the pair's receive row (or -1); pp its partition
//   src   the token's row of x; send_s / recv: row bases
// `loaded`, if given, is the segment already in registers.
// Stores x's segment to every slot < cap_send, then, B partitions at a time,
// reads back the send row of each partition holding pairs and stores it to
// those pairs' rows.  A partition whose slot is missing (< 0, an inconsistent
// layout) or past cap_send gives its pairs zero rows, as the permute does.
template <int U, int B>
__device__ __forceinline__ void move_token_segment(const int4 *__restrict__ src, int4 *send_s,
                                                   int4 *recv, int V, int v0, int ts, int pr,
                                                   int pp, int P, int cap_send, bool &bad_slot,
                                                   bool &cap_flag, bool report,
                                                   const int4 *loaded = nullptr)
{
    int4 xr[U];
#pragma unroll
    for (int u = 0; u < U; u++) {
        const int vi = v0 + 32 * u;
        xr[u] = make_int4(0, 0, 0, 0);
        if (loaded) xr[u] = loaded[u];
        else if (vi < V) xr[u] = ld_stream(src + vi);
    }
    const int lane = threadIdx.x & 31;
    unsigned smask = __ballot_sync(kFull, lane < P && ts >= 0 && ts < cap_send);
    while (smask) {
        const int p = __ffs(smask) - 1;
        smask &= smask - 1;
        const int sl = __shfl_sync(kFull, ts, p);
        store_seg<U>(send_s + (int64_t)sl * V, xr, v0, V);
    }
    unsigned rmask = __ballot_sync(kFull, pr >= 0);
    while (rmask) {
        int4 rb[B][U];
        unsigned gm[B];
#pragma unroll
        for (int b = 0; b < B; b++) {
            gm[b] = 0u;
            if (rmask) {
                const int j0 = __ffs(rmask) - 1;
                const int p0 = __shfl_sync(kFull, pp, j0);
                const unsigned gmask = __ballot_sync(kFull, pr >= 0 && pp == p0);
                rmask &= ~gmask;
                gm[b] = gmask;
                const int sl = __shfl_sync(kFull, ts, p0);
                const bool ok = sl >= 0 && sl < cap_send;
                if (!ok && report && lane == 0) {
                    if (sl < 0) bad_slot = true;
                    else cap_flag = true;
                }
                const int4 *row = send_s + (int64_t)(ok ? sl : 0) * V;
#pragma unroll
                for (int u = 0; u < U; u++) {
                    const int vi = v0 + 32 * u;
                    rb[b][u] = make_int4(0, 0, 0, 0);
                    if (ok && vi < V) rb[b][u] = ld_stream(row + vi);
                }
            }
        }
#pragma unroll
        for (int b = 0; b < B; b++) {
            unsigned dm = gm[b];
            while (dm) {
                const int j = __ffs(dm) - 1;
                dm &= dm - 1;
                const int row = __shfl_sync(kFull, pr, j);
                store_seg<U>(recv + (int64_t)row * V, rb[b], v0, V);
            }
        }
    }
}

}  // namespace moe
