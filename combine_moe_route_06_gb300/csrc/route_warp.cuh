// route_warp.cuh -- top-k routing of one token by one warp (device function).
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 1.1: for
// every token the router produces the ids of the chosen experts and one weight
// per expert.  Chosen: the k largest logits, in descending order, equal logits
// resolved to the lower id.  Weights: softmax over the k chosen logits in fp32.
//
// Lane l holds logits l, l+32, l+64, ... in registers (coalesced 128-byte
// loads) and tracks its own two best; k rounds of a warp arg-max (value desc,
// id asc) pick the experts (one redux.sync max over order-preserving keys, one
// redux.sync min over the tied ids), and the winning lane promotes its second
// best, rescanning only when that is used up.  Both the routing kernel and the
// one-launch dispatch call this function, so their ids and weights are the
// same bits.
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe {

// Routes the token whose E logits start at `row`.  On return lane j < k holds
// choice j (id, weight); other lanes hold id -1, weight 0.  The whole warp
// must call it.
template <int VPL>
__device__ __forceinline__ void route_token_warp(const float *__restrict__ row, int E, int k,
                                                 int &out_id, float &out_w)
{
    const int lane = threadIdx.x & 31;
    // order-preserving keys; 0 marks "out of range"
    unsigned key[VPL];
#pragma unroll
    for (int i = 0; i < VPL; i++) {
        const int e = lane + 32 * i;
        key[i] = (e < E) ? float_key(__ldcs(row + e)) : 0u;
    }

    // This lane's two best live elements, ordered by (key desc, index asc): a
    // strict comparison while i ascends keeps the lower index first on ties.
    // A lane whose best is chosen promotes its second; only a lane chosen a
    // third time rescans its remaining elements (retired ones are in rmask).
    unsigned k1 = 0, k2 = 0, rmask = 0;
    int i1 = 0, i2 = 0;
    bool have2 = true;
#pragma unroll
    for (int i = 0; i < VPL; i++) {
        const unsigned v = key[i];
        if (v > k1) {
            k2 = k1;
            i2 = i1;
            k1 = v;
            i1 = i;
        } else if (v > k2) {
            k2 = v;
            i2 = i;
        }
    }

    unsigned my_key = 0;
    int my_id = -1;
    for (int r = 0; r < k; r++) {
        // warp arg-max: largest key, then the lowest id holding it
        const unsigned mx = __reduce_max_sync(kFull, k1);
        const unsigned cand = (k1 == mx) ? (unsigned)(lane + 32 * i1) : 0xffffffffu;
        const unsigned win = __reduce_min_sync(kFull, cand);
        if (lane == r) {
            my_key = mx;
            my_id = (int)win;
        }
        bool rescan = false;
        if ((int)(win & 31u) == lane) {
            rmask |= 1u << i1;
            if (have2) {
                k1 = k2;
                i1 = i2;
                have2 = false;
            } else {
                rescan = true;
            }
        }
        if (__any_sync(kFull, rescan) && rescan) {
            k1 = 0;
            k2 = 0;
            i1 = 0;
            i2 = 0;
#pragma unroll
            for (int i = 0; i < VPL; i++) {
                const unsigned v = ((rmask >> i) & 1u) ? 0u : key[i];
                if (v > k1) {
                    k2 = k1;
                    i2 = i1;
                    k1 = v;
                    i1 = i;
                } else if (v > k2) {
                    k2 = v;
                    i2 = i;
                }
            }
            have2 = true;
        }
    }

    // softmax over the k chosen logits: lane j < k holds choice j
    const float my_v = key_float(my_key);
    const float lmax = __shfl_sync(kFull, my_v, 0);
    const float ex = (lane < k) ? expf(my_v - lmax) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    out_id = (lane < k) ? my_id : -1;
    out_w = (lane < k) ? ex / sum : 0.f;
}

}  // namespace moe
