// route.cu -- top-k routing: router logits -> expert ids + renormalised weights.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 1.1: for
// every token the router produces the ids of the chosen experts and one weight
// per expert.  Chosen: the k largest logits, in descending order, equal logits
// resolved to the lower id.  Weights: softmax over the k chosen logits in fp32.
//
// One warp per token row.  Lane l holds logits l, l+32, l+64, ... in registers
// (coalesced 128-byte loads) and tracks its own two best; k rounds of a warp
// arg-max (value desc, id asc) pick the experts (one redux.sync max over
// order-preserving keys, one redux.sync min over the tied ids), and the
// winning lane promotes its second best, rescanning only when that is used up.
#include <float.h>
#include <limits.h>
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "trace.h"

namespace moe {

template <int VPL>
__global__ void __launch_bounds__(256) k_route_topk(const float *__restrict__ logits, int64_t N,
                                                    int E, int k, int32_t *__restrict__ ids,
                                                    float *__restrict__ w)
{
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (n >= N) return;  // uniform per warp
    const float *row = logits + n * E;

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
    if (lane < k) {
        ids[n * k + lane] = my_id;
        w[n * k + lane] = ex / sum;
    }
}

cudaError_t launch_route_topk(const float *logits, int64_t N, int E, int k, int32_t *ids,
                              float *w, cudaStream_t st)
{
    if (N == 0) return cudaSuccess;
    const int warps_per_block = 8;
    const unsigned blocks = (unsigned)((N + warps_per_block - 1) / warps_per_block);
    const int vpl = (E + 31) / 32;
#define MOE_ROUTE_CASE(V)                                                              \
    if (vpl <= V) {                                                                    \
        cudaError_t err;                                                               \
        MOE_TRACED_LAUNCH("k_route_topk", st,                                            \
            err = launch_pdl(k_route_topk<V>, dim3(blocks), dim3(warps_per_block * 32), 0, st, \
                             logits, N, E, k, ids, w));                                \
        return err;                                                                    \
    }
    MOE_ROUTE_CASE(1)
    MOE_ROUTE_CASE(2)
    MOE_ROUTE_CASE(4)
    MOE_ROUTE_CASE(8)
    MOE_ROUTE_CASE(12)
    MOE_ROUTE_CASE(16)
    MOE_ROUTE_CASE(24)
    MOE_ROUTE_CASE(32)
#undef MOE_ROUTE_CASE
    return cudaErrorInvalidValue;
}

}  // namespace moe
