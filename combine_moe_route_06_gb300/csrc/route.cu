// route.cu -- top-k routing: router logits -> expert ids + renormalised weights.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 1.1: for
// every token the router produces the ids of the chosen experts and one weight
// per expert.  Chosen: the k largest logits, in descending order, equal logits
// resolved to the lower id.  Weights: softmax over the k chosen logits in fp32.
//
// One warp per token row (route_token_warp in route_warp.cuh: every lane keeps
// its two best logits, k rounds of a warp arg-max pick the experts).
#include "common.cuh"
#include "launch.h"
#include "route_warp.cuh"
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
    int id;
    float wt;
    route_token_warp<VPL>(logits + n * E, E, k, id, wt);
    if (lane < k) {
        ids[n * k + lane] = id;
        w[n * k + lane] = wt;
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
