// common.cuh -- device helpers shared by the kernels of libmoeroute.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_route.h"

namespace moe {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kMaxP = 32;

// Tokens per CTA in the counting/ranking kernels of layout and permute.
constexpr int kChunk = 256;
constexpr int kChunkWarps = kChunk / 32;

__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ int warp_inclusive_scan(int v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(kFull, v, off);
        if (lane >= off) v += o;
    }
    return v;
}

// Whether expert e (of E, L per partition) is held by the receiving set:
// partition recv_part, or every partition when recv_part < 0.
__device__ __forceinline__ bool in_recv(int e, int E, int L, int recv_part)
{
    return e >= 0 && e < E && (recv_part < 0 || e / L == recv_part);
}

// Exclusive scan of n <= 1024 values in shared memory by a 256-thread CTA;
// returns the total.  `a` is overwritten with the exclusive prefix.
__device__ __forceinline__ int block_exclusive_scan_1024(int *a, int n)
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

// Set a status bit (MOE_STATUS_BIT(code)) in the caller's word.
__device__ __forceinline__ void flag_status(uint32_t *dev_status, int code)
{
    if (dev_status) atomicOr(dev_status, MOE_STATUS_BIT(code));
}

// 16-byte global accesses with explicit cache policy.
// Read-once streams: evict-first in L2, no L1 allocation.
__device__ __forceinline__ int4 ld_stream(const int4 *p)
{
    int4 v;
    asm volatile("ld.global.cs.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ld_stream(const uint2 *p)
{
    uint2 v;
    asm volatile("ld.global.cs.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
// Intermediate buffers that the next kernel reads: keep in L2 (cache global).
__device__ __forceinline__ int4 ld_cg(const int4 *p)
{
    int4 v;
    asm volatile("ld.global.cg.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void st_cg(int4 *p, int4 v)
{
    asm volatile("st.global.cg.v4.s32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}
// Final outputs: streaming store.
__device__ __forceinline__ void st_stream(int4 *p, int4 v)
{
    asm volatile("st.global.cs.v4.s32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Programmatic dependent launch (sm_90+): a kernel launched with
// launch_pdl() may start while the previous kernel of the stream drains; it
// must call pdl_wait() before touching memory that earlier work reads or
// writes.  pdl_trigger() lets the next kernel's CTAs be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;"); }

// Float -> uint32 key with the same order (-0.0 is folded onto +0.0, so equal
// floats give equal keys).  Key 0 never comes from a finite float.
__device__ __forceinline__ unsigned float_key(float v)
{
    const unsigned u = __float_as_uint(v == 0.f ? 0.f : v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(unsigned k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

}  // namespace moe

#ifndef __CUDACC_RTC__
#include <utility>
namespace moe {
// Launch with programmatic stream serialization allowed (see pdl_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_pdl with the grid split into thread-block clusters of `cluster_x` CTAs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      unsigned cluster_x, cudaStream_t st, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
}  // namespace moe
#endif
