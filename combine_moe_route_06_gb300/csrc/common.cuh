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

__device__ __forceinline__ int warp_sum(int v)
{
#pragma unroll
    for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    return v;
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

}  // namespace moe
