// quant.cuh -- one 16-byte vector of bf16 values quantized into an MXFP8 or
// NVFP4 record piece (device functions shared by the quantized pack and the
// quantized pack + permute, so both write the same bytes).
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 7.2: rows
// are converted before they are sent; an FP8 row of 5,120 values is 5,280
// bytes (one scale byte per 32 values), an NVFP4 row 2,880 bytes (one per 16).
#pragma once

#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

// E8M0 exponent of an MXFP8 block whose largest magnitude is amax:
// floor(log2 amax) - 8 (the largest E4M3 binade), clamped to [-127, 127];
// -127 for an all-zero block.
__device__ __forceinline__ int mx_shared_exp(float amax)
{
    if (amax == 0.f) return -127;
    const unsigned bits = __float_as_uint(amax);
    const int field = (int)((bits >> 23) & 0xFFu);
    const int e = field ? field - 127 : (31 - __clz((int)(bits & 0x7FFFFFu))) - 149;
    const int se = e - 8;
    return se < -127 ? -127 : (se > 127 ? 127 : se);
}

// MXFP8: lanes 4b .. 4b+3 hold the 32 values of one block (8 each, `v`); every
// lane of the warp must call.  Returns this lane's 8 E4M3 codes (the pair's
// first value in the low byte of each 16 bits) and the block's E8M0 scale
// byte X = 2^(scale - 127): code = e4m3_rn_satfinite(value / X).  Finite
// inputs give se <= 120, so the 2^-se factor is a normal float.
__device__ __forceinline__ void mxfp8_quantize(int4 v, uint2 &code, uint8_t &scale)
{
    const uint32_t w4[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
    float f[8];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        f[2 * i] = __uint_as_float(w4[i] << 16);
        f[2 * i + 1] = __uint_as_float(w4[i] & 0xffff0000u);
        amax = fmaxf(amax, fmaxf(fabsf(f[2 * i]), fabsf(f[2 * i + 1])));
    }
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    const int se = mx_shared_exp(amax);
    const float inv = __uint_as_float((uint32_t)(127 - se) << 23);   // 2^-se, exact
    // two values per conversion (round to nearest even, saturate to finite)
    uint32_t c2[4];
#pragma unroll
    for (int i = 0; i < 4; i++)
        c2[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(f[2 * i] * inv, f[2 * i + 1] * inv),
                                                   __NV_SATFINITE, __NV_E4M3);
    code = make_uint2(c2[0] | (c2[1] << 16), c2[2] | (c2[3] << 16));
    scale = (uint8_t)(se + 127);
}

// NVFP4: lanes 2b, 2b+1 hold the 16 values of one block (8 each); every lane
// of the warp must call.  g is the per-tensor scale and d = fp32(6 g).  Block
// scale s = e4m3(amax / d), code = e2m1_rn_satfinite(value / (s g)) (0 if
// s g = 0), in fp32 with correctly rounded division; element 2i of the lane's
// 8 values lands in the low nibble of byte i.
__device__ __forceinline__ void nvfp4_quantize(int4 v, float g, float d, uint32_t &code,
                                               uint8_t &scale)
{
    const uint32_t w4[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
    float f[8];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        f[2 * i] = __uint_as_float(w4[i] << 16);
        f[2 * i + 1] = __uint_as_float(w4[i] & 0xffff0000u);
        amax = fmaxf(amax, fmaxf(fabsf(f[2 * i]), fabsf(f[2 * i + 1])));
    }
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    const __nv_fp8_storage_t sb = __nv_cvt_float_to_fp8(__fdiv_rn(amax, d), __NV_SATFINITE,
                                                        __NV_E4M3);
    const __half_raw sh = __nv_cvt_fp8_to_halfraw(sb, __NV_E4M3);
    const float sg = __fmul_rn(__half2float(*reinterpret_cast<const __half *>(&sh)), g);
    uint32_t c = 0;
    if (sg != 0.f) {
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const float2 q = make_float2(__fdiv_rn(f[2 * i], sg), __fdiv_rn(f[2 * i + 1], sg));
            c |= (uint32_t)__nv_cvt_float2_to_fp4x2(q, __NV_E2M1, cudaRoundNearest) << (8 * i);
        }
    }
    code = c;
    scale = (uint8_t)sb;
}

}  // namespace moe

namespace moe {

// Wider lane mappings for passes that store one record piece to several
// places: each lane produces 16 contiguous code bytes (one 16-byte store per
// destination) and the block scales travel as packed 32-bit words.  Same block
// arithmetic as mxfp8_quantize / nvfp4_quantize, so the same bytes.

// MXFP8, 16 values per lane (`v[0..1]`, consecutive): lanes 2b, 2b+1 hold one
// 32-value block; every lane of the warp must call.  code = the 16 E4M3 bytes
// in value order; scale = the block's E8M0 byte.
__device__ __forceinline__ void mxfp8_quantize16(const int4 *v, uint4 &code, uint32_t &scale)
{
    float f[16];
    float amax = 0.f;
#pragma unroll
    for (int h = 0; h < 2; h++) {
        const uint32_t w4[4] = {(uint32_t)v[h].x, (uint32_t)v[h].y, (uint32_t)v[h].z,
                                (uint32_t)v[h].w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            f[8 * h + 2 * i] = __uint_as_float(w4[i] << 16);
            f[8 * h + 2 * i + 1] = __uint_as_float(w4[i] & 0xffff0000u);
            amax = fmaxf(amax, fmaxf(fabsf(f[8 * h + 2 * i]), fabsf(f[8 * h + 2 * i + 1])));
        }
    }
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    const int se = mx_shared_exp(amax);
    const float inv = __uint_as_float((uint32_t)(127 - se) << 23);   // 2^-se, exact
    uint32_t c2[8];
#pragma unroll
    for (int i = 0; i < 8; i++)
        c2[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(f[2 * i] * inv, f[2 * i + 1] * inv),
                                                   __NV_SATFINITE, __NV_E4M3);
    code = make_uint4(c2[0] | (c2[1] << 16), c2[2] | (c2[3] << 16), c2[4] | (c2[5] << 16),
                      c2[6] | (c2[7] << 16));
    scale = (uint32_t)(se + 127);
}

// NVFP4, 32 values per lane (`v[0..3]`, consecutive) = two 16-value blocks,
// lane-local.  code = the 16 code bytes (value 2i in the low nibble of byte
// i); scales = the two E4M3 block scale bytes (first block in the low byte).
__device__ __forceinline__ void nvfp4_quantize32(const int4 *v, float g, float d, uint4 &code,
                                                 uint32_t &scales)
{
    uint32_t cw[4];
    scales = 0u;
#pragma unroll
    for (int b = 0; b < 2; b++) {
        float f[16];
        float amax = 0.f;
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int4 q = v[2 * b + h];
            const uint32_t w4[4] = {(uint32_t)q.x, (uint32_t)q.y, (uint32_t)q.z, (uint32_t)q.w};
#pragma unroll
            for (int i = 0; i < 4; i++) {
                f[8 * h + 2 * i] = __uint_as_float(w4[i] << 16);
                f[8 * h + 2 * i + 1] = __uint_as_float(w4[i] & 0xffff0000u);
                amax = fmaxf(amax, fmaxf(fabsf(f[8 * h + 2 * i]), fabsf(f[8 * h + 2 * i + 1])));
            }
        }
        const __nv_fp8_storage_t sb = __nv_cvt_float_to_fp8(__fdiv_rn(amax, d), __NV_SATFINITE,
                                                            __NV_E4M3);
        const __half_raw sh = __nv_cvt_fp8_to_halfraw(sb, __NV_E4M3);
        const float sg = __fmul_rn(__half2float(*reinterpret_cast<const __half *>(&sh)), g);
#pragma unroll
        for (int h = 0; h < 2; h++) {
            uint32_t c = 0;
            if (sg != 0.f) {
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const float2 q = make_float2(__fdiv_rn(f[8 * h + 2 * i], sg),
                                                 __fdiv_rn(f[8 * h + 2 * i + 1], sg));
                    c |= (uint32_t)__nv_cvt_float2_to_fp4x2(q, __NV_E2M1, cudaRoundNearest)
                         << (8 * i);
                }
            }
            cw[2 * b + h] = c;
        }
        scales |= (uint32_t)sb << (8 * b);
    }
    code = make_uint4(cw[0], cw[1], cw[2], cw[3]);
}

}  // namespace moe
