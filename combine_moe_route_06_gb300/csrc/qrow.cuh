// qrow.cuh -- one warp's piece of a quantized record (MXFP8 or NVFP4) for one
// 1,024-value row segment: quantize it once, store it to a record, load it
// back.  Shared by the quantized pack + permute pass and the one-launch
// quantized dispatch.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 7.2: rows
// are converted to a low-precision format before they are sent.  The record
// holds the codes at their value offset (one byte per MXFP8 value, one per
// pair of NVFP4 values) and all block scale bytes after the codes, as the
// quantized packs lay them out (quant.cuh holds the block arithmetic).
#pragma once

#include "common.cuh"
#include "quant.cuh"

namespace moe {

// 4-byte global accesses that bypass L1 (the read-back of a record piece the
// same thread has just stored is a real load, served from L2).
__device__ __forceinline__ void st_cg4(void *p, uint32_t v)
{
    asm volatile("st.global.cg.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_cg4(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

constexpr int kQFmtMxfp8 = 1;
constexpr int kQFmtNvfp4 = 2;
constexpr int kQSegVec = 128;                 // 16-byte x vectors (1,024 values) per segment

// One warp's piece of a record for one 1,024-value segment.  MXFP8: lane l
// owns values 16l + 512u (u = 0, 1) -> code[u], 16 E4M3 bytes each; lanes 0..7
// carry the segment's 32 scale bytes as words (lane j: pass j / 4, blocks
// 4 (j % 4) .. +3).  NVFP4: lane l owns values 32l .. 32l + 31 -> code[0], 16
// bytes of E2M1 pairs; lanes 0..15 carry the 64 scale bytes as words (lane j:
// blocks 4j .. 4j + 3).  The record holds codes at value offset / (1 or 2)
// and the scales after all codes, as the quantized packs lay them out.
struct QPiece {
    uint4 code[2];
    uint32_t sw;
};

template <int FMT> struct QLayout;
template <> struct QLayout<kQFmtMxfp8> {
    static constexpr int kCodePerVec = 8;      // code bytes per 16-byte x vector
    static constexpr int kVecPerScale = 4;     // x vectors per scale byte
    static constexpr int kScaleLanes = 8;
};
template <> struct QLayout<kQFmtNvfp4> {
    static constexpr int kCodePerVec = 4;
    static constexpr int kVecPerScale = 2;
    static constexpr int kScaleLanes = 16;
};

// x vector of this lane's i-th 16-byte piece (i < 4) of the segment that
// starts at vector vb: MXFP8 lanes take two adjacent vectors in each half of
// the segment, NVFP4 lanes four adjacent vectors.
template <int FMT>
__device__ __forceinline__ int piece_vec(int vb, int i)
{
    const int lane = threadIdx.x & 31;
    return FMT == kQFmtMxfp8 ? vb + 64 * (i >> 1) + 2 * lane + (i & 1) : vb + 4 * lane + i;
}

// Quantizes this lane's four pieces v (piece_vec order; zero past the row) of
// a segment (every lane of the warp must call).
template <int FMT>
__device__ __forceinline__ QPiece quantize_loaded(const int4 (&v)[4], float g, float d)
{
    const int lane = threadIdx.x & 31;
    QPiece q;
    q.sw = 0u;
    if (FMT == kQFmtMxfp8) {
        uint32_t sc[2];
#pragma unroll
        for (int u = 0; u < 2; u++) mxfp8_quantize16(v + 2 * u, q.code[u], sc[u]);
        const int w = lane & 3;
        uint32_t a = 0u, b = 0u;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            a |= __shfl_sync(kFull, sc[0], 8 * w + 2 * i) << (8 * i);
            b |= __shfl_sync(kFull, sc[1], 8 * w + 2 * i) << (8 * i);
        }
        q.sw = (lane < 4) ? a : b;
    } else {
        uint32_t sp;
        nvfp4_quantize32(v, g, d, q.code[0], sp);
        q.code[1] = make_uint4(0u, 0u, 0u, 0u);
        const int j = lane & 15;
        q.sw = __shfl_sync(kFull, sp, 2 * j) | (__shfl_sync(kFull, sp, 2 * j + 1) << 16);
    }
    return q;
}

// Quantizes the segment starting at vector vb of the token's row (every lane
// of the warp must call).
template <int FMT>
__device__ __forceinline__ QPiece quantize_piece(const int4 *__restrict__ row, int V, int vb,
                                                 float g, float d)
{
    int4 v[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int vi = piece_vec<FMT>(vb, i);
        v[i] = (vi < V) ? ld_stream(row + vi) : make_int4(0, 0, 0, 0);
    }
    return quantize_loaded<FMT>(v, g, d);
}

// Byte offsets of this lane's code vector(s) and scale word in a record, and
// whether they lie inside the row.
template <int FMT>
__device__ __forceinline__ bool code_at(int V, int vb, int u, int64_t &off)
{
    const int lane = threadIdx.x & 31;
    const int vi = (FMT == kQFmtMxfp8) ? vb + 64 * u + 2 * lane : vb + 4 * lane;
    off = (int64_t)vi * QLayout<FMT>::kCodePerVec;
    return vi < V;
}
template <int FMT>
__device__ __forceinline__ bool scale_at(int V, int vb, int64_t &off)
{
    using QL = QLayout<FMT>;
    const int lane = threadIdx.x & 31;
    if (lane >= QL::kScaleLanes) return false;
    // first x vector the word's four blocks cover, and the word's place
    const int v0 = (FMT == kQFmtMxfp8) ? vb + 64 * (lane >> 2) + 16 * (lane & 3) : vb + 8 * lane;
    off = (int64_t)V * QL::kCodePerVec + v0 / QL::kVecPerScale;
    return v0 < V;
}

template <int FMT>
__device__ __forceinline__ void store_piece(uint8_t *rec, int V, int vb, const QPiece &q)
{
    int64_t off;
#pragma unroll
    for (int u = 0; u < (FMT == kQFmtMxfp8 ? 2 : 1); u++)
        if (code_at<FMT>(V, vb, u, off))
            st_cg(reinterpret_cast<int4 *>(rec + off),
                  make_int4((int)q.code[u].x, (int)q.code[u].y, (int)q.code[u].z, (int)q.code[u].w));
    if (scale_at<FMT>(V, vb, off)) st_cg4(rec + off, q.sw);
}

template <int FMT>
__device__ __forceinline__ QPiece load_piece(const uint8_t *rec, int V, int vb)
{
    QPiece q;
    q.code[0] = q.code[1] = make_uint4(0u, 0u, 0u, 0u);
    q.sw = 0u;
    int64_t off;
#pragma unroll
    for (int u = 0; u < (FMT == kQFmtMxfp8 ? 2 : 1); u++)
        if (code_at<FMT>(V, vb, u, off)) {
            const int4 c = ld_cg(reinterpret_cast<const int4 *>(rec + off));
            q.code[u] = make_uint4((uint32_t)c.x, (uint32_t)c.y, (uint32_t)c.z, (uint32_t)c.w);
        }
    if (scale_at<FMT>(V, vb, off)) q.sw = ld_cg4(rec + off);
    return q;
}

}  // namespace moe
