// combine.cu -- weighted combine back to token order, and the stand-in expert.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 1.1 (the MoE
// output of a token is the sum of its experts' outputs, each multiplied by its
// router weight), section 7.1 (the home GPU adds the returned rows in 32-bit
// floats) and section 7.2 (combine travels as bf16).
//
// One warp per (token, 1 KiB column segment): the lanes gather the segment of
// each of the token's k expert rows (up to 8 rows, 16 loads of 16 bytes per
// lane in flight), accumulate weight * value with fp32 FMAs in j order, round
// once to bf16 and stream the result out.
#include <cuda_bf16.h>

#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"
#include "trace.h"

namespace moe {

namespace {

constexpr int kCombUnroll = 2;                  // int4 (8 bf16) per lane per segment
constexpr int kCombSegVec = 32 * kCombUnroll;   // int4 per segment (1 KiB)
constexpr int kCombBatch = 8;                   // rows whose loads are issued together
constexpr int kCombThreads = 256;
// The stage kernels read one or a few rows per warp task, so they take wider
// segments (2 KiB) and smaller batches than k_combine to keep enough bytes in
// flight at the occupancy their registers allow.
constexpr int kStageUnroll = 4;
constexpr int kRoutedUnroll = 8;
constexpr int kStageBatch = 2;
constexpr int kStage2Unroll = 2;
constexpr int kStage2Batch = 8;

__device__ __forceinline__ void fma_bf16x8(float *acc, int4 v, float w)
{
    const uint32_t u[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float lo = __uint_as_float(u[i] << 16);
        const float hi = __uint_as_float(u[i] & 0xffff0000u);
        acc[2 * i] = fmaf(w, lo, acc[2 * i]);
        acc[2 * i + 1] = fmaf(w, hi, acc[2 * i + 1]);
    }
}

__device__ __forceinline__ int4 pack_bf16x8(const float *a)
{
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
        u[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_int4((int)u[0], (int)u[1], (int)u[2], (int)u[3]);
}

__global__ void __launch_bounds__(kCombThreads) k_combine(const int4 *__restrict__ y, int y_rows,
                                                          const int32_t *__restrict__ pair_row,
                                                          const float *__restrict__ w,
                                                          int64_t N, int k, int V,
                                                          int4 *__restrict__ out,
                                                          uint32_t *dev_status)
{
    pdl_wait();
    pdl_trigger();
    bool bad_row = false;
    const int lane = threadIdx.x & 31;
    const int64_t gwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nseg = (V + kCombSegVec - 1) / kCombSegVec;
    const int64_t ntask = N * nseg;
    const bool narrow = ntask <= 0xffffffffll;  // task indices fit a 32-bit division
    for (int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < ntask;
         task += gwarps) {
        const int64_t n = narrow ? (int64_t)((uint32_t)task / (uint32_t)nseg) : task / nseg;
        const int g = (int)(task - n * nseg);
        int pr = -1;
        float wj = 0.f;
        if (lane < k) {
            pr = __ldg(pair_row + n * k + lane);
            wj = __ldg(w + n * k + lane);
            if (pr >= y_rows) {
                if (g == 0) bad_row = true;
                pr = -1;
            }
        }
        unsigned vmask = __ballot_sync(kFull, pr >= 0);
        const int v0 = g * kCombSegVec + lane;
        float acc[8 * kCombUnroll];
#pragma unroll
        for (int i = 0; i < 8 * kCombUnroll; i++) acc[i] = 0.f;

        while (vmask) {
            // issue the loads of up to kCombBatch rows, then accumulate in j order
            int4 r[kCombBatch][kCombUnroll];
            float wb[kCombBatch];
            int nb = 0;
#pragma unroll
            for (int b = 0; b < kCombBatch; b++) {
                if (vmask) {
                    const int j = __ffs(vmask) - 1;
                    vmask &= vmask - 1;
                    const int row = __shfl_sync(kFull, pr, j);
                    wb[b] = __shfl_sync(kFull, wj, j);
                    const int4 *src = y + (int64_t)row * V;
#pragma unroll
                    for (int u = 0; u < kCombUnroll; u++) {
                        const int vi = v0 + 32 * u;
                        r[b][u] = (vi < V) ? ld_stream(src + vi) : make_int4(0, 0, 0, 0);
                    }
                    nb = b + 1;
                }
            }
#pragma unroll
            for (int b = 0; b < kCombBatch; b++) {
                if (b < nb) {
#pragma unroll
                    for (int u = 0; u < kCombUnroll; u++) fma_bf16x8(acc + 8 * u, r[b][u], wb[b]);
                }
            }
        }
        int4 *dst = out + n * V;
#pragma unroll
        for (int u = 0; u < kCombUnroll; u++) {
            const int vi = v0 + 32 * u;
            if (vi < V) st_stream(dst + vi, pack_bf16x8(acc + 8 * u));
        }
    }
    if (bad_row) flag_status(dev_status, MOE_ERR_INVALID_ARG);
}

// Stage 1 of the split combine (a2a-backends section 7.1): one warp per
// (token, 1 KiB segment); for every partition of the receiving set that holds
// a send slot of the token, the weighted sum of the token's experts in that
// partition (fp32 FMAs in j order) is rounded once to bf16 and written to the
// slot's row of `ret` (send layout: the rows travel back the way they came).
template <int U, int B>
__global__ void __launch_bounds__(kCombThreads) k_combine_stage1(
    const int4 *__restrict__ y, int y_rows, const int32_t *__restrict__ pair_row,
    const float *__restrict__ w, const int32_t *__restrict__ ids,
    const int32_t *__restrict__ token_slot, int64_t N, int T, int k, int E, int L, int P, int V,
    int recv_part, int cap_send, int4 *__restrict__ ret, uint32_t *dev_status)
{
    pdl_wait();
    pdl_trigger();
    bool bad_row = false, cap_flag = false;
    const int lane = threadIdx.x & 31;
    const int64_t gwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nseg = (V + (32 * U) - 1) / (32 * U);
    const int64_t ntask = N * nseg;
    for (int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < ntask;
         task += gwarps) {
        const int64_t n = task / nseg;
        const int g = (int)(task - n * nseg);
        const int s = (int)(n / T);
        int pr = -1, pj = -1, slot = -1;
        float wj = 0.f;
        if (lane < k) {
            pr = __ldg(pair_row + n * k + lane);
            wj = __ldg(w + n * k + lane);
            const int e = __ldg(ids + n * k + lane);
            if (e >= 0 && e < E) pj = e / L;
            if (pr >= y_rows) {
                if (g == 0) bad_row = true;
                pr = -1;
            }
        }
        bool in_r = false;
        if (lane < P) {
            slot = __ldg(token_slot + n * P + lane);
            in_r = (recv_part < 0 || lane == recv_part) && slot >= 0;
            if (in_r && slot >= cap_send) {
                if (g == 0) cap_flag = true;
                in_r = false;
            }
        }
        unsigned smask = __ballot_sync(kFull, in_r);
        const int v0 = g * (32 * U) + lane;
        while (smask) {
            const int p0 = __ffs(smask) - 1;
            smask &= smask - 1;
            const int slot0 = __shfl_sync(kFull, slot, p0);
            unsigned jmask = __ballot_sync(kFull, pr >= 0 && pj == p0);
            float acc[8 * U];
#pragma unroll
            for (int i = 0; i < 8 * U; i++) acc[i] = 0.f;
            while (jmask) {
                int4 r[B][U];
                float wb[B];
                int nb = 0;
#pragma unroll
                for (int b = 0; b < B; b++) {
                    if (jmask) {
                        const int j = __ffs(jmask) - 1;
                        jmask &= jmask - 1;
                        const int row = __shfl_sync(kFull, pr, j);
                        wb[b] = __shfl_sync(kFull, wj, j);
                        const int4 *src = y + (int64_t)row * V;
#pragma unroll
                        for (int u = 0; u < U; u++) {
                            const int vi = v0 + 32 * u;
                            r[b][u] = (vi < V) ? ld_stream(src + vi) : make_int4(0, 0, 0, 0);
                        }
                        nb = b + 1;
                    }
                }
#pragma unroll
                for (int b = 0; b < B; b++) {
                    if (b < nb) {
#pragma unroll
                        for (int u = 0; u < U; u++) fma_bf16x8(acc + 8 * u, r[b][u], wb[b]);
                    }
                }
            }
            int4 *dst = ret + ((int64_t)s * cap_send + slot0) * V;
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int vi = v0 + 32 * u;
                if (vi < V) st_cg(dst + vi, pack_bf16x8(acc + 8 * u));
            }
        }
    }
    if (bad_row) flag_status(dev_status, MOE_ERR_INVALID_ARG);
    if (cap_flag) flag_status(dev_status, MOE_ERR_CAPACITY);
}

// Routed expert with the stage-1 pre-add (a2a-backends section 6.1: the rows
// arrive in sender order with their routing and a routed expert kernel picks
// its experts from the ids; section 7.1: it already produces the weighted sum
// per GPU).  Stand-in expert y_j = bf16(x * scale[e_j]) (x itself when scale
// is null).  One warp per (send row, 1 KiB segment): the row is read once and
// each of its experts on the row's partition adds w_j * y_j in ascending j
// with fp32 FMAs -- the same operations, in the same order, as the stand-in
// expert followed by k_combine_stage1, so the two paths give the same bytes.
template <int U, bool SCALED>
__global__ void __launch_bounds__(kCombThreads) k_routed_stage1(
    const int4 *__restrict__ send, const int32_t *__restrict__ send_ids,
    const float *__restrict__ send_w, const int32_t *__restrict__ part_offsets, int S,
    int cap_send, int span, int k, int E, int L, int P, int V, int recv_part,
    const float *__restrict__ scale, int4 *__restrict__ ret, uint32_t *dev_status)
{
    pdl_wait();
    pdl_trigger();
    bool bad_id = false;
    const int lane = threadIdx.x & 31;
    const int64_t gwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nseg = (V + (32 * U) - 1) / (32 * U);
    // Tasks: (source, i, segment) for i < span.  With one receiving partition
    // i indexes that partition's region of the source (span = at most T rows);
    // otherwise i is the send row itself (span = cap_send).
    const int64_t ntask = (int64_t)S * span * nseg;
    for (int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < ntask;
         task += gwarps) {
        const int64_t q = task / nseg;
        const int g = (int)(task - q * nseg);
        const int s = (int)(q / span);
        const int i = (int)(q - (int64_t)s * span);
        const int32_t *po = part_offsets + (int64_t)s * (P + 1);
        int r, p;
        if (recv_part >= 0) {
            r = __ldg(po + recv_part) + i;
            if (r >= __ldg(po + recv_part + 1) || r >= cap_send) continue;
            p = recv_part;
        } else {
            // partition of the row: the number of region ends at or below it
            r = i;
            const int end = lane < P ? __ldg(po + lane + 1) : 0x7fffffff;
            p = __popc(__ballot_sync(kFull, end <= r));
            if (p >= P) continue;                                   // empty row
        }
        const int64_t row = (int64_t)s * cap_send + r;
        int e = -1;
        float wj = 0.f, sj = 1.f;
        if (lane < k) {
            e = __ldg(send_ids + row * k + lane);
            wj = __ldg(send_w + row * k + lane);
            if (e >= E && g == 0) bad_id = true;
            if (e >= 0 && e < E && e / L == p) {
                if (SCALED) sj = __ldg(scale + e);
            } else {
                e = -1;
            }
        }
        unsigned jmask = __ballot_sync(kFull, e >= 0);
        const int v0 = g * (32 * U) + lane;
        int4 x[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int vi = v0 + 32 * u;
            x[u] = (vi < V && jmask) ? ld_stream(send + row * V + vi) : make_int4(0, 0, 0, 0);
        }
        // column-outer: each 16-byte column is finished over all the row's experts
        // before the next, so only 8 accumulators are live (the per-element order
        // of the sum over j is unchanged)
#pragma unroll
        for (int u = 0; u < U; u++) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; i++) acc[i] = 0.f;
            for (unsigned m = jmask; m; m &= m - 1) {
                const int j = __ffs(m) - 1;
                const float wb = __shfl_sync(kFull, wj, j);
                int4 y = x[u];
                if (SCALED) {
                    const float sb = __shfl_sync(kFull, sj, j);
                    float a[8];
                    const uint32_t uu[4] = {(uint32_t)y.x, (uint32_t)y.y, (uint32_t)y.z, (uint32_t)y.w};
#pragma unroll
                    for (int i = 0; i < 4; i++) {
                        a[2 * i] = __uint_as_float(uu[i] << 16) * sb;
                        a[2 * i + 1] = __uint_as_float(uu[i] & 0xffff0000u) * sb;
                    }
                    y = pack_bf16x8(a);
                }
                fma_bf16x8(acc, y, wb);
            }
            const int vi = v0 + 32 * u;
            if (vi < V) st_cg(ret + row * V + vi, pack_bf16x8(acc));
        }
    }
    if (bad_id) flag_status(dev_status, MOE_ERR_BAD_EXPERT_ID);
}

// Stage 2: one warp per (token, 1 KiB segment); the token's returned rows (one
// per send slot, partitions in ascending order) summed with fp32 adds, one bf16
// rounding.
template <int U, int B>
__global__ void __launch_bounds__(kCombThreads) k_combine_stage2(
    const int4 *__restrict__ ret, const int32_t *__restrict__ token_slot, int64_t N, int T,
    int P, int V, int recv_part, int cap_send, int4 *__restrict__ out, uint32_t *dev_status)
{
    pdl_wait();
    pdl_trigger();
    bool cap_flag = false;
    const int lane = threadIdx.x & 31;
    const int64_t gwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int nseg = (V + (32 * U) - 1) / (32 * U);
    const int64_t ntask = N * nseg;
    for (int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < ntask;
         task += gwarps) {
        const int64_t n = task / nseg;
        const int g = (int)(task - n * nseg);
        const int s = (int)(n / T);
        int slot = -1;
        if (lane < P && (recv_part < 0 || lane == recv_part)) slot = __ldg(token_slot + n * P + lane);
        if (slot >= cap_send) {
            if (g == 0) cap_flag = true;
            slot = -1;
        }
        unsigned vmask = __ballot_sync(kFull, slot >= 0);
        const int v0 = g * (32 * U) + lane;
        if constexpr (B == 1) {
            // launched only when one partition returns rows: at most one row per
            // token, so each 16-byte column is finished on its own (8 accumulators)
            int4 r[U];
            int sl = -1;
            if (vmask) sl = __shfl_sync(kFull, slot, __ffs(vmask) - 1);
            const int4 *src = ret + ((int64_t)s * cap_send + (sl < 0 ? 0 : sl)) * V;
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int vi = v0 + 32 * u;
                r[u] = (vi < V && sl >= 0) ? ld_stream(src + vi) : make_int4(0, 0, 0, 0);
            }
            int4 *dst = out + n * V;
#pragma unroll
            for (int u = 0; u < U; u++) {
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; i++) acc[i] = 0.f;
                if (sl >= 0) fma_bf16x8(acc, r[u], 1.f);
                const int vi = v0 + 32 * u;
                if (vi < V) st_stream(dst + vi, pack_bf16x8(acc));
            }
            continue;
        }
        float acc[8 * U];
#pragma unroll
        for (int i = 0; i < 8 * U; i++) acc[i] = 0.f;
        while (vmask) {
            int4 r[B][U];
            int nb = 0;
#pragma unroll
            for (int b = 0; b < B; b++) {
                if (vmask) {
                    const int p = __ffs(vmask) - 1;
                    vmask &= vmask - 1;
                    const int sl = __shfl_sync(kFull, slot, p);
                    const int4 *src = ret + ((int64_t)s * cap_send + sl) * V;
#pragma unroll
                    for (int u = 0; u < U; u++) {
                        const int vi = v0 + 32 * u;
                        r[b][u] = (vi < V) ? ld_stream(src + vi) : make_int4(0, 0, 0, 0);
                    }
                    nb = b + 1;
                }
            }
#pragma unroll
            for (int b = 0; b < B; b++) {
                if (b < nb) {
#pragma unroll
                    for (int u = 0; u < U; u++) fma_bf16x8(acc + 8 * u, r[b][u], 1.f);
                }
            }
        }
        int4 *dst = out + n * V;
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int vi = v0 + 32 * u;
            if (vi < V) st_stream(dst + vi, pack_bf16x8(acc + 8 * u));
        }
    }
    if (cap_flag) flag_status(dev_status, MOE_ERR_CAPACITY);
}

// The expert whose run holds `row`: the last e < E with off[e] <= row (off is
// the ascending run starts, off[0] = 0).  Two warp ballots over at most 32
// run starts each (E <= 1024) instead of a serial binary search.
__device__ __forceinline__ int expert_of_row(const int *off, int E, int row, int lane)
{
    const int step = (E + 31) >> 5;
    const int i1 = lane * step;
    const unsigned b1 = __ballot_sync(kFull, i1 < E && off[i1] <= row);
    const int base = (31 - __clz(b1)) * step;
    const int i2 = base + lane;
    const unsigned b2 = __ballot_sync(kFull, lane < step && i2 < E && off[i2] <= row);
    return base + (31 - __clz(b2));
}

// Stand-in expert: one warp per (row, 2 KiB segment); expert of the row from
// the run starts.
__global__ void __launch_bounds__(256) k_expert_scale(const int4 *__restrict__ recv,
                                                      const int32_t *__restrict__ expert_offsets,
                                                      const float *__restrict__ scale, int E,
                                                      int V, int cap_recv,
                                                      int4 *__restrict__ y)
{
    extern __shared__ int off[];  // [E + 1]
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i <= E; i += blockDim.x) off[i] = __ldg(expert_offsets + i);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int rows = off[E] < cap_recv ? off[E] : cap_recv;
    const int nseg = (V + 127) / 128;
    const int64_t ntask = (int64_t)rows * nseg;
    const int64_t gwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < ntask;
         task += gwarps) {
        const int row = (int)(task / nseg);
        const int g = (int)(task - (int64_t)row * nseg);
        const int lo = expert_of_row(off, E, row, lane);
        const float sc = __ldg(scale + lo);
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const int vi = g * 128 + u * 32 + lane;
            if (vi < V) {
                const int4 v = recv[(int64_t)row * V + vi];
                float a[8];
                const uint32_t uu[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    a[2 * i] = __uint_as_float(uu[i] << 16) * sc;
                    a[2 * i + 1] = __uint_as_float(uu[i] & 0xffff0000u) * sc;
                }
                y[(int64_t)row * V + vi] = pack_bf16x8(a);
            }
        }
    }
}

// Stand-in expert on MXFP8 records (codes, then one E8M0 byte per 32 values):
//   y = bf16( s_e * e4m3(code) * 2^(scale - 127) )
// One warp per (row, 1,024-value segment); each lane decodes 8 codes.  The
// code times s_e is rounded once to fp32; the power of two is applied in two
// exact halves so that only a result below the normal range rounds again.
__global__ void __launch_bounds__(256) k_expert_scale_mxfp8(
    const uint8_t *__restrict__ recv_q, const int32_t *__restrict__ expert_offsets,
    const float *__restrict__ scale, int E, int V, int cap_recv, int4 *__restrict__ y)
{
    extern __shared__ int off[];  // [E + 1]
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i <= E; i += blockDim.x) off[i] = __ldg(expert_offsets + i);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int rows = off[E] < cap_recv ? off[E] : cap_recv;
    const int64_t rb = (int64_t)V * 8 + V / 4;
    const int nseg = (V + 127) / 128;
    const int64_t ntask = (int64_t)rows * nseg;
    const int64_t gwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < ntask;
         task += gwarps) {
        const int row = (int)(task / nseg);
        const int g = (int)(task - (int64_t)row * nseg);
        const uint8_t *rec = recv_q + (int64_t)row * rb;
        uint2 c[4];
        int sb[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const int vi = g * 128 + u * 32 + lane;
            c[u] = make_uint2(0, 0);
            sb[u] = 127;
            if (vi < V) {
                c[u] = ld_stream(reinterpret_cast<const uint2 *>(rec) + vi);
                sb[u] = __ldg(rec + (int64_t)V * 8 + (vi >> 2));
            }
        }
        // the row's expert, while the loads are in flight
        const float sc = __ldg(scale + expert_of_row(off, E, row, lane));
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const int vi = g * 128 + u * 32 + lane;
            if (vi >= V) continue;
            const int k2 = sb[u] - 127;
            const int k1 = k2 / 2;
            const float f1 = __uint_as_float((uint32_t)(127 + k1) << 23);
            const float f2 = __uint_as_float((uint32_t)(127 + k2 - k1) << 23);
            const uint32_t w[2] = {c[u].x, c[u].y};
            float a[8];
#pragma unroll
            for (int i = 0; i < 2; i++) {
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(
                        (__nv_fp8x2_storage_t)(w[i] >> (16 * h)), __NV_E4M3);
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
                    a[4 * i + 2 * h] = (f.x * sc) * f1 * f2;
                    a[4 * i + 2 * h + 1] = (f.y * sc) * f1 * f2;
                }
            }
            st_cg(y + (int64_t)row * V + vi, pack_bf16x8(a));
        }
    }
}

// Stand-in expert on NVFP4 records (H/2 code bytes, then one E4M3 scale per
// 16 values):  y = bf16( s_e * e2m1(code) * e4m3(scale) * g ).  The product
// code * scale is exact in fp32; the two factors g and s_e are applied as one
// fp32 product, so y may differ from the exactly rounded value by one bf16 unit.
__global__ void __launch_bounds__(256) k_expert_scale_nvfp4(
    const uint8_t *__restrict__ recv_q, const int32_t *__restrict__ expert_offsets,
    const float *__restrict__ scale, int E, int V, float g, int cap_recv, int4 *__restrict__ y)
{
    extern __shared__ int off[];  // [E + 1]
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i <= E; i += blockDim.x) off[i] = __ldg(expert_offsets + i);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int rows = off[E] < cap_recv ? off[E] : cap_recv;
    const int64_t rb = (int64_t)V * 4 + V / 2;
    const int nseg = (V + 127) / 128;
    const int64_t ntask = (int64_t)rows * nseg;
    const int64_t gwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < ntask;
         task += gwarps) {
        const int row = (int)(task / nseg);
        const int gs = (int)(task - (int64_t)row * nseg);
        const uint8_t *rec = recv_q + (int64_t)row * rb;
        uint32_t c[4];
        uint8_t sb[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const int vi = gs * 128 + u * 32 + lane;
            c[u] = 0;
            sb[u] = 0;
            if (vi < V) {
                c[u] = __ldg(reinterpret_cast<const uint32_t *>(rec) + vi);
                sb[u] = __ldg(rec + (int64_t)V * 4 + (vi >> 1));
            }
        }
        // the row's expert, while the loads are in flight
        const float f = __fmul_rn(__ldg(scale + expert_of_row(off, E, row, lane)), g);
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const int vi = gs * 128 + u * 32 + lane;
            if (vi >= V) continue;
            const __half_raw shr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)sb[u], __NV_E4M3);
            const float sd = __half2float(*reinterpret_cast<const __half *>(&shr));
            float a[8];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const __half2_raw hr =
                    __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)(c[u] >> (8 * i)), __NV_E2M1);
                const float2 q = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
                a[2 * i] = __fmul_rn(__fmul_rn(q.x, sd), f);
                a[2 * i + 1] = __fmul_rn(__fmul_rn(q.y, sd), f);
            }
            st_cg(y + (int64_t)row * V + vi, pack_bf16x8(a));
        }
    }
}

}  // namespace

cudaError_t launch_combine(const uint16_t *y, int y_rows, const int32_t *pair_row, const float *w,
                           int64_t N, int k, int H, uint16_t *out, uint32_t *dev_status,
                           cudaStream_t st)
{
    if (N == 0) return cudaSuccess;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int V = H / 8;
    const int nseg = (V + kCombSegVec - 1) / kCombSegVec;
    const int64_t warps = N * nseg;
    int64_t blocks = (warps + (kCombThreads / 32) - 1) / (kCombThreads / 32);
    const int resident = resident_grid((const void *)k_combine, kCombThreads, 0);
    const int64_t wave = resident > 0 ? resident : (int64_t)di.sm_count * (2048 / kCombThreads);
    if (blocks > wave) blocks = wave;
    MOE_TRACED_LAUNCH("k_combine", st,
                      e = launch_pdl(k_combine, dim3((unsigned)blocks), dim3(kCombThreads), 0, st,
                                     (const int4 *)y, y_rows, pair_row, w, N, k, V, (int4 *)out,
                                     dev_status));
    return e;
}

cudaError_t launch_expert_scale(const uint16_t *recv, const int32_t *expert_offsets,
                                const float *scale, int E, int H, int cap_recv, uint16_t *y,
                                cudaStream_t st)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int blocks = di.sm_count * 8;
    MOE_TRACED_LAUNCH("k_expert_scale", st,
                      e = launch_pdl(k_expert_scale, dim3(blocks), dim3(256),
                                     (size_t)(E + 1) * sizeof(int), st, (const int4 *)recv,
                                     expert_offsets, scale, E, H / 8, cap_recv, (int4 *)y));
    return e;
}

cudaError_t launch_combine_stage1(const uint16_t *y, int y_rows, const int32_t *pair_row,
                                  const float *w, const int32_t *ids, const int32_t *token_slot,
                                  int S, int T, int k, int E, int P, int H, int recv_part,
                                  int cap_send, uint16_t *ret, uint32_t *dev_status, cudaStream_t st)
{
    const int64_t N = (int64_t)S * T;
    if (N == 0) return cudaSuccess;
    const int V = H / 8;
    constexpr int U = kStageUnroll, B = kStageBatch;
    const int nseg = (V + 32 * U - 1) / (32 * U);
    int64_t blocks = (N * nseg + (kCombThreads / 32) - 1) / (kCombThreads / 32);
    const int resident = resident_grid((const void *)k_combine_stage1<U, B>, kCombThreads, 0);
    if (resident > 0 && blocks > resident) blocks = resident;
    cudaError_t e;
    MOE_TRACED_LAUNCH("k_combine_stage1", st,
                      e = launch_pdl(k_combine_stage1<U, B>, dim3((unsigned)blocks), dim3(kCombThreads),
                                     0, st, (const int4 *)y, y_rows, pair_row, w, ids, token_slot,
                                     N, T, k, E, E / P, P, V, recv_part, cap_send, (int4 *)ret,
                                     dev_status));
    return e;
}

cudaError_t launch_combine_stage2(const uint16_t *ret, const int32_t *token_slot, int S, int T,
                                  int P, int H, int recv_part, int cap_send, uint16_t *out,
                                  uint32_t *dev_status, cudaStream_t st)
{
    const int64_t N = (int64_t)S * T;
    if (N == 0) return cudaSuccess;
    const int V = H / 8;
    // one returned row per token from a single receiving partition, up to P otherwise
    const bool one = recv_part >= 0 || P == 1;
    const void *kfn = one ? (const void *)k_combine_stage2<kRoutedUnroll, 1>
                          : (const void *)k_combine_stage2<kStage2Unroll, kStage2Batch>;
    const int U = one ? kRoutedUnroll : kStage2Unroll;
    const int nseg = (V + 32 * U - 1) / (32 * U);
    int64_t blocks = (N * nseg + (kCombThreads / 32) - 1) / (kCombThreads / 32);
    const int resident = resident_grid(kfn, kCombThreads, 0);
    if (resident > 0 && blocks > resident) blocks = resident;
    cudaError_t e;
    if (one) {
        MOE_TRACED_LAUNCH("k_combine_stage2", st,
                          e = launch_pdl(k_combine_stage2<kRoutedUnroll, 1>, dim3((unsigned)blocks),
                                         dim3(kCombThreads), 0, st, (const int4 *)ret, token_slot,
                                         N, T, P, V, recv_part, cap_send, (int4 *)out, dev_status));
    } else {
        MOE_TRACED_LAUNCH("k_combine_stage2", st,
                          e = launch_pdl(k_combine_stage2<kStage2Unroll, kStage2Batch>,
                                         dim3((unsigned)blocks), dim3(kCombThreads), 0, st,
                                         (const int4 *)ret, token_slot, N, T, P, V, recv_part,
                                         cap_send, (int4 *)out, dev_status));
    }
    return e;
}

cudaError_t launch_expert_scale_mxfp8(const uint8_t *recv_q, const int32_t *expert_offsets,
                                      const float *scale, int E, int H, int cap_recv, uint16_t *y,
                                      cudaStream_t st)
{
    if (cap_recv == 0) return cudaSuccess;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int blocks = di.sm_count * 8;
    MOE_TRACED_LAUNCH("k_expert_scale_mxfp8", st,
                      e = launch_pdl(k_expert_scale_mxfp8, dim3(blocks), dim3(256),
                                     (size_t)(E + 1) * sizeof(int), st, recv_q, expert_offsets,
                                     scale, E, H / 8, cap_recv, (int4 *)y));
    return e;
}

cudaError_t launch_routed_stage1(const uint16_t *send, const int32_t *send_ids,
                                 const float *send_w, const int32_t *part_offsets, int S, int T,
                                 int cap_send, int k, int E, int P, int H, int recv_part,
                                 const float *scale, uint16_t *ret, uint32_t *dev_status,
                                 cudaStream_t st)
{
    const int span = recv_part >= 0 ? (T < cap_send ? T : cap_send) : cap_send;
    const int64_t rows = (int64_t)S * span;
    if (rows == 0) return cudaSuccess;
    const int V = H / 8;
    constexpr int U = kRoutedUnroll;
    const int nseg = (V + 32 * U - 1) / (32 * U);
    int64_t blocks = (rows * nseg + (kCombThreads / 32) - 1) / (kCombThreads / 32);
    const void *kfn = scale ? (const void *)k_routed_stage1<U, true>
                            : (const void *)k_routed_stage1<U, false>;
    const int resident = resident_grid(kfn, kCombThreads, 0);
    if (resident > 0 && blocks > resident) blocks = resident;
    cudaError_t e;
    if (scale) {
        MOE_TRACED_LAUNCH("k_routed_stage1", st,
                          e = launch_pdl(k_routed_stage1<U, true>, dim3((unsigned)blocks),
                                         dim3(kCombThreads), 0, st, (const int4 *)send, send_ids,
                                         send_w, part_offsets, S, cap_send, span, k, E, E / P, P, V,
                                         recv_part, scale, (int4 *)ret, dev_status));
    } else {
        MOE_TRACED_LAUNCH("k_routed_stage1", st,
                          e = launch_pdl(k_routed_stage1<U, false>, dim3((unsigned)blocks),
                                         dim3(kCombThreads), 0, st, (const int4 *)send, send_ids,
                                         send_w, part_offsets, S, cap_send, span, k, E, E / P, P, V,
                                         recv_part, scale, (int4 *)ret, dev_status));
    }
    return e;
}

cudaError_t launch_expert_scale_nvfp4(const uint8_t *recv_q, const int32_t *expert_offsets,
                                      const float *scale, int E, int H, float g, int cap_recv,
                                      uint16_t *y, cudaStream_t st)
{
    if (cap_recv == 0) return cudaSuccess;
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int blocks = di.sm_count * 8;
    MOE_TRACED_LAUNCH("k_expert_scale_nvfp4", st,
                      e = launch_pdl(k_expert_scale_nvfp4, dim3(blocks), dim3(256),
                                     (size_t)(E + 1) * sizeof(int), st, recv_q, expert_offsets,
                                     scale, E, H / 8, g, cap_recv, (int4 *)y));
    return e;
}

}  // namespace moe
