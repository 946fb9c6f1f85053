// pack.cu -- sender side of dispatch: bit copies of bf16 rows into the send
// region of every partition that needs the token.
//
// a2a-backends page (vincentzed.com/writing/a2a-backends), section 3.2 (fourth
// step: the rows move), section 5.1 (a region per sender, rows written straight
// into place) and section 6.1 (one copy per GPU that needs the token).
//
// Work unit: one warp per (token, 2 KiB column segment).  The warp reads the
// segment of x once (16-byte vectors, four per lane in flight) and stores it
// to each of the token's c <= min(k, P) destination rows.  HBM traffic is the
// minimum: x read once, c copies written.
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"
#include "quant.cuh"
#include "trace.h"

namespace moe {

namespace {

constexpr int kPackUnroll = 4;                   // int4 per lane per segment
constexpr int kPackSegVec = 32 * kPackUnroll;    // int4 per segment (2 KiB)
constexpr int kPackThreads = 256;

// ROUTED: each written row also carries the token's k expert ids and weights
// (a2a-backends section 6.1: payloads are the hidden state, the top-k ids and
// the top-k weights); rows no slot names carry id -1 and weight 0 (section
// 6.3: empty slots have an invalid expert id).
template <bool ROUTED>
__global__ void __launch_bounds__(kPackThreads) k_pack(const int4 *__restrict__ x, int S, int T,
                                                       int V, int P,
                                                       const int32_t *__restrict__ token_slot,
                                                       const int32_t *__restrict__ part_offsets,
                                                       int cap_send, int4 *__restrict__ send,
                                                       int32_t *__restrict__ send_src,
                                                       uint32_t *dev_status,
                                                       const int32_t *__restrict__ ids,
                                                       const float *__restrict__ w, int k,
                                                       int32_t *__restrict__ send_ids,
                                                       float *__restrict__ send_w)
{
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t gthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;

    // rows of send_src past the last used row of each source
    for (int64_t i = gtid; i < (int64_t)S * cap_send; i += gthreads) {
        const int s = (int)(i / cap_send);
        const int r = (int)(i - (int64_t)s * cap_send);
        if (r >= __ldg(part_offsets + (int64_t)s * (P + 1) + P)) {
            send_src[i] = -1;
            if (ROUTED) {
                for (int j = 0; j < k; j++) {
                    send_ids[i * k + j] = -1;
                    send_w[i * k + j] = 0.f;
                }
            }
        }
    }

    const int nseg = (V + kPackSegVec - 1) / kPackSegVec;
    const int64_t ntask = (int64_t)S * T * nseg;
    const int64_t gwarps = gthreads >> 5;
    bool overflow = false;
    for (int64_t task = gtid >> 5; task < ntask; task += gwarps) {
        const int64_t n = task / nseg;          // token index s*T + t
        const int g = (int)(task - n * nseg);   // column segment
        const int s = (int)(n / T);
        int slot = -1;
        if (lane < P) slot = __ldg(token_slot + n * P + lane);
        const bool ok = slot >= 0 && slot < cap_send;
        if (slot >= cap_send) overflow = true;
        unsigned dmask = __ballot_sync(kFull, ok);
        if (g == 0 && ok) send_src[(int64_t)s * cap_send + slot] = (int32_t)(n - (int64_t)s * T);
        if (dmask == 0) continue;
        if (ROUTED && g == 0) {
            int id = -1;
            float wt = 0.f;
            if (lane < k) {
                id = __ldg(ids + n * k + lane);
                wt = __ldg(w + n * k + lane);
            }
            for (unsigned m = dmask; m; m &= m - 1) {
                const int sl = __shfl_sync(kFull, slot, __ffs(m) - 1);
                if (lane < k) {
                    const int64_t o = ((int64_t)s * cap_send + sl) * k + lane;
                    send_ids[o] = id;
                    send_w[o] = wt;
                }
            }
        }

        const int4 *src = x + n * V;
        const int v0 = g * kPackSegVec + lane;
        int4 r[kPackUnroll];
#pragma unroll
        for (int u = 0; u < kPackUnroll; u++) {
            const int vi = v0 + 32 * u;
            if (vi < V) r[u] = ld_stream(src + vi);
        }
        while (dmask) {
            const int p = __ffs(dmask) - 1;
            dmask &= dmask - 1;
            const int sl = __shfl_sync(kFull, slot, p);
            int4 *dst = send + ((int64_t)s * cap_send + sl) * V;
#pragma unroll
            for (int u = 0; u < kPackUnroll; u++) {
                const int vi = v0 + 32 * u;
                if (vi < V) st_cg(dst + vi, r[u]);
            }
        }
    }
    if (__any_sync(kFull, overflow) && lane == 0) flag_status(dev_status, MOE_ERR_CAPACITY);
}

// Pack with MXFP8 records (a2a-backends section 7.2: tokens are converted
// before they are sent; an FP8 row is 5,280 bytes for 5,120 values, one scale
// byte per 32).  A record is H E4M3 codes followed by H/32 E8M0 scales,
//   X = 2^(floor(log2 max|v|) - 8), code = e4m3_rn_satfinite(v / X).
// One warp per (token, 1,024-value segment); lanes 4b..4b+3 hold one 32-value
// block for each of the four 16-byte loads (mxfp8_quantize in quant.cuh).  The
// row is quantized once and stored to every destination slot.
constexpr int kQSegVec = 32 * kPackUnroll;   // int4 (8 values) per segment

__global__ void __launch_bounds__(kPackThreads) k_pack_mxfp8(
    const int4 *__restrict__ x, int S, int T, int V, int P, const int32_t *__restrict__ token_slot,
    const int32_t *__restrict__ part_offsets, int cap_send, uint8_t *__restrict__ send_q,
    int32_t *__restrict__ send_src, uint32_t *dev_status)
{
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t gthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t i = gtid; i < (int64_t)S * cap_send; i += gthreads) {
        const int s = (int)(i / cap_send);
        const int r = (int)(i - (int64_t)s * cap_send);
        if (r >= __ldg(part_offsets + (int64_t)s * (P + 1) + P)) send_src[i] = -1;
    }
    const int64_t rb = (int64_t)V * 8 + V / 4;  // record bytes: codes, then scales
    const int nseg = (V + kQSegVec - 1) / kQSegVec;
    const int64_t ntask = (int64_t)S * T * nseg;
    const int64_t gwarps = gthreads >> 5;
    bool overflow = false;
    for (int64_t task = gtid >> 5; task < ntask; task += gwarps) {
        const int64_t n = task / nseg;
        const int g = (int)(task - n * nseg);
        const int s = (int)(n / T);
        int slot = -1;
        if (lane < P) slot = __ldg(token_slot + n * P + lane);
        const bool ok = slot >= 0 && slot < cap_send;
        if (slot >= cap_send) overflow = true;
        unsigned dmask = __ballot_sync(kFull, ok);
        if (g == 0 && ok) send_src[(int64_t)s * cap_send + slot] = (int32_t)(n - (int64_t)s * T);
        if (dmask == 0) continue;

        const int v0 = g * kQSegVec + lane;
        uint2 code[kPackUnroll];
        uint8_t scale[kPackUnroll];
#pragma unroll
        for (int u = 0; u < kPackUnroll; u++) {
            const int vi = v0 + 32 * u;
            int4 v = make_int4(0, 0, 0, 0);
            if (vi < V) v = ld_stream(x + n * V + vi);
            mxfp8_quantize(v, code[u], scale[u]);
        }
        while (dmask) {
            const int p = __ffs(dmask) - 1;
            dmask &= dmask - 1;
            const int sl = __shfl_sync(kFull, slot, p);
            uint8_t *rec = send_q + ((int64_t)s * cap_send + sl) * rb;
#pragma unroll
            for (int u = 0; u < kPackUnroll; u++) {
                const int vi = v0 + 32 * u;
                if (vi < V) {
                    reinterpret_cast<uint2 *>(rec)[vi] = code[u];
                    if ((vi & 3) == 0) rec[(int64_t)V * 8 + (vi >> 2)] = scale[u];
                }
            }
        }
    }
    if (__any_sync(kFull, overflow) && lane == 0) flag_status(dev_status, MOE_ERR_CAPACITY);
}

// Pack with NVFP4 records (a2a-backends section 7.2: an NVFP4 row is 2,880
// bytes for 5,120 values, one scale byte per 16).  A record is H/2 bytes of
// E2M1 codes (element 2i in the low nibble) followed by H/16 E4M3 block
// scales; with the tensor scale g,
//   s = e4m3(amax / (6 g)),  code = e2m1_rn_satfinite(v / (s g))   (0 if s = 0)
// all in fp32 with correctly rounded division.  One warp per (token, 1,024
// values); lanes 2b, 2b+1 hold one 16-value block for each 16-byte load.
__global__ void __launch_bounds__(kPackThreads) k_pack_nvfp4(
    const int4 *__restrict__ x, int S, int T, int V, int P, float g,
    const int32_t *__restrict__ token_slot, const int32_t *__restrict__ part_offsets,
    int cap_send, uint8_t *__restrict__ send_q, int32_t *__restrict__ send_src,
    uint32_t *dev_status)
{
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t gthreads = (int64_t)gridDim.x * blockDim.x;
    const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (int64_t i = gtid; i < (int64_t)S * cap_send; i += gthreads) {
        const int s = (int)(i / cap_send);
        const int r = (int)(i - (int64_t)s * cap_send);
        if (r >= __ldg(part_offsets + (int64_t)s * (P + 1) + P)) send_src[i] = -1;
    }
    const int64_t rb = (int64_t)V * 4 + V / 2;  // record bytes: codes, then scales
    const float d = __fmul_rn(6.0f, g);
    const int nseg = (V + kQSegVec - 1) / kQSegVec;
    const int64_t ntask = (int64_t)S * T * nseg;
    const int64_t gwarps = gthreads >> 5;
    bool overflow = false;
    for (int64_t task = gtid >> 5; task < ntask; task += gwarps) {
        const int64_t n = task / nseg;
        const int gseg = (int)(task - n * nseg);
        const int s = (int)(n / T);
        int slot = -1;
        if (lane < P) slot = __ldg(token_slot + n * P + lane);
        const bool ok = slot >= 0 && slot < cap_send;
        if (slot >= cap_send) overflow = true;
        unsigned dmask = __ballot_sync(kFull, ok);
        if (gseg == 0 && ok) send_src[(int64_t)s * cap_send + slot] = (int32_t)(n - (int64_t)s * T);
        if (dmask == 0) continue;

        const int v0 = gseg * kQSegVec + lane;
        uint32_t code[kPackUnroll];
        uint8_t scale[kPackUnroll];
#pragma unroll
        for (int u = 0; u < kPackUnroll; u++) {
            const int vi = v0 + 32 * u;
            int4 v = make_int4(0, 0, 0, 0);
            if (vi < V) v = ld_stream(x + n * V + vi);
            nvfp4_quantize(v, g, d, code[u], scale[u]);
        }
        while (dmask) {
            const int p = __ffs(dmask) - 1;
            dmask &= dmask - 1;
            const int sl = __shfl_sync(kFull, slot, p);
            uint8_t *rec = send_q + ((int64_t)s * cap_send + sl) * rb;
#pragma unroll
            for (int u = 0; u < kPackUnroll; u++) {
                const int vi = v0 + 32 * u;
                if (vi < V) {
                    reinterpret_cast<uint32_t *>(rec)[vi] = code[u];
                    if ((vi & 1) == 0) rec[(int64_t)V * 4 + (vi >> 1)] = scale[u];
                }
            }
        }
    }
    if (__any_sync(kFull, overflow) && lane == 0) flag_status(dev_status, MOE_ERR_CAPACITY);
}

}  // namespace

cudaError_t launch_dispatch_pack(const uint16_t *x, int S, int T, int H, int P,
                                 const int32_t *token_slot, const int32_t *part_offsets,
                                 int cap_send, uint16_t *send, int32_t *send_src,
                                 uint32_t *dev_status, cudaStream_t st, const int32_t *ids,
                                 const float *w, int k, int32_t *send_ids, float *send_w)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int V = H / 8;
    const int nseg = (V + kPackSegVec - 1) / kPackSegVec;
    const int64_t warps = (int64_t)S * T * nseg;
    const int64_t want = (warps + (kPackThreads / 32) - 1) / (kPackThreads / 32);
    const int resident = resident_grid((const void *)k_pack<false>, kPackThreads, 0);
    int64_t blocks = resident > 0 ? resident : (int64_t)di.sm_count * (2048 / kPackThreads);
    if (want < blocks) blocks = want;
    const int64_t tail_blocks = ((int64_t)S * cap_send + kPackThreads - 1) / kPackThreads;
    if (blocks < 1) blocks = tail_blocks < 1 ? 1 : (tail_blocks < di.sm_count ? tail_blocks : di.sm_count);
    if (send_ids == nullptr) {
        MOE_TRACED_LAUNCH("k_pack", st,
                          e = launch_pdl(k_pack<false>, dim3((unsigned)blocks), dim3(kPackThreads), 0,
                                         st, (const int4 *)x, S, T, V, P, token_slot, part_offsets,
                                         cap_send, (int4 *)send, send_src, dev_status,
                                         (const int32_t *)nullptr, (const float *)nullptr, 0,
                                         (int32_t *)nullptr, (float *)nullptr));
    } else {
        MOE_TRACED_LAUNCH("k_pack_routed", st,
                          e = launch_pdl(k_pack<true>, dim3((unsigned)blocks), dim3(kPackThreads), 0,
                                         st, (const int4 *)x, S, T, V, P, token_slot, part_offsets,
                                         cap_send, (int4 *)send, send_src, dev_status, ids, w, k,
                                         send_ids, send_w));
    }
    return e;
}

cudaError_t launch_dispatch_pack_mxfp8(const uint16_t *x, int S, int T, int H, int P,
                                       const int32_t *token_slot, const int32_t *part_offsets,
                                       int cap_send, uint8_t *send_q, int32_t *send_src,
                                       uint32_t *dev_status, cudaStream_t st)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int V = H / 8;
    const int nseg = (V + kQSegVec - 1) / kQSegVec;
    const int64_t warps = (int64_t)S * T * nseg;
    const int64_t want = (warps + (kPackThreads / 32) - 1) / (kPackThreads / 32);
    const int resident = resident_grid((const void *)k_pack_mxfp8, kPackThreads, 0);
    int64_t blocks = resident > 0 ? resident : (int64_t)di.sm_count * (2048 / kPackThreads);
    if (want < blocks) blocks = want;
    const int64_t tail_blocks = ((int64_t)S * cap_send + kPackThreads - 1) / kPackThreads;
    if (blocks < 1) blocks = tail_blocks < 1 ? 1 : (tail_blocks < di.sm_count ? tail_blocks : di.sm_count);
    MOE_TRACED_LAUNCH("k_pack_mxfp8", st,
                      e = launch_pdl(k_pack_mxfp8, dim3((unsigned)blocks), dim3(kPackThreads), 0, st,
                                     (const int4 *)x, S, T, V, P, token_slot, part_offsets,
                                     cap_send, send_q, send_src, dev_status));
    return e;
}

cudaError_t launch_dispatch_pack_nvfp4(const uint16_t *x, int S, int T, int H, int P, float g,
                                       const int32_t *token_slot, const int32_t *part_offsets,
                                       int cap_send, uint8_t *send_q, int32_t *send_src,
                                       uint32_t *dev_status, cudaStream_t st)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int V = H / 8;
    const int nseg = (V + kQSegVec - 1) / kQSegVec;
    const int64_t warps = (int64_t)S * T * nseg;
    const int64_t want = (warps + (kPackThreads / 32) - 1) / (kPackThreads / 32);
    const int resident = resident_grid((const void *)k_pack_nvfp4, kPackThreads, 0);
    int64_t blocks = resident > 0 ? resident : (int64_t)di.sm_count * (2048 / kPackThreads);
    if (want < blocks) blocks = want;
    const int64_t tail_blocks = ((int64_t)S * cap_send + kPackThreads - 1) / kPackThreads;
    if (blocks < 1) blocks = tail_blocks < 1 ? 1 : (tail_blocks < di.sm_count ? tail_blocks : di.sm_count);
    MOE_TRACED_LAUNCH("k_pack_nvfp4", st,
                      e = launch_pdl(k_pack_nvfp4, dim3((unsigned)blocks), dim3(kPackThreads), 0, st,
                                     (const int4 *)x, S, T, V, P, g, token_slot, part_offsets,
                                     cap_send, send_q, send_src, dev_status));
    return e;
}

}  // namespace moe
