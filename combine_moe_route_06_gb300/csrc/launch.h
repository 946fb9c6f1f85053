// launch.h -- internal launchers (one per kernel family); arguments are
// validated by api.cu before any of these is called.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe_route.h"

namespace moe {

// Per-device launch geometry, queried once per device.
struct DeviceInfo {
    int sm_count;
    int max_smem_optin;
};
cudaError_t device_info(DeviceInfo *out);

// CTAs of `kernel` that fit on the whole device at once (SM count x blocks
// per SM for this block size and dynamic shared memory); cached per device
// and kernel.  Persistent grid-stride kernels launch exactly this many, so no
// second wave leaves a tail.  Returns 0 if the query fails.
int resident_grid(const void *kernel, int threads, size_t smem);

// Record `message` as the calling thread's last error text and return `code`.
moe_status_t report(moe_status_t code, const char *message);

cudaError_t launch_route_topk(const float *logits, int64_t N, int E, int k, int32_t *ids,
                              float *w, cudaStream_t st);

size_t layout_ws_bytes(int S, int T, int E, int P);
// Kernels launch_dispatch_layout enqueues for these sizes on the current device.
cudaError_t layout_kernel_count(int T, int k, int E, int P, int *n);
cudaError_t launch_dispatch_layout(const int32_t *ids, int S, int T, int k, int E, int P,
                                   int32_t *expert_counts, int32_t *expert_rank, int32_t *part_counts,
                                   int32_t *part_offsets, int32_t *token_slot, void *ws,
                                   uint32_t *dev_status, cudaStream_t st);

// With send_ids != nullptr the rows also carry the tokens' ids and weights.
cudaError_t launch_dispatch_pack(const uint16_t *x, int S, int T, int H, int P,
                                 const int32_t *token_slot, const int32_t *part_offsets,
                                 int cap_send, uint16_t *send, int32_t *send_src,
                                 uint32_t *dev_status, cudaStream_t st,
                                 const int32_t *ids = nullptr, const float *w = nullptr, int k = 0,
                                 int32_t *send_ids = nullptr, float *send_w = nullptr);
cudaError_t launch_routed_stage1(const uint16_t *send, const int32_t *send_ids,
                                 const float *send_w, const int32_t *part_offsets, int S, int T,
                                 int cap_send, int k, int E, int P, int H, int recv_part,
                                 const float *scale, uint16_t *ret, uint32_t *dev_status,
                                 cudaStream_t st);

cudaError_t launch_dispatch_pack_mxfp8(const uint16_t *x, int S, int T, int H, int P,
                                       const int32_t *token_slot, const int32_t *part_offsets,
                                       int cap_send, uint8_t *send_q, int32_t *send_src,
                                       uint32_t *dev_status, cudaStream_t st);
cudaError_t launch_dispatch_pack_nvfp4(const uint16_t *x, int S, int T, int H, int P, float g,
                                       const int32_t *token_slot, const int32_t *part_offsets,
                                       int cap_send, uint8_t *send_q, int32_t *send_src,
                                       uint32_t *dev_status, cudaStream_t st);
cudaError_t launch_expert_scale_nvfp4(const uint8_t *recv_q, const int32_t *expert_offsets,
                                      const float *scale, int E, int H, float g, int cap_recv,
                                      uint16_t *y, cudaStream_t st);
cudaError_t launch_expert_scale_mxfp8(const uint8_t *recv_q, const int32_t *expert_offsets,
                                      const float *scale, int E, int H, int cap_recv, uint16_t *y,
                                      cudaStream_t st);

// Expert placement by load with redundant copies (host) and the layout over a
// placement (device).  plan_placement returns the number of slots used.
int plan_placement(const int64_t *load, int E, int P, int R, int32_t *copy_offsets,
                   int32_t *copy_slots, int32_t *slot_expert, int64_t *part_load);
size_t mapped_ws_bytes(int S, int T, int k, int E, int P, int E_phys);
cudaError_t launch_dispatch_layout_mapped(const int32_t *ids, int S, int T, int k, int E, int P,
                                          int E_phys, const int32_t *copy_offsets,
                                          const int32_t *copy_slots, int n_copies,
                                          int32_t *phys, int32_t *expert_counts,
                                          int32_t *expert_rank, int32_t *part_counts,
                                          int32_t *part_offsets, int32_t *token_slot, void *ws,
                                          uint32_t *dev_status, cudaStream_t st);

size_t permute_ws_bytes(int S, int T, int E);
// Whether launch_permute runs its map step inside the copy kernel (one launch).
bool permute_map_fused(int S, int E);
cudaError_t launch_permute(const uint16_t *send, const int32_t *token_slot, const int32_t *ids,
                           const int32_t *expert_counts, const int32_t *expert_rank,
                           int S, int T, int k, int E, int P, int H, int recv_part, int align,
                           int cap_send, int cap_recv, uint16_t *recv, int32_t *expert_offsets,
                           int32_t *pair_row, int32_t *recv_pair, void *ws,
                           uint32_t *dev_status, cudaStream_t st);

cudaError_t launch_permute_masked(const uint16_t *send, const int32_t *token_slot,
                                  const int32_t *ids, const int32_t *expert_counts,
                                  const int32_t *expert_rank, int S, int T, int k, int E, int P,
                                  int H, int recv_part, int block_rows, int cap_send,
                                  uint16_t *recv, int32_t *masked_counts, int32_t *pair_row,
                                  int32_t *recv_pair, uint32_t *dev_status, cudaStream_t st);

cudaError_t launch_combine(const uint16_t *y, int y_rows, const int32_t *pair_row, const float *w,
                           int64_t N, int k, int H, uint16_t *out, uint32_t *dev_status,
                           cudaStream_t st);

cudaError_t launch_combine_stage1(const uint16_t *y, int y_rows, const int32_t *pair_row,
                                  const float *w, const int32_t *ids, const int32_t *token_slot,
                                  int S, int T, int k, int E, int P, int H, int recv_part,
                                  int cap_send, uint16_t *ret, uint32_t *dev_status,
                                  cudaStream_t st);
cudaError_t launch_combine_stage2(const uint16_t *ret, const int32_t *token_slot, int S, int T,
                                  int P, int H, int recv_part, int cap_send, uint16_t *out,
                                  uint32_t *dev_status, cudaStream_t st);

// The dispatch side in one launch for one source of at most 256 tokens
// (dispatch_small.cu): whether that form runs for these sizes on the current
// device (cached attributes only, so the answer holds inside a stream
// capture), and its launch.  With masked_counts (non-null) the receive rows
// take the masked layout (block_rows rows per receiving expert; expert_offsets
// and align unused), else the contiguous runs.
cudaError_t dispatch_small_form(int S, int T, int k, int E, int P, bool *out);
cudaError_t launch_dispatch_small(const float *logits, const uint16_t *x, int T, int H, int E,
                                  int k, int P, int recv_part, int align, int cap_send,
                                  int cap_recv, int32_t *topk_ids, float *topk_w,
                                  int32_t *expert_counts, int32_t *expert_rank,
                                  int32_t *part_counts, int32_t *part_offsets,
                                  int32_t *token_slot, uint16_t *send, int32_t *send_src,
                                  uint16_t *recv, int32_t *expert_offsets, int32_t *pair_row,
                                  int32_t *recv_pair, uint32_t *dev_status,
                                  int32_t *masked_counts, int block_rows, cudaStream_t st);

// The quantized dispatch side in one launch for one source of at most 256
// tokens (dispatch_small_q.cu; format 1: MXFP8 records, 2: NVFP4, g the NVFP4
// tensor scale); the form runs where dispatch_small_form says so.
cudaError_t launch_dispatch_small_q(const float *logits, const uint16_t *x, int T, int H, int E,
                                    int k, int P, int format, float g, int recv_part, int align,
                                    int cap_send, int cap_recv, int32_t *topk_ids, float *topk_w,
                                    int32_t *expert_counts, int32_t *expert_rank,
                                    int32_t *part_counts, int32_t *part_offsets,
                                    int32_t *token_slot, uint8_t *send_q, int32_t *send_src,
                                    uint8_t *recv_q, int32_t *expert_offsets, int32_t *pair_row,
                                    int32_t *recv_pair, uint32_t *dev_status, cudaStream_t st);

// The dispatch side in one call with the masked receive layout (dispatch.cu):
// one launch for one source of at most 256 tokens, else route, layout and the
// masked pack + permute.
int dispatch_masked_kernel_count(int S, int T, int k, int E, int P, int recv_part);
cudaError_t launch_dispatch_masked(const float *logits, const uint16_t *x, int S, int T, int H,
                                   int E, int k, int P, int recv_part, int block_rows,
                                   int cap_send, int32_t *topk_ids, float *topk_w,
                                   int32_t *expert_counts, int32_t *expert_rank,
                                   int32_t *part_counts, int32_t *part_offsets,
                                   int32_t *token_slot, uint16_t *send, int32_t *send_src,
                                   uint16_t *recv, int32_t *masked_counts, int32_t *pair_row,
                                   int32_t *recv_pair, void *ws, uint32_t *dev_status,
                                   cudaStream_t st);

// The dispatch side in one call (dispatch.cu): route, layout, pack and permute.
cudaError_t dispatch_kernel_count(int S, int T, int k, int E, int P, int *n);
cudaError_t launch_dispatch(const float *logits, const uint16_t *x, int S, int T, int H, int E,
                            int k, int P, int recv_part, int align, int cap_send, int cap_recv,
                            int32_t *topk_ids, float *topk_w, int32_t *expert_counts,
                            int32_t *expert_rank, int32_t *part_counts, int32_t *part_offsets,
                            int32_t *token_slot, uint16_t *send, int32_t *send_src,
                            uint16_t *recv, int32_t *expert_offsets, int32_t *pair_row,
                            int32_t *recv_pair, void *ws, uint32_t *dev_status, cudaStream_t st);

// Pack and permute in one pass given a layout (x_before_wait: the launcher
// guarantees that x was complete before the previous kernel passed its grid
// dependency wait); the kernels it enqueues.
int pack_permute_kernel_count(int S, int T, int E);
cudaError_t launch_pack_permute(const uint16_t *x, const int32_t *token_slot,
                                const int32_t *part_offsets, const int32_t *topk_ids,
                                const int32_t *expert_counts, const int32_t *expert_rank, int S,
                                int T, int k, int E, int P, int H, int recv_part, int align,
                                int cap_send, int cap_recv, uint16_t *send, int32_t *send_src,
                                uint16_t *recv, int32_t *expert_offsets, int32_t *pair_row,
                                int32_t *recv_pair, void *ws, uint32_t *dev_status,
                                cudaStream_t st, bool x_before_wait);

// Pack and the masked receive layout in one pass (x_before_wait as for
// launch_pack_permute); the kernels it enqueues.
int pack_permute_masked_kernel_count(int S, int T, int E, int P, int recv_part);
cudaError_t launch_pack_permute_masked(const uint16_t *x, const int32_t *token_slot,
                                       const int32_t *part_offsets, const int32_t *topk_ids,
                                       const int32_t *expert_counts, const int32_t *expert_rank,
                                       int S, int T, int k, int E, int P, int H, int recv_part,
                                       int block_rows, int cap_send, uint16_t *send,
                                       int32_t *send_src, uint16_t *recv, int32_t *masked_counts,
                                       int32_t *pair_row, int32_t *recv_pair,
                                       uint32_t *dev_status, cudaStream_t st, bool x_before_wait);

// The dispatch side with quantized rows (format 1: MXFP8 records, 2: NVFP4).
cudaError_t dispatch_quantized_kernel_count(int S, int T, int k, int E, int P, int *n);
cudaError_t launch_dispatch_quantized(const float *logits, const uint16_t *x, int S, int T, int H,
                                      int E, int k, int P, int format, float g, int recv_part,
                                      int align, int cap_send, int cap_recv, int32_t *topk_ids,
                                      float *topk_w, int32_t *expert_counts, int32_t *expert_rank,
                                      int32_t *part_counts, int32_t *part_offsets,
                                      int32_t *token_slot, uint8_t *send_q, int32_t *send_src,
                                      uint8_t *recv_q, int32_t *expert_offsets, int32_t *pair_row,
                                      int32_t *recv_pair, void *ws, uint32_t *dev_status,
                                      cudaStream_t st);

cudaError_t launch_expert_scale(const uint16_t *recv, const int32_t *expert_offsets,
                                const float *scale, int E, int H, int cap_recv, uint16_t *y,
                                cudaStream_t st);

}  // namespace moe
