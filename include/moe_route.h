/*
 * moe_route.h -- C ABI of the GB300 MoE token-path library (libmoeroute.so).
 *
 * The library implements, on one GPU, the data-parallel hot path of
 * expert-parallel MoE serving as described on the a2a-backends page
 * (vincentzed.com/writing/a2a-backends):
 *
 *   moe_route_topk          router logits -> top-k expert ids + weights      (section 1.1)
 *   moe_dispatch_layout     per-expert / per-partition counts, one copy per
 *                           destination partition, prefix-sum layout        (sections 1.3, 3.2)
 *   moe_dispatch_pack       bf16 rows -> per-partition send regions          (sections 3.2, 5.1, 6.1)
 *   moe_permute_to_experts  receiver side: rows -> expert-contiguous runs    (sections 1.5, 3.3, 5.1)
 *   moe_combine             weighted sum of expert outputs back in token
 *                           order, fp32 accumulation, bf16 out               (sections 7.1, 7.2)
 *   moe_dispatch            route + layout + pack + permute in one call,
 *                           one launch for a decode-sized batch              (section 1.4)
 *   moe_dispatch_pack_permute  pack + permute in one pass, any layout        (sections 3.2, 5.1)
 *   moe_dispatch_pack_permute_masked  the same into the masked layout        (sections 4.1, 4.2)
 *   moe_dispatch_masked     moe_dispatch into the masked layout, one launch
 *                           for a decode-sized batch                       (sections 1.4, 4.1, 4.2)
 *
 * Further forms of the same round trip, each declared below with its source:
 *   moe_permute_to_experts_masked   a fixed block per expert plus a count     (sections 4.1, 4.2)
 *   moe_combine_stage1 / _stage2    pre-add per partition, then a home sum    (section 7.1)
 *   moe_dispatch_pack_routed,       rows that carry their ids and weights,
 *   moe_routed_expert_stage1        and the routed expert's per-partition sum (sections 6.1, 7.1)
 *   moe_dispatch_pack_mxfp8 / _nvfp4  rows quantized once before they are sent (section 7.2)
 *   moe_dispatch_quantized          moe_dispatch with MXFP8 or NVFP4 records  (section 7.2)
 *   moe_plan_placement (host),      experts placed by load with copies of the
 *   moe_dispatch_layout_mapped      hot ones ("Beyond One GPU", section 6)
 *   moe_dispatch_layout_static      the layout for callers that cannot allocate
 *   moe_expert_scale(_mxfp8/_nvfp4) stand-in experts for tests and benchmarks
 *   moe_trace_*                     optional CUDA-event timing of launches
 *   moe_dispatch_layout_kernels,    kernels one call enqueues for given sizes
 *   moe_permute_to_experts_kernels  (for counting launches per step)
 *
 * Expert-parallel ranks are emulated as partitions of buffers in one GPU's
 * memory: partition p holds the L = E/P experts p*L .. p*L+L-1 (contiguous
 * blocks, section 2.1 of the same page) unless a placement maps them.  There
 * is no peer traffic.
 *
 * Conventions for every call
 * --------------------------
 * - All array pointers are DEVICE pointers into memory the caller owns.  The
 *   library never allocates, frees or synchronises; every call is enqueued
 *   on `stream` and returns without waiting, so a chain of calls can be
 *   captured in a CUDA graph (fixed shapes, fixed addresses, no host reads of
 *   device counts -- section 1.4 of the page).
 * - bf16 arrays are passed as uint16_t bit patterns.  Row-major throughout.
 *   bf16 row arrays (x, send, recv, y, out) must be 16-byte aligned and H must
 *   be a multiple of 8 (rows are moved in 16-byte vectors).  int32/float
 *   arrays must be 4-byte aligned.
 * - Sizes: S >= 1 sources (emulated sending ranks), T >= 0 tokens per source,
 *   1 <= k <= 32 experts per token, k <= E <= 1024 experts, 1 <= P <= 32
 *   partitions with E % P == 0, H >= 8, S*T*k < 2^31, row counts < 2^31.
 *   T == 0 is a valid call that only writes the count/offset outputs.
 * - Expert ids < 0 mean "not routed": no copy is made and the slot adds
 *   nothing to the combine (section 2.1, the -1 convention; section 6.3).
 * - Host return value: MOE_OK, MOE_ERR_INVALID_ARG (bad pointer, size or
 *   alignment -- nothing is enqueued) or MOE_ERR_CUDA (a launch failed).
 *   moe_last_error_message() describes the last non-OK return of the
 *   calling thread.
 * - Data errors are found on the device and OR-ed into the caller's
 *   `dev_status` word (device pointer to one uint32_t) as MOE_STATUS_BIT(code):
 *     MOE_STATUS_BIT(MOE_ERR_INVALID_ARG)   an index input is inconsistent
 *                                           (a routed pair whose token has no
 *                                           slot in its partition)
 *     MOE_STATUS_BIT(MOE_ERR_CAPACITY)      a row did not fit under cap_send or
 *                                           cap_recv; it was dropped, never
 *                                           written out of bounds (section 4.3,
 *                                           9.2: the cap)
 *     MOE_STATUS_BIT(MOE_ERR_BAD_EXPERT_ID) an id >= E was skipped
 *   The library only sets bits; the caller clears the word when it wants.
 *   `dev_status` may be NULL, in which case data errors are not reported.
 * - Results are deterministic: the same inputs give the same bytes.
 * - Calls may be made from several host threads on different streams; the
 *   only shared state is moe_dispatch_layout_static's built-in scratch (see
 *   there) and the optional trace.  Every call opens an NVTX range named after
 *   it, so profiler timelines show which call launched which kernels.
 */
#ifndef MOE_ROUTE_H
#define MOE_ROUTE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,
    MOE_ERR_CAPACITY = 2,
    MOE_ERR_BAD_EXPERT_ID = 3,
    MOE_ERR_TIMEOUT = 4,
    MOE_ERR_CUDA = 5
} moe_status_t;

#define MOE_STATUS_BIT(code) (1u << (code))

/* Row formats of moe_dispatch_quantized. */
#define MOE_FORMAT_MXFP8 1
#define MOE_FORMAT_NVFP4 2

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int moe_version(void);

/* Static description of a status code ("ok", "invalid argument", ...). */
const char *moe_status_string(moe_status_t code);

/* Human-readable reason for the calling thread's last non-OK return
 * ("" if none).  The string is owned by the library and valid until the
 * thread's next call. */
const char *moe_last_error_message(void);

/*
 * Scratch bytes that moe_dispatch_layout and moe_permute_to_experts need for
 * the given sizes (the larger of the two).  The caller allocates it (any
 * device memory, 256-byte aligned) and may reuse it across calls that are
 * ordered on one stream.  Returns 0 for invalid sizes.
 */
size_t moe_workspace_bytes(int S, int T, int k, int E, int P);

/*
 * Number of kernels one moe_dispatch_layout call with these sizes enqueues on
 * the calling thread's current device: 1 (one chunk per source, or one
 * thread-block cluster per source) or 2 (more chunks per source than a
 * cluster of that device holds).  For counting launches, e.g. per step of a
 * captured graph.  Returns -1 for invalid sizes or a failed device query.
 */
int moe_dispatch_layout_kernels(int S, int T, int k, int E, int P);

/*
 * Number of kernels one moe_permute_to_experts call with these sizes
 * enqueues: 1 when the map step (run starts, pair rows) runs inside the copy
 * kernel, which is whenever S*E + 2*E + 1 counts fit in 48 KiB of shared
 * memory, else 2.  Returns -1 for invalid sizes.
 */
int moe_permute_to_experts_kernels(int S, int T, int k, int E, int P);

/*
 * Top-k routing (a2a-backends section 1.1: the router gives each token the
 * ids of its chosen experts and one weight per expert).
 *   logits  [S][T][E] float32, finite.
 *   topk_ids[S][T][k] int32 out: the k largest logits of the row in
 *           descending order; equal logits go to the lower expert id.
 *   topk_w  [S][T][k] float32 out: softmax over the k chosen logits,
 *           w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max), computed in fp32.
 */
moe_status_t moe_route_topk(const float *logits, int S, int T, int E, int k,
                            int32_t *topk_ids, float *topk_w, cudaStream_t stream);

/*
 * Dispatch layout (a2a-backends section 1.3, third answer, and section 3.2,
 * first step: the set of GPUs that hold at least one of a token's experts
 * and the number of rows each GPU gets).
 *   topk_ids      [S][T][k] int32 in.
 *   expert_counts [S][E]    int32 out: pairs (t, j) routed to expert e.
 *   expert_rank   [S][T][k] int32 out: place of pair (t, j) in source s's run
 *                           of its expert, i.e. #{(t', j') before (t, j) in
 *                           (token, slot) order with the same expert}; -1 for
 *                           ids < 0 or >= E.  The receiver's runs (section 1.5)
 *                           are built from it by moe_permute_to_experts.
 *   part_counts   [S][P]    int32 out: tokens with >= 1 expert in partition p
 *                           (one de-duplicated copy per token and partition).
 *   part_offsets  [S][P+1]  int32 out: exclusive prefix sum of part_counts;
 *                           part_offsets[s][P] = copies of source s.
 *   token_slot    [S][T][P] int32 out: row of token t in source s's send
 *                           buffer for partition p, or -1.  Within a
 *                           partition's region rows are in ascending token
 *                           order: token_slot = part_offsets[s][p] +
 *                           #{t' < t : t' needs p}.
 *   ws, ws_bytes  scratch, ws_bytes >= moe_workspace_bytes(S, T, k, E, P).
 *   dev_status    device uint32 status word (bad ids).
 * Work is cut into 256-token chunks, one CTA each; with 2 to 16 chunks per
 * source the chunks of a source form one thread-block cluster and exchange
 * their counts in distributed shared memory (one launch); a longer source of
 * at most 16 chunks of 1,024 tokens takes the same form with 1,024-token chunks
 * where their shared memory fits; otherwise the counts go through `ws` (two
 * launches).  Counting uses order-free integer adds and
 * ranks follow the fixed (token, slot) order, so the outputs are the same
 * bytes on every run.  The first call on a device asks the device once which
 * cluster sizes it schedules; make it before capturing a stream (a query
 * refused during a capture is asked again on the next call, and that call
 * takes the two-launch form).
 */
moe_status_t moe_dispatch_layout(const int32_t *topk_ids, int S, int T, int k, int E, int P,
                                 int32_t *expert_counts, int32_t *expert_rank,
                                 int32_t *part_counts, int32_t *part_offsets, int32_t *token_slot,
                                 void *ws, size_t ws_bytes, uint32_t *dev_status,
                                 cudaStream_t stream);

/*
 * moe_dispatch_layout without a workspace argument.  The pages have no
 * counterpart to this call; it exists for callers that have no way to
 * allocate device memory when they call the layout -- for example a plugin
 * inside a serving engine whose own pool owns every byte of device memory and
 * forbids side allocations, or plain C code with no allocator at hand.
 *
 * Same arguments, outputs and errors as moe_dispatch_layout, minus ws and
 * ws_bytes.  The scratch is a 4 MiB array built into the library (every GPU
 * that loads the library keeps it until the process exits); calls whose
 * moe_workspace_bytes(S, T, k, E, P) exceeds 4 MiB are rejected with
 * MOE_ERR_INVALID_ARG and a message naming the sizes (with E = 384 and P = 8
 * that is past about 680,000 tokens in all).  The first call on a device looks
 * up the array's device address (with that device current) and caches it;
 * make that first call before capturing any stream.  The cached address
 * belongs to the device's primary context: after cudaDeviceReset (or any
 * other teardown of that context) in the same process, do not call this entry
 * point again.  Only sizes that take the layout's two-launch form (more
 * chunks per source than one thread-block cluster holds, see
 * moe_dispatch_layout_kernels) read or write the array.  All calls share the one
 * array and it keeps the last call's contents (nothing in it needs to start
 * at zero): calls that can overlap on the GPU -- on different streams, or from
 * different threads -- race on it and must be ordered by the caller.
 */
moe_status_t moe_dispatch_layout_static(const int32_t *topk_ids, int S, int T, int k, int E,
                                        int P, int32_t *expert_counts, int32_t *expert_rank,
                                        int32_t *part_counts, int32_t *part_offsets,
                                        int32_t *token_slot, uint32_t *dev_status,
                                        cudaStream_t stream);

/*
 * Pack (a2a-backends section 3.2, fourth step; section 5.1: a region for every
 * sender, rows written straight into place; section 6.1: one copy per GPU
 * that needs the token).
 *   x            [S][T][H] bf16 in.
 *   token_slot   [S][T][P] int32 in (from moe_dispatch_layout).
 *   part_offsets [S][P+1]  int32 in (from moe_dispatch_layout).
 *   cap_send     rows of send buffer per source; T*min(k,P) always suffices.
 *   send         [S][cap_send][H] bf16 out: send[s][token_slot[s][t][p]] =
 *                x[s][t] (bit copy) for every slot >= 0.  Rows at or beyond
 *                part_offsets[s][P] are not written.
 *   send_src     [S][cap_send] int32 out: source token of each row; -1 for
 *                rows at or beyond part_offsets[s][P].
 *   Slots >= cap_send are dropped and flag MOE_ERR_CAPACITY.
 */
moe_status_t moe_dispatch_pack(const uint16_t *x, int S, int T, int H, int P,
                               const int32_t *token_slot, const int32_t *part_offsets,
                               int cap_send, uint16_t *send, int32_t *send_src,
                               uint32_t *dev_status, cudaStream_t stream);

/*
 * Routed payload (a2a-backends section 6.1: next to the hidden state the
 * sender writes the token's expert ids and weights -- payloads = hidden
 * state, top-k ids, top-k weights -- so the receiver groups nothing and hands
 * the rows to a routed expert kernel; section 6.3: empty slots carry an
 * invalid expert id so the kernel skips them).
 * moe_dispatch_pack_routed: moe_dispatch_pack plus, for every written row,
 *   send_ids[s][slot][j] = topk_ids[s][t][j], send_w[s][slot][j] = topk_w[s][t][j]
 * and id -1 / weight 0 for rows no slot names.
 *   topk_ids, topk_w [S][T][k]; send_ids [S][cap_send][k] int32 out;
 *   send_w [S][cap_send][k] float32 out; the rest as moe_dispatch_pack.
 * Rows stay where moe_dispatch_pack puts them: partition p's rows from source
 * s are [part_offsets[s][p], part_offsets[s][p+1]) in token order -- the
 * page's block of rows per sender, without padding to the largest batch.
 */
moe_status_t moe_dispatch_pack_routed(const uint16_t *x, const int32_t *topk_ids,
                                      const float *topk_w, int S, int T, int H, int k, int P,
                                      const int32_t *token_slot, const int32_t *part_offsets,
                                      int cap_send, uint16_t *send, int32_t *send_src,
                                      int32_t *send_ids, float *send_w, uint32_t *dev_status,
                                      cudaStream_t stream);

/*
 * Routed expert with the first combine stage (a2a-backends section 6.1: the
 * routed expert kernel reads each row's ids and selects its experts itself;
 * section 7.1: it already produces the weighted sum per GPU, which the home
 * side then adds up with moe_combine_stage2).  Stand-in expert (tests and
 * benchmarks, like moe_expert_scale): y_j = bf16(x * scale[e_j]), or x when
 * scale is NULL.  For every row r of partition p's region of source s, p in
 * the receiving set (recv_part, or all partitions if -1):
 *   ret[s][r] = bf16_rne( sum over ascending j with send_ids[s][r][j] in
 *               partition p of send_w[s][r][j] * y_j ), fp32 fused multiply-adds
 * -- the same bytes as moe_expert_scale + moe_combine_stage1 over the
 * permuted rows.  Rows outside the receiving regions are not written; ids >= E
 * are skipped and flag MOE_ERR_BAD_EXPERT_ID.
 *   send [S][cap_send][H] bf16; send_ids, send_w [S][cap_send][k];
 *   part_offsets [S][P+1]; scale [E] float32 or NULL; ret [S][cap_send][H] bf16 out.
 *   T: tokens per source (a partition's region of one source holds at most T
 *   rows, which bounds the work when one partition receives).
 */
moe_status_t moe_routed_expert_stage1(const uint16_t *send, const int32_t *send_ids,
                                      const float *send_w, const int32_t *part_offsets, int S,
                                      int T, int cap_send, int k, int E, int P, int H,
                                      int recv_part, const float *scale, uint16_t *ret,
                                      uint32_t *dev_status, cudaStream_t stream);

/*
 * Expert placement by load with redundant copies of the hot experts ("Beyond
 * One GPU", section 6, "The fix: place experts by load, and copy the hot
 * ones").  HOST function: all pointers are host memory; no GPU is used.
 *  1. Heaviest expert first (equal loads: lower id first), each onto the
 *     least-loaded partition (equal loads: lower index) that still has one of
 *     its E/P regular slots free.
 *  2. Every partition also has R spare slots.  Repeatedly: take the busiest
 *     partition (ties: lower index) and its expert with the largest share
 *     (ties: lower id); copy it to the least-loaded partition that has a
 *     spare slot free and no copy of it yet.  The copy is kept only if that
 *     partition's new load stays below the busiest partition's load; the
 *     first copy that fails this, or the lack of a free spare slot, ends it.
 * Loads are integer pair counts split over an expert's n copies as the
 * mapped layout splits them: copy c carries ceil((load - c) / n).
 *   load          [E] int64 in: pairs per logical expert in a past batch.
 *   copy_offsets  [E+1] int32 out; copy_slots [E + P*R] int32 out: the slots
 *                 of expert e are copy_slots[copy_offsets[e] .. copy_offsets[e+1]),
 *                 the original first, then its copies in the order made.
 *   slot_expert   [P*(E/P+R)] int32 out: logical expert in each physical slot,
 *                 -1 if empty.  Partition p owns slots [p*Lp, (p+1)*Lp),
 *                 Lp = E/P + R, filled in the order experts arrive there.
 *   part_load     [P] int64 out: pairs per partition after the copies.
 * Errors: MOE_ERR_INVALID_ARG (E % P != 0, P*Lp > 1024, a negative load, null).
 */
moe_status_t moe_plan_placement(const int64_t *load, int E, int P, int R, int32_t *copy_offsets,
                                int32_t *copy_slots, int32_t *slot_expert, int64_t *part_load);

/*
 * Dispatch layout over a placement (same section: a replicated expert's
 * tokens are split evenly between its copies).  For each source, the r-th
 * pair of logical expert e in (token, choice) order goes to physical slot
 *   phys_ids[s][t][j] = copy_slots[copy_offsets[e] + (r mod n_e)],
 * n_e = copy_offsets[e+1] - copy_offsets[e]; ids < 0 give -1, ids >= E give
 * P*Lp (flagged MOE_ERR_BAD_EXPERT_ID).  The outputs are then exactly those
 * of moe_dispatch_layout over phys_ids with P*Lp experts (partition of a
 * slot = slot / Lp), so moe_permute_to_experts and the combine run unchanged
 * with E = P*Lp and topk_ids = phys_ids.
 *   copy_offsets [E+1], copy_slots [n_copies] int32 device arrays (from
 *   moe_plan_placement or the caller); a copy list that leaves
 *   [0, n_copies) or a slot outside [0, P*Lp) flags MOE_ERR_INVALID_ARG and
 *   the pair becomes -1.
 *   expert_counts [S][P*Lp]; the other outputs as moe_dispatch_layout.
 *   ws: moe_workspace_bytes_mapped(S, T, k, E, P, Lp) bytes, 256-byte aligned.
 * n_copies must equal copy_offsets[E].  Five kernels: the layout over logical
 * ids (for the ranks r), the map, the layout over physical ids; three when
 * n_copies == E (no expert has copies, so no ranks are needed).
 */
size_t moe_workspace_bytes_mapped(int S, int T, int k, int E, int P, int Lp);
moe_status_t moe_dispatch_layout_mapped(const int32_t *topk_ids, int S, int T, int k, int E,
                                        int P, int Lp, const int32_t *copy_offsets,
                                        const int32_t *copy_slots, int n_copies,
                                        int32_t *phys_ids, int32_t *expert_counts,
                                        int32_t *expert_rank, int32_t *part_counts,
                                        int32_t *part_offsets, int32_t *token_slot, void *ws,
                                        size_t ws_bytes, uint32_t *dev_status,
                                        cudaStream_t stream);

/*
 * Pack with the rows quantized on the way (a2a-backends section 7.2: expert
 * kernels that quantize their input anyway can take rows already quantized,
 * so a token is converted before it is sent; a DeepSeek-V4.1-Flash FP8 row is
 * 5,280 bytes: 5,120 one-byte values and a one-byte scale per 32 values).
 * A quantized row is one record of H + H/32 bytes: the H E4M3 codes, then the
 * H/32 E8M0 block scales.  Encoding (the page fixes only the sizes): OCP
 * MXFP8, per block of 32 values
 *   X = 2^(floor(log2 max|v|) - 8), clamped to [2^-127, 2^127]; scale byte = log2 X + 127
 *   code_i = e4m3(v_i / X), round to nearest even, magnitudes above 448 -> 448
 * An all-zero block gets scale byte 0.  x must be finite.
 *   x            [S][T][H] bf16 in; H a multiple of 256 (8-byte aligned records).
 *   send_q       [S][cap_send][H + H/32] uint8 out, 8-byte aligned.  Rows that no
 *                slot names are not written.
 *   token_slot, part_offsets, cap_send, send_src, dev_status: as moe_dispatch_pack.
 * The records move through moe_permute_to_experts(_masked) as opaque rows of
 * (H + H/32)/2 bf16 slots, which needs H % 512 == 0.
 * Errors: as moe_dispatch_pack.
 */
moe_status_t moe_dispatch_pack_mxfp8(const uint16_t *x, int S, int T, int H, int P,
                                     const int32_t *token_slot, const int32_t *part_offsets,
                                     int cap_send, uint8_t *send_q, int32_t *send_src,
                                     uint32_t *dev_status, cudaStream_t stream);

/*
 * Pack with NVFP4 records (a2a-backends section 7.2: FlashInfer's all-to-all
 * sends NVFP4 rows when the expert kernel takes them; an NVFP4 row of a
 * DeepSeek-V4.1-Flash token is 2,880 bytes, a one-byte scale for every 16 of
 * its 5,120 values).  Encoding (the page fixes only the size): NVIDIA's NVFP4
 * with the per-tensor fp32 scale g = global_scale given by the caller (it is
 * not part of a row).  Per block of 16 values, in fp32 with correctly
 * rounded division:
 *   s = e4m3_rn_satfinite( amax / (6 g) ),  code_i = e2m1_rn_satfinite( v_i / (s g) )
 * and all codes 0 when s is 0.  A record is H/2 bytes of E2M1 codes (element
 * 2i in the low nibble), then H/16 bytes of E4M3 scales.
 *   x       [S][T][H] bf16 in; H a multiple of 256.
 *   send_q  [S][cap_send][H/2 + H/16] uint8 out, 16-byte aligned; rows no slot
 *           names are not written.
 *   token_slot, part_offsets, cap_send, send_src, dev_status: as moe_dispatch_pack.
 * The records move through moe_permute_to_experts as opaque rows of
 * (H/2 + H/16)/2 bf16 slots.  Errors: as moe_dispatch_pack; g must be positive.
 */
moe_status_t moe_dispatch_pack_nvfp4(const uint16_t *x, int S, int T, int H, int P,
                                     float global_scale, const int32_t *token_slot,
                                     const int32_t *part_offsets, int cap_send, uint8_t *send_q,
                                     int32_t *send_src, uint32_t *dev_status, cudaStream_t stream);

/*
 * Receiver permute into expert-contiguous runs (a2a-backends section 1.5:
 * the contiguous layout, runs optionally padded to a multiple of `align`
 * rows as DeepGEMM wants 128; section 3.3: one row per (token, local
 * expert); section 5.1: the copy epilogue with device-side offsets).
 *   send, token_slot, topk_ids   as produced/consumed above; cap_send as in pack.
 *   expert_counts, expert_rank   from moe_dispatch_layout for the same topk_ids
 *              (a pair whose rank is outside [0, expert_counts) is skipped
 *              and flags MOE_ERR_INVALID_ARG).
 *   recv_part  receiving partition in [0, P), or -1 for all partitions.
 *   align      run alignment in rows, 1 <= align <= 1024.
 *   cap_recv   rows of recv; S*T*k + E*(align-1) always suffices.
 *   recv       [cap_recv][H] bf16 out.  For each expert e of the receiving
 *              set in ascending order, its run starts at expert_offsets[e]
 *              and holds the pairs (s, t, j) with topk_ids[s][t][j] == e in
 *              ascending (s, t, j) order, each a copy of
 *              send[s][token_slot[s][t][e / L]]; padding rows are zero.
 *              Rows at or beyond min(expert_offsets[E], cap_recv) are not
 *              written.
 *   expert_offsets [E+1] int32 out: run starts; experts outside the
 *              receiving set have empty runs.  expert_offsets[E] = rows used
 *              (may exceed cap_recv, then MOE_ERR_CAPACITY is flagged).
 *   pair_row   [S][T][k] int32 out: recv row of each pair, or -1 (id < 0,
 *              expert outside the receiving set, or row >= cap_recv).
 *   recv_pair  [cap_recv] int32 out: (s*T + t)*k + j for pair rows, -1 for
 *              padding rows and rows >= expert_offsets[E].
 *   ws, ws_bytes  scratch, ws_bytes >= moe_workspace_bytes(S, T, k, E, P).
 * A routed pair whose slot is -1 (inconsistent inputs) or >= cap_send gets a
 * zero row and flags MOE_ERR_INVALID_ARG or MOE_ERR_CAPACITY respectively.
 * One kernel both places and copies the rows while the S*E counts fit in its
 * shared memory (moe_permute_to_experts_kernels), else a placement kernel
 * runs first; the results are the same.
 */
moe_status_t moe_permute_to_experts(const uint16_t *send, const int32_t *token_slot,
                                    const int32_t *topk_ids, const int32_t *expert_counts,
                                    const int32_t *expert_rank, int S, int T, int k, int E,
                                    int P, int H, int recv_part, int align, int cap_send,
                                    int cap_recv, uint16_t *recv, int32_t *expert_offsets,
                                    int32_t *pair_row, int32_t *recv_pair, void *ws,
                                    size_t ws_bytes, uint32_t *dev_status, cudaStream_t stream);

/*
 * The dispatch side in one call: moe_route_topk, moe_dispatch_layout,
 * moe_dispatch_pack and moe_permute_to_experts on the same arguments, with
 * the same outputs byte for byte, in fewer launches (a2a-backends section 1.4:
 * a decode step makes a round trip per MoE layer, so its fixed cost per call
 * matters; sections 1.1, 1.3, 3.2, 3.3, 5.1 for the steps).
 *   logits [S][T][E] fp32 in; x [S][T][H] bf16 in.
 *   topk_ids, topk_w                   out, as moe_route_topk.
 *   expert_counts, expert_rank, part_counts, part_offsets, token_slot
 *                                      out, as moe_dispatch_layout.
 *   send, send_src, cap_send           as moe_dispatch_pack.
 *   recv, expert_offsets, pair_row, recv_pair, recv_part, align, cap_recv
 *                                      as moe_permute_to_experts.
 *   ws, ws_bytes  scratch, ws_bytes >= moe_workspace_bytes(S, T, k, E, P).
 * Forms (moe_dispatch_kernels reports the launch count):
 *   - one source of 1..256 tokens: one kernel.  Clusters of 8 CTAs route the
 *     batch, every CTA lays it out in its own shared memory, then the grid
 *     moves the rows;
 *   - otherwise: the routing kernel, the layout's kernel(s), then one kernel
 *     that packs and permutes in the same pass (or the separate pack and
 *     permute when the S*E counts do not fit its shared memory, and for T = 0).
 * In both, the receive rows are read from the send rows of the receiving
 * partitions right after they are stored (by the same warp), so the bytes
 * placed in recv are the bytes in send, as in the separate calls.
 * Errors: those of the four calls.  Routing never produces an id < 0 or >= E.
 */
moe_status_t moe_dispatch(const float *logits, const uint16_t *x, int S, int T, int H, int E,
                          int k, int P, int recv_part, int align, int cap_send, int cap_recv,
                          int32_t *topk_ids, float *topk_w, int32_t *expert_counts,
                          int32_t *expert_rank, int32_t *part_counts, int32_t *part_offsets,
                          int32_t *token_slot, uint16_t *send, int32_t *send_src, uint16_t *recv,
                          int32_t *expert_offsets, int32_t *pair_row, int32_t *recv_pair,
                          void *ws, size_t ws_bytes, uint32_t *dev_status, cudaStream_t stream);

/*
 * Kernels one moe_dispatch call with these sizes enqueues on the calling
 * thread's current device (1 for the one-launch form); -1 for invalid sizes.
 */
int moe_dispatch_kernels(int S, int T, int k, int E, int P);

/*
 * Pack and permute in one call, for a layout the caller computed (for example
 * moe_dispatch_layout_mapped over a placement with expert copies): the outputs
 * of moe_dispatch_pack followed by moe_permute_to_experts with the same
 * arguments, byte for byte, from one pass over the rows while the S*E counts
 * fit one CTA's shared memory (each row segment read once from x, stored to
 * the token's send rows, the receiving partitions' send rows read back right
 * after and stored to the pair rows); otherwise, and for T = 0, the two
 * separate calls' kernels.  Arguments and errors as those two calls (x, part_offsets
 * and send_src from moe_dispatch_pack; the rest from moe_permute_to_experts).
 * moe_dispatch_pack_permute_kernels reports the kernels it enqueues (-1 for
 * invalid sizes).
 */
moe_status_t moe_dispatch_pack_permute(const uint16_t *x, const int32_t *token_slot,
                                       const int32_t *part_offsets, const int32_t *topk_ids,
                                       const int32_t *expert_counts, const int32_t *expert_rank,
                                       int S, int T, int k, int E, int P, int H, int recv_part,
                                       int align, int cap_send, int cap_recv, uint16_t *send,
                                       int32_t *send_src, uint16_t *recv,
                                       int32_t *expert_offsets, int32_t *pair_row,
                                       int32_t *recv_pair, void *ws, size_t ws_bytes,
                                       uint32_t *dev_status, cudaStream_t stream);
int moe_dispatch_pack_permute_kernels(int S, int T, int k, int E, int P);

/*
 * Pack and the masked receive layout in one call: the outputs of
 * moe_dispatch_pack followed by moe_permute_to_experts_masked with the same
 * arguments, byte for byte (a2a-backends sections 4.1, 4.2), from one pass
 * over the rows while the per-block counts of all sources fit one CTA's
 * shared memory ((2 + S) * blocks ints <= 48 KiB), else (and for T = 0) the
 * separate calls' kernels; moe_dispatch_pack_permute_masked_kernels reports
 * the count (-1 for invalid sizes).  Arguments and errors as those two calls.
 */
moe_status_t moe_dispatch_pack_permute_masked(const uint16_t *x, const int32_t *token_slot,
                                              const int32_t *part_offsets,
                                              const int32_t *topk_ids,
                                              const int32_t *expert_counts,
                                              const int32_t *expert_rank, int S, int T, int k,
                                              int E, int P, int H, int recv_part, int block_rows,
                                              int cap_send, uint16_t *send, int32_t *send_src,
                                              uint16_t *recv, int32_t *masked_counts,
                                              int32_t *pair_row, int32_t *recv_pair,
                                              uint32_t *dev_status, cudaStream_t stream);
int moe_dispatch_pack_permute_masked_kernels(int S, int T, int k, int E, int P, int recv_part);

/*
 * The dispatch side in one call with the masked receive layout: the outputs of
 * moe_route_topk, moe_dispatch_layout, moe_dispatch_pack and
 * moe_permute_to_experts_masked on the same arguments, byte for byte
 * (a2a-backends sections 4.1, 4.2: the layout a decode step records in a CUDA
 * graph, fixed blocks per expert and a count per block; section 1.4 for the
 * launch count).
 *   logits [S][T][E] fp32 in; x [S][T][H] bf16 in.
 *   topk_ids, topk_w                   out, as moe_route_topk.
 *   expert_counts, expert_rank, part_counts, part_offsets, token_slot
 *                                      out, as moe_dispatch_layout.
 *   send, send_src, cap_send           as moe_dispatch_pack.
 *   recv, masked_counts, pair_row, recv_pair, recv_part, block_rows
 *                                      as moe_permute_to_experts_masked.
 *   ws, ws_bytes  scratch, ws_bytes >= moe_workspace_bytes(S, T, k, E, P).
 * Forms (moe_dispatch_masked_kernels reports the launch count, -1 for invalid
 * sizes): one source of 1..256 tokens, one kernel (as moe_dispatch's one-launch
 * form, each pair placed in its expert's block); otherwise the routing kernel,
 * the layout's kernel(s) and moe_dispatch_pack_permute_masked's kernel(s).
 * Errors: those of the four calls.  Routing never produces an id < 0 or >= E.
 */
moe_status_t moe_dispatch_masked(const float *logits, const uint16_t *x, int S, int T, int H,
                                 int E, int k, int P, int recv_part, int block_rows,
                                 int cap_send, int32_t *topk_ids, float *topk_w,
                                 int32_t *expert_counts, int32_t *expert_rank,
                                 int32_t *part_counts, int32_t *part_offsets,
                                 int32_t *token_slot, uint16_t *send, int32_t *send_src,
                                 uint16_t *recv, int32_t *masked_counts, int32_t *pair_row,
                                 int32_t *recv_pair, void *ws, size_t ws_bytes,
                                 uint32_t *dev_status, cudaStream_t stream);
int moe_dispatch_masked_kernels(int S, int T, int k, int E, int P, int recv_part);

/*
 * moe_dispatch with the rows sent as quantized records (a2a-backends section
 * 7.2: tokens are converted before they are sent): the outputs of
 * moe_route_topk, moe_dispatch_layout, moe_dispatch_pack_mxfp8 (format
 * MOE_FORMAT_MXFP8, H a multiple of 512) or moe_dispatch_pack_nvfp4 (format
 * MOE_FORMAT_NVFP4, H a multiple of 256, global_scale its tensor scale g) and
 * moe_permute_to_experts of the records as opaque rows, byte for byte.
 *   send_q  [S][cap_send][rb] uint8 out, recv_q [cap_recv][rb] uint8 out, both
 *           16-byte aligned; rb = H + H/32 (MXFP8) or H/2 + H/16 (NVFP4).
 *   The other arguments and the errors are those of moe_dispatch (plus a bad
 *   format, H or global_scale: MOE_ERR_INVALID_ARG).
 * Kernels: for one source of 1..256 tokens one kernel (as moe_dispatch's
 * one-launch form, each row segment quantized once); otherwise the routing
 * kernel, the layout's kernel(s), then one pass that quantizes each row
 * segment once, stores the piece to the token's send records, reads each
 * receiving partition's piece back and stores it to the pair records (the
 * separate pack and permute for T = 0 or when the S*E counts do not fit one
 * CTA's shared memory); moe_dispatch_quantized_kernels reports the count (-1
 * for invalid sizes).
 */
moe_status_t moe_dispatch_quantized(const float *logits, const uint16_t *x, int S, int T, int H,
                                    int E, int k, int P, int format, float global_scale,
                                    int recv_part, int align, int cap_send, int cap_recv,
                                    int32_t *topk_ids, float *topk_w, int32_t *expert_counts,
                                    int32_t *expert_rank, int32_t *part_counts,
                                    int32_t *part_offsets, int32_t *token_slot, uint8_t *send_q,
                                    int32_t *send_src, uint8_t *recv_q, int32_t *expert_offsets,
                                    int32_t *pair_row, int32_t *recv_pair, void *ws,
                                    size_t ws_bytes, uint32_t *dev_status, cudaStream_t stream);
int moe_dispatch_quantized_kernels(int S, int T, int k, int E, int P);

/*
 * Masked receive layout (a2a-backends section 4.1: a region per (local expert,
 * sender) with room for the cap; section 4.2: the receiver packs each expert's
 * rows together, writes a per-expert count on the device, and the output has a
 * fixed shape -- 48 x 8 x 128 rows for the decode example; section 5.2: the
 * masked expert kernel reads fixed-size blocks).
 *   Same inputs as moe_permute_to_experts.  The receiving set (recv_part, or
 *   all experts if -1) has nb experts; expert b of the set owns rows
 *   [b*block_rows, (b+1)*block_rows) of recv.
 *   recv          [nb*block_rows][H] bf16 out: the pairs of each expert in
 *                 ascending (s, t, j) order from the first row of its block;
 *                 rows past masked_counts[b] are not written.
 *   masked_counts [nb] int32 out: rows of each block in use (<= block_rows).
 *   pair_row      [S][T][k] int32 out: row of each pair or -1.
 *   recv_pair     [nb*block_rows] int32 out: pair id of used rows, -1 otherwise.
 * Pairs past a block's end are dropped and flag MOE_ERR_CAPACITY (the page's
 * "the call fails if the batch is larger than the cap", here without failing).
 * Needs no workspace.  moe_combine reads this layout through pair_row.
 */
moe_status_t moe_permute_to_experts_masked(const uint16_t *send, const int32_t *token_slot,
                                           const int32_t *topk_ids, const int32_t *expert_counts,
                                           const int32_t *expert_rank, int S, int T, int k,
                                           int E, int P, int H, int recv_part, int block_rows,
                                           int cap_send, uint16_t *recv, int32_t *masked_counts,
                                           int32_t *pair_row, int32_t *recv_pair,
                                           uint32_t *dev_status, cudaStream_t stream);

/*
 * Weighted combine (a2a-backends section 1.1: the MoE output is the sum of
 * the chosen experts' outputs, each multiplied by its weight; section 7.1:
 * the home side sums in 32-bit floats; section 7.2: bf16 on the wire).
 *   y        [y_rows][H] bf16 in: expert outputs in the recv layout.
 *   pair_row [S][T][k] int32 in (from moe_permute_to_experts); entries
 *            >= y_rows are skipped and flag MOE_ERR_INVALID_ARG.
 *   topk_w   [S][T][k] float32 in.
 *   out      [S][T][H] bf16 out: out[s][t] = bf16_rne( sum over j in
 *            ascending order with pair_row >= 0 of topk_w * float(y[row]) ),
 *            accumulated with fp32 fused multiply-adds; +0 if no pair.
 * With a single receiving partition this is that partition's partial
 * (stage-1) combine; the partials of all partitions add up to the full one.
 */
moe_status_t moe_combine(const uint16_t *y, int y_rows, const int32_t *pair_row,
                         const float *topk_w, int S, int T, int k, int H, uint16_t *out,
                         uint32_t *dev_status, cudaStream_t stream);

/*
 * Two-stage combine (a2a-backends section 7.1: the weighted sum over a token's
 * experts splits into a sum over the experts that sit on one GPU, taken before
 * the rows travel back -- DeepEP's combine and FlashInfer's routed kernel
 * pre-add there -- and a sum over GPUs at home; each token then returns as
 * many rows as it sent, about 4.43 instead of 6 for the page's model;
 * section 7.2: the returned rows are bf16).
 *
 * moe_combine_stage1 (expert side), for every (s, t, p) with p in the
 * receiving set (recv_part, or all partitions if -1) and a send slot
 * 0 <= token_slot[s][t][p] < cap_send:
 *   ret[s][slot] = bf16_rne( sum over j in ascending order with pair_row >= 0
 *                  and topk_ids[s][t][j] in partition p of topk_w * float(y[row]) )
 *   y [y_rows][H] bf16 (expert outputs, contiguous or masked layout, addressed
 *   by pair_row); ret [S][cap_send][H] bf16 (the send layout).  Rows of ret
 *   without such a slot are not written.  pair_row >= y_rows is skipped and
 *   flags MOE_ERR_INVALID_ARG.
 * moe_combine_stage2 (home side): over the partitions p of the receiving set
 * (recv_part, or all if -1 -- with one receiving partition only its rows come
 * back, so the result is that partition's partial combine):
 *   out[s][t] = bf16_rne( sum over p ascending with 0 <= token_slot < cap_send
 *               of float(ret[s][token_slot[s][t][p]]) ), fp32 adds; +0 if none.
 * Slots >= cap_send flag MOE_ERR_CAPACITY in both stages.
 */
moe_status_t moe_combine_stage1(const uint16_t *y, int y_rows, const int32_t *pair_row,
                                const float *topk_w, const int32_t *topk_ids,
                                const int32_t *token_slot, int S, int T, int k, int E, int P,
                                int H, int recv_part, int cap_send, uint16_t *ret,
                                uint32_t *dev_status, cudaStream_t stream);
moe_status_t moe_combine_stage2(const uint16_t *ret, const int32_t *token_slot, int S, int T,
                                int P, int H, int recv_part, int cap_send, uint16_t *out,
                                uint32_t *dev_status, cudaStream_t stream);

/*
 * Stand-in expert for tests and benchmarks -- NOT a step of the method (the
 * pages time dispatch and combine without the expert kernel, a2a-backends
 * section 8.1).  y[r] = bf16_rne(float(recv[r]) * scale[e]) for every row r
 * of expert e's run, r < min(expert_offsets[E], cap_recv).
 *   recv, y [cap_recv][H] bf16; expert_offsets [E+1] int32; scale [E] float32.
 */
moe_status_t moe_expert_scale(const uint16_t *recv, const int32_t *expert_offsets,
                              const float *scale, int E, int H, int cap_recv, uint16_t *y,
                              cudaStream_t stream);

/*
 * Stand-in expert on MXFP8 records (harness, like moe_expert_scale): for each
 * row r of expert e's run, y[r][h] = bf16( scale[e] * e4m3(code[r][h]) *
 * 2^(scale_byte[r][h/32] - 127) ).  The product code * scale[e] is rounded to
 * fp32 before the power of two, so y may differ from the exactly rounded value
 * by one bf16 unit.
 *   recv_q  [cap_recv][H + H/32] uint8 records (moe_dispatch_pack_mxfp8), 8-byte aligned.
 *   y       [cap_recv][H] bf16 out, 16-byte aligned; rows at or beyond
 *           min(expert_offsets[E], cap_recv) are not written.
 *   H a multiple of 256.  Errors: MOE_ERR_INVALID_ARG / MOE_ERR_CUDA.
 */
moe_status_t moe_expert_scale_mxfp8(const uint8_t *recv_q, const int32_t *expert_offsets,
                                    const float *scale, int E, int H, int cap_recv, uint16_t *y,
                                    cudaStream_t stream);

/*
 * Stand-in expert on NVFP4 records (harness, like moe_expert_scale):
 *   y[r][h] = bf16( scale[e] * e2m1(code) * e4m3(block scale) * global_scale )
 * code * block scale is exact in fp32; scale[e] * global_scale is one fp32
 * product, so y may differ from the exactly rounded value by one bf16 unit.
 *   recv_q [cap_recv][H/2 + H/16] uint8 (16-byte aligned); y [cap_recv][H] bf16 out.
 */
moe_status_t moe_expert_scale_nvfp4(const uint8_t *recv_q, const int32_t *expert_offsets,
                                    const float *scale, int E, int H, float global_scale,
                                    int cap_recv, uint16_t *y, cudaStream_t stream);

/*
 * Per-kernel timing (tracing aid; off by default).  While enabled, every
 * kernel launch of this library whose name contains `kernel_filter` (all of
 * them if NULL or "") is bracketed by two CUDA events recorded on the
 * launch's stream, up to max_records launches.  moe_trace_enable creates the
 * events (host handles only, no device memory) and clears earlier records;
 * moe_trace_get(i) waits for record i to finish and returns the kernel name
 * (static string) and its duration in ms.  Launches captured into a CUDA graph
 * while tracing is on get event nodes in the graph; each replay re-records
 * them and moe_trace_get returns the latest replay's duration.
 */
moe_status_t moe_trace_enable(const char *kernel_filter, int max_records);
void moe_trace_disable(void);
void moe_trace_reset(void);
int moe_trace_count(void);
moe_status_t moe_trace_get(int i, const char **kernel_name, float *ms);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTE_H */
