// placement.cu -- experts placed by load with redundant copies of the hot
// ones, and the dispatch layout over such a placement ("Beyond One GPU",
// section 6, "The fix: place experts by load, and copy the hot ones").
//
// The plan is host code: it runs when the load statistics are refreshed, not
// per step.  Per step, a placement changes only which physical expert slot
// each (token, choice) pair goes to; every later call of the path (pack,
// permute, combine) works on physical slots exactly as on experts.
//
// Split rule: the r-th pair of logical expert e from one source, in (token,
// choice) order, goes to copy r mod n_e.  Copy c therefore receives
// #{r < load : r mod n = c} = ceil((load - c) / n) pairs, the same integer
// share the planner uses to predict loads.
#include <algorithm>
#include <numeric>
#include <vector>

#include "common.cuh"
#include "launch.h"
#include "trace.h"

namespace moe {

namespace {

int64_t copy_share(int64_t load, int n, int c)
{
    return load > c ? (load - c + n - 1) / n : 0;
}

struct Plan {
    int E, P, R, Lb, Lp;
    std::vector<std::vector<int>> slots;    // per expert: its slots, original first
    std::vector<int> used;                  // slots filled per partition
    std::vector<int64_t> pload;             // pairs per partition under the split rule
    std::vector<int32_t> slot_expert;

    // partition load contributed by expert e's copies (added with sign +1/-1)
    void account(const int64_t *load, int e, int sign)
    {
        const int n = (int)slots[e].size();
        for (int c = 0; c < n; c++) pload[slots[e][c] / Lp] += sign * copy_share(load[e], n, c);
    }
    bool holds(int p, int e) const
    {
        for (int s : slots[e])
            if (s / Lp == p) return true;
        return false;
    }
    int take_slot(int p, int e)
    {
        const int s = p * Lp + used[p]++;
        slot_expert[s] = e;
        slots[e].push_back(s);
        return s;
    }
};

}  // namespace

int plan_placement(const int64_t *load, int E, int P, int R, int32_t *copy_offsets,
                   int32_t *copy_slots, int32_t *slot_expert, int64_t *part_load)
{
    Plan pl;
    pl.E = E;
    pl.P = P;
    pl.R = R;
    pl.Lb = E / P;
    pl.Lp = E / P + R;
    pl.slots.assign(E, {});
    pl.used.assign(P, 0);
    pl.pload.assign(P, 0);
    pl.slot_expert.assign((size_t)P * pl.Lp, -1);

    // 1. heaviest expert first (stable: equal loads keep the lower id first),
    //    each onto the least-loaded partition with a regular slot free
    std::vector<int> order(E);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return load[a] > load[b]; });
    for (int e : order) {
        int q = -1;
        for (int p = 0; p < P; p++)
            if (pl.used[p] < pl.Lb && (q < 0 || pl.pload[p] < pl.pload[q])) q = p;
        pl.take_slot(q, e);
        pl.pload[q] += load[e];
    }

    // 2. copies of the busiest partition's busiest expert into spare slots
    for (;;) {
        const int g = (int)(std::max_element(pl.pload.begin(), pl.pload.end()) - pl.pload.begin());
        int hot = -1;
        int64_t hot_share = -1;
        for (int i = 0; i < pl.Lp; i++) {
            const int e = pl.slot_expert[(size_t)g * pl.Lp + i];
            if (e < 0) continue;
            const int n = (int)pl.slots[e].size();
            int c = 0;
            while (pl.slots[e][c] / pl.Lp != g) c++;
            const int64_t sh = copy_share(load[e], n, c);
            if (sh > hot_share || (sh == hot_share && e < hot)) {
                hot_share = sh;
                hot = e;
            }
        }
        if (hot < 0) break;
        int tgt = -1;
        for (int p = 0; p < P; p++) {
            if (pl.used[p] >= pl.Lp || pl.holds(p, hot)) continue;
            if (tgt < 0 || pl.pload[p] < pl.pload[tgt]) tgt = p;
        }
        if (tgt < 0) break;
        const int n1 = (int)pl.slots[hot].size() + 1;
        // kept only if the receiving partition stays below the busiest one
        if (!(pl.pload[tgt] + copy_share(load[hot], n1, n1 - 1) < pl.pload[g])) break;
        pl.account(load, hot, -1);
        pl.take_slot(tgt, hot);
        pl.account(load, hot, +1);
    }

    int o = 0;
    for (int e = 0; e < E; e++) {
        copy_offsets[e] = o;
        for (int s : pl.slots[e]) copy_slots[o++] = s;
    }
    copy_offsets[E] = o;
    std::copy(pl.slot_expert.begin(), pl.slot_expert.end(), slot_expert);
    std::copy(pl.pload.begin(), pl.pload.end(), part_load);
    return o;
}

namespace {

// Physical slot of every pair from the pair's rank among its source's pairs
// of the same logical expert (computed by the layout over logical ids); with
// rank == nullptr every expert has one slot and the rank is not needed.
__global__ void __launch_bounds__(256) k_map_replicas(
    const int32_t *__restrict__ ids, const int32_t *__restrict__ rank, int64_t n_pairs, int E,
    int E_phys, const int32_t *__restrict__ copy_offsets, const int32_t *__restrict__ copy_slots,
    int n_copies, int32_t *__restrict__ phys, uint32_t *dev_status)
{
    pdl_wait();
    pdl_trigger();
    bool bad = false;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_pairs;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int e = __ldg(ids + i);
        int out = -1;
        if (e >= E) {
            out = E_phys;                   // the layout over physical ids flags it
        } else if (e >= 0) {
            const int r = rank ? __ldg(rank + i) : 0;
            const int o0 = __ldg(copy_offsets + e), n = __ldg(copy_offsets + e + 1) - o0;
            if (r < 0 || n < 1 || o0 < 0 || o0 + n > n_copies) {
                bad = true;
            } else {
                const int s = __ldg(copy_slots + o0 + r % n);
                if (s < 0 || s >= E_phys) bad = true;
                else out = s;
            }
        }
        phys[i] = out;
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(dev_status, MOE_ERR_INVALID_ARG);
}

// Scratch of the mapped layout, carved from the caller's workspace.
struct MappedWs {
    int32_t *ec1, *rk1, *pc1, *po1, *ts1;
    void *inner;
};

size_t up256(size_t b) { return (b + 255) / 256 * 256; }

MappedWs carve(void *ws, int S, int T, int k, int E)
{
    char *p = (char *)ws;
    MappedWs m;
    m.ec1 = (int32_t *)p;
    p += up256((size_t)S * E * 4);
    m.rk1 = (int32_t *)p;
    p += up256((size_t)S * T * k * 4);
    m.pc1 = (int32_t *)p;
    p += up256((size_t)S * 4);
    m.po1 = (int32_t *)p;
    p += up256((size_t)S * 2 * 4);
    m.ts1 = (int32_t *)p;
    p += up256((size_t)S * T * 4);
    m.inner = p;
    return m;
}

}  // namespace

size_t mapped_ws_bytes(int S, int T, int k, int E, int P, int E_phys)
{
    const size_t a = layout_ws_bytes(S, T, E, 1), b = layout_ws_bytes(S, T, E_phys, P);
    return up256((size_t)S * E * 4) + up256((size_t)S * T * k * 4) + up256((size_t)S * 4) +
           up256((size_t)S * 2 * 4) + up256((size_t)S * T * 4) + up256(a > b ? a : b);
}

cudaError_t launch_dispatch_layout_mapped(const int32_t *ids, int S, int T, int k, int E, int P,
                                          int E_phys, const int32_t *copy_offsets,
                                          const int32_t *copy_slots, int n_copies,
                                          int32_t *phys, int32_t *expert_counts,
                                          int32_t *expert_rank, int32_t *part_counts,
                                          int32_t *part_offsets, int32_t *token_slot, void *ws,
                                          uint32_t *dev_status, cudaStream_t st)
{
    const MappedWs m = carve(ws, S, T, k, E);
    // ranks among each source's pairs of each logical expert -- needed only
    // when some expert has copies (n_copies > E; every expert has at least one)
    const bool copies = n_copies > E;
    cudaError_t e = cudaSuccess;
    if (copies) {
        e = launch_dispatch_layout(ids, S, T, k, E, 1, m.ec1, m.rk1, m.pc1, m.po1, m.ts1, m.inner,
                                   dev_status, st);
        if (e != cudaSuccess) return e;
    }
    const int64_t n_pairs = (int64_t)S * T * k;
    if (n_pairs > 0) {
        DeviceInfo di;
        if ((e = device_info(&di)) != cudaSuccess) return e;
        int64_t blocks = (n_pairs + 255) / 256;
        if (blocks > (int64_t)di.sm_count * 8) blocks = (int64_t)di.sm_count * 8;
        MOE_TRACED_LAUNCH("k_map_replicas", st,
                          e = launch_pdl(k_map_replicas, dim3((unsigned)blocks), dim3(256), 0, st,
                                         ids, copies ? (const int32_t *)m.rk1 : nullptr, n_pairs,
                                         E, E_phys,
                                         copy_offsets, copy_slots, n_copies, phys, dev_status));
        if (e != cudaSuccess) return e;
    }
    // the ordinary layout over physical slots
    return launch_dispatch_layout(phys, S, T, k, E_phys, P, expert_counts, expert_rank,
                                  part_counts, part_offsets, token_slot, m.inner, dev_status, st);
}

}  // namespace moe
