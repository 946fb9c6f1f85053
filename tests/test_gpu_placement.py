"""Layout over a placement with replicated experts ("Beyond One GPU", section 6)
on the GPU vs the oracle.

The placement is planned from the routing of a different batch (the plan is
made from past load and used on new traffic).  Physical ids, counts, ranks,
offsets and slots are integers and must be bit-exact; the whole path with a
placement must give the same output bytes as without one, because a copy of
an expert computes what its original computes.
"""
import dataclasses

import numpy as np
import pytest
import torch

import combine_moe_route_06_gb300 as m
import moe_synth as ms
import oracle
from gpu_util import DEV, bf16_dev, bf16_host, close_bf16, f32_dev, host, i32_dev

pytestmark = pytest.mark.gpu
KEYS = ("expert_counts", "expert_rank", "part_counts", "part_offsets", "token_slot")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load_library()


def _plan(w_, R, learn_seed=7919):
    """Plan from the routing of another batch of the same workload."""
    past = dataclasses.replace(w_, index=w_.index + learn_seed)
    ids, _ = oracle.route_topk(ms.gen_logits(past), past.k)
    load = np.bincount(ids[ids >= 0].ravel(), minlength=w_.E).astype(np.int64)
    return m.moe_plan_placement(load, w_.P, R)


def _mapped_gpu(ids, E, P, pl, cs=None):
    S, T, k = ids.shape
    Ep = pl.E_phys
    i32 = dict(dtype=torch.int32, device=DEV)
    out = {"phys": torch.full((S, T, k), -9, **i32),
           "expert_counts": torch.full((S, Ep), -7, **i32),
           "expert_rank": torch.full((S, T, k), -7, **i32),
           "part_counts": torch.full((S, P), -7, **i32),
           "part_offsets": torch.full((S, P + 1), -7, **i32),
           "token_slot": torch.full((S, T, P), -7, **i32)}
    ws = torch.empty(max(m.moe_workspace_bytes_mapped(S, T, k, E, P, pl.Lp), 256),
                     dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, **i32)
    co, cs_d, _ = pl.to(DEV)
    if cs is not None:
        cs_d = i32_dev(cs)
    m.moe_dispatch_layout_mapped(i32_dev(ids), E, P, pl.Lp, co, cs_d, out["phys"],
                                 out["expert_counts"], out["expert_rank"], out["part_counts"],
                                 out["part_offsets"], out["token_slot"], ws, st)
    torch.cuda.synchronize()
    res = {key: host(t) for key, t in out.items()}
    res["status"] = int(st.item())
    return res


def _mapped_ref(ids, E, P, pl, cs=None):
    phys = oracle.map_replicas(ids, E, pl.copy_offsets, pl.copy_slots if cs is None else cs,
                               pl.E_phys)
    lay = oracle.dispatch_layout(phys, pl.E_phys, P)
    return phys, lay


# one expert per partition with Zipf popularity: placement cannot help there and
# the planner makes copies (22 of them for this batch), so the split is exercised
ONE_PER_PART = dict(E=32, P=32, k=4, zipf_s=1.2, T=2048)
FEW_PER_PART = dict(E=64, P=8, k=4, zipf_s=1.2, T=1000, H=512)


@pytest.mark.parametrize("name,over,R", [("tiny", {}, 2), ("decode", {}, 4), ("prefill", {}, 4),
                                         ("prefill", {}, 0), ("skewed", {}, 4), ("large", {}, 8),
                                         ("tiny", ONE_PER_PART, 2), ("tiny", FEW_PER_PART, 4),
                                         ("tiny", dict(ONE_PER_PART, S=3, T=700), 3)])
def test_mapped_layout_parity(name, over, R):
    w_ = ms.workload(name, **over)
    pl = _plan(w_, R)
    ids, _ = oracle.route_topk(ms.gen_logits(w_), w_.k)
    got = _mapped_gpu(ids, w_.E, w_.P, pl)
    phys, lay = _mapped_ref(ids, w_.E, w_.P, pl)
    assert np.array_equal(got["phys"], phys)
    for key in KEYS:
        assert np.array_equal(got[key], lay[key]), key
    assert got["status"] == lay["status"] == 0
    # the plan's partition loads are those of the batch it was learned from; on this
    # batch every pair still lands on a copy of its own expert
    assert np.array_equal(pl.slot_expert[got["phys"]], ids)


def test_mapped_layout_skips_bad_ids_and_ragged():
    rng = np.random.default_rng(5)
    E, P, R = 16, 4, 2
    load = rng.integers(1, 50, E).astype(np.int64)
    pl = m.moe_plan_placement(load, P, R)
    for S, T, k in ((2, 300, 3), (1, 1, 1), (3, 257, 2)):
        ids = rng.integers(-2, E + 3, size=(S, T, k)).astype(np.int32)
        got = _mapped_gpu(ids, E, P, pl)
        phys, lay = _mapped_ref(ids, E, P, pl)
        assert np.array_equal(got["phys"], phys)
        for key in KEYS:
            assert np.array_equal(got[key], lay[key]), (S, T, k, key)
        assert got["status"] == lay["status"]
        assert got["status"] & m.status_bit(m.MOE_ERR_BAD_EXPERT_ID)


def test_mapped_layout_empty_batch():
    E, P = 16, 4
    pl = m.moe_plan_placement(np.arange(E, dtype=np.int64), P, 1)
    got = _mapped_gpu(np.zeros((2, 0, 2), np.int32), E, P, pl)
    assert np.all(got["expert_counts"] == 0) and np.all(got["part_offsets"] == 0)
    assert got["status"] == 0


def test_mapped_layout_flags_a_slot_outside_the_placement():
    E, P = 16, 4
    pl = m.moe_plan_placement(np.arange(E, dtype=np.int64) + 1, P, 1)
    cs = pl.copy_slots.copy()
    cs[pl.copy_offsets[3]] = pl.E_phys + 5           # expert 3's original points nowhere
    ids = np.full((1, 8, 2), 3, np.int32)
    ids[0, :, 1] = 4
    got = _mapped_gpu(ids, E, P, pl, cs=cs)
    assert got["status"] & m.status_bit(m.MOE_ERR_INVALID_ARG)
    n3 = pl.copy_offsets[4] - pl.copy_offsets[3]
    # pairs of expert 3 that would use the bad slot become "not routed"; the rest map
    r = np.arange(8)
    assert np.all(got["phys"][0, r % n3 == 0, 0] == -1)
    assert np.array_equal(got["phys"][0, :, 1],
                          pl.copy_slots[pl.copy_offsets[4] + r % (pl.copy_offsets[5] - pl.copy_offsets[4])])


@pytest.mark.parametrize("name,over,combine", [("tiny", {}, "single"), ("decode", {}, "single"),
                                               ("prefill", {}, "single"),
                                               ("decode", {}, "two_stage"),
                                               ("tiny", ONE_PER_PART, "single"),
                                               ("tiny", FEW_PER_PART, "two_stage")])
@pytest.mark.parametrize("dispatch", ["fused", "separate"])
def test_path_with_placement_equals_path_without(name, over, combine, dispatch):
    """The placed path (mapped layout, then pack + permute in one call or the two
    separate calls) against the unplaced path and the oracle."""
    w_ = ms.workload(name, **over)
    inp = ms.gen_inputs(w_)
    pl = _plan(w_, 4)
    if over:
        assert pl.copy_offsets[-1] > w_.E            # copies made: the split is exercised
    lg, xx, sc = f32_dev(inp["logits"]), bf16_dev(inp["x"]), f32_dev(inp["scales"])
    plain = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, combine=combine)
    placed = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, combine=combine, placement=pl,
                       dispatch=dispatch)
    out0 = bf16_host(plain.step(lg, xx, sc)).copy()
    out1 = bf16_host(placed.step(lg, xx, sc)).copy()
    torch.cuda.synchronize()
    assert int(placed.dev_status.item()) == 0
    if combine == "single":
        assert np.array_equal(out1, out0)          # same rows, same weights, same j order
    # and against the oracle of the whole placed path
    ids, wts = oracle.route_topk(inp["logits"], w_.k)
    phys, lay = _mapped_ref(ids, w_.E, w_.P, pl)
    assert np.array_equal(host(placed.phys_ids), phys)
    assert np.array_equal(host(placed.token_slot), lay["token_slot"])
    cap_send = w_.T * min(w_.k, w_.P)
    send, _, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap_send)
    per = oracle.permute_to_experts(send, lay["token_slot"], phys, pl.E_phys)
    assert np.array_equal(host(placed.pair_row), per["pair_row"])
    rows = int(per["expert_offsets"][-1])
    assert np.array_equal(bf16_host(placed.recv)[:rows], per["recv"][:rows])
    slot_scale = np.where(pl.slot_expert >= 0, inp["scales"][np.maximum(pl.slot_expert, 0)], 0)
    y = oracle.expert_scale(per["recv"], per["expert_offsets"], slot_scale.astype(np.float32))
    if combine == "single":
        assert close_bf16(out1, oracle.combine(y, per["pair_row"], wts))
    else:
        # stage 1 rounds each partition's pre-sum to bf16 and the placement changes the
        # partitions, so the reference is the two-stage combine over the placed layout
        ret, _ = oracle.combine_stage1(y, per["pair_row"], wts, phys, lay["token_slot"],
                                       pl.E_phys, cap_send)
        ref2, _ = oracle.combine_stage2(ret, lay["token_slot"])
        assert close_bf16(out1, ref2)


def test_placed_bound_calls_and_graph_replay():
    w_ = ms.workload("decode")
    inp = ms.gen_inputs(w_)
    pl = _plan(w_, 2)
    path = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, placement=pl)
    lg, xx = f32_dev(inp["logits"]), bf16_dev(inp["x"])
    ref = bf16_host(path.step(lg, xx)).copy()
    stream = torch.cuda.Stream()
    calls = path.bind(lg, xx, stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        m.MoePath.run_bound(calls)
    path.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(path.out), ref)
    assert np.array_equal(ref, inp["x"])            # identity expert: the round trip is exact
