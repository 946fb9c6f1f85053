"""Seeded random shapes through the whole path on the GPU vs the oracle.

Every case draws S, T (up to 2,500 tokens: up to 10 layout chunks per source,
so the layout's cluster form too), H, E, k, P, align, the receiving partition
and the path's form (contiguous, masked, two-stage, routed; the contiguous
and two-stage forms through moe_dispatch or the separate calls) from a fixed seed, with
the logits sometimes quantised so that equal logits (ties) are common.  Index
outputs and moved rows are compared bit for bit; the output is compared
within the combine tolerance against the oracle's combine of the same expert
rows.
"""
import numpy as np
import pytest
import torch

import combine_moe_route_06_gb300 as m
import moe_synth as ms
import oracle
from gpu_util import bf16_dev, bf16_host, close_bf16, f32_dev, host, worst_rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load_library()


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    P = int(rng.choice([1, 2, 3, 4, 8, 16, 32]))
    L = int(rng.integers(1, max(2, 512 // P) + 1))
    E = min(P * L, 1024)
    E -= E % P
    k = int(rng.integers(1, min(E, 32) + 1))
    S = int(rng.integers(1, 4))
    T = int(rng.choice([0, 1, 7, 64, 255, 256, 257, 600, 1000, 2500]))
    H = 8 * int(rng.integers(1, 160)) if T <= 600 else 8 * int(rng.integers(1, 40))
    form = str(rng.choice(["contiguous", "contiguous", "masked", "two_stage", "routed"]))
    align = int(rng.choice([1, 1, 2, 128])) if form == "contiguous" else 1
    recv_part = int(rng.integers(-1, P)) if rng.random() < 0.5 else -1
    ties = rng.random() < 0.3
    # contiguous and two-stage forms: moe_dispatch (default) or the four separate calls
    dispatch = "separate" if rng.random() < 0.35 else None
    return dict(S=S, T=T, H=H, E=E, k=k, P=P, form=form, align=align, recv_part=recv_part,
                ties=ties, seed=seed, dispatch=dispatch)


@pytest.mark.parametrize("seed", range(120))
def test_random_shapes(seed):
    c = _draw(seed)
    S, T, H, E, k, P = c["S"], c["T"], c["H"], c["E"], c["k"], c["P"]
    w_ = ms.workload("tiny", S=S, T=T, H=H, E=E, k=k, P=P)
    inp = ms.gen_inputs(w_)
    logits = inp["logits"]
    if c["ties"]:
        logits = np.round(logits * 2.0).astype(np.float32) / 2.0   # many equal logits
    ids, wts = oracle.route_topk(logits, k)
    kw = {}
    if c["form"] == "masked":
        kw = dict(layout="masked", block_rows=max(1, (S * T * k) // max(E, 1) + 3))
    elif c["form"] == "two_stage":
        kw = dict(combine="two_stage")
    elif c["form"] == "routed":
        kw = dict(layout="routed")
    if c["form"] in ("contiguous", "two_stage"):
        kw["dispatch"] = c["dispatch"]
    path = m.MoePath(S, T, H, E, k, P, recv_part=c["recv_part"], align=c["align"], **kw)
    out = path.step(f32_dev(logits), bf16_dev(inp["x"]))          # identity expert
    torch.cuda.synchronize()
    got_out = bf16_host(out)

    assert np.array_equal(host(path.topk_ids), ids), c
    lay = oracle.dispatch_layout(ids, E, P)
    for key in ("expert_counts", "expert_rank", "part_counts", "part_offsets", "token_slot"):
        assert np.array_equal(host(getattr(path, key)), lay[key]), (key, c)
    cap_send = T * min(k, P)
    send, src, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap_send)
    used = lay["part_offsets"][:, -1]
    for s in range(S):
        assert np.array_equal(bf16_host(path.send)[s, :used[s]], send[s, :used[s]]), c
    st = int(path.dev_status.item())

    if c["form"] == "routed":
        ret, _ = oracle.routed_expert_stage1(send, *oracle.dispatch_pack_routed(
            inp["x"], ids, wts.astype(np.float32), lay["token_slot"], cap_send)[2:4],
            lay["part_offsets"], E, c["recv_part"])
        only = lay["token_slot"] if c["recv_part"] < 0 else np.where(
            np.arange(P) == c["recv_part"], lay["token_slot"], -1)
        want, _ = oracle.combine_stage2(ret, only)
        assert close_bf16(got_out, want), (worst_rel(got_out, want), c)
        assert st == 0, c
        return

    if c["form"] == "masked":
        per = oracle.permute_masked(send, lay["token_slot"], ids, E, c["recv_part"],
                                    path.block_rows)
        assert np.array_equal(host(path.masked_counts), per["masked_counts"]), c
    else:
        per = oracle.permute_to_experts(send, lay["token_slot"], ids, E,
                                        recv_part=c["recv_part"], align=c["align"])
        assert np.array_equal(host(path.expert_offsets), per["expert_offsets"]), c
    assert np.array_equal(host(path.pair_row), per["pair_row"]), c
    y = bf16_host(path.recv)
    valid = per["recv_pair"] >= 0
    assert np.array_equal(y[valid], per["recv"][valid]), c
    if c["form"] == "two_stage":
        ret, _ = oracle.combine_stage1(y, per["pair_row"], wts.astype(np.float32), ids,
                                       lay["token_slot"], E, cap_send, recv_part=c["recv_part"])
        only = lay["token_slot"] if c["recv_part"] < 0 else np.where(
            np.arange(P) == c["recv_part"], lay["token_slot"], -1)
        want, _ = oracle.combine_stage2(ret, only)
    else:
        want = oracle.combine(y, per["pair_row"], wts.astype(np.float32))
    assert close_bf16(got_out, want), (worst_rel(got_out, want), c)
    assert st == per["status"], (st, per["status"], c)
