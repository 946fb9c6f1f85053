"""Routed payload layout (a2a-backends sections 6.1, 7.1) on the GPU vs the oracle.

The routed pack writes each row with its token's ids and weights; the routed
stand-in expert pre-adds per partition straight from the rows in arrival
order.  Rows, ids, weights and send_src are compared bit for bit; the
stage-1 rows equal the GPU's own permute + expert + stage-1 path byte for byte
(same operations in the same order) and the oracle within the combine
tolerance.
"""
import numpy as np
import pytest
import torch

import combine_moe_route_06_gb300 as m
import moe_synth as ms
import oracle
from gpu_util import DEV, bf16_dev, bf16_host, close_bf16, f32_dev, host, i32_dev

pytestmark = pytest.mark.gpu
FILL = 0x2B2B


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load_library()


def _case(name, **over):
    w_ = ms.workload(name, **over)
    inp = ms.gen_inputs(w_)
    ids, wts = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    return w_, inp, ids, wts.astype(np.float32), lay


def _pack_routed_gpu(x, ids, wts, lay, cap_send):
    S, T, H = x.shape
    k = ids.shape[2]
    send = bf16_dev(np.full((S, cap_send, H), FILL, np.uint16))
    src = torch.full((S, cap_send), -5, dtype=torch.int32, device=DEV)
    sid = torch.full((S, cap_send, k), -5, dtype=torch.int32, device=DEV)
    sw = torch.full((S, cap_send, k), -5.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.moe_dispatch_pack_routed(bf16_dev(x), i32_dev(ids), f32_dev(wts), i32_dev(lay["token_slot"]),
                               i32_dev(lay["part_offsets"]), send, src, sid, sw, st)
    torch.cuda.synchronize()
    return send, src, sid, sw, int(st.item())


@pytest.mark.parametrize("name,over,extra", [("tiny", {}, 0), ("tiny", {"S": 3, "T": 77}, 5),
                                             ("decode", {}, 3), ("prefill", {}, 0),
                                             ("large", {}, 0)])
def test_pack_routed_parity(name, over, extra):
    w_, inp, ids, wts, lay = _case(name, **over)
    cap = w_.T * min(w_.k, w_.P) + extra
    send, src, sid, sw, st = _pack_routed_gpu(inp["x"], ids, wts, lay, cap)
    r_send, r_src, r_sid, r_sw, r_st = oracle.dispatch_pack_routed(
        inp["x"], ids, wts, lay["token_slot"], cap,
        send=np.full((w_.S, cap, w_.H), FILL, np.uint16))
    assert st == r_st == 0
    assert np.array_equal(bf16_host(send), r_send)
    assert np.array_equal(host(src), r_src)
    assert np.array_equal(host(sid), r_sid)
    assert np.array_equal(host(sw), r_sw)


@pytest.mark.parametrize("name,over,recv_part,scaled", [("tiny", {}, -1, True),
                                                        ("tiny", {"S": 3, "T": 77}, 2, True),
                                                        ("decode", {}, -1, True),
                                                        ("decode", {}, 5, False),
                                                        ("prefill", {}, -1, True)])
def test_routed_stage1_parity(name, over, recv_part, scaled):
    w_, inp, ids, wts, lay = _case(name, **over)
    cap = w_.T * min(w_.k, w_.P) + 2
    send, _, sid, sw, _ = _pack_routed_gpu(inp["x"], ids, wts, lay, cap)
    scale = inp["scales"] if scaled else None
    ret = bf16_dev(np.full((w_.S, cap, w_.H), FILL, np.uint16))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.moe_routed_expert_stage1(send, sid, sw, i32_dev(lay["part_offsets"]), w_.T, w_.E, recv_part,
                               None if scale is None else f32_dev(scale), ret, st)
    torch.cuda.synchronize()
    got = bf16_host(ret)
    r_send, _, r_sid, r_sw, _ = oracle.dispatch_pack_routed(inp["x"], ids, wts, lay["token_slot"], cap)
    want, r_st = oracle.routed_expert_stage1(r_send, r_sid, r_sw, lay["part_offsets"], w_.E,
                                             recv_part, scale,
                                             ret=np.full((w_.S, cap, w_.H), FILL, np.uint16))
    assert int(st.item()) == r_st == 0
    # rows of the receiving partitions' regions are written, every other row is not
    written = np.zeros((w_.S, cap), bool)
    for s_ in range(w_.S):
        po = lay["part_offsets"][s_]
        for p_ in range(w_.P):
            if recv_part < 0 or p_ == recv_part:
                written[s_, po[p_]:po[p_ + 1]] = True
    assert np.all(got[~written] == FILL) and np.all(want[~written] == FILL)
    # The stand-in computes x*s in fp32 and then rounds to bf16, the oracle rounds the
    # exact product once: y may differ by one bf16 unit (2^-7 relative; e.g. x = 1.734375,
    # s = 7/48: the fp32 product is a bf16 tie, the exact one lies just below it).  A row
    # whose partition holds a single expert of its token keeps that whole error, and the
    # row's own rounding adds up to one more unit of the result: 2^-7 + 2^-8 < 2^-6.
    tol = 2.0 ** -6 if scaled else 1e-2
    assert close_bf16(got[written], want[written], rel=tol)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill"])
def test_routed_path_equals_permuted_two_stage_path(name):
    """Same rows, same expert, same pre-add order: the routed path and the permute
    path with a two-stage combine give the same bytes."""
    w_ = ms.workload(name)
    inp = ms.gen_inputs(w_)
    lg, xx, sc = f32_dev(inp["logits"]), bf16_dev(inp["x"]), f32_dev(inp["scales"])
    perm = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, combine="two_stage")
    routed = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, layout="routed")
    out0 = bf16_host(perm.step(lg, xx, sc)).copy()
    out1 = bf16_host(routed.step(lg, xx, sc)).copy()
    torch.cuda.synchronize()
    assert int(routed.dev_status.item()) == 0
    assert np.array_equal(out1, out0)
    ref = oracle.run_path(inp["x"], inp["logits"], w_.E, w_.k, w_.P, inp["scales"])
    assert close_bf16(out1, ref["out"])


def test_routed_skewed_receiver():
    w_ = ms.workload("skewed", T=1024)
    inp = ms.gen_inputs(w_)
    path = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, recv_part=w_.recv_part, layout="routed")
    path.step(f32_dev(inp["logits"]), bf16_dev(inp["x"]))
    torch.cuda.synchronize()
    ids, wts = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    send, _, sid, sw, _ = oracle.dispatch_pack_routed(inp["x"], ids, wts, lay["token_slot"],
                                                      path.cap_send)
    ret, _ = oracle.routed_expert_stage1(send, sid, sw, lay["part_offsets"], w_.E, w_.recv_part)
    # stage 2 over partition 0's returned rows only: the partial combine of its experts
    only = np.where(np.arange(w_.P) == w_.recv_part, lay["token_slot"], -1)
    want, _ = oracle.combine_stage2(ret, only)
    got = bf16_host(path.out)
    assert close_bf16(got, want)
    assert int(path.dev_status.item()) == 0


def test_routed_bound_calls_in_a_graph():
    w_ = ms.workload("decode")
    inp = ms.gen_inputs(w_)
    path = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, layout="routed")
    lg, xx = f32_dev(inp["logits"]), bf16_dev(inp["x"])
    stream = torch.cuda.Stream()
    calls = path.bind(lg, xx, stream)
    assert len(calls) == 5 and path.launches_per_step() == 5
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        m.MoePath.run_bound(calls)
    g.replay()
    torch.cuda.synchronize()
    x = ms.f32_from_bf16_bits(inp["x"]).astype(np.float64)
    got = ms.f32_from_bf16_bits(bf16_host(path.out)).astype(np.float64)
    assert np.all(np.abs(got - x) <= 2.0 ** -6 * np.maximum(np.abs(x), 1e-3))
