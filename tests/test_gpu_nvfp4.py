"""Pack with NVFP4 records (a2a-backends section 7.2) on the GPU vs the oracle.

Codes and block scales are integer results of decisions both sides take in
fp32 (the scale amax / (6 g), the quotient v / (s g), then one rounding each),
so records are compared bit for bit, over the workloads, over every finite
bf16 pattern, on rounding ties and with several tensor scales g.  The records
then travel through the permute and the dequantizing stand-in expert.
"""
import numpy as np
import pytest
import torch

import combine_moe_route_06_gb300 as m
import moe_synth as ms
import oracle
from gpu_util import DEV, bf16_dev, bf16_host, close_bf16, f32_dev, host, i32_dev, worst_rel

pytestmark = pytest.mark.gpu
QFILL = 0x5C


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load_library()


def _finite_bf16_bits(rng, shape):
    b = rng.integers(0, 1 << 16, size=shape, dtype=np.uint32).astype(np.uint16)
    inf_nan = (b & 0x7F80) == 0x7F80
    b[inf_nan] &= 0xBFFF
    return b


def _case(name, **over):
    w_ = ms.workload(name, **over)
    inp = ms.gen_inputs(w_)
    ids, _ = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    return w_, inp["x"], ids, lay


def _check_pack(x, lay, cap_send, g=1.0, guard=2):
    S, T, H = x.shape
    rb = m.nvfp4_record_bytes(H)
    q_full = torch.full((S, cap_send + guard, rb), QFILL, dtype=torch.uint8, device=DEV)
    if S == 1:
        q = q_full[:, :cap_send]
    else:
        q_full = q_full[:, :cap_send].contiguous()
        q = q_full
    src = torch.full((S, cap_send), -5, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.moe_dispatch_pack_nvfp4(bf16_dev(x), i32_dev(lay["token_slot"]), i32_dev(lay["part_offsets"]),
                              q, src, g, st)
    torch.cuda.synchronize()
    gq, gsrc, gst = host(q_full), host(src), int(st.item())
    rq, rsrc, rst = oracle.dispatch_pack_nvfp4(x, lay["token_slot"], cap_send, g,
                                               send_q=np.full((S, cap_send, rb), QFILL, np.uint8))
    if not np.array_equal(gq[:, :cap_send], rq):
        bad = np.argwhere(gq[:, :cap_send] != rq)[:5]
        raise AssertionError(f"records differ at {bad.tolist()}: gpu "
                             f"{[int(gq[tuple(b)]) for b in bad]} oracle {[int(rq[tuple(b)]) for b in bad]}")
    assert np.all(gq[:, cap_send:] == QFILL)
    assert np.array_equal(gsrc, rsrc)
    assert gst == rst
    return gq[:, :cap_send], rst


@pytest.mark.parametrize("name,over,g", [("tiny", {}, 1.0), ("decode", {}, 1.0),
                                         ("prefill", {}, 1.0), ("large", {}, 2.0 ** -12),
                                         ("skewed", {"T": 512}, 0.37), ("tiny", {"T": 77}, 3.0)])
def test_pack_nvfp4_parity(name, over, g):
    w_, x, ids, lay = _case(name, **over)
    _, st = _check_pack(x, lay, w_.T * min(w_.k, w_.P), g)
    assert st == 0


@pytest.mark.parametrize("H,g", [(256, 1.0), (768, 2.0 ** -20), (1280, 1e-3), (2304, 5.0)])
def test_pack_nvfp4_every_finite_bf16(H, g):
    w_, _, ids, lay = _case("tiny", H=H, T=150)
    x = _finite_bf16_bits(np.random.default_rng(H), (w_.S, w_.T, H))
    _check_pack(x, lay, w_.T * min(w_.k, w_.P), g)


def test_pack_nvfp4_ties_and_special_blocks():
    w_, _, ids, lay = _case("tiny", H=256, T=64)
    rng = np.random.default_rng(9)
    v = rng.standard_normal((w_.S, w_.T, 256)).astype(np.float32)
    # rows 0-7: a 6 in every block (s = 1 exactly) beside the E2M1 midpoints
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    for t in range(8):
        row = np.resize(np.concatenate([mids, -mids]), 256).astype(np.float32)
        row[::16] = 6.0
        v[:, t] = row * (2.0 ** (t - 4))           # other binades: s = 2^(t-4)
    x = ms.bf16_bits_from_f32(v)
    x[:, 8, :] = 0                                   # zeros: scale byte 0
    x[:, 9, :] = 0x8000                              # negative zeros
    x[:, 10, :16] = 0x7F7F                           # largest bf16: scale saturates at 448
    x[:, 10, 16:32] = 0x0001                         # smallest subnormal: flushes
    for g in (1.0, 0.75, 2.0 ** -8):
        _check_pack(x, lay, w_.T * min(w_.k, w_.P), g)


def test_pack_nvfp4_capacity_and_rejects():
    w_, x, ids, lay = _case("tiny", T=200)
    _, st = _check_pack(x, lay, 150)
    assert st & m.status_bit(m.MOE_ERR_CAPACITY)
    S = x.shape[0]
    for H, g in ((96, 1.0), (256, 0.0), (256, -1.0)):
        xx = torch.zeros((S, 8, H), dtype=torch.bfloat16, device=DEV)
        q = torch.zeros((S, 8, m.nvfp4_record_bytes(H)), dtype=torch.uint8, device=DEV)
        src = torch.zeros((S, 8), dtype=torch.int32, device=DEV)
        w8, _, _, lay8 = _case("tiny", T=8)
        with pytest.raises(m.MoeError) as ei:
            m.moe_dispatch_pack_nvfp4(xx, i32_dev(lay8["token_slot"]),
                                      i32_dev(lay8["part_offsets"]), q, src, g)
        assert ei.value.code == m.MOE_ERR_INVALID_ARG


def _oracle_path(w_, inp, scales, g):
    ids, wts = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    q, _, st = oracle.dispatch_pack_nvfp4(inp["x"], lay["token_slot"], w_.T * min(w_.k, w_.P), g)
    per = oracle.permute_to_experts(q.view(np.uint16), lay["token_slot"], ids, w_.E)
    recv_q = per["recv"].view(np.uint8)
    y = oracle.expert_scale_nvfp4(recv_q, per["expert_offsets"], scales, g)
    return dict(layout=lay, send=q, permute=per, recv_q=recv_q, y=y,
                out=oracle.combine(y, per["pair_row"], wts), status=st | per["status"])


@pytest.mark.parametrize("dispatch", ["fused", "separate"])
@pytest.mark.parametrize("name,g", [("tiny", 1.0), ("decode", 1.0), ("prefill", 0.02)])
def test_nvfp4_path(name, g, dispatch):
    """The NVFP4 path through moe_dispatch_quantized or the separate calls."""
    w_ = ms.workload(name)
    inp = ms.gen_inputs(w_)
    ref = _oracle_path(w_, inp, inp["scales"], g)
    path = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, quant="nvfp4", nvfp4_scale=g,
                     dispatch=dispatch)
    out = path.step(f32_dev(inp["logits"]), bf16_dev(inp["x"]), f32_dev(inp["scales"]))
    torch.cuda.synchronize()
    used = int(ref["layout"]["part_offsets"][0, -1])
    assert np.array_equal(host(path.send)[0, :used], ref["send"][0, :used])
    rows = int(ref["permute"]["expert_offsets"][-1])
    assert np.array_equal(host(path.recv)[:rows], ref["recv_q"][:rows])
    assert close_bf16(bf16_host(path.y)[:rows], ref["y"][:rows], rel=2.0 ** -7, floor=1e-30)
    assert close_bf16(bf16_host(out), ref["out"]), worst_rel(bf16_host(out), ref["out"])
    assert int(path.dev_status.item()) == 0 == ref["status"]
    calls = path.bind(f32_dev(inp["logits"]), bf16_dev(inp["x"]), scale=f32_dev(inp["scales"]))
    assert len(calls) == (6 if dispatch == "separate" else 3)
