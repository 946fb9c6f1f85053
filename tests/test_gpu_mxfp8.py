"""Pack with MXFP8 records (a2a-backends section 7.2) on the GPU vs the oracle.

The codes and scale bytes are integer results of a decision the two sides take
in the same way (a power-of-two scale, then one rounding to E4M3), so the
records are compared bit for bit, as are send_src, the status word and every
byte the pack must not touch.  The records then go through the permute as
opaque rows, the dequantizing stand-in expert and the combine, each against
the oracle.
"""
import numpy as np
import pytest
import torch

import combine_moe_route_06_gb300 as m
import moe_synth as ms
import oracle
from gpu_util import DEV, bf16_dev, bf16_host, close_bf16, f32_dev, host, i32_dev, worst_rel

pytestmark = pytest.mark.gpu
QFILL = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load_library()


def _finite_bf16_bits(rng, shape):
    """Uniform over every finite bf16 bit pattern (zeros, subnormals, both signs, max)."""
    b = rng.integers(0, 1 << 16, size=shape, dtype=np.uint32).astype(np.uint16)
    inf_nan = (b & 0x7F80) == 0x7F80
    b[inf_nan] &= 0xBFFF            # exponent 255 -> 127: finite
    return b


def _case(name, **over):
    w_ = ms.workload(name, **over)
    inp = ms.gen_inputs(w_)
    ids, _ = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    return w_, inp["x"], ids, lay


def _pack_gpu(x, token_slot, part_offsets, cap_send, guard=2):
    S, T, H = x.shape
    rb = m.mxfp8_record_bytes(H)
    q_full = torch.full((S, cap_send + guard, rb), QFILL, dtype=torch.uint8, device=DEV)
    src = torch.full((S, cap_send), -5, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    # the pack writes [S][cap_send] rows: hand it exactly that many (S == 1 keeps the
    # leading slice contiguous; S > 1 runs without a guard band)
    if S == 1:
        q = q_full[:, :cap_send]
    else:
        q_full = q_full[:, :cap_send].contiguous()
        q = q_full
    m.moe_dispatch_pack_mxfp8(bf16_dev(x), i32_dev(token_slot), i32_dev(part_offsets), q, src, st)
    torch.cuda.synchronize()
    return host(q_full), host(src), int(st.item())


def _check_pack(x, lay, cap_send):
    S, T, H = x.shape
    gq, gsrc, gst = _pack_gpu(x, lay["token_slot"], lay["part_offsets"], cap_send)
    rq, rsrc, rst = oracle.dispatch_pack_mxfp8(
        x, lay["token_slot"], cap_send,
        send_q=np.full((S, cap_send, m.mxfp8_record_bytes(H)), QFILL, np.uint8))
    assert np.array_equal(gq[:, :cap_send], rq)
    assert np.all(gq[:, cap_send:] == QFILL)
    assert np.array_equal(gsrc, rsrc)
    assert gst == rst
    return gq[:, :cap_send], rst


@pytest.mark.parametrize("name,over", [("tiny", {}), ("decode", {}), ("prefill", {}),
                                       ("large", {}), ("skewed", {"T": 512}),
                                       ("tiny", {"T": 77})])
def test_pack_mxfp8_parity(name, over):
    w_, x, ids, lay = _case(name, **over)
    cap_send = w_.T * min(w_.k, w_.P)
    _, st = _check_pack(x, lay, cap_send)
    assert st == 0


@pytest.mark.parametrize("H", [256, 768, 1280, 2304])
def test_pack_mxfp8_every_finite_bf16(H):
    # widths with a ragged last 1,024-value segment; values drawn over all finite
    # bf16 patterns so blocks see zeros, subnormals, saturation and rounding ties
    w_, _, ids, lay = _case("tiny", H=H, T=150)
    x = _finite_bf16_bits(np.random.default_rng(H), (w_.S, w_.T, H))
    _check_pack(x, lay, w_.T * min(w_.k, w_.P))


def test_pack_mxfp8_special_blocks():
    w_, _, ids, lay = _case("tiny", H=256, T=64)
    rng = np.random.default_rng(7)
    x = ms.bf16_bits_from_f32(rng.standard_normal((w_.S, w_.T, 256)).astype(np.float32))
    x[:, 0, :] = 0                                   # all-zero row: scale byte 0
    x[:, 1, :] = 0x8000                              # negative zeros
    x[:, 2, :32] = 0x7F7F                            # largest finite bf16
    x[:, 2, 32:64] = 0x0001                          # smallest subnormal
    x[:, 3, :] = 0x43E0                              # 448: E4M3's largest value at X = 1
    x[:, 4, ::32] = 0x43F0                           # 480 beside small values
    q, _ = _check_pack(x, lay, w_.T * min(w_.k, w_.P))


def test_pack_mxfp8_capacity_overflow():
    w_, x, ids, lay = _case("tiny", T=200)
    _, st = _check_pack(x, lay, 150)
    assert st & m.status_bit(m.MOE_ERR_CAPACITY)


def test_pack_mxfp8_empty_source():
    w_, x, ids, lay = _case("tiny", T=64)
    lay = dict(lay)
    lay["token_slot"] = np.full_like(lay["token_slot"], -1)
    lay["part_offsets"] = np.zeros_like(lay["part_offsets"])
    gq, st = _check_pack(x, lay, 16)
    assert st == 0 and np.all(gq == QFILL)


@pytest.mark.parametrize("H", [96, 1000])
def test_pack_mxfp8_rejects_width(H):
    w_, x, ids, lay = _case("tiny", T=8)
    S = x.shape[0]
    xx = torch.zeros((S, 8, H), dtype=torch.bfloat16, device=DEV)
    q = torch.zeros((S, 8, m.mxfp8_record_bytes(H)), dtype=torch.uint8, device=DEV)
    src = torch.zeros((S, 8), dtype=torch.int32, device=DEV)
    with pytest.raises(m.MoeError) as ei:
        m.moe_dispatch_pack_mxfp8(xx, i32_dev(lay["token_slot"]), i32_dev(lay["part_offsets"]),
                                  q, src)
    assert ei.value.code == m.MOE_ERR_INVALID_ARG


def _oracle_quant_path(w_, inp, scales, recv_part=-1, align=1):
    """Oracle path with MXFP8 rows: records travel through the permute as opaque rows."""
    ids, wts = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    cap_send = w_.T * min(w_.k, w_.P)
    q, src, st = oracle.dispatch_pack_mxfp8(inp["x"], lay["token_slot"], cap_send)
    per = oracle.permute_to_experts(q.view(np.uint16), lay["token_slot"], ids, w_.E,
                                    recv_part=recv_part, align=align)
    recv_q = per["recv"].view(np.uint8)
    y = oracle.expert_scale_mxfp8(recv_q, per["expert_offsets"], scales)
    out = oracle.combine(y, per["pair_row"], wts)
    return dict(ids=ids, w=wts, layout=lay, send=q, permute=per, recv_q=recv_q, y=y, out=out,
                status=st | per["status"])


@pytest.mark.parametrize("dispatch", ["fused", "separate"])
@pytest.mark.parametrize("name", ["tiny", "decode", "prefill"])
def test_mxfp8_path(name, dispatch):
    """The quantized path through moe_dispatch_quantized or the separate calls."""
    over = {"H": 512} if name == "tiny" else {}
    w_ = ms.workload(name, **over)
    inp = ms.gen_inputs(w_)
    ref = _oracle_quant_path(w_, inp, inp["scales"])
    path = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, quant="mxfp8", dispatch=dispatch)
    out = path.step(f32_dev(inp["logits"]), bf16_dev(inp["x"]), f32_dev(inp["scales"]))
    torch.cuda.synchronize()
    assert np.array_equal(host(path.pair_row), ref["permute"]["pair_row"])
    assert np.array_equal(host(path.expert_offsets), ref["permute"]["expert_offsets"])
    used = int(ref["layout"]["part_offsets"][0, -1])
    assert np.array_equal(host(path.send)[0, :used], ref["send"][0, :used])
    rows = int(ref["permute"]["expert_offsets"][-1])
    assert np.array_equal(host(path.recv)[:rows], ref["recv_q"][:rows])
    # the stand-in rounds code * s_e to fp32 before bf16: at most one bf16 unit apart
    assert close_bf16(bf16_host(path.y)[:rows], ref["y"][:rows], rel=2.0 ** -7, floor=1e-30)
    assert close_bf16(bf16_host(out), ref["out"]), worst_rel(bf16_host(out), ref["out"])
    assert int(path.dev_status.item()) == 0 == ref["status"]


@pytest.mark.parametrize("dispatch", ["fused", "separate"])
def test_mxfp8_path_bound_calls_and_identity_scale(dispatch):
    """The pre-marshalled calls give the same bytes as the checked calls; with unit
    scales the output is the combine of the dequantized rows."""
    w_ = ms.workload("decode")
    inp = ms.gen_inputs(w_)
    path = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, quant="mxfp8", dispatch=dispatch)
    lg, xx = f32_dev(inp["logits"]), bf16_dev(inp["x"])
    out1 = bf16_host(path.step(lg, xx)).copy()
    calls = path.bind(lg, xx)
    if dispatch == "separate":
        # route, layout, pack, permute, expert, combine; at T = 64 the layout is one
        # kernel, and the permute one (its map step runs inside the copy kernel)
        assert len(calls) == 6 and path.launches_per_step() == 6
    else:
        # moe_dispatch_quantized (one launch for a decode batch), expert, combine
        assert len(calls) == 3 and path.launches_per_step() == 3
    path.out.zero_()
    m.MoePath.run_bound(calls)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(path.out), out1)
    ref = _oracle_quant_path(w_, inp, np.ones(w_.E, np.float32))
    assert close_bf16(out1, ref["out"])
