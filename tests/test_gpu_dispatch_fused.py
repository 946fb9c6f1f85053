"""moe_dispatch (route + layout + pack + permute in one call) against the four
separate calls and the CPU oracle.

Every output buffer starts filled with a sentinel, and the fused call must
leave every byte of every output exactly as the separate calls leave it
(written values and untouched sentinels alike), including under capacity
overflow; where nothing overflows the outputs are also compared with the
oracle.  The one-launch form (one source of 1..256 tokens) is covered at its
edges (1, 63, 64, 65, 255, 256 tokens; E from 16 to 1024; k and P up to 32;
8-value and ragged rows; run alignment; a receiving partition), and the
launch counts the library reports are checked against the launch trace.
moe_dispatch_quantized (MXFP8 and NVFP4 records) is held to the separate
quantized pack and permute the same way, and its records to the oracle's;
moe_dispatch_pack_permute (pack + permute for a layout already made) to
moe_dispatch_pack followed by moe_permute_to_experts.
"""
import numpy as np
import pytest
import torch

import combine_moe_route_06_gb300 as m
import moe_synth as ms
import oracle
from gpu_util import bf16_dev, bf16_host, f32_dev, host

pytestmark = pytest.mark.gpu

OUT_I32 = ("topk_ids", "expert_counts", "expert_rank", "part_counts", "part_offsets",
           "token_slot", "send_src", "expert_offsets", "pair_row", "recv_pair")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load_library()


def _dispatch(mode, w_, inp, recv_part=-1, align=1, cap_send=None, cap_recv=None, trace=False):
    """One dispatch through `mode` with sentinel-filled outputs; returns the outputs
    as host arrays (and the traced kernel names)."""
    path = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, recv_part=recv_part, align=align,
                     cap_send=cap_send, cap_recv=cap_recv, dispatch=mode)
    for name in OUT_I32:
        getattr(path, name).fill_(-7)
    path.topk_w.fill_(-9.0)
    path.send.view(torch.int16).fill_(0x5A5A)
    path.recv.view(torch.int16).fill_(0x3C3C)
    logits, x = f32_dev(inp["logits"]), bf16_dev(inp["x"])
    torch.cuda.synchronize()
    if trace:
        m.trace_enable(None, 64)
        m.trace_reset()
    try:
        if mode == "fused":
            path.dispatch_fused(logits, x)
        else:
            path.route(logits)
            path.dispatch(x)
        torch.cuda.synchronize()
        kernels = [n for n, _ in m.trace_records()] if trace else None
    finally:
        if trace:
            m.trace_disable()
    out = {name: host(getattr(path, name)) for name in OUT_I32}
    out["topk_w"] = host(path.topk_w).view(np.uint32)
    out["send"] = bf16_host(path.send)
    out["recv"] = bf16_host(path.recv)
    out["status"] = int(path.dev_status.item())
    return out, kernels, path


def _same(a, b):
    for key in a:
        if key in ("status",):
            assert a[key] == b[key], (key, a[key], b[key])
        else:
            assert np.array_equal(a[key], b[key]), key


def _against_oracle(got, w_, inp, recv_part=-1, align=1):
    ref = oracle.run_path(inp["x"], inp["logits"], w_.E, w_.k, w_.P, None, recv_part=recv_part,
                          align=align)
    assert np.array_equal(got["topk_ids"], ref["ids"])
    assert np.max(np.abs(got["topk_w"].view(np.float32) - ref["w"])) <= 2e-6
    for key in ("expert_counts", "part_counts", "part_offsets", "token_slot"):
        assert np.array_equal(got[key], ref["layout"][key]), key
    for key in ("expert_offsets", "pair_row", "recv_pair"):
        assert np.array_equal(got[key], ref["permute"][key]), key
    for s in range(w_.S):
        used = int(ref["layout"]["part_offsets"][s, -1])
        assert np.array_equal(got["send"][s, :used], ref["send"][s, :used])
        assert np.array_equal(got["send_src"][s], ref["send_src"][s])
    rows = int(ref["permute"]["expert_offsets"][-1])
    assert np.array_equal(got["recv"][:rows], ref["permute"]["recv"][:rows])
    assert got["status"] == ref["status"] == 0


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "large"])
def test_fused_equals_separate_and_oracle(name):
    w_ = ms.workload(name)
    inp = ms.gen_inputs(w_)
    fused, kf, path = _dispatch("fused", w_, inp, trace=True)
    sep, ks, _ = _dispatch("separate", w_, inp, trace=True)
    _same(fused, sep)
    _against_oracle(fused, w_, inp)
    assert len(kf) == m.moe_dispatch_kernels(w_.S, w_.T, w_.k, w_.E, w_.P), kf
    if w_.S == 1 and w_.T <= 256:
        assert kf == ["k_dispatch_small"]
    else:
        assert kf[-1] == "k_pack_permute" and len(ks) > len(kf), (kf, ks)


@pytest.mark.parametrize("name", ["skewed", "skewed_perm"])
def test_fused_skewed_receiver_equals_separate(name):
    """The receiver view of the skewed workloads (popularity ranks equal to the
    expert ids, or a seeded permutation of them): every output of the fused
    call equals the separate calls'; the routing and layout equal the
    oracle's."""
    w_ = ms.workload(name)
    inp = ms.gen_inputs(w_)
    fused, kf, _ = _dispatch("fused", w_, inp, recv_part=w_.recv_part, trace=True)
    sep, _, _ = _dispatch("separate", w_, inp, recv_part=w_.recv_part)
    _same(fused, sep)
    assert kf[-1] == "k_pack_permute"
    assert fused["status"] == 0
    ids, _ = oracle.route_topk(inp["logits"], w_.k)
    assert np.array_equal(fused["topk_ids"], ids)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    for key in ("expert_counts", "part_counts", "part_offsets", "token_slot"):
        assert np.array_equal(fused[key], lay[key]), key


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 255, 256, 257])
def test_one_launch_edges_in_tokens(T):
    w_ = ms.workload("decode", T=T, index=100 + T)
    inp = ms.gen_inputs(w_)
    fused, kf, _ = _dispatch("fused", w_, inp, trace=True)
    sep, _, _ = _dispatch("separate", w_, inp)
    _same(fused, sep)
    _against_oracle(fused, w_, inp)
    assert (kf == ["k_dispatch_small"]) == (T <= 256), kf


@pytest.mark.parametrize("T,H,E,k,P,align,recv_part", [
    (100, 8, 16, 2, 4, 1, -1),        # 8-value rows, E < 32 (one logit per lane)
    (130, 520, 1024, 32, 32, 1, -1),  # the ABI's largest E, k, P; ragged segments
    (256, 256, 64, 8, 8, 128, -1),    # run alignment: zero padding rows
    (77, 5120, 384, 6, 8, 1, 3),      # one receiving partition
    (200, 64, 96, 3, 1, 8, 0),        # a single partition
    (33, 2048, 992, 7, 32, 4, 5),
    # wide rows: 255 tokens x 256 segments is the largest task index the
    # multiply-high division takes (65,279 < 2^16); 256 x 256 reaches 2^16 and
    # takes the plain division
    (255, 131072, 64, 2, 4, 1, -1),
    (256, 131072, 64, 2, 4, 1, -1),
])
def test_one_launch_shapes(T, H, E, k, P, align, recv_part):
    w_ = ms.workload("tiny", T=T, H=H, E=E, k=k, P=P, index=7 * T + k)
    inp = ms.gen_inputs(w_)
    fused, kf, _ = _dispatch("fused", w_, inp, recv_part=recv_part, align=align, trace=True)
    sep, _, _ = _dispatch("separate", w_, inp, recv_part=recv_part, align=align)
    _same(fused, sep)
    _against_oracle(fused, w_, inp, recv_part=recv_part, align=align)
    assert kf == ["k_dispatch_small"]


@pytest.mark.parametrize("name,T", [("decode", 64), ("decode", 200), ("prefill", 1000)])
def test_capacity_overflow_matches_separate(name, T):
    """Caps too small for the batch: rows past them are dropped and flagged the
    same way (send past cap_send, receive rows past cap_recv)."""
    w_ = ms.workload(name, T=T, index=300 + T)
    inp = ms.gen_inputs(w_)
    for cap_send, cap_recv in ((T, None), (None, T * 2), (T // 2, T)):
        fused, _, _ = _dispatch("fused", w_, inp, cap_send=cap_send, cap_recv=cap_recv)
        sep, _, _ = _dispatch("separate", w_, inp, cap_send=cap_send, cap_recv=cap_recv)
        _same(fused, sep)
        assert fused["status"] & m.status_bit(m.MOE_ERR_CAPACITY)


def test_several_sources_take_the_pack_permute_kernel():
    w_ = ms.workload("decode", S=3, T=50, index=55)
    inp = ms.gen_inputs(w_)
    for recv_part in (-1, 2):
        fused, kf, _ = _dispatch("fused", w_, inp, recv_part=recv_part, trace=True)
        sep, _, _ = _dispatch("separate", w_, inp, recv_part=recv_part)
        _same(fused, sep)
        _against_oracle(fused, w_, inp, recv_part=recv_part)
        assert kf[0] == "k_route_topk" and kf[-1] == "k_pack_permute", kf


def test_empty_batch():
    w_ = ms.workload("decode", T=0)
    inp = ms.gen_inputs(w_)
    fused, kf, _ = _dispatch("fused", w_, inp, trace=True)
    sep, _, _ = _dispatch("separate", w_, inp)
    _same(fused, sep)
    assert len(kf) == m.moe_dispatch_kernels(1, 0, w_.k, w_.E, w_.P)


def test_fused_decode_step_in_a_cuda_graph():
    """The fused decode step (moe_dispatch + moe_combine) captured once and
    replayed on new inputs at the same addresses."""
    w_ = ms.workload("decode")
    inp = ms.gen_inputs(w_)
    path = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, dispatch="fused")
    logits, x = f32_dev(inp["logits"]), bf16_dev(inp["x"])
    s = torch.cuda.Stream()
    calls = path.bind(logits, x, s)
    assert [fn.__name__ for fn, _ in calls] == ["moe_dispatch", "moe_combine"]
    with torch.cuda.stream(s):
        m.MoePath.run_bound(calls)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        m.MoePath.run_bound(calls)
    inp2 = ms.gen_inputs(ms.workload("decode", index=9))
    logits.copy_(f32_dev(inp2["logits"]))
    x.copy_(bf16_dev(inp2["x"]))
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        ref = oracle.run_path(inp2["x"], inp2["logits"], w_.E, w_.k, w_.P, None)
        assert np.array_equal(host(path.pair_row), ref["permute"]["pair_row"])
        # identity expert: the combine of a token's own row with weights summing to 1
        got = ms.f32_from_bf16_bits(bf16_host(path.out)).astype(np.float64)
        want = ms.f32_from_bf16_bits(ref["out"]).astype(np.float64)
        assert np.all(np.abs(got - want) <= 1e-2 * np.maximum(np.abs(want), 1e-3))
    assert int(path.dev_status.item()) == 0


# ------------------------------------------------------ quantized records --

def _dispatch_q(mode, quant, w_, inp, g=1.0, recv_part=-1, align=1, cap_send=None,
                cap_recv=None, trace=False):
    """One quantized dispatch through `mode` with sentinel-filled outputs."""
    path = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, recv_part=recv_part, align=align,
                     cap_send=cap_send, cap_recv=cap_recv, quant=quant, nvfp4_scale=g,
                     dispatch=mode)
    for name in OUT_I32:
        getattr(path, name).fill_(-7)
    path.topk_w.fill_(-9.0)
    path.send.fill_(0x5A)
    path.recv.fill_(0x3C)
    logits, x = f32_dev(inp["logits"]), bf16_dev(inp["x"])
    torch.cuda.synchronize()
    if trace:
        m.trace_enable(None, 64)
        m.trace_reset()
    try:
        if mode == "fused":
            path.dispatch_fused(logits, x)
        else:
            path.route(logits)
            path.dispatch(x)
        torch.cuda.synchronize()
        kernels = [n for n, _ in m.trace_records()] if trace else None
    finally:
        if trace:
            m.trace_disable()
    out = {name: host(getattr(path, name)) for name in OUT_I32}
    out["topk_w"] = host(path.topk_w).view(np.uint32)
    out["send"] = host(path.send)
    out["recv"] = host(path.recv)
    out["status"] = int(path.dev_status.item())
    return out, kernels


def _q_oracle(quant, w_, inp, g=1.0, recv_part=-1, align=1):
    ids, _ = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    cap_send = w_.T * min(w_.k, w_.P)
    if quant == "mxfp8":
        q, src, st = oracle.dispatch_pack_mxfp8(inp["x"], lay["token_slot"], cap_send)
    else:
        q, src, st = oracle.dispatch_pack_nvfp4(inp["x"], lay["token_slot"], cap_send, g)
    per = oracle.permute_to_experts(q.view(np.uint16), lay["token_slot"], ids, w_.E,
                                    recv_part=recv_part, align=align)
    return lay, q, src, per


@pytest.mark.parametrize("quant,g", [("mxfp8", 1.0), ("nvfp4", 1.0), ("nvfp4", 0.02)])
@pytest.mark.parametrize("name,over,recv_part,align", [
    ("decode", {}, -1, 1), ("prefill", {}, -1, 1), ("large", {}, -1, 1),
    ("tiny", {"S": 2, "T": 300, "H": 512, "E": 64, "k": 8, "P": 8}, 2, 8),
    # one source past the one-launch form: x staged before the wait, a ragged
    # last segment (192 vectors = 128 + 64)
    ("tiny", {"T": 700, "H": 1536, "E": 64, "k": 8, "P": 8}, -1, 1),
    # one launch: one token, the largest batch, ragged segments with run alignment
    ("decode", {"T": 1}, 4, 1), ("decode", {"T": 256}, -1, 1),
    ("tiny", {"T": 200, "H": 1536, "E": 64, "k": 8, "P": 8}, 2, 8)])
def test_quantized_fused_equals_separate_and_oracle(quant, g, name, over, recv_part, align):
    w_ = ms.workload(name, index=900 + len(over), **over)
    inp = ms.gen_inputs(w_)
    fused, kf = _dispatch_q("fused", quant, w_, inp, g, recv_part, align, trace=True)
    sep, _ = _dispatch_q("separate", quant, w_, inp, g, recv_part, align)
    _same(fused, sep)
    if w_.S == 1 and w_.T <= 256:
        assert kf == [f"k_dispatch_small_{quant}"], kf
    else:
        assert kf[-1] == f"k_pack_permute_{quant}", kf
    assert len(kf) == m.moe_dispatch_quantized_kernels(w_.S, w_.T, w_.k, w_.E, w_.P), kf
    lay, q, src, per = _q_oracle(quant, w_, inp, g, recv_part, align)
    for key in ("token_slot", "part_offsets", "expert_counts"):
        assert np.array_equal(fused[key], lay[key]), key
    for key in ("expert_offsets", "pair_row", "recv_pair"):
        assert np.array_equal(fused[key], per[key]), key
    for s in range(w_.S):
        used = int(lay["part_offsets"][s, -1])
        assert np.array_equal(fused["send"][s, :used], q[s, :used])
        assert np.array_equal(fused["send_src"][s], src[s])
    rows = int(per["expert_offsets"][-1])
    assert np.array_equal(fused["recv"][:rows], per["recv"].view(np.uint8)[:rows])
    assert fused["status"] == 0


@pytest.mark.parametrize("quant", ["mxfp8", "nvfp4"])
@pytest.mark.parametrize("T", [600, 64])
def test_quantized_capacity_overflow_matches_separate(quant, T):
    w_ = ms.workload("prefill", T=T, index=41)
    inp = ms.gen_inputs(w_)
    for cap_send, cap_recv in ((T, None), (None, 2 * T)):
        fused, _ = _dispatch_q("fused", quant, w_, inp, 1.0, cap_send=cap_send, cap_recv=cap_recv)
        sep, _ = _dispatch_q("separate", quant, w_, inp, 1.0, cap_send=cap_send, cap_recv=cap_recv)
        _same(fused, sep)
        assert fused["status"] & m.status_bit(m.MOE_ERR_CAPACITY)


# ------------------------------------------- pack + permute for any layout --

@pytest.mark.parametrize("S,T,H,E,k,P,recv_part,align", [
    (1, 1000, 5120, 384, 6, 8, -1, 1), (3, 700, 520, 96, 4, 8, 1, 128), (2, 0, 256, 16, 2, 4, -1, 1),
    (12, 64, 64, 1024, 8, 8, -1, 1)])          # S*E too large for the in-kernel map
def test_pack_permute_equals_pack_then_permute(S, T, H, E, k, P, recv_part, align):
    """moe_dispatch_pack_permute on a layout made by moe_dispatch_layout: every
    output byte as moe_dispatch_pack followed by moe_permute_to_experts."""
    w_ = ms.workload("tiny", S=S, T=T, H=H, E=E, k=k, P=P, index=S * 1000 + T)
    inp = ms.gen_inputs(w_)
    outs = []
    for mode in ("one_call", "two_calls"):
        path = m.MoePath(S, T, H, E, k, P, recv_part=recv_part, align=align, dispatch="separate")
        path.route(f32_dev(inp["logits"]))
        m.moe_dispatch_layout(path.topk_ids, E, P, path.expert_counts, path.expert_rank,
                              path.part_counts, path.part_offsets, path.token_slot, path.ws,
                              path.dev_status)
        path.send.view(torch.int16).fill_(0x5A5A)
        path.recv.view(torch.int16).fill_(0x3C3C)
        for name in ("send_src", "expert_offsets", "pair_row", "recv_pair"):
            getattr(path, name).fill_(-7)
        x = bf16_dev(inp["x"])
        m.trace_enable(None, 16)
        m.trace_reset()
        try:
            if mode == "one_call":
                m.moe_dispatch_pack_permute(x, path.token_slot, path.part_offsets, path.topk_ids,
                                            path.expert_counts, path.expert_rank, E, recv_part,
                                            align, path.send, path.send_src, path.recv,
                                            path.expert_offsets, path.pair_row, path.recv_pair,
                                            path.ws, path.dev_status)
            else:
                m.moe_dispatch_pack(x, path.token_slot, path.part_offsets, path.send,
                                    path.send_src, path.dev_status)
                m.moe_permute_to_experts(path.send, path.token_slot, path.topk_ids,
                                         path.expert_counts, path.expert_rank, E, recv_part, align,
                                         path.recv, path.expert_offsets, path.pair_row,
                                         path.recv_pair, path.ws, path.dev_status)
            torch.cuda.synchronize()
            kernels = [n for n, _ in m.trace_records()]
        finally:
            m.trace_disable()
        if mode == "one_call":
            assert len(kernels) == m.moe_dispatch_pack_permute_kernels(S, T, k, E, P), kernels
            if T > 0 and S * E <= 8 * 1024:
                assert kernels == ["k_pack_permute"], kernels
        outs.append({"send": bf16_host(path.send), "recv": bf16_host(path.recv),
                     "send_src": host(path.send_src), "expert_offsets": host(path.expert_offsets),
                     "pair_row": host(path.pair_row), "recv_pair": host(path.recv_pair),
                     "status": int(path.dev_status.item())})
    _same(outs[0], outs[1])
    assert outs[0]["status"] == 0
