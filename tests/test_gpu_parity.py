"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Index outputs (ids, counts, offsets, slots, pair rows) and moved rows must be
bit-identical; routing weights agree within 2e-6 absolute (fp32 expf on the
GPU, double in the oracle); combine outputs within 1e-2 relative per element
(|gpu - ref| <= 1e-2 * max(|ref|, 1e-3)): bf16 out, fp32 accumulation.
"""
import numpy as np
import pytest
import torch

import combine_moe_route_06_gb300 as m
import moe_synth as ms
import oracle
from gpu_util import (DEV, bf16_dev, bf16_host, close_bf16, combine_within_fp32_bound, f32_dev,
                      host, i32_dev, run_layout, worst_rel)

pytestmark = pytest.mark.gpu

W_TOL = 2e-6
CAP = m.status_bit(m.MOE_ERR_CAPACITY)
BAD = m.status_bit(m.MOE_ERR_BAD_EXPERT_ID)
INC = m.status_bit(m.MOE_ERR_INVALID_ARG)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load_library()


# ------------------------------------------------------------------- route --

def _route_gpu(logits: np.ndarray, k: int):
    S, T, E = logits.shape
    ids = torch.full((S, T, k), -9, dtype=torch.int32, device=DEV)
    w = torch.full((S, T, k), -9.0, dtype=torch.float32, device=DEV)
    m.moe_route_topk(f32_dev(logits), ids, w)
    torch.cuda.synchronize()
    return host(ids), host(w)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "skewed", "large"])
def test_route_parity(name):
    w_ = ms.workload(name)
    logits = ms.gen_logits(w_)
    ids, w = _route_gpu(logits, w_.k)
    rid, rw = oracle.route_topk(logits, w_.k)
    assert np.array_equal(ids, rid)
    assert np.max(np.abs(w - rw)) <= W_TOL


@pytest.mark.parametrize("E,k,T", [(50, 3, 33), (7, 7, 5), (1024, 32, 40), (64, 1, 257),
                                   (384, 6, 1), (33, 4, 100)])
def test_route_shapes_and_ties(E, k, T):
    rng = np.random.default_rng(E * 131 + k)
    logits = rng.integers(-3, 4, size=(2, T, E)).astype(np.float32)  # heavy ties
    ids, w = _route_gpu(logits, k)
    rid, rw = oracle.route_topk(logits, k)
    assert np.array_equal(ids, rid)
    assert np.max(np.abs(w - rw)) <= W_TOL


def test_route_empty():
    ids, w = _route_gpu(np.zeros((1, 0, 16), np.float32), 2)
    assert ids.shape == (1, 0, 2)


# ------------------------------------------------------------------ layout --

def _check_layout(ids, E, P):
    got = run_layout(ids, E, P)
    ref = oracle.dispatch_layout(ids, E, P)
    for key in ("expert_counts", "expert_rank", "part_counts", "part_offsets", "token_slot"):
        assert np.array_equal(got[key], ref[key]), key
    assert got["status"] == ref["status"]


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "skewed", "large"])
def test_layout_parity(name):
    w_ = ms.workload(name)
    ids, _ = oracle.route_topk(ms.gen_logits(w_), w_.k)
    _check_layout(ids, w_.E, w_.P)


@pytest.mark.parametrize("S,T,k,E,P", [(1, 1, 2, 16, 4), (1, 255, 3, 12, 3), (1, 257, 3, 12, 3),
                                       (3, 513, 2, 32, 32), (2, 1000, 8, 64, 1),
                                       (1, 700, 32, 1024, 32), (2, 0, 2, 16, 4),
                                       (4, 200, 3, 12, 3), (3, 256, 6, 384, 8)])
def test_layout_ragged_and_extremes(S, T, k, E, P):
    rng = np.random.default_rng(S * 1000 + T)
    ids = rng.integers(0, E, size=(S, T, k)).astype(np.int32)
    _check_layout(ids, E, P)


def test_layout_skipped_and_bad_ids():
    rng = np.random.default_rng(3)
    ids = rng.integers(-2, 20, size=(2, 300, 3)).astype(np.int32)  # -2, -1 skipped; 16..19 bad
    _check_layout(ids, 16, 4)
    all_skip = -np.ones((1, 64, 4), np.int32)
    _check_layout(all_skip, 16, 4)


# -------------------------------------------------------------------- pack --

def _pack_case(name, T=None, cap=None, S=None):
    w_ = ms.workload(name) if T is None else ms.workload(name, T=T)
    if S is not None:
        w_ = ms.workload(name, S=S, T=w_.T)
    inp = ms.gen_inputs(w_)
    ids, _ = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    cap_send = w_.T * min(w_.k, w_.P) if cap is None else cap
    return w_, inp, ids, lay, cap_send


@pytest.mark.parametrize("name,T,cap", [("tiny", None, None), ("decode", None, None),
                                        ("prefill", None, None), ("large", None, None),
                                        ("tiny", 77, None), ("tiny", 200, 150)])
def test_pack_parity(name, T, cap):
    w_, inp, ids, lay, cap_send = _pack_case(name, T, cap)
    S = w_.S
    guard = 3
    canary = np.full((S, cap_send + guard, w_.H), 0x7A5B, np.uint16)
    d_send_full = bf16_dev(canary)
    assert S == 1  # with one source the leading slice below stays contiguous
    d_send = d_send_full[:, :cap_send]
    d_src = torch.full((S, cap_send), -5, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.moe_dispatch_pack(bf16_dev(inp["x"]), i32_dev(lay["token_slot"]), i32_dev(lay["part_offsets"]),
                        d_send, d_src, st)
    torch.cuda.synchronize()
    ref_send, ref_src, ref_st = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap_send,
                                                     send=canary[:, :cap_send].copy())
    got = bf16_host(d_send_full)
    assert np.array_equal(got[:, :cap_send], ref_send)          # written rows and untouched rows
    assert np.all(got[:, cap_send:] == 0x7A5B)                    # guard band
    assert np.array_equal(host(d_src), ref_src)
    assert int(st.item()) == ref_st


# ----------------------------------------------------------------- permute --

def _permute_gpu(send: np.ndarray, token_slot, ids, E, recv_part, align, cap_recv, guard=2,
                 fill=0x3C3C, counts=None, ranks=None):
    S, cap_send, H = send.shape
    _, T, P = token_slot.shape
    k = ids.shape[2]
    recv_full = bf16_dev(np.full((cap_recv + guard, H), fill, np.uint16))
    recv = recv_full[:cap_recv]
    eo = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
    pr = torch.full((S, T, k), -7, dtype=torch.int32, device=DEV)
    rp_full = torch.full((cap_recv + guard,), -7, dtype=torch.int32, device=DEV)
    rp = rp_full[:cap_recv]
    ws = torch.empty(max(m.moe_workspace_bytes(S, T, k, E, P), 256), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    if counts is None:
        # counts and ranks of the pairs come from the oracle's layout
        lay = oracle.dispatch_layout(ids, E, P)
        counts, ranks = lay["expert_counts"], lay["expert_rank"]
    m.moe_permute_to_experts(bf16_dev(send), i32_dev(token_slot), i32_dev(ids), i32_dev(counts),
                             i32_dev(ranks), E, recv_part, align, recv, eo, pr, rp, ws, st)
    torch.cuda.synchronize()
    full = bf16_host(recv_full)
    rpf = host(rp_full)
    assert np.all(full[cap_recv:] == fill) and np.all(rpf[cap_recv:] == -7), "guard band written"
    return {"recv": full[:cap_recv], "expert_offsets": host(eo), "pair_row": host(pr),
            "recv_pair": rpf[:cap_recv], "status": int(st.item())}


def _check_permute(send, token_slot, ids, E, recv_part, align, cap_recv, fill=0x3C3C, counts=None,
                   ranks=None):
    got = _permute_gpu(send, token_slot, ids, E, recv_part, align, cap_recv, fill=fill,
                       counts=counts, ranks=ranks)
    H = send.shape[2]
    ref = oracle.permute_to_experts(send, token_slot, ids, E, recv_part=recv_part, align=align,
                                    cap_recv=cap_recv, recv=np.full((cap_recv, H), fill, np.uint16))
    for key in ("expert_offsets", "pair_row", "recv_pair"):
        assert np.array_equal(got[key], ref[key]), key
    assert np.array_equal(got["recv"], ref["recv"])
    assert got["status"] == ref["status"]
    return got


@pytest.mark.parametrize("name,recv_part,align", [("tiny", -1, 1), ("tiny", -1, 128), ("tiny", 2, 8),
                                                  ("decode", -1, 1), ("decode", 5, 128),
                                                  ("prefill", -1, 1), ("prefill", 0, 128),
                                                  ("large", -1, 1)])
def test_permute_parity(name, recv_part, align):
    w_, inp, ids, lay, cap_send = _pack_case(name)
    send, _, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap_send)
    cap_recv = w_.S * w_.T * w_.k + w_.E * (align - 1)
    _check_permute(send, lay["token_slot"], ids, w_.E, recv_part, align, cap_recv)


def test_permute_multi_source_ragged():
    w_, inp, ids, lay, cap_send = _pack_case("tiny", T=301, S=3)
    send, _, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap_send)
    for rp, al in ((-1, 1), (1, 4), (3, 128)):
        _check_permute(send, lay["token_slot"], ids, w_.E, rp, al, w_.S * w_.T * w_.k + w_.E * (al - 1))


@pytest.mark.parametrize("S,E,recv_part,align,kernels", [
    (1, 16, -1, 1, ["k_perm_copy"]), (3, 64, 2, 8, ["k_perm_copy"]),
    (12, 1024, -1, 1, ["k_perm_map", "k_perm_copy"]), (12, 1024, 5, 128, ["k_perm_map", "k_perm_copy"])])
def test_permute_map_in_copy_or_separate(S, E, recv_part, align, kernels):
    """The map step runs inside the copy kernel while the counts' prefix sums fit in its shared
    memory (S*E + 2E + 1 ints <= 48 KiB), else as its own kernel first; both give the oracle's
    rows, offsets and pair rows, and the library reports the launch count it uses."""
    w_ = ms.workload("tiny", S=S, T=40, H=64, E=E, k=8, P=8)
    inp = ms.gen_inputs(w_)
    ids, _ = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    cap_send = w_.T * min(w_.k, w_.P)
    send, _, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap_send)
    torch.cuda.synchronize()
    m.trace_enable("k_perm", 8)
    try:
        _check_permute(send, lay["token_slot"], ids, w_.E, recv_part, align,
                       S * w_.T * w_.k + w_.E * (align - 1))
        names = [name for name, _ in m.trace_records()]
    finally:
        m.trace_disable()
    assert names == kernels
    assert m.moe_permute_to_experts_kernels(S, w_.T, w_.k, w_.E, w_.P) == len(kernels)


def test_permute_capacity_and_bad_inputs():
    w_, inp, ids, lay, cap_send = _pack_case("tiny")
    ids = ids.copy()
    ids[0, 3, 0] = 99       # bad id
    ids[0, 4, 1] = -1       # skipped
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    send, _, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap_send)
    # too small a receive buffer: pairs beyond it are dropped and flagged
    _check_permute(send, lay["token_slot"], ids, w_.E, -1, 1, 100)
    _check_permute(send, lay["token_slot"], ids, w_.E, -1, 32, 200)
    # a slot beyond cap_send (source row dropped at pack) and an inconsistent slot
    ts = lay["token_slot"].copy()
    p0 = int(np.nonzero(ts[0, 10] >= 0)[0][0])
    ts[0, 10, p0] = cap_send + 5
    p1 = int(np.nonzero(ts[0, 11] >= 0)[0][0])
    ts[0, 11, p1] = -1
    got = _check_permute(send, ts, ids, w_.E, -1, 1, w_.T * w_.k)
    assert got["status"] & CAP and got["status"] & INC and got["status"] & BAD


def test_permute_rejects_inconsistent_ranks():
    """A rank outside [0, expert_counts) is skipped and flagged, never written out of place."""
    w_, inp, ids, lay, cap_send = _pack_case("tiny")
    send, _, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap_send)
    ranks = lay["expert_rank"].copy()
    ranks[0, 9, 0] = 10_000
    ranks[0, 12, 1] = -1
    got = _permute_gpu(send, lay["token_slot"], ids, w_.E, -1, 1, w_.T * w_.k,
                       counts=lay["expert_counts"], ranks=ranks)
    ref = oracle.permute_to_experts(send, lay["token_slot"], ids, w_.E)
    assert got["status"] & INC
    bad = np.zeros(ids.shape, bool)
    bad[0, 9, 0] = bad[0, 12, 1] = True
    assert np.all(got["pair_row"][bad] == -1)
    assert np.array_equal(got["pair_row"][~bad], ref["pair_row"][~bad])


def test_permute_empty():
    send = np.zeros((1, 0, 16), np.uint16)
    ts = np.zeros((1, 0, 4), np.int32)
    ids = np.zeros((1, 0, 2), np.int32)
    got = _check_permute(send, ts, ids, 16, -1, 1, 5)
    assert np.all(got["expert_offsets"] == 0) and np.all(got["recv_pair"] == -1)


# ----------------------------------------------------------------- combine --

def _combine_gpu(y, pair_row, w, H):
    S, T, k = pair_row.shape
    out = torch.full((S, T, H), 1.5, dtype=torch.bfloat16, device=DEV)
    m.moe_combine(bf16_dev(y), i32_dev(pair_row), f32_dev(w), out)
    torch.cuda.synchronize()
    return bf16_host(out)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "large"])
def test_combine_parity(name):
    w_ = ms.workload(name)
    inp = ms.gen_inputs(w_)
    ref = oracle.run_path(inp["x"], inp["logits"], w_.E, w_.k, w_.P, inp["scales"])
    w32 = ref["w"].astype(np.float32)
    got = _combine_gpu(ref["y"], ref["permute"]["pair_row"], w32, w_.H)
    assert close_bf16(got, ref["out"]), worst_rel(got, ref["out"])


def test_combine_random_rows_and_holes():
    rng = np.random.default_rng(9)
    S, T, k, H, R = 2, 300, 5, 264, 900
    y = ms.bf16_bits_from_f32(rng.standard_normal((R, H)).astype(np.float32))
    pr = rng.integers(-1, R, size=(S, T, k)).astype(np.int32)
    pr[0, 7] = -1                                      # token with no pair -> zeros
    w = rng.uniform(0.01, 1.0, size=(S, T, k)).astype(np.float32)
    got = _combine_gpu(y, pr, w, H)
    ref = oracle.combine(y, pr, w)
    assert close_bf16(got, ref), worst_rel(got, ref)
    assert np.all(got[0, 7] == 0)


def test_combine_rejects_rows_beyond_y():
    rng = np.random.default_rng(4)
    S, T, k, H, R = 1, 50, 3, 64, 40
    y = ms.bf16_bits_from_f32(rng.standard_normal((R, H)).astype(np.float32))
    pr = rng.integers(0, R, size=(S, T, k)).astype(np.int32)
    pr[0, 5, 1] = R + 1000                              # out of range: skipped and flagged
    w = rng.uniform(0.1, 1.0, size=(S, T, k)).astype(np.float32)
    out = torch.zeros((S, T, H), dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.moe_combine(bf16_dev(y), i32_dev(pr), f32_dev(w), out, st)
    torch.cuda.synchronize()
    pr_ref = pr.copy()
    pr_ref[0, 5, 1] = -1
    ref = oracle.combine(y, pr_ref, w)
    assert close_bf16(bf16_host(out), ref)
    assert int(st.item()) == INC


# ------------------------------------------------------------- whole path --

def _gpu_path(w_, inp, recv_part=-1, align=1, scales=None, dispatch=None):
    path = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, recv_part=recv_part, align=align,
                     dispatch=dispatch)
    out = path.step(f32_dev(inp["logits"]), bf16_dev(inp["x"]),
                    None if scales is None else f32_dev(scales))
    torch.cuda.synchronize()
    return path, bf16_host(out)


@pytest.mark.parametrize("dispatch", ["fused", "separate"])
@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "large"])
def test_path_full_size(name, dispatch):
    """The whole path, with moe_dispatch or the four separate calls, against the oracle."""
    w_ = ms.workload(name)
    inp = ms.gen_inputs(w_)
    path, out = _gpu_path(w_, inp, scales=inp["scales"], dispatch=dispatch)
    ref = oracle.run_path(inp["x"], inp["logits"], w_.E, w_.k, w_.P, inp["scales"])
    assert np.array_equal(host(path.topk_ids), ref["ids"])
    assert np.array_equal(host(path.token_slot), ref["layout"]["token_slot"])
    assert np.array_equal(host(path.part_offsets), ref["layout"]["part_offsets"])
    assert np.array_equal(host(path.expert_offsets), ref["permute"]["expert_offsets"])
    assert np.array_equal(host(path.pair_row), ref["permute"]["pair_row"])
    used = int(ref["layout"]["part_offsets"][0, -1])
    assert np.array_equal(bf16_host(path.send)[0, :used], ref["send"][0, :used])
    rows = int(ref["permute"]["expert_offsets"][-1])
    assert np.array_equal(bf16_host(path.recv)[:rows], ref["permute"]["recv"][:rows])
    y = bf16_host(path.y)[:rows]
    # the stand-in expert rounds fp32 products; the oracle rounds exact ones: at most 1 ulp apart
    assert close_bf16(y, ref["y"][:rows], rel=2.0 ** -7, floor=1e-30)
    assert close_bf16(out, ref["out"]), worst_rel(out, ref["out"])
    # the combine's own accuracy on the rows and weights it was given: within the
    # fp32 accumulation bound plus one bf16 unit of the oracle's exact sum
    S, T, H, k = w_.S, w_.T, w_.H, w_.k
    y_all = bf16_host(path.y)
    pr = host(path.pair_row).reshape(-1, k)
    wg = host(path.topk_w).reshape(-1, k)
    want = oracle.combine(y_all, pr.reshape(S, T, k), wg.reshape(S, T, k)).reshape(-1, H)
    ok, excess = combine_within_fp32_bound(out.reshape(-1, H), want, y_all, pr, wg)
    assert ok, excess
    assert int(path.dev_status.item()) == 0


@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_identity_round_trip(name):
    w_ = ms.workload(name)
    inp = ms.gen_inputs(w_)
    for align in (1, 128):
        _, out = _gpu_path(w_, inp, align=align)
        assert np.array_equal(out, inp["x"])


def _skewed_reference(w_, inp):
    """Oracle index outputs of the skewed workload.  Indices do not depend on
    the row width, so the oracle permutes 8-wide stand-in rows; the moved rows
    are then checked against the source tokens' rows of x."""
    ids, w64 = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    cap_send = w_.T * min(w_.k, w_.P)
    narrow = np.zeros((w_.S, cap_send, 8), np.uint16)
    per = oracle.permute_to_experts(narrow, lay["token_slot"], ids, w_.E, recv_part=w_.recv_part)
    return ids, w64, lay, per


@pytest.mark.parametrize("expert,dispatch", [("identity", "fused"), ("scale", "separate")])
def test_skewed_receiver_full_size(expert, dispatch):
    """Skewed workload (8 sources x 4096 tokens, Zipf(1.2), partition 0 receives),
    compared in full: every index output; every used receive row bit-exact
    against its source token's row of x (recv[r] = x[s, t] for the pair
    recv_pair[r] = (s*T + t)*k + j); every one of the 32,768 partial-combine
    outputs against the oracle's combine.  With the stand-in expert
    (y = bf16(recv * s_e)) every expert row is held to one bf16 unit of the
    oracle's, and the combine to the oracle's combine of the rows it read.  The
    identity case runs moe_dispatch, the stand-in expert case the separate calls."""
    w_ = ms.workload("skewed")
    inp = ms.gen_inputs(w_)
    ids, w64, lay, per = _skewed_reference(w_, inp)
    scales = inp["scales"] if expert == "scale" else None
    path, out = _gpu_path(w_, inp, recv_part=w_.recv_part, scales=scales, dispatch=dispatch)
    assert np.array_equal(host(path.topk_ids), ids)
    assert np.max(np.abs(host(path.topk_w) - w64)) <= W_TOL
    assert np.array_equal(host(path.token_slot), lay["token_slot"])
    assert np.array_equal(host(path.expert_counts), lay["expert_counts"])
    assert np.array_equal(host(path.part_offsets), lay["part_offsets"])
    assert np.array_equal(host(path.expert_offsets), per["expert_offsets"])
    assert np.array_equal(host(path.pair_row), per["pair_row"])
    assert np.array_equal(host(path.recv_pair), per["recv_pair"])
    H, k = w_.H, w_.k
    x_flat = inp["x"].reshape(-1, H)
    rows_used = int(per["expert_offsets"][-1])
    recv_pair = per["recv_pair"]
    assert rows_used > 150_000 and np.all(recv_pair[:rows_used] >= 0)
    # every used receive row (and, with the stand-in expert, every expert row)
    y_dev = path.recv if scales is None else path.y
    y_all = np.empty((rows_used, H), np.uint16)
    eoff = per["expert_offsets"]
    for r0 in range(0, rows_used, 16384):
        r1 = min(rows_used, r0 + 16384)
        src = x_flat[recv_pair[r0:r1] // k]
        assert np.array_equal(bf16_host(path.recv[r0:r1]), src), (r0, r1)
        y_all[r0:r1] = bf16_host(y_dev[r0:r1])
        if scales is not None:
            # the oracle's stand-in expert on these rows (run starts relative to r0)
            want_y = oracle.expert_scale(src, np.clip(eoff - r0, 0, r1 - r0), scales)
            # the kernel rounds the fp32 product, the oracle the exact one: one
            # bf16 unit apart at most
            assert close_bf16(y_all[r0:r1], want_y, rel=2.0 ** -7, floor=1e-30), (r0, r1)
    # every partial-combine output (tokens with no pair in partition 0 give exact 0)
    pr_all = per["pair_row"].reshape(-1, k)
    w_all = w64.reshape(-1, k).astype(np.float32)
    out_all = out.reshape(-1, H)
    for n0 in range(0, w_.S * w_.T, 4096):
        n1 = n0 + 4096
        pr = pr_all[n0:n1]
        want = oracle.combine(y_all, pr[None], w_all[n0:n1][None])[0]
        assert close_bf16(out_all[n0:n1], want), (n0, worst_rel(out_all[n0:n1], want))
        ok, excess = combine_within_fp32_bound(out_all[n0:n1], want, y_all, pr, w_all[n0:n1])
        assert ok, (n0, excess)
    assert int(path.dev_status.item()) == 0


def test_deterministic_bytes():
    w_ = ms.workload("decode")
    inp = ms.gen_inputs(w_)
    p1, o1 = _gpu_path(w_, inp, scales=inp["scales"])
    p2, o2 = _gpu_path(w_, inp, scales=inp["scales"])
    assert np.array_equal(o1, o2)
    assert np.array_equal(bf16_host(p1.recv), bf16_host(p2.recv))
    assert np.array_equal(host(p1.topk_w).view(np.uint32), host(p2.topk_w).view(np.uint32))


def test_cuda_graph_replay_decode():
    w_ = ms.workload("decode")
    inp = ms.gen_inputs(w_)
    path = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P)
    logits = f32_dev(inp["logits"])
    x = bf16_dev(inp["x"])
    scale = f32_dev(inp["scales"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        path.step(logits, x, scale, stream=s)   # warm-up (allocates y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        path.step(logits, x, scale, stream=s)
    # new inputs at the same addresses, then replay
    inp2 = ms.gen_inputs(ms.workload("decode", index=7))
    logits.copy_(f32_dev(inp2["logits"]))
    x.copy_(bf16_dev(inp2["x"]))
    g.replay()
    torch.cuda.synchronize()
    ref = oracle.run_path(inp2["x"], inp2["logits"], w_.E, w_.k, w_.P, inp2["scales"])
    assert np.array_equal(host(path.pair_row), ref["permute"]["pair_row"])
    got = bf16_host(path.out)
    assert close_bf16(got, ref["out"]), worst_rel(got, ref["out"])


def test_bound_calls_match_checked_calls():
    """The pre-marshalled call list (used by the benchmark) gives the same bytes."""
    w_ = ms.workload("decode")
    inp = ms.gen_inputs(w_)
    p1, o1 = _gpu_path(w_, inp)
    p2 = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P)
    calls = p2.bind(f32_dev(inp["logits"]), bf16_dev(inp["x"]))
    m.MoePath.run_bound(calls)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(p2.out), o1)
    assert np.array_equal(host(p2.pair_row), host(p1.pair_row))


def test_trace_inside_cuda_graph():
    """With tracing on during capture, each replay re-records the traced kernel's events."""
    w_ = ms.workload("decode")
    inp = ms.gen_inputs(w_)
    path = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, dispatch="separate")
    logits, x = f32_dev(inp["logits"]), bf16_dev(inp["x"])
    s = torch.cuda.Stream()
    calls = path.bind(logits, x, s)
    with torch.cuda.stream(s):
        m.MoePath.run_bound(calls)
    torch.cuda.synchronize()
    m.trace_enable("k_perm_copy", 4)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            m.MoePath.run_bound(calls)
        for _ in range(2):
            g.replay()
            torch.cuda.synchronize()
            recs = m.trace_records()
            assert [r[0] for r in recs] == ["k_perm_copy"] and recs[0][1] > 0
        del g
        torch.cuda.synchronize()
    finally:
        m.trace_disable()
    ref = oracle.run_path(inp["x"], inp["logits"], w_.E, w_.k, w_.P, None)
    assert close_bf16(bf16_host(path.out), ref["out"])


@pytest.mark.parametrize("S,T,H,E,k,P,align", [(2, 300, 8, 1024, 32, 32, 1),
                                               (3, 257, 24, 64, 8, 4, 128),
                                               (1, 1, 8, 16, 2, 4, 1),
                                               (2, 513, 520, 96, 3, 32, 8)])
def test_path_at_the_limits(S, T, H, E, k, P, align):
    """The whole path at the ABI's extremes (E = 1024, k = 32, P = 32, the smallest row of
    8 values, a single token, ragged T over chunks) against the oracle."""
    w_ = ms.workload("tiny", S=S, T=T, H=H, E=E, k=k, P=P)
    inp = ms.gen_inputs(w_)
    path, out = _gpu_path(w_, inp, align=align, scales=inp["scales"])
    ref = oracle.run_path(inp["x"], inp["logits"], E, k, P, inp["scales"], align=align)
    assert np.array_equal(host(path.topk_ids), ref["ids"])
    assert np.array_equal(host(path.token_slot), ref["layout"]["token_slot"])
    assert np.array_equal(host(path.expert_offsets), ref["permute"]["expert_offsets"])
    assert np.array_equal(host(path.pair_row), ref["permute"]["pair_row"])
    rows = int(ref["permute"]["expert_offsets"][-1])
    assert np.array_equal(bf16_host(path.recv)[:rows], ref["permute"]["recv"][:rows])
    # the stand-in expert (not a step of the method) rounds x*s in fp32 first: one bf16 unit;
    # the combine is then held to its tolerance on the expert rows it was given
    y = bf16_host(path.y)
    assert close_bf16(y[:rows], ref["y"][:rows], rel=2.0 ** -7, floor=1e-30)
    want = oracle.combine(y, ref["permute"]["pair_row"], ref["w"].astype(np.float32))
    assert close_bf16(out, want), worst_rel(out, want)
    assert int(path.dev_status.item()) == 0
