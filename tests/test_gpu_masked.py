"""Masked receive layout (a2a-backends sections 4.1-4.2) on the GPU vs the oracle.

Bit-exact: counts, pair rows, recv_pair and every used row; rows past each
block's count are not written (checked with a canary fill on both sides).
"""
import numpy as np
import pytest
import torch

import combine_moe_route_06_gb300 as m
import moe_synth as ms
import oracle
from gpu_util import DEV, bf16_dev, bf16_host, close_bf16, host, i32_dev

pytestmark = pytest.mark.gpu

CAP = m.status_bit(m.MOE_ERR_CAPACITY)
FILL = 0x5A5A


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load_library()


def _case(name, S=None, index=None):
    kw = {}
    if S is not None:
        kw["S"] = S
    if index is not None:
        kw["index"] = index
    w_ = ms.workload(name, **kw)
    inp = ms.gen_inputs(w_)
    ids, wt = oracle.route_topk(inp["logits"], w_.k)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    cap_send = w_.T * min(w_.k, w_.P)
    send, _, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap_send)
    return w_, inp, ids, wt, lay, send


def _masked_gpu(send, lay, ids, E, recv_part, block_rows):
    S, cap_send, H = send.shape
    _, T, P = lay["token_slot"].shape
    k = ids.shape[2]
    nb = E if recv_part < 0 else E // P
    recv = bf16_dev(np.full((nb * block_rows, H), FILL, np.uint16))
    counts = torch.full((nb,), -7, dtype=torch.int32, device=DEV)
    pr = torch.full((S, T, k), -7, dtype=torch.int32, device=DEV)
    rp = torch.full((nb * block_rows,), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.moe_permute_to_experts_masked(bf16_dev(send), i32_dev(lay["token_slot"]), i32_dev(ids),
                                    i32_dev(lay["expert_counts"]), i32_dev(lay["expert_rank"]), E,
                                    recv_part, block_rows, recv, counts, pr, rp, st)
    torch.cuda.synchronize()
    return {"recv": bf16_host(recv), "masked_counts": host(counts), "pair_row": host(pr),
            "recv_pair": host(rp), "status": int(st.item()), "recv_dev": recv, "pair_row_dev": pr}


def _check(send, lay, ids, E, recv_part, block_rows):
    got = _masked_gpu(send, lay, ids, E, recv_part, block_rows)
    H = send.shape[2]
    nb = E if recv_part < 0 else E // lay["token_slot"].shape[2]
    ref = oracle.permute_masked(send, lay["token_slot"], ids, E, recv_part, block_rows,
                                recv=np.full((nb * block_rows, H), FILL, np.uint16))
    for key in ("masked_counts", "pair_row", "recv_pair"):
        assert np.array_equal(got[key], ref[key]), key
    assert np.array_equal(got["recv"], ref["recv"])
    assert got["status"] == ref["status"]
    return got, ref


@pytest.mark.parametrize("recv_part,block_rows", [(0, 1024), (5, 1024), (-1, 64), (3, 4)])
def test_masked_decode_from_8_sources(recv_part, block_rows):
    w_, inp, ids, wt, lay, send = _case("decode", S=8, index=11)
    got, ref = _check(send, lay, ids, w_.E, recv_part, block_rows)
    if block_rows == 4:
        assert got["status"] & CAP


@pytest.mark.parametrize("block_rows", [128, 32])
def test_masked_prefill_all_experts(block_rows):
    w_, inp, ids, wt, lay, send = _case("prefill")
    _check(send, lay, ids, w_.E, -1, block_rows)


def test_masked_tiny_ragged():
    w_, inp, ids, wt, lay, send = _case("tiny", S=3)
    for rp, br in ((-1, 40), (1, 200), (2, 7)):
        _check(send, lay, ids, w_.E, rp, br)


def test_combine_over_masked_equals_combine_over_contiguous():
    """The combine reads either layout through pair_row and returns the same bytes."""
    w_, inp, ids, wt, lay, send = _case("decode")
    got = _masked_gpu(send, lay, ids, w_.E, -1, 64)
    assert got["status"] == 0
    w32 = torch.from_numpy(wt.astype(np.float32)).to(DEV)
    out_m = torch.zeros((w_.S, w_.T, w_.H), dtype=torch.bfloat16, device=DEV)
    m.moe_combine(got["recv_dev"], got["pair_row_dev"], w32, out_m)
    per = oracle.permute_to_experts(send, lay["token_slot"], ids, w_.E)
    out_c = torch.zeros_like(out_m)
    m.moe_combine(bf16_dev(per["recv"]), i32_dev(per["pair_row"]), w32, out_c)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host(out_m), bf16_host(out_c))
    ref = oracle.combine(per["recv"], per["pair_row"], wt.astype(np.float32))
    assert close_bf16(bf16_host(out_m), ref)


# ------------------------------------------ pack + masked layout in one call --

def _pack_masked_gpu(x, lay, ids, E, recv_part, block_rows, cap_send):
    """moe_dispatch_pack_permute_masked on the oracle's layout, outputs canary-filled."""
    S, T, H = x.shape
    P = lay["token_slot"].shape[2]
    k = ids.shape[2]
    nb = E if recv_part < 0 else E // P
    send = bf16_dev(np.full((S, cap_send, H), FILL, np.uint16))
    src = torch.full((S, cap_send), -7, dtype=torch.int32, device=DEV)
    recv = bf16_dev(np.full((nb * block_rows, H), FILL, np.uint16))
    counts = torch.full((nb,), -7, dtype=torch.int32, device=DEV)
    pr = torch.full((S, T, k), -7, dtype=torch.int32, device=DEV)
    rp = torch.full((nb * block_rows,), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.trace_enable(None, 16)
    m.trace_reset()
    try:
        m.moe_dispatch_pack_permute_masked(
            bf16_dev(x), i32_dev(lay["token_slot"]), i32_dev(lay["part_offsets"]), i32_dev(ids),
            i32_dev(lay["expert_counts"]), i32_dev(lay["expert_rank"]), E, recv_part, block_rows,
            send, src, recv, counts, pr, rp, st)
        torch.cuda.synchronize()
        kernels = [n for n, _ in m.trace_records()]
    finally:
        m.trace_disable()
    return {"send": bf16_host(send), "send_src": host(src), "recv": bf16_host(recv),
            "masked_counts": host(counts), "pair_row": host(pr), "recv_pair": host(rp),
            "status": int(st.item()), "kernels": kernels}


@pytest.mark.parametrize("name,S,recv_part,block_rows", [
    ("decode", 8, 0, 1024), ("decode", 8, 5, 1024), ("decode", 8, -1, 64), ("decode", 8, 3, 4),
    ("prefill", None, -1, 128), ("tiny", 3, -1, 40), ("tiny", 3, 1, 200), ("tiny", 3, 2, 7),
    ("tiny", 12, -1, 16)])
def test_pack_permute_masked_equals_oracle(name, S, recv_part, block_rows):
    """Pack + the masked layout in one call against the oracle's pack followed by its
    masked permute: send rows, send_src, counts, pair rows, recv_pair and every recv row
    (canary included) bit-exact, and the same status bits."""
    over = {"E": 1024, "k": 8, "P": 8} if (name == "tiny" and S == 12) else {}
    w_, inp, ids, wt, lay, send = _case(name, S=S)
    if over:                                   # blocks of all 1,024 experts from 12 sources
        w_ = ms.workload("tiny", S=S, **over)
        inp = ms.gen_inputs(w_)
        ids, wt = oracle.route_topk(inp["logits"], w_.k)
        lay = oracle.dispatch_layout(ids, w_.E, w_.P)
        send, _, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], w_.T * min(w_.k, w_.P))
    cap_send = w_.T * min(w_.k, w_.P)
    got = _pack_masked_gpu(inp["x"], lay, ids, w_.E, recv_part, block_rows, cap_send)
    nb = w_.E if recv_part < 0 else w_.E // w_.P
    _, src, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap_send)
    ref = oracle.permute_masked(send, lay["token_slot"], ids, w_.E, recv_part, block_rows,
                                recv=np.full((nb * block_rows, w_.H), FILL, np.uint16))
    for s in range(w_.S):
        used = int(lay["part_offsets"][s, -1])
        assert np.array_equal(got["send"][s, :used], send[s, :used])
    assert np.array_equal(got["send_src"], src)
    for key in ("masked_counts", "pair_row", "recv_pair", "recv"):
        assert np.array_equal(got[key], ref[key]), key
    assert got["status"] == ref["status"]
    if block_rows == 4:
        assert got["status"] & CAP
    n_expected = m.moe_dispatch_pack_permute_masked_kernels(w_.S, w_.T, w_.k, w_.E, w_.P, recv_part)
    assert len(got["kernels"]) == n_expected, got["kernels"]
    if (2 + w_.S) * nb * 4 <= 48 * 1024:
        assert got["kernels"] == ["k_pack_permute_masked"]


# ------------------------- route + layout + pack + masked layout in one call --

def _dispatch_masked_gpu(w_, inp, recv_part, block_rows):
    """moe_dispatch_masked from the logits, every output canary-filled first."""
    S, T, H, E, k, P = w_.S, w_.T, w_.H, w_.E, w_.k, w_.P
    nb = E if recv_part < 0 else E // P
    cap_send = T * min(k, P)
    i32 = lambda *shape: torch.full(shape, -7, dtype=torch.int32, device=DEV)  # noqa: E731
    o = {"topk_ids": i32(S, T, k), "expert_counts": i32(S, E), "expert_rank": i32(S, T, k),
         "part_counts": i32(S, P), "part_offsets": i32(S, P + 1), "token_slot": i32(S, T, P),
         "send_src": i32(S, cap_send), "masked_counts": i32(nb), "pair_row": i32(S, T, k),
         "recv_pair": i32(nb * block_rows)}
    topk_w = torch.full((S, T, k), -9.0, dtype=torch.float32, device=DEV)
    send = bf16_dev(np.full((S, cap_send, H), FILL, np.uint16))
    recv = bf16_dev(np.full((nb * block_rows, H), FILL, np.uint16))
    ws = torch.empty(max(m.moe_workspace_bytes(S, T, k, E, P), 256), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    logits = torch.from_numpy(np.ascontiguousarray(inp["logits"])).to(DEV)
    m.trace_enable(None, 16)
    m.trace_reset()
    try:
        m.moe_dispatch_masked(logits, bf16_dev(inp["x"]), E, P, recv_part, block_rows,
                              o["topk_ids"], topk_w, o["expert_counts"], o["expert_rank"],
                              o["part_counts"], o["part_offsets"], o["token_slot"], send,
                              o["send_src"], recv, o["masked_counts"], o["pair_row"],
                              o["recv_pair"], ws, st)
        torch.cuda.synchronize()
        kernels = [n for n, _ in m.trace_records()]
    finally:
        m.trace_disable()
    got = {key: host(v) for key, v in o.items()}
    got.update({"topk_w": host(topk_w), "send": bf16_host(send), "recv": bf16_host(recv),
                "status": int(st.item()), "kernels": kernels})
    return got


@pytest.mark.parametrize("name,over,recv_part,block_rows", [
    ("decode", {}, -1, 64),
    ("decode", {}, 3, 1024),
    ("decode", {}, -1, 1),                                  # most pairs dropped
    ("decode", {"T": 1}, 6, 8),
    ("decode", {"T": 255}, 5, 16),
    ("decode", {"T": 256}, -1, 4),
    ("decode", {"T": 257}, -1, 64),                         # past the one-launch form
    ("decode", {"T": 0}, -1, 64),                           # an empty batch
    ("decode", {"T": 0}, 2, 0),
    ("tiny", {"T": 100, "E": 1024, "k": 32, "P": 32}, 7, 8),
    ("tiny", {"S": 3}, 1, 200),
    ("prefill", {}, -1, 128),
])
def test_dispatch_masked_equals_oracle(name, over, recv_part, block_rows):
    """moe_dispatch_masked against the oracle's route, layout, pack and masked
    permute: ids and layout bit-exact, weights within 2e-6, send rows, send_src,
    counts, pair rows, recv_pair and every recv row (canary included) bit-exact,
    the same status bits; one kernel for one source of at most 256 tokens."""
    w_ = ms.workload(name, index=500 + len(over) + block_rows, **over)
    inp = ms.gen_inputs(w_)
    got = _dispatch_masked_gpu(w_, inp, recv_part, block_rows)
    ids, wt = oracle.route_topk(inp["logits"], w_.k)
    assert np.array_equal(got["topk_ids"], ids)
    assert np.all(np.abs(got["topk_w"] - wt) <= 2e-6)
    lay = oracle.dispatch_layout(ids, w_.E, w_.P)
    for key in ("expert_counts", "expert_rank", "part_counts", "part_offsets", "token_slot"):
        assert np.array_equal(got[key], lay[key]), key
    cap_send = w_.T * min(w_.k, w_.P)
    send, src, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap_send)
    for s in range(w_.S):
        used = int(lay["part_offsets"][s, -1])
        assert np.array_equal(got["send"][s, :used], send[s, :used])
    assert np.array_equal(got["send_src"], src)
    nb = w_.E if recv_part < 0 else w_.E // w_.P
    ref = oracle.permute_masked(send, lay["token_slot"], ids, w_.E, recv_part, block_rows,
                                recv=np.full((nb * block_rows, w_.H), FILL, np.uint16))
    for key in ("masked_counts", "pair_row", "recv_pair", "recv"):
        assert np.array_equal(got[key], ref[key]), key
    assert got["status"] == ref["status"]
    n = m.moe_dispatch_masked_kernels(w_.S, w_.T, w_.k, w_.E, w_.P, recv_part)
    assert len(got["kernels"]) == n, got["kernels"]
    assert (got["kernels"] == ["k_dispatch_small"]) == (w_.S == 1 and 1 <= w_.T <= 256), \
        got["kernels"]


def test_masked_path_one_call_equals_separate():
    """MoePath with the masked layout: the fused step (moe_dispatch_masked, then the
    combine) leaves every output as the separate calls do, in two launches at decode."""
    w_ = ms.workload("decode", index=77)
    inp = ms.gen_inputs(w_)
    outs = {}
    for mode in ("fused", "separate"):
        path = m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, layout="masked", block_rows=64,
                         dispatch=mode)
        path.recv.view(torch.int16).fill_(FILL)
        path.recv_pair.fill_(-7)
        out = path.step(torch.from_numpy(inp["logits"]).to(DEV), bf16_dev(inp["x"]))
        torch.cuda.synchronize()
        outs[mode] = {"out": bf16_host(out), "recv": bf16_host(path.recv),
                      "pair_row": host(path.pair_row), "recv_pair": host(path.recv_pair),
                      "masked_counts": host(path.masked_counts),
                      "status": int(path.dev_status.item()),
                      "launches": path.launches_per_step()}
    for key in ("out", "recv", "pair_row", "recv_pair", "masked_counts", "status"):
        assert np.array_equal(outs["fused"][key], outs["separate"][key]), key
    assert outs["fused"]["launches"] == 2
