"""Decode as an engine runs it: several layers' moe_dispatch + moe_combine
recorded in one CUDA graph and replayed (a2a-backends page, section 1.4: a
decode step makes ~40 round trips, recorded once and replayed).

Layer l + 1 dispatches the rows layer l's combine wrote (x of layer l + 1 is
layer l's `out` buffer), every launch chained to the one before it by
programmatic dependent launch; the receive rows take the contiguous runs or
the masked layout (a2a-backends sections 4.1, 4.2).  The one-launch dispatch asks L2 for its logits
before its grid-dependency wait and loads its first x segment right after the
wait, so each layer's received rows must be, byte for byte, the previous
layer's combine output of the same replay: the test rewrites every layer's
logits and the first layer's x between replays, so a read that ran ahead of
the previous layer would return the last replay's bytes.  Index outputs are
held to the oracle bit for bit and each combine to the oracle within the
combine's fp32 bound.
"""
import numpy as np
import pytest
import torch

import combine_moe_route_06_gb300 as m
import moe_synth as ms
import oracle
from gpu_util import bf16_dev, bf16_host, combine_within_fp32_bound, f32_dev, host

pytestmark = pytest.mark.gpu

LAYERS = 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    m.load_library()


def _inputs(w_, batch):
    """Logits for every layer and x for the first, rows of one larger batch."""
    wb = ms.workload("decode", index=batch)
    lg = ms.gen_logits(wb, T=w_.T * LAYERS).reshape(LAYERS, w_.S, w_.T, w_.E)
    x0 = ms.gen_x(wb, T=w_.T).reshape(w_.S, w_.T, w_.H)
    return lg, x0


def _check_layers(w_, paths, x0_bits, logits, layout):
    x_bits = x0_bits
    for l, p in enumerate(paths):
        ref = oracle.run_path(x_bits, logits[l], w_.E, w_.k, w_.P, None)
        pair_row = host(p.pair_row)
        assert np.array_equal(host(p.topk_ids), ref["ids"]), l
        if layout == "masked":
            cap_send = w_.T * min(w_.k, w_.P)
            mref = oracle.permute_masked(ref["send"], ref["layout"]["token_slot"], ref["ids"],
                                         w_.E, -1, p.block_rows)
            assert np.array_equal(pair_row, mref["pair_row"]), l
            assert np.array_equal(host(p.masked_counts), mref["masked_counts"]), l
            assert ref["send"].shape[1] == cap_send
        else:
            assert np.array_equal(pair_row, ref["permute"]["pair_row"]), l
        assert np.array_equal(host(p.token_slot), ref["layout"]["token_slot"]), l
        # the received rows are the bytes of this layer's x: for l > 0 the
        # previous layer's combine output of this replay
        recv = bf16_host(p.recv)
        xr = x_bits.reshape(w_.T, w_.H)
        pr = pair_row.reshape(w_.T, w_.k)
        t_idx, j_idx = np.nonzero(pr >= 0)
        assert np.array_equal(recv[pr[t_idx, j_idx]], xr[t_idx]), l
        out = bf16_host(p.out).reshape(w_.T, w_.H)
        ok, worst = combine_within_fp32_bound(out, ref["out"].reshape(w_.T, w_.H), recv, pr,
                                              ref["w"].astype(np.float32).reshape(w_.T, w_.k))
        assert ok, (l, worst)
        assert int(p.dev_status.item()) == 0, l
        x_bits = out.reshape(w_.S, w_.T, w_.H)


@pytest.mark.parametrize("layout", ["contiguous", "masked"])
def test_decode_layers_in_one_graph(layout):
    w_ = ms.workload("decode")
    kw = {"layout": "masked", "block_rows": 64} if layout == "masked" else {}
    paths = [m.MoePath(w_.S, w_.T, w_.H, w_.E, w_.k, w_.P, dispatch="fused", **kw)
             for _ in range(LAYERS)]
    lg, x0 = _inputs(w_, 11)
    logits = [f32_dev(lg[l]) for l in range(LAYERS)]
    x_first = bf16_dev(x0)
    xs = [x_first] + [paths[l - 1].out for l in range(1, LAYERS)]
    s = torch.cuda.Stream()
    calls = [p.bind(logits[l], xs[l], s) for l, p in enumerate(paths)]
    first = "moe_dispatch_masked" if layout == "masked" else "moe_dispatch"
    for c in calls:
        assert [fn.__name__ for fn, _ in c] == [first, "moe_combine"]
    with torch.cuda.stream(s):
        for c in calls:
            m.MoePath.run_bound(c)
    torch.cuda.synchronize()
    _check_layers(w_, paths, x0, lg, layout)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for c in calls:
            m.MoePath.run_bound(c)
    for batch in (12, 13):
        lg, x0 = _inputs(w_, batch)
        for l in range(LAYERS):
            logits[l].copy_(f32_dev(lg[l]))
        x_first.copy_(bf16_dev(x0))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        _check_layers(w_, paths, x0, lg, layout)
