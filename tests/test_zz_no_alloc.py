"""moe_dispatch_layout_static: the layout for callers that cannot allocate.

Some callers have no way to allocate device memory at the moment they call
the layout (a plugin whose host engine owns all device memory, plain C code
without an allocator), so this entry point keeps its scratch in an array built
into the library.  These tests call it through the C ABI and check that it
gives exactly the bytes that moe_dispatch_layout gives with a caller-provided
workspace, on two calls in a row with different shapes (the second call reuses
the array after the first one filled it), and that sizes beyond the built-in
array are refused.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import combine_moe_route_06_gb300 as m
import moe_synth as ms
import oracle

pytestmark = pytest.mark.gpu

KEYS = ("expert_counts", "expert_rank", "part_counts", "part_offsets", "token_slot")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    m.build()
    return m.load_library()


def _outputs(S, T, k, E, P):
    i32 = dict(dtype=torch.int32, device="cuda")
    return {"expert_counts": torch.full((S, E), -7, **i32),
            "expert_rank": torch.full((S, T, k), -7, **i32),
            "part_counts": torch.full((S, P), -7, **i32),
            "part_offsets": torch.full((S, P + 1), -7, **i32),
            "token_slot": torch.full((S, T, P), -7, **i32),
            "dev_status": torch.zeros((1,), **i32)}


def _static_layout(lib, ids, E, P):
    S, T, k = ids.shape
    o = _outputs(S, T, k, E, P)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.moe_dispatch_layout_static(p(ids), S, T, k, E, P, p(o["expert_counts"]),
                                        p(o["expert_rank"]), p(o["part_counts"]),
                                        p(o["part_offsets"]), p(o["token_slot"]),
                                        p(o["dev_status"]), stream)
    assert rc == m.MOE_OK, lib.moe_last_error_message().decode()
    torch.cuda.synchronize()
    return {key: t.cpu().numpy() for key, t in o.items()}


def _workspace_layout(ids, E, P):
    S, T, k = ids.shape
    o = _outputs(S, T, k, E, P)
    ws = torch.empty(m.moe_workspace_bytes(S, T, k, E, P), dtype=torch.uint8, device="cuda")
    m.moe_dispatch_layout(ids, E, P, o["expert_counts"], o["expert_rank"], o["part_counts"],
                          o["part_offsets"], o["token_slot"], ws, o["dev_status"])
    torch.cuda.synchronize()
    return {key: t.cpu().numpy() for key, t in o.items()}


def test_static_layout_matches_workspace_layout_twice(lib):
    # first call: 8 sources x 4096 tokens (the larger scratch footprint);
    # second call: one source of 64 tokens, reading what the first left behind
    for name in ("skewed", "decode"):
        w = ms.workload(name)
        ids_np, _ = oracle.route_topk(ms.gen_logits(w), w.k)
        ids = torch.from_numpy(ids_np).cuda()
        got = _static_layout(lib, ids, w.E, w.P)
        want = _workspace_layout(ids, w.E, w.P)
        for key in KEYS:
            assert np.array_equal(got[key], want[key]), (name, key)
        assert int(got["dev_status"][0]) == int(want["dev_status"][0]) == 0


def test_static_layout_refuses_sizes_beyond_its_scratch(lib):
    fake = ctypes.c_void_p(1 << 20)      # never dereferenced: the call is refused first
    rc = lib.moe_dispatch_layout_static(fake, 8, 40000, 2, 1024, 32, fake, fake, fake, fake,
                                        fake, fake, ctypes.c_void_p(0))
    assert rc == m.MOE_ERR_INVALID_ARG
    assert "scratch" in lib.moe_last_error_message().decode()
